/* tq_oracle.c -- plain CPU oracle of the TurboQuant KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY (see tq_oracle.h): used by the tests, the smoke
 * check and the benchmark's CPU baseline; never by the product path.
 *
 * Each function names the op of page "@mlx-bun/inference 0.0.0-stage ->
 * 1.0.0", file package/src/kernels/turboquant/ops.ts, that it restates. The
 * arithmetic is IEEE binary32, one rounding per operation, in the order the
 * page applies its ops. Build: -O2 -ffp-contract=off, no fast-math.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

#define GROUP 32 /* BLOCK_SIZE: quantisation groups of 32 along head_dim */

/* fp32 value of the page's eps scalar (scalarLike(1e-8, fp32 array)). */
static const float kEps = 1e-8f;

/* ------------------------------------------------------------------------ */
/* packedDim: dim*bits/8 bytes, error on a non-byte-aligned product.        */
int64_t oracle_packed_dim(int64_t dim, int bits) {
    if (dim < 0 || bits <= 0) return -1;
    if ((dim * bits) % 8 != 0) return -1;
    return dim * bits / 8;
}

static int supported_head_dim(int64_t d) {
    return d == 64 || d == 128 || d == 256 || d == 512;
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 conversions, written from the binary16/bfloat16 formats:        */
/* binary16 = 1 sign, 5 exponent (bias 15), 10 fraction bits.               */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    int32_t exp = (int32_t)((x >> 23) & 0xFFu);
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFF) { /* Inf or NaN; NaN stays a quiet NaN */
        return (uint16_t)(sign | 0x7C00u | (man ? (0x200u | (man >> 13)) : 0u));
    }
    int32_t e = exp - 127 + 15; /* re-biased exponent */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u); /* |x| >= 2^16: overflow */
    if (e <= 0) {
        /* binary16 subnormal (or zero): value = m * 2^-24 */
        if (e < -10) return (uint16_t)sign; /* |x| < 2^-25 rounds to zero */
        uint32_t sig = man | 0x800000u;      /* 24-bit significand */
        int shift = 14 - e;                  /* sig * 2^(e-15-23) / 2^-24 */
        uint32_t m = sig >> shift;
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (m & 1u))) m++; /* may carry to normal */
        return (uint16_t)(sign | m);
    }
    uint32_t h = sign | ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h++; /* carry may give Inf */
    return (uint16_t)h;
}

float oracle_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t man = (uint32_t)h & 0x3FFu;
    uint32_t x;
    if (exp == 0x1F) {
        x = sign | 0x7F800000u | (man << 13);
    } else if (exp == 0) {
        if (man == 0) {
            x = sign;
        } else { /* subnormal: normalise */
            int e = -14;
            while (!(man & 0x400u)) { man <<= 1; e--; }
            man &= 0x3FFu;
            x = sign | ((uint32_t)(e + 127) << 23) | (man << 13);
        }
    } else {
        x = sign | ((exp - 15 + 127) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &x, 4);
    return f;
}

/* bfloat16 = the upper 16 bits of binary32; round to nearest even. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu)) {
        return (uint16_t)((x >> 16) | 0x40u); /* quiet NaN */
    }
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7FFFu + lsb;
    return (uint16_t)(x >> 16);
}

float oracle_bf16_to_f32(uint16_t h) {
    uint32_t x = (uint32_t)h << 16;
    float f;
    memcpy(&f, &x, 4);
    return f;
}

/* ops.round: round half to even. */
float oracle_round(float x) { return nearbyintf(x); }

void oracle_f32_to_f16_n(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_f16(x[i]);
}
void oracle_f16_to_f32_n(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_to_f32(h[i]);
}
void oracle_f32_to_bf16_n(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* fwht: rotation. The Hadamard transform of n = 2^k values by radix-2      */
/* butterflies; stage h pairs element i0+j with i0+j+h into (a+b, a-b).     */
void oracle_hadamard_unnormalized(float* x, int n) {
    for (int h = 1; h < n; h *= 2) {
        for (int i0 = 0; i0 < n; i0 += 2 * h) {
            for (int j = 0; j < h; j++) {
                float a = x[i0 + j];
                float b = x[i0 + j + h];
                x[i0 + j] = a + b;
                x[i0 + j + h] = a - b;
            }
        }
    }
}

void oracle_hadamard(float* x, int n) {
    oracle_hadamard_unnormalized(x, n);
    const float c = (float)(1.0 / sqrt((double)n));
    for (int i = 0; i < n; i++) x[i] = x[i] * c;
}

/* fwht(x, encode): encode multiplies by the signs, then transforms; decode
 * transforms, then multiplies by the signs. */
int oracle_fwht(float* x, int d, int encode) {
    const signed char* s = oracle_sign_vector(d);
    if (!s) return -1;
    if (encode) {
        for (int i = 0; i < d; i++) x[i] = x[i] * (float)s[i];
        oracle_hadamard(x, d);
    } else {
        oracle_hadamard(x, d);
        for (int i = 0; i < d; i++) x[i] = x[i] * (float)s[i];
    }
    return 0;
}

void oracle_hadamard_rows(float* x, int64_t n_rows, int n, int normalised) {
    for (int64_t r = 0; r < n_rows; r++) {
        if (normalised) oracle_hadamard(x + r * n, n);
        else oracle_hadamard_unnormalized(x + r * n, n);
    }
}

int oracle_fwht_rows(float* x, int64_t n_rows, int d, int encode) {
    if (!oracle_sign_vector(d)) return -1;
    for (int64_t r = 0; r < n_rows; r++) oracle_fwht(x + r * d, d, encode);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* searchsorted: index = count(boundaries < x).                            */
void oracle_searchsorted(const float* b, int nb, const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) {
        int c = 0;
        for (int j = 0; j < nb; j++) c += (x[i] > b[j]) ? 1 : 0;
        out[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------------ */
/* packBits / unpackBits: element i occupies bits [i*b, i*b+b) of a flat    */
/* little-endian bitstream (LSB of byte 0 first). bits == 8 is a copy.      */
static int valid_pack_bits(int bits) {
    return bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 8;
}

int oracle_pack_bits(const uint8_t* codes, int64_t n, int bits, uint8_t* out) {
    if (!valid_pack_bits(bits)) return -1;
    int64_t nbytes = oracle_packed_dim(n, bits);
    if (nbytes < 0) return -1;
    memset(out, 0, (size_t)nbytes);
    for (int64_t i = 0; i < n; i++) {
        for (int k = 0; k < bits; k++) {
            int64_t pos = i * bits + k;
            uint8_t bit = (uint8_t)((codes[i] >> k) & 1u);
            out[pos >> 3] = (uint8_t)(out[pos >> 3] | (bit << (pos & 7)));
        }
    }
    return 0;
}

int oracle_unpack_bits(const uint8_t* packed, int64_t n, int bits, uint8_t* codes) {
    if (!valid_pack_bits(bits)) return -1;
    if (oracle_packed_dim(n, bits) < 0) return -1;
    for (int64_t i = 0; i < n; i++) {
        uint8_t v = 0;
        for (int k = 0; k < bits; k++) {
            int64_t pos = i * bits + k;
            v = (uint8_t)(v | (((packed[pos >> 3] >> (pos & 7)) & 1u) << k));
        }
        codes[i] = v;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* encodeKeys: per 32-group affine min/max quantisation, in fp32.          */
/* unsigned (bits 2/4/5/8): maxVal = 2^b-1, scale = (max-min)/maxVal,       */
/*   zp = round(min/(scale+eps)), q = clip(round(x/(scale+eps) - zp), 0, maxVal) */
/* signed (bits 8 only): maxVal = 2^(b-1)-1, scale = (max-min)/(2*maxVal),  */
/*   zp = round((max+min)/(2*(scale+eps))), q = clip(..., -maxVal, maxVal)  */
/* scale and zp are cast to fp16 last.                                       */
static int valid_key_bits(int bits, int is_signed) {
    if (is_signed) return bits == 8;
    return bits == 2 || bits == 4 || bits == 5 || bits == 8;
}

int oracle_encode_keys_row(const float* x, int d, int bits, int is_signed,
                           uint8_t* codes, uint16_t* scales, uint16_t* zeros) {
    if (d <= 0 || d % GROUP != 0) return ORACLE_ERR_HEAD_DIM;
    if (!valid_key_bits(bits, is_signed)) return ORACLE_ERR_BITS;
    const int max_val = is_signed ? (1 << (bits - 1)) - 1 : (1 << bits) - 1;
    for (int g = 0; g < d / GROUP; g++) {
        const float* xg = x + g * GROUP;
        /* ops.minAxis / ops.maxAxis. A NaN anywhere in the group makes both
         * NaN (the reductions propagate NaN, as IEEE 754-2019 minimum and
         * maximum do); otherwise a left-to-right scan that keeps the first of
         * equal values (only +0 / -0 can tell). */
        float mn = xg[0], mx = xg[0];
        int has_nan = 0;
        for (int i = 0; i < GROUP; i++) has_nan |= (xg[i] != xg[i]);
        for (int i = 1; i < GROUP; i++) {
            if (xg[i] < mn) mn = xg[i];
            if (xg[i] > mx) mx = xg[i];
        }
        if (has_nan) {
            mn = NAN;
            mx = NAN;
        }
        float scale, zp, lo, hi;
        if (is_signed) {
            float range = mx - mn;
            scale = range / (float)(2 * max_val);
            float scale_eps = scale + kEps;
            float denom = 2.0f * scale_eps;
            float sum_min_max = mx + mn;
            zp = oracle_round(sum_min_max / denom);
            lo = (float)(-max_val);
            hi = (float)max_val;
        } else {
            float range = mx - mn;
            scale = range / (float)max_val;
            float scale_eps = scale + kEps;
            zp = oracle_round(mn / scale_eps);
            lo = 0.0f;
            hi = (float)max_val;
        }
        float scale_eps2 = scale + kEps;
        for (int i = 0; i < GROUP; i++) {
            float shifted = xg[i] / scale_eps2 - zp;
            float r = oracle_round(shifted);
            if (r < lo) r = lo;
            if (r > hi) r = hi;
            /* astype(int8 / uint8): clip keeps a NaN, which converts to 0 (the
             * reading taken for a conversion IEEE leaves invalid). */
            int q = (r != r) ? 0 : (int)r;
            codes[g * GROUP + i] = (uint8_t)(q & 0xFF); /* int8 two's complement */
        }
        scales[g] = oracle_f32_to_f16(scale);
        zeros[g] = oracle_f32_to_f16(zp);
    }
    return ORACLE_OK;
}

/* decodeKeys: x = (indices + zero) * scale, fp32 (zero, scale from fp16). */
int oracle_decode_keys_row(const uint8_t* codes, int d, int is_signed,
                           const uint16_t* scales, const uint16_t* zeros, float* out) {
    if (d <= 0 || d % GROUP != 0) return ORACLE_ERR_HEAD_DIM;
    for (int g = 0; g < d / GROUP; g++) {
        float z = oracle_f16_to_f32(zeros[g]);
        float s = oracle_f16_to_f32(scales[g]);
        for (int i = 0; i < GROUP; i++) {
            uint8_t c = codes[g * GROUP + i];
            float q = is_signed ? (float)(int8_t)c : (float)c;
            float sum = q + z;
            out[g * GROUP + i] = sum * s;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* encodeValues: fwht(encode), then per 32-group scale = sqrt(mean(x^2)),   */
/* xNorm = x / (scale + eps), idx = searchsorted(boundaries, xNorm).        */
static float pairwise_sum(const float* a, int n) {
    if (n == 1) return a[0];
    return pairwise_sum(a, n / 2) + pairwise_sum(a + n / 2, n / 2);
}

int oracle_encode_values_row(const float* x, int d, int bits, uint8_t* idx, uint16_t* scales) {
    if (!supported_head_dim(d)) return ORACLE_ERR_HEAD_DIM;
    const float *cent, *bnd;
    int nc = oracle_lloyd_max(bits, &cent, &bnd);
    if (!nc) return ORACLE_ERR_BITS;
    float y[512];
    memcpy(y, x, sizeof(float) * (size_t)d);
    oracle_fwht(y, d, 1);
    for (int g = 0; g < d / GROUP; g++) {
        const float* yg = y + g * GROUP;
        float sq[GROUP];
        for (int i = 0; i < GROUP; i++) sq[i] = yg[i] * yg[i];
        float mean_sq = pairwise_sum(sq, GROUP) / (float)GROUP;
        float scale = sqrtf(mean_sq);
        float scale_eps = scale + kEps;
        float xnorm[GROUP];
        for (int i = 0; i < GROUP; i++) xnorm[i] = yg[i] / scale_eps;
        oracle_searchsorted(bnd, nc - 1, xnorm, GROUP, idx + g * GROUP);
        scales[g] = oracle_f32_to_f16(scale);
    }
    return ORACLE_OK;
}

/* dequantScaled: centroids[idx] * scale, in the rotated domain. */
int oracle_decode_values_rotated_row(const uint8_t* idx, int d, int bits,
                                     const uint16_t* scales, float* out) {
    if (!supported_head_dim(d)) return ORACLE_ERR_HEAD_DIM;
    const float *cent, *bnd;
    int nc = oracle_lloyd_max(bits, &cent, &bnd);
    if (!nc) return ORACLE_ERR_BITS;
    for (int g = 0; g < d / GROUP; g++) {
        float s = oracle_f16_to_f32(scales[g]);
        for (int i = 0; i < GROUP; i++) {
            int c = idx[g * GROUP + i];
            if (c >= nc) return ORACLE_ERR_INVALID_ARG;
            out[g * GROUP + i] = cent[c] * s;
        }
    }
    return ORACLE_OK;
}

/* decodeValues: dequantScaled, then fwht(decode). */
int oracle_decode_values_row(const uint8_t* idx, int d, int bits, const uint16_t* scales, float* out) {
    int st = oracle_decode_values_rotated_row(idx, d, bits, scales, out);
    if (st) return st;
    oracle_fwht(out, d, 0);
    return ORACLE_OK;
}

/* unrotateValues: fwht(decode) on fp32 rows. */
int oracle_unrotate_rows(const float* x, int64_t n, int d, float* out) {
    if (!supported_head_dim(d)) return ORACLE_ERR_HEAD_DIM;
    for (int64_t r = 0; r < n; r++) {
        memcpy(out + r * d, x + r * d, sizeof(float) * (size_t)d);
        oracle_fwht(out + r * d, d, 0);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Whole tensors, row by row.                                               */
static void load_row(const void* base, int dtype, int64_t row, int64_t d, float* out) {
    if (dtype == ORACLE_F32) {
        memcpy(out, (const float*)base + row * d, sizeof(float) * (size_t)d);
    } else {
        const uint16_t* p = (const uint16_t*)base + row * d;
        for (int64_t i = 0; i < d; i++) out[i] = oracle_bf16_to_f32(p[i]);
    }
}

static void store_row(void* base, int dtype, int64_t row, int64_t d, const float* in) {
    if (dtype == ORACLE_F32) {
        memcpy((float*)base + row * d, in, sizeof(float) * (size_t)d);
    } else {
        uint16_t* p = (uint16_t*)base + row * d;
        for (int64_t i = 0; i < d; i++) p[i] = oracle_f32_to_bf16(in[i]);
    }
}

static int check_shapes(int64_t B, int64_t H, int64_t T, int64_t D, int k_bits, int k_signed,
                        int v_bits, int64_t t_cap, int64_t t_off) {
    if (B < 0 || H < 0 || T < 0 || t_off < 0 || t_cap < 0) return ORACLE_ERR_INVALID_ARG;
    if (!supported_head_dim(D)) return ORACLE_ERR_HEAD_DIM;
    if (!valid_key_bits(k_bits, k_signed)) return ORACLE_ERR_BITS;
    const float *c, *b;
    if (!oracle_lloyd_max(v_bits, &c, &b)) return ORACLE_ERR_BITS;
    if (t_off + T > t_cap) return ORACLE_ERR_INVALID_ARG;
    return ORACLE_OK;
}

int oracle_encode_kv(const void* k, const void* v, int in_dtype,
                     int64_t B, int64_t H, int64_t T, int64_t D,
                     int k_bits, int k_signed, int v_bits,
                     uint8_t* k_codes, uint16_t* k_scales, uint16_t* k_zeros,
                     uint8_t* v_codes, uint16_t* v_scales,
                     int64_t t_cap, int64_t t_off) {
    int st = check_shapes(B, H, T, D, k_bits, k_signed, v_bits, t_cap, t_off);
    if (st) return st;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return ORACLE_ERR_DTYPE;
    const int64_t G = D / GROUP;
    const int64_t pk = oracle_packed_dim(D, k_bits), pv = oracle_packed_dim(D, v_bits);
    float row[512];
    uint8_t codes[512];
    for (int64_t bh = 0; bh < B * H; bh++) {
        for (int64_t t = 0; t < T; t++) {
            const int64_t in_row = bh * T + t;
            const int64_t out_row = bh * t_cap + t_off + t;
            load_row(k, in_dtype, in_row, D, row);
            oracle_encode_keys_row(row, (int)D, k_bits, k_signed, codes,
                                   k_scales + out_row * G, k_zeros + out_row * G);
            oracle_pack_bits(codes, D, k_bits, k_codes + out_row * pk);
            load_row(v, in_dtype, in_row, D, row);
            oracle_encode_values_row(row, (int)D, v_bits, codes, v_scales + out_row * G);
            oracle_pack_bits(codes, D, v_bits, v_codes + out_row * pv);
        }
    }
    return ORACLE_OK;
}

int oracle_decode_kv(const uint8_t* k_codes, const uint16_t* k_scales, const uint16_t* k_zeros,
                     const uint8_t* v_codes, const uint16_t* v_scales,
                     int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                     int k_bits, int k_signed, int v_bits,
                     void* k_out, void* v_out, int out_dtype, int rotated_v) {
    int st = check_shapes(B, H, T, D, k_bits, k_signed, v_bits, t_cap, 0);
    if (st) return st;
    if (out_dtype != ORACLE_F32 && out_dtype != ORACLE_BF16) return ORACLE_ERR_DTYPE;
    const int64_t G = D / GROUP;
    const int64_t pk = oracle_packed_dim(D, k_bits), pv = oracle_packed_dim(D, v_bits);
    float row[512];
    uint8_t codes[512];
    for (int64_t bh = 0; bh < B * H; bh++) {
        for (int64_t t = 0; t < T; t++) {
            const int64_t in_row = bh * t_cap + t;
            const int64_t out_row = bh * T + t;
            oracle_unpack_bits(k_codes + in_row * pk, D, k_bits, codes);
            oracle_decode_keys_row(codes, (int)D, k_signed, k_scales + in_row * G,
                                   k_zeros + in_row * G, row);
            store_row(k_out, out_dtype, out_row, D, row);
            oracle_unpack_bits(v_codes + in_row * pv, D, v_bits, codes);
            if (rotated_v) {
                oracle_decode_values_rotated_row(codes, (int)D, v_bits, v_scales + in_row * G, row);
            } else {
                oracle_decode_values_row(codes, (int)D, v_bits, v_scales + in_row * G, row);
            }
            store_row(v_out, out_dtype, out_row, D, row);
        }
    }
    return ORACLE_OK;
}
