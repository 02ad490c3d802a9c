/* tq_oracle_attention.c -- oracle of decode attention over a packed
 * TurboQuant KV cache.
 *
 * TEST INFRASTRUCTURE ONLY, like the rest of this directory: the CUDA library
 * never includes, links or calls it.
 *
 * What it follows:
 *   - page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
 *     package/src/kernels/turboquant/ops.ts: tryDecodePackedKv with deferV
 *     decodes the keys with decodeKeys and the values with
 *     decodeValuesRotated, both returned as bf16; attention runs over those
 *     rows; unrotateValues then applies the inverse rotation once to the
 *     attention output (the decodeValuesRotated comment: attention is linear
 *     in V, so rotating the weighted sum back equals weighting the rotated-
 *     back rows);
 *   - page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
 *     package/src/model/batched-mask.ts (and the quantized cache wrapper in
 *     batched-quant.ts): a batch row padded on the left by leftPad[b] tokens
 *     never attends to its pad columns.
 *
 * The attention itself is the textbook definition, o = softmax(scale * q K^T) V
 * over the valid keys, evaluated in double precision from the bf16 decoded
 * rows, and the inverse rotation of the output is the exact orthogonal map
 * (Sylvester Hadamard / sqrt(d), then the signs), also in double. The
 * readings taken where the pages leave this open:
 *   - grouped-query attention: query head hq reads kv head hq / (Hq / Hkv);
 *   - Nq query tokens per head (a decode step of Nq new tokens already
 *     written to the cache): query token n sits at position T - Nq + n and
 *     attends to keys t with leftPad[b] <= t <= T - Nq + n;
 *   - a query row with no valid key outputs zeros;
 *   - a NaN score (a constant key group decodes to NaN) makes its row NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "tq_oracle.h"

/* Unnormalised Sylvester Hadamard transform in double (radix-2 stages). */
static void hadamard_double(double* x, int n) {
    for (int h = 1; h < n; h *= 2) {
        for (int i0 = 0; i0 < n; i0 += 2 * h) {
            for (int j = 0; j < h; j++) {
                const double a = x[i0 + j], b = x[i0 + j + h];
                x[i0 + j] = a + b;
                x[i0 + j + h] = a - b;
            }
        }
    }
}

int oracle_decode_attention(const uint16_t* q, int64_t B, int64_t Hq, int64_t Nq,
                            const uint8_t* k_codes, const uint16_t* k_scales, const uint16_t* k_zeros,
                            const uint8_t* v_codes, const uint16_t* v_scales,
                            int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                            int k_bits, int k_signed, int v_bits,
                            const int32_t* left_pad, double scale, double* out) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || T < 0 || Hq % Hkv != 0) return ORACLE_ERR_INVALID_ARG;
    const signed char* sign = oracle_sign_vector((int)D);
    if (!sign) return ORACLE_ERR_HEAD_DIM;
    const int64_t G = Hq / Hkv;
    const int64_t pk = oracle_packed_dim(D, k_bits), pv = oracle_packed_dim(D, v_bits);
    if (pk < 0 || pv < 0) return ORACLE_ERR_BITS;
    const int64_t ng = D / 32;
    const int64_t rows = T > 0 ? T : 1;
    uint16_t* kb = malloc(sizeof(uint16_t) * rows * D);
    uint16_t* vb = malloc(sizeof(uint16_t) * rows * D);
    double* kd = malloc(sizeof(double) * rows * D);
    double* vd = malloc(sizeof(double) * rows * D);
    double* s = malloc(sizeof(double) * rows);
    double qd[512], o[512];
    int st = (kb && vb && kd && vd && s) ? ORACLE_OK : ORACLE_ERR_INVALID_ARG;
    for (int64_t b = 0; b < B && st == ORACLE_OK; b++) {
        for (int64_t h = 0; h < Hkv && st == ORACLE_OK; h++) {
            /* the (b, h) block of the cache, decoded as tryDecodePackedKv
             * with deferV returns it: bf16 keys, bf16 values still rotated */
            const int64_t blk = b * Hkv + h;
            if (T > 0) {
                st = oracle_decode_kv(k_codes + blk * t_cap * pk, k_scales + blk * t_cap * ng,
                                      k_zeros + blk * t_cap * ng, v_codes + blk * t_cap * pv,
                                      v_scales + blk * t_cap * ng, 1, 1, T, D, t_cap, k_bits, k_signed,
                                      v_bits, kb, vb, ORACLE_BF16, 1);
                if (st) break;
            }
            for (int64_t i = 0; i < T * D; i++) {
                kd[i] = (double)oracle_bf16_to_f32(kb[i]);
                vd[i] = (double)oracle_bf16_to_f32(vb[i]);
            }
            for (int64_t g = 0; g < G; g++) {
                const int64_t hq = h * G + g;
                for (int64_t n = 0; n < Nq; n++) {
                    const int64_t row = (b * Hq + hq) * Nq + n;
                    for (int64_t d = 0; d < D; d++) qd[d] = (double)oracle_bf16_to_f32(q[row * D + d]);
                    int64_t lo = left_pad ? (int64_t)left_pad[b] : 0;
                    int64_t hi = T - Nq + n; /* inclusive */
                    if (lo < 0) lo = 0;
                    if (hi > T - 1) hi = T - 1;
                    double* orow = out + row * D;
                    if (lo > hi) { /* no valid key */
                        for (int64_t d = 0; d < D; d++) orow[d] = 0.0;
                        continue;
                    }
                    /* scores and their largest (NaN scores are skipped here
                     * and poison the sum below) */
                    double m = -INFINITY;
                    for (int64_t t = lo; t <= hi; t++) {
                        double acc = 0.0;
                        for (int64_t d = 0; d < D; d++) acc += qd[d] * kd[t * D + d];
                        s[t] = scale * acc;
                        if (s[t] > m) m = s[t];
                    }
                    double den = 0.0;
                    for (int64_t d = 0; d < D; d++) o[d] = 0.0;
                    for (int64_t t = lo; t <= hi; t++) {
                        const double p = exp(s[t] - m);
                        den += p;
                        for (int64_t d = 0; d < D; d++) o[d] += p * vd[t * D + d];
                    }
                    for (int64_t d = 0; d < D; d++) o[d] /= den;
                    /* unrotateValues: Hadamard / sqrt(d), then the signs */
                    hadamard_double(o, (int)D);
                    const double c = 1.0 / sqrt((double)D);
                    for (int64_t d = 0; d < D; d++) orow[d] = o[d] * c * (double)sign[d];
                }
            }
        }
    }
    free(kb);
    free(vb);
    free(kd);
    free(vd);
    free(s);
    return st;
}
