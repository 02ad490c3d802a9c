/* tq_oracle.h -- plain, slow, single-threaded CPU oracle of the TurboQuant
 * KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY. The product (the CUDA library) never includes,
 * links or calls this code; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it, to check the GPU path and to time a CPU
 * reference. It shares no code, header, table or helper with the CUDA path.
 *
 * What it follows: page "@mlx-bun/inference 0.0.0-stage -> 1.0.0", file
 * package/src/kernels/turboquant/ops.ts (the codec ops: packedDim, fwht,
 * searchsorted, encodeKeys, decodeKeys, encodeValues, dequantScaled,
 * decodeValues, decodeValuesRotated, unrotateValues, packBits, unpackBits) and
 * page "mlx-bun 0.0.9 -> 0.0.11", file package/src/mlx/turboquant-tables.ts
 * (SIGN_VECTORS, LLOYD_MAX). Every step is computed in IEEE binary32 with one
 * rounding per operation (built with -ffp-contract=off, no fast-math): the
 * pages fix fp32 for all codec arithmetic (keys are upcast to fp32 first; the
 * value path is promoted to fp32 by the sign multiply) and fp16 for the stored
 * scales and zero points.
 *
 * Readings taken where the pages leave a step open (each is listed again in
 * the design notes):
 *   - round() is round-half-to-even (nearbyintf in the default rounding mode).
 *   - float->fp16 and float->bf16 casts are IEEE round-to-nearest-even with
 *     overflow to +-Inf (this is what makes a constant key group's zero point
 *     become +Inf, which the codec header comment on the ops.ts page requires).
 *   - The Hadamard transform is the Sylvester-ordered one, computed by radix-2
 *     butterflies with strides 1, 2, 4, ..., d/2 in ascending order, then one
 *     multiply by fp32(1/sqrt(d)).
 *   - The mean of squares over a 32-group is the pairwise-tree sum of the 32
 *     squares (pairs (0,1),(2,3),... first), divided by 32.
 *   - searchsorted counts boundaries strictly below x (the page's
 *     x > boundaries comparison); NaN counts nothing.
 *   - Packed rows are independent; each row is a flat LSB-first bitstream.
 *
 * Parity pins: every function here is checked by the -m "not gpu" tests
 * against something other than itself (library routines, closed forms,
 * brute force, hand-evaluated page formulas, the page's stated special case).
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes of the tensor-level oracle calls (0 = ok). */
enum {
    ORACLE_OK = 0,
    ORACLE_ERR_INVALID_ARG = 1,
    ORACLE_ERR_HEAD_DIM = 2,
    ORACLE_ERR_BITS = 3,
    ORACLE_ERR_ALIGNMENT = 4,
    ORACLE_ERR_DTYPE = 5
};
/* Element types of K/V tensors: 0 = fp32, 1 = bf16 (raw 16-bit patterns). */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* ---- constants (tq_oracle_tables.c) ------------------------------------ */
/* +-1 sign table for head_dim 64/128/256/512, NULL otherwise. */
const signed char* oracle_sign_vector(int head_dim);
/* Lloyd-Max table for bits 2/3/4/5/8: sets the pointers, returns the number
 * of centroids (2^bits); boundaries has one entry fewer. Returns 0 for an
 * unsupported width. */
int oracle_lloyd_max(int bits, const float** centroids, const float** boundaries);

/* ---- packedDim (ops.ts, packedDim) ------------------------------------- */
/* dim*bits/8, or -1 when dim*bits is not a multiple of 8. */
int64_t oracle_packed_dim(int64_t dim, int bits);

/* ---- scalar conversions (IEEE 754 binary16 / bfloat16, RNE) ------------ */
uint16_t oracle_f32_to_f16(float x);
float oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float x);
float oracle_bf16_to_f32(uint16_t h);
/* round half to even, in fp32 */
float oracle_round(float x);
/* the same conversions over arrays of n elements */
void oracle_f32_to_f16_n(const float* x, int64_t n, uint16_t* out);
void oracle_f16_to_f32_n(const uint16_t* h, int64_t n, float* out);
void oracle_f32_to_bf16_n(const float* x, int64_t n, uint16_t* out);

/* ---- rotation (ops.ts, fwht) ------------------------------------------- */
/* In-place unnormalised Sylvester Hadamard transform of n = 2^k floats. */
void oracle_hadamard_unnormalized(float* x, int n);
/* The normalised transform H x / sqrt(n), as one more multiply by
 * fp32(1/sqrt(n)). */
void oracle_hadamard(float* x, int n);
/* fwht(x, encode): encode = signs then normalised Hadamard; decode =
 * normalised Hadamard then signs. Returns -1 for an unsupported d. */
int oracle_fwht(float* x, int d, int encode);
/* oracle_hadamard (normalised=1) or oracle_hadamard_unnormalized on each of
 * n_rows contiguous rows of n floats; oracle_fwht on rows of d floats. */
void oracle_hadamard_rows(float* x, int64_t n_rows, int n, int normalised);
int oracle_fwht_rows(float* x, int64_t n_rows, int d, int encode);

/* ---- searchsorted (ops.ts, searchsorted) ------------------------------- */
/* out[i] = number of boundaries b_j with b_j < x[i]. */
void oracle_searchsorted(const float* boundaries, int nb, const float* x, int64_t n,
                         uint8_t* out);

/* ---- bit packing (ops.ts, packBits / unpackBits) ----------------------- */
/* n codes (low `bits` bits used) -> packed_dim(n, bits) bytes; bits == 8
 * copies bytes. Returns -1 for an unsupported width or misalignment. */
int oracle_pack_bits(const uint8_t* codes, int64_t n, int bits, uint8_t* out);
int oracle_unpack_bits(const uint8_t* packed, int64_t n, int bits, uint8_t* codes);

/* ---- one row of head_dim d (ops.ts, encodeKeys ... decodeValues) ------- */
/* Keys: affine min/max quantisation per 32-group. Codes are unpacked, one
 * byte per element (two's complement when is_signed). scales/zeros: fp16
 * bit patterns, d/32 each. */
int oracle_encode_keys_row(const float* x, int d, int bits, int is_signed,
                           uint8_t* codes, uint16_t* scales, uint16_t* zeros);
int oracle_decode_keys_row(const uint8_t* codes, int d, int is_signed,
                           const uint16_t* scales, const uint16_t* zeros, float* out);
/* Values: rotate, per-32-group RMS scale, Lloyd-Max index. idx unpacked. */
int oracle_encode_values_row(const float* x, int d, int bits, uint8_t* idx,
                             uint16_t* scales);
/* Eager decode: centroid * scale, inverse rotation. */
int oracle_decode_values_row(const uint8_t* idx, int d, int bits,
                             const uint16_t* scales, float* out);
/* Deferred decode: centroid * scale only (still in the rotated domain). */
int oracle_decode_values_rotated_row(const uint8_t* idx, int d, int bits,
                                     const uint16_t* scales, float* out);

/* ---- whole tensors, same conventions as the library's C ABI ------------ */
/* k, v: [B,H,T,D] contiguous, element type in_dtype. Packed outputs are
 * [B,H,t_cap,X] with X = packed_dim(D,bits) (codes) or D/32 (fp16 scales,
 * zeros); tokens [t_off, t_off+T) are written, nothing else is touched. */
int oracle_encode_kv(const void* k, const void* v, int in_dtype,
                     int64_t B, int64_t H, int64_t T, int64_t D,
                     int k_bits, int k_signed, int v_bits,
                     uint8_t* k_codes, uint16_t* k_scales, uint16_t* k_zeros,
                     uint8_t* v_codes, uint16_t* v_scales,
                     int64_t t_cap, int64_t t_off);
/* Reads tokens [0,T) of caches with capacity t_cap; writes [B,H,T,D] outputs
 * of element type out_dtype. rotated_v != 0 leaves V in the rotated domain. */
int oracle_decode_kv(const uint8_t* k_codes, const uint16_t* k_scales, const uint16_t* k_zeros,
                     const uint8_t* v_codes, const uint16_t* v_scales,
                     int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                     int k_bits, int k_signed, int v_bits,
                     void* k_out, void* v_out, int out_dtype, int rotated_v);
/* unrotateValues: inverse rotation of n rows of d values (fp32 in, fp32 out). */
int oracle_unrotate_rows(const float* x, int64_t n, int d, float* out);

/* ---- decode attention over a packed cache (tq_oracle_attention.c) ----- */
/* q: [B,Hq,Nq,D] bf16 bit patterns; cache: [B,Hkv,t_cap,X], tokens [0,T)
 * valid; left_pad: B entries or NULL; out: [B,Hq,Nq,D] doubles, the attention
 * output after the inverse rotation. Query head hq reads kv head hq/(Hq/Hkv);
 * query token n attends to keys left_pad[b] <= t <= T-Nq+n; a row with no
 * valid key is zero. */
int oracle_decode_attention(const uint16_t* q, int64_t B, int64_t Hq, int64_t Nq,
                            const uint8_t* k_codes, const uint16_t* k_scales, const uint16_t* k_zeros,
                            const uint8_t* v_codes, const uint16_t* v_scales,
                            int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                            int k_bits, int k_signed, int v_bits,
                            const int32_t* left_pad, double scale, double* out);

#ifdef __cplusplus
}
#endif
#endif
