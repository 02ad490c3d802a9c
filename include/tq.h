/* tq.h -- C ABI of the GB300 TurboQuant KV-cache codec (libtq.so).
 *
 * The codec is the one on page "@mlx-bun/inference 0.0.0-stage -> 1.0.0",
 * file package/src/kernels/turboquant/ops.ts, with the constants of page
 * "mlx-bun 0.0.9 -> 0.0.11", file package/src/mlx/turboquant-tables.ts:
 *   keys   -> per-32-group affine min/max quantisation along head_dim in fp32,
 *             scale and zero point stored as fp16 (encodeKeys / decodeKeys);
 *   values -> sign flip, normalised Hadamard transform, per-32-group RMS scale
 *             (fp16), Lloyd-Max index (encodeValues / decodeValues);
 *   codes  -> byte-aligned LSB-first bit packing per row (packBits / unpackBits).
 *
 * Conventions shared by every call:
 *   - K and V tensors are contiguous [B, H, T, D] (batch, kv heads, tokens,
 *     head_dim), element type tq_dtype.
 *   - A packed cache is five contiguous buffers, each [B, H, t_cap, X]:
 *       k_codes  X = tq_packed_dim(D, k_bits) bytes (int8 two's complement
 *                when k_signed, else unsigned codes),
 *       k_scales X = D/32 fp16, k_zeros X = D/32 fp16,
 *       v_codes  X = tq_packed_dim(D, v_bits) bytes, v_scales X = D/32 fp16.
 *     Rows (b, h, t) are packed independently, so a token is a whole row of
 *     each buffer and appends never touch another token's bytes.
 *   - All buffer pointers are device-accessible pointers owned by the caller
 *     (device memory, or pinned host memory mapped into the device's address
 *     space, which the kernels then read or write over the CPU-GPU link); the
 *     library never allocates, frees or keeps them. Every buffer pointer must
 *     be 16-byte aligned. A decode whose buffers are all device memory moves
 *     its data with bulk asynchronous copies; one with a buffer in host memory
 *     takes per-thread loads and stores.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously; the call returns once it is enqueued.
 *   - Arguments are checked on the host before anything is launched; a
 *     non-OK status means nothing was enqueued, except TQ_ERR_CUDA, which
 *     reports the launch error (cudaGetLastError) of the kernel just enqueued.
 *   - Numerics: fp32 with one IEEE rounding per operation in the pages' order;
 *     round() is round-half-to-even; fp16/bf16 stores round to nearest even.
 */
#ifndef TQ_H
#define TQ_H

#include <stdint.h>

/* The entry points are the library's only exported symbols (it is built
 * with hidden visibility for everything else). */
#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, t_off + T > t_cap, size overflow */
    TQ_ERR_HEAD_DIM = 2,    /* D not in {64, 128, 256, 512} */
    TQ_ERR_BITS = 3,        /* v_bits not in {2,3,4,5,8}; k_bits not in {2,4,5,8};
                               k_signed with k_bits != 8 */
    TQ_ERR_ALIGNMENT = 4,   /* dim*bits not a multiple of 8; a buffer not 16-byte aligned */
    TQ_ERR_DTYPE = 5,       /* unknown tq_dtype */
    TQ_ERR_CUDA = 6,        /* the CUDA runtime reported an error */
    TQ_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (tq_lloyd_max_fit_status, tq_device_status) */
    TQ_ERR_DEVICE_CHECK = 8 /* a debug build's device-side index check failed (tq_device_status) */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1 } tq_dtype;

/* packedDim (ops.ts, packedDim): bytes of one packed row of `dim` codes of
 * `bits` bits, dim*bits/8. Returns -TQ_ERR_ALIGNMENT when dim*bits is not a
 * multiple of 8 and -TQ_ERR_INVALID_ARG for dim < 0 or bits < 1. */
TQ_API int64_t tq_packed_dim(int64_t dim, int bits);

/* Encode (ops.ts: encodeKeys + packBits for K, encodeValues + packBits for V),
 * one fused kernel.
 *   k, v        [B,H,T,D] inputs of type in_dtype (read only).
 *   k_bits      2, 4, 5 or 8; k_signed = 1 selects the symmetric int8 form
 *               (k_bits must be 8).
 *   v_bits      2, 3, 4, 5 or 8 (Lloyd-Max table width).
 *   k_codes, k_scales, k_zeros, v_codes, v_scales: the packed cache, capacity
 *               t_cap tokens; tokens [t_off, t_off + T) are written, nothing
 *               else is touched.
 * T == 0 (or B*H == 0) is a no-op that returns TQ_OK. B*H*T above
 * 2^31 - 1 - 2^24 rows returns TQ_ERR_INVALID_ARG (as for tq_decode_kv). */
TQ_API tq_status tq_encode_kv(const void* k, const void* v, tq_dtype in_dtype,
                       int64_t B, int64_t H, int64_t T, int64_t D,
                       int k_bits, int k_signed, int v_bits,
                       void* k_codes, void* k_scales, void* k_zeros,
                       void* v_codes, void* v_scales,
                       int64_t t_cap, int64_t t_off, void* stream);

/* Decode (ops.ts: unpackBits + decodeKeys for K; unpackBits + decodeValues,
 * i.e. centroid * scale followed by the inverse rotation, for V), one fused
 * kernel. Reads tokens [0, T) of a cache of capacity t_cap >= T and writes
 * k_out, v_out as contiguous [B,H,T,D] of type out_dtype. A key group whose
 * stored zero point is infinite (a constant group, see the ops.ts header)
 * decodes to NaN, as the page's formula (q + zero) * scale gives. */
TQ_API tq_status tq_decode_kv(const void* k_codes, const void* k_scales, const void* k_zeros,
                       const void* v_codes, const void* v_scales,
                       int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                       int k_bits, int k_signed, int v_bits,
                       void* k_out, void* v_out, tq_dtype out_dtype, void* stream);

/* Deferred-V decode (ops.ts: decodeValuesRotated, the deferV branch of
 * tryDecodePackedKv). Same arguments, checks and K output as tq_decode_kv;
 * v_out holds the values still in the rotated domain, centroid[idx] * scale
 * per element (fp32 product of the centroid and the stored fp16 scale),
 * rounded to out_dtype, with no inverse Hadamard transform and no signs.
 * Attention over V is linear in V, so a caller may attend over these values
 * and undo the rotation once per output row with tq_unrotate. */
TQ_API tq_status tq_decode_kv_rotated(const void* k_codes, const void* k_scales, const void* k_zeros,
                               const void* v_codes, const void* v_scales,
                               int64_t B, int64_t H, int64_t T, int64_t D, int64_t t_cap,
                               int k_bits, int k_signed, int v_bits,
                               void* k_out, void* v_out, tq_dtype out_dtype, void* stream);

/* Inverse value rotation (ops.ts: unrotateValues, i.e. fwht(x, false)):
 * for each of n_rows contiguous rows of D elements of type dtype, convert to
 * fp32, apply the normalised Hadamard transform (ascending radix-2
 * butterflies, then * fp32(1/sqrt(D))), multiply by the sign vector of D,
 * and store in the same dtype. x and out are device pointers, 16-byte
 * aligned, [n_rows, D], and must not overlap (the input is read through
 * the read-only data path).
 * D in {64,128,256,512}; n_rows == 0 is a no-op; n_rows <= 2^31 - 1 - 2^24. */
TQ_API tq_status tq_unrotate(const void* x, tq_dtype dtype, int64_t n_rows, int64_t D, void* out, void* stream);

/* Lloyd-Max index (ops.ts, searchsorted): idx[i] = number of boundaries of
 * the v_bits table strictly below u[i] (NaN -> 0), for n fp32 values already
 * in the rotated, RMS-normalised domain. u and idx are device pointers
 * (u 4-byte aligned, idx unaligned bytes). The same device routine the
 * encode kernel uses. */
TQ_API tq_status tq_lloyd_max_index(const float* u, int64_t n, int v_bits, uint8_t* idx, void* stream);

/* Fused decode attention over a packed cache (ops.ts: the deferV branch of
 * tryDecodePackedKv, i.e. decodeKeys and decodeValuesRotated returning bf16,
 * attention over those rows, then unrotateValues on the output; the left-pad
 * key mask of batched decode, batched-mask.ts). The decoded cache is never
 * written to memory.
 *   q        [B, Hq, Nq, D] bf16, contiguous: Nq query tokens per head. Query
 *            head hq attends with kv head hq / (Hq / Hkv).
 *   cache    five buffers [B, Hkv, t_cap, X] as for tq_decode_kv; tokens
 *            [0, T) are read. t_cap must be a multiple of 16.
 *   left_pad NULL, or B int32 device values: batch row b never attends to
 *            tokens t < left_pad[b].
 *   Query token n of a head sits at position T - Nq + n and attends to the
 *   keys t with left_pad[b] <= t <= T - Nq + n. For those,
 *     o = H( sum_t softmax_t(scale * q . K[t]) * Vrot[t] ) / sqrt(D) * signs
 *   with K[t] = bf16 of the decoded key row, Vrot[t] = bf16 of centroid *
 *   scale (rotated domain), scores and weights in fp32, products of bf16
 *   operands exact, the weights split into two bf16 parts (exact to about
 *   2^-18 relative), and the inverse rotation in fp32. A row with no valid
 *   key is zero; a key row that decodes to NaN (a constant key group, see
 *   the ops.ts header) makes every row that attends to it NaN.
 *   out      [B, Hq, Nq, D] of out_dtype, contiguous.
 *   scale    the softmax scale (1/sqrt(D) for standard attention).
 *   workspace, workspace_bytes: caller-owned device scratch of at least
 *            tq_decode_attention_workspace_size(B, Hkv, T, D) bytes (16-byte
 *            aligned) for the partial results of the split pass (one record
 *            per split block and kv head it covers) and, when a head can
 *            have more than 32 records, the combine's per-chunk results and
 *            ticket counters (zeroed by the split pass); it must not be in
 *            use by another call still running, and needs no initialisation.
 * Limits: D in {64, 128, 256, 512} (else TQ_ERR_HEAD_DIM; at 256 and 512 two
 * warps share each token tile, one per half of head_dim); Hq a multiple of Hkv
 * and (Hq / Hkv) * Nq <= 16 (else TQ_ERR_INVALID_ARG); t_cap % 16 == 0
 * (else TQ_ERR_ALIGNMENT). B == 0 is a no-op. Two kernels are enqueued on
 * `stream`: the split pass, which cuts the (batch, kv head, 16-token tile)
 * space evenly over one wave of blocks, and the combine pass. */
TQ_API tq_status tq_decode_attention(const void* q, int64_t B, int64_t Hq, int64_t Nq,
                              const void* k_codes, const void* k_scales, const void* k_zeros,
                              const void* v_codes, const void* v_scales,
                              int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                              int k_bits, int k_signed, int v_bits,
                              const int32_t* left_pad, float scale, void* out, tq_dtype out_dtype,
                              void* workspace, int64_t workspace_bytes, void* stream);

/* Bytes of scratch tq_decode_attention needs for these sizes on the current
 * device (the token chunking follows the device's SM count, so query it with
 * the same device current). Negative: -TQ_ERR_HEAD_DIM or -TQ_ERR_INVALID_ARG. */
TQ_API int64_t tq_decode_attention_workspace_size(int64_t B, int64_t Hkv, int64_t T, int64_t D);

/* tq_decode_attention for callers that cannot allocate device memory: no
 * counterpart on the pages (an interface addition of this library). Some
 * callers may not call cudaMalloc: a plugin inside a serving runtime that
 * reserves the device's memory budget at start-up and owns every allocation
 * afterwards, or code on a latency-bound path where an allocation (which can
 * synchronize the device) is not acceptable. Such a caller cannot provide the
 * workspace tq_decode_attention needs. This call takes the same arguments
 * minus the workspace and uses a fixed scratch array compiled into the
 * library instead (TQ_ATTENTION_NOALLOC_SCRATCH_BYTES of device memory, held
 * on every GPU that loads the library until the process exits). It allocates
 * nothing.
 *   - Returns TQ_ERR_INVALID_ARG when the scratch these sizes need,
 *     tq_decode_attention_workspace_size(B, Hkv, T, D), is larger than
 *     TQ_ATTENTION_NOALLOC_SCRATCH_BYTES; every other check and result is
 *     that of tq_decode_attention (an empty batch, B == 0, returns TQ_OK
 *     without looking at the scratch). The need is one partial record of
 *     16 * (D + 2) floats per split block and per (batch, kv head) pair, with
 *     at most 8 split blocks per SM (plus, for fewer than 8 * SMs / 30
 *     pairs, at most 8 * 34 * 32 floats per 1024 / D output rows for the
 *     combine), so the largest B * Hkv served is
 *     floor(TQ_ATTENTION_NOALLOC_SCRATCH_BYTES / (64 * (D + 2))) - 8 * SMs:
 *     on a 152-SM GB300 that is 14671, 6849, 2848 and 824 pairs at head_dim
 *     64, 128, 256 and 512, independent of the number of tokens.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture. TQ_ERR_CUDA if the lookup fails.
 *   - All calls share the one array: two calls whose work can overlap on the
 *     GPU (streams with no ordering between them) race. Order them on one
 *     stream or with events. Nothing in the array needs clearing between
 *     calls: each call writes every scratch record it reads. */
#define TQ_ATTENTION_NOALLOC_SCRATCH_BYTES (64LL << 20)
TQ_API tq_status tq_decode_attention_noalloc(const void* q, int64_t B, int64_t Hq, int64_t Nq,
                                      const void* k_codes, const void* k_scales, const void* k_zeros,
                                      const void* v_codes, const void* v_scales,
                                      int64_t Hkv, int64_t T, int64_t D, int64_t t_cap,
                                      int k_bits, int k_signed, int v_bits,
                                      const int32_t* left_pad, float scale, void* out, tq_dtype out_dtype,
                                      void* stream);

/* One source row of tq_cache_assemble: tokens [t_start, t_start + len) of
 * batch row b of a packed cache (five buffers [B, H, t_cap, X], as above,
 * with the destination's H, D and bit widths). Pointers may be NULL when
 * len == 0 (an all-padding row). */
typedef struct {
    const void* k_codes;
    const void* k_scales;
    const void* k_zeros;
    const void* v_codes;
    const void* v_scales;
    int64_t B;       /* batch rows of the source cache */
    int64_t b;       /* the batch row read, 0 <= b < B */
    int64_t t_cap;   /* token capacity of the source cache */
    int64_t t_start; /* first token read */
    int64_t len;     /* tokens read, 0 <= len <= width, t_start + len <= t_cap */
} tq_row_source;

/* Batched packed-cache row assembly, the byte-preserving primitive behind
 * the continuous-batching cache operations of page "@mlx-bun/inference
 * 0.0.0-stage -> 1.0.0", file batched-quant.ts (mergeQuantRows,
 * extendQuantRows, extractQuantRow, filterQuantRows): destination batch row
 * r (of n_rows) receives, for every head and each of the five buffers,
 * width - rows[r].len zero tokens followed by the source's tokens
 * [t_start, t_start + len), i.e. the row right-justified in a window of
 * `width` tokens with its left padding zeroed. Tokens [width, t_cap) of the
 * destination are not touched. Quantization packs along head_dim only, so
 * this copies whole token rows and never alters a quantization group.
 *   rows      host array of n_rows descriptors (read during the call).
 *   destination: five buffers [n_rows, H, t_cap, X], 16-byte aligned; X from
 *             D, k_bits, v_bits as for tq_encode_kv. Source and destination
 *             memory must not overlap.
 * Sizes and descriptors are checked on the host (TQ_ERR_INVALID_ARG,
 * TQ_ERR_HEAD_DIM, TQ_ERR_BITS, TQ_ERR_ALIGNMENT) before anything is
 * enqueued; one kernel is enqueued per 48 destination rows. */
TQ_API tq_status tq_cache_assemble(const tq_row_source* rows, int64_t n_rows, int64_t H, int64_t D,
                            int k_bits, int v_bits, void* k_codes, void* k_scales, void* k_zeros,
                            void* v_codes, void* v_scales, int64_t t_cap, int64_t width, void* stream);

/* Lloyd-Max fit of a scalar quantizer table, the procedure the tables page
 * (page "mlx-bun 0.0.9 -> 0.0.11", turboquant-tables.ts header) names for
 * the LLOYD_MAX value tables: `iters` Lloyd iterations on the fp32 sample
 * x[0..n) starting from the ascending centroids init[0..levels). One
 * iteration: boundaries are the fp32 midpoints RN(c_k + c_{k+1}) / 2; each
 * sample joins cell count(boundaries < x) (the codec's searchsorted); each
 * centroid becomes its cell's mean (sum / count in float64, rounded once to
 * fp32); a cell with no samples keeps its centroid. Cell sums are exact
 * integers in units of 2^-32 (samples of magnitude below 2^-9 are rounded to
 * that unit), so the result does not depend on the order of additions.
 *   x          n finite fp32 samples with sum |x| < 2^31 (device).
 *   levels     2, 4, ..., 256; init, centroids: levels fp32 (device);
 *              boundaries: levels - 1 fp32 (device), the final midpoints.
 *   workspace  device scratch of tq_lloyd_max_fit_workspace_size(levels)
 *              bytes (16-byte aligned; the call clears it first).
 * One cooperative kernel runs every iteration (its blocks meet at a bounded
 * grid barrier per iteration; if a wait gives up, centroids and boundaries
 * are left NaN and tq_lloyd_max_fit_status reports TQ_ERR_TIMEOUT);
 * n < 2^31. Returns once the work is enqueued. */
TQ_API tq_status tq_lloyd_max_fit(const float* x, int64_t n, int levels, int iters, const float* init,
                           float* centroids, float* boundaries, void* workspace, int64_t workspace_bytes,
                           void* stream);

/* tq_lloyd_max_fit with the grid barrier's give-up made explicit (no
 * counterpart on the pages: failure detection of this library's
 * cooperative kernel).
 *   spin_limit    polls (about 64 ns each) a block waits at a grid barrier
 *                 before it gives up; 0 takes the default 2^22 (about a
 *                 quarter of a second). At most 2^32 - 1.
 *   absent_block  -1, or a test hook: the index of a block that leaves the
 *                 kernel at its first barrier without arriving, as a block
 *                 that died would; every other block's wait then runs out,
 *                 the error word is set and centroids and boundaries are
 *                 left NaN. Every wait stays bounded either way. */
TQ_API tq_status tq_lloyd_max_fit_bounded(const float* x, int64_t n, int levels, int iters, const float* init,
                                   float* centroids, float* boundaries, void* workspace, int64_t workspace_bytes,
                                   int64_t spin_limit, int absent_block, void* stream);

/* Outcome of the last fit enqueued with `workspace`: waits for `stream`,
 * then reads the fit's error word from the workspace (byte offset 8).
 * TQ_OK, or TQ_ERR_TIMEOUT when a block gave up at a grid barrier (the
 * results are then NaN); TQ_ERR_CUDA if the wait or the copy failed. */
TQ_API tq_status tq_lloyd_max_fit_status(const void* workspace, void* stream);

/* Bytes of scratch tq_lloyd_max_fit needs (64 + 48 * levels), or
 * -TQ_ERR_INVALID_ARG for a level count that is not a power of two in
 * [2, 256]. */
TQ_API int64_t tq_lloyd_max_fit_workspace_size(int levels);

/* Device-side failures of the library's kernels on the current device (no
 * counterpart on the pages: failure detection of this library). Kernels that
 * wait on an asynchronous copy (the decode's bulk-copy path) bound the wait;
 * one that gives up sets the device error word, stops early and leaves its
 * outputs incomplete. A debug build of the library (compiled with
 * -DTQ_DEBUG_CHECKS) also checks the row and record indices of its kernels'
 * global accesses against the buffers' extents, and an index outside them
 * sets the word and skips the access (no trap). This call waits for
 * `stream`, then returns TQ_OK; or TQ_ERR_DEVICE_CHECK (an index check
 * failed) or TQ_ERR_TIMEOUT (a wait gave up), clearing the word; or
 * TQ_ERR_CUDA if the wait or the copies failed. The first call of a kernel on
 * a device looks up the word's address (make it before any stream capture). */
TQ_API tq_status tq_device_status(void* stream);

/* 1 in a debug build of the library (device-side index checks), else 0. */
TQ_API int tq_debug_checks(void);

/* Human-readable name of a status code (static string). */
TQ_API const char* tq_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif
