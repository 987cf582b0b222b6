/*
 * fp8gemm.h -- C ABI of the GB300 (sm_103a) FP8 block-scaled GEMM library.
 *
 * What is computed.  FP8 e4m3 operands with fine-grained block scales, FP32
 * accumulation and a BF16 result:
 *
 *     D[m, n] = bf16( sum_kb  P_kb[m, n] * sA[kb][m] * sB[n / 128][kb] )
 *     P_kb[m, n] = sum_{k in K block kb} A[m, k] * B[n, k]       (128-wide K blocks)
 *
 * Calls (declared below in this order):
 *   quantisation   fp8_quantize_1x128, fp8_quantize_1x128_masked, fp8_route_gather_quantize_1x128,
 *                  fp8_quantize_128x128
 *   GEMMs          fp8_gemm_nt, fp8_gemm_nt_noalloc, fp8_grouped_gemm_contiguous,
 *                  fp8_grouped_gemm_masked
 *   per-tensor / per-token / per-channel scales
 *                  fp8_quantize_per_row, fp8_quantize_per_tensor, fp8_gemm_nt_scaled,
 *                  fp8_grouped_gemm_contiguous_scaled, fp8_grouped_gemm_masked_scaled
 *   backward (e5m2 gradients)
 *                  fp8_quantize_1x128_e5m2, fp8_gemm_nt_dgrad, fp8_grouped_gemm_contiguous_dgrad,
 *                  fp8_grouped_gemm_wgrad
 *   status         fp8g_get_status, fp8g_status_string, fp8g_selftest_bounded_waits, fp8g_last_config,
 *                  fp8g_last_split, fp8g_last_swap_ab, fp8g_last_cluster_k
 *
 * Sources (page title, section):
 *  - "DeepGEMM FP8 walk-through" (m.czchanglian.com/news/60438), sec. 2.2: per-token
 *    scales for the activations A, per-channel scales for the weights B, K cut
 *    into blocks; scales handled inside the GEMM pipeline.  Sec. 2.3: FP32
 *    accumulation across the whole K, rounding to the output type only on write.
 *  - "DeepGEMM explainer" (nxmr.cn/news/131680), sec. 3.1: a block's scale is its
 *    amax divided by the largest FP8 value; sec. 3.2: the MoE grouped GEMM runs
 *    experts with different token counts in one kernel; sec. 3.3: operands are
 *    taken without a transpose (A and B both K-contiguous, "NT"); sec. 4.2: the
 *    call takes FP8 a and b, their scales and the group sizes; sec. 5.1: the
 *    scale shapes must match the blocking (1x128 rows of A, 128x128 blocks of B).
 *  - "Production FP8 GEMM alignment and Tensor Core peak tuning" (gtnt.cn/news/117510),
 *    "E4M3 vs E5M2": e4m3 range +-448.
 *
 * Conventions for every call:
 *  - Every pointer is CUDA device memory on the current device, owned by the
 *    caller.  The library never allocates, frees or synchronises caller
 *    buffers, and never synchronises the stream (except fp8g_get_status).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Work is enqueued on it; results are valid once the stream reaches that point.
 *  - The return value is an fp8g_status.  Arguments are validated on the host
 *    before anything is launched; an invalid call launches nothing and returns
 *    FP8G_ERR_INVALID_ARG or FP8G_ERR_ALIGNMENT.  Calls never throw.
 *  - Errors found on the device (a bounded wait that ran out, out-of-contract
 *    group offsets or counts) are recorded in a per-device status word that
 *    fp8g_get_status reads and clears; the kernel returns early instead of
 *    trapping, so the CUDA context stays usable.
 *  - e4m3 bytes use the OCP "e4m3fn" encoding (no infinities, 0x7F/0xFF NaN,
 *    max 448); e5m2 bytes (gradients) the OCP "E5M2" encoding (max 57344, with
 *    infinities and NaN in the top exponent).  Inputs must be finite.
 *  - Only sm_103 devices are supported; anything else returns
 *    FP8G_ERR_UNSUPPORTED_DEVICE (there is no fallback path).
 *  - Calls are thread-safe; calls on different streams may run concurrently.
 *  - GEMM workspace.  When a GEMM's tiles do not fill whole rounds of the grid, the
 *    K blocks of the last, partial round may be split across all SMs (stream-K;
 *    FP8G_STREAMK=0 turns this off).  The first such call on a stream allocates an
 *    internal workspace for it -- 128 KiB per SM plus one flag per SM, about 19 MiB
 *    on GB300 -- which the library keeps for the life of the process.  A call made
 *    while its stream is being captured never allocates: if that stream has no
 *    workspace yet, the call runs without the split.  fp8_gemm_nt_noalloc is the
 *    variant that never allocates.
 */
#ifndef FP8GEMM_H_
#define FP8GEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8G_OK = 0,
  FP8G_ERR_INVALID_ARG = 1,        /* a size, count or leading dimension out of range */
  FP8G_ERR_ALIGNMENT = 2,          /* a pointer or stride not 16-byte aligned */
  FP8G_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 */
  FP8G_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed (launch, attribute, ...) */
  FP8G_ERR_TIMEOUT = 5,            /* device: a pipeline wait ran past its cycle budget */
  FP8G_ERR_DEVICE_ASSERT = 6       /* device: out-of-contract group offsets / masked counts */
} fp8g_status;

/*
 * fp8_quantize_1x128 -- activation quantisation, one scale per row and 128-wide
 * K block ("DeepGEMM explainer" sec. 3.1; "DeepGEMM FP8 walk-through" sec. 5.2).
 *
 * For every row m and block kb (columns 128*kb .. 128*kb+127):
 *     amax = max |x|;  s = fp32(amax / 448);  q = e4m3(fp32(x / s))
 * with IEEE fp32 division, round-to-nearest-even, saturation to +-448 and the
 * sign kept.  A block with amax == 0 gets s = 0 and all codes 0x00.
 *
 *   x     bf16 [M, K], row stride ldx elements (ldx >= K, ldx % 8 == 0)
 *   q     e4m3 [M, K] (one byte each), row stride ldq bytes (ldq >= K, ldq % 16 == 0)
 *   sA    fp32 [K/128][ld_sa], K-block-major: sA[kb * ld_sa + m]
 *         (ld_sa >= M, ld_sa % 4 == 0; entries m >= M are not written)
 *   M >= 0 (M == 0: no-op), K > 0, K % 128 == 0, M * (K/128) < 2^31.  Pointers 16-byte aligned.
 */
int fp8_quantize_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                       float* sA, int64_t ld_sa, void* stream);

/*
 * fp8_quantize_1x128_masked -- fp8_quantize_1x128 for the masked layout: x and q are [E, cap, K]
 * (contiguous), and only rows m < masked_m[e] of each expert are quantised -- the rows
 * fp8_grouped_gemm_masked reads for its output.  The other rows of q and their scales are left
 * as they are (each output row of the masked GEMM depends only on its own row of A and its
 * scales, and rows past the count are never stored).
 *
 *   x         bf16 [E, cap, K], contiguous
 *   masked_m  int32 [E], DEVICE memory; values are clamped to [0, cap]
 *   q         e4m3 [E, cap, K], contiguous
 *   sA        fp32 [K/128][ld_sa] with row index e*cap + m (ld_sa >= E*cap, ld_sa % 4 == 0)
 *   1 <= E <= 65535, cap >= 0 (cap == 0: no-op), K % 128 == 0, E*cap*(K/128) < 2^31.  x, q, sA 16-byte
 *   aligned.
 */
int fp8_quantize_1x128_masked(const void* x, int32_t E, int64_t cap, int64_t K, const int32_t* masked_m,
                              void* q, float* sA, int64_t ld_sa, void* stream);

/*
 * fp8_route_gather_quantize_1x128 -- builds the contiguous grouped layout that
 * fp8_grouped_gemm_contiguous reads, straight from routed tokens, and quantises it
 * ("DeepGEMM explainer" sec. 3.2 and 4.2; "DeepGEMM FP8 walk-through" sec. 5.3:
 * each expert's rows contiguous and block-loadable, described by group offsets).
 *
 *   x              bf16 [T, K] tokens, row stride ldx elements (ldx >= K, ldx % 8 == 0)
 *   topk_ids       int32 [T, topk], DEVICE memory: the experts each token is routed to
 *   q, sA          outputs as fp8_quantize_1x128 writes them, for M_cap rows:
 *                  e4m3 [M_cap, K] (row stride ldq bytes) and fp32 [K/128][ld_sa >= M_cap]
 *   group_offsets  int32 [E+1], DEVICE memory, output: expert e owns rows
 *                  group_offsets[e] .. group_offsets[e+1]-1 (multiples of 128)
 *   row_token      int32 [M_cap], DEVICE memory, output: the token of each row, -1 for a
 *                  padding row
 *   entry_row      int32 [T*topk], DEVICE memory, output: the row of each entry (token t,
 *                  slot j at t*topk + j), -1 for a dropped entry -- the inverse of row_token,
 *                  the map a combine step needs to bring the experts' output rows back to
 *                  their tokens (may be null when T == 0)
 *   M_cap          rows of q / sA / row_token: a multiple of 128 and at least
 *                  T*topk + 127*E (every group padded to 128 fits)
 *
 * Each token row is read and quantised once and its codes and scales are stored to every
 * row of the token (its 1x128 scales depend only on the row's own values).
 * Inside a group the rows hold the expert's tokens in ascending order (a token that names
 * one expert twice gets two rows), then zero rows up to the next multiple of 128.  Every
 * row with token -1 -- padding, and the rows from group_offsets[E] to M_cap -- has scale
 * 0 and codes 0.  Call the grouped GEMM with M_total = M_cap: rows outside every group
 * are skipped and their output rows left untouched.  Expert ids outside [0, E) are
 * dropped and set FP8G_ERR_DEVICE_ASSERT.  T >= 0, topk >= 1, 1 <= E <= 2048,
 * K % 128 == 0, M_cap * (K/128) < 2^31.  x, q, sA 16-byte aligned (x may be null when
 * T == 0); the int32 arrays 4-byte aligned.
 */
int fp8_route_gather_quantize_1x128(const void* x, int64_t T, int64_t K, int64_t ldx,
                                    const int32_t* topk_ids, int32_t topk, int32_t E, void* q,
                                    int64_t ldq, float* sA, int64_t ld_sa, int32_t* group_offsets,
                                    int32_t* row_token, int32_t* entry_row, int64_t M_cap,
                                    void* stream);

/*
 * fp8_quantize_128x128 -- weight quantisation, one scale per 128x128 block
 * ("DeepGEMM explainer" sec. 5.1; "DeepGEMM FP8 walk-through" sec. 2.2).
 * Same rule as fp8_quantize_1x128 with amax taken over the block's rows that
 * exist (N need not be a multiple of 128).
 *
 *   w     bf16 [E, N, K], contiguous
 *   q     e4m3 [E, N, K], contiguous
 *   sB    fp32 [E][ceil(N/128)][K/128], contiguous
 *   E >= 1, N >= 1, K > 0, K % 128 == 0.  Pointers 16-byte aligned.
 */
int fp8_quantize_128x128(const void* w, int64_t E, int64_t N, int64_t K, void* q, float* sB,
                         void* stream);

/*
 * fp8_gemm_nt -- dense D = A * B^T with 1x128 scales on A and 128x128 scales on B
 * ("DeepGEMM FP8 walk-through" sec. 2.2-2.3; "DeepGEMM explainer" sec. 3.3).
 *
 *   A     e4m3 [M, K], row stride lda bytes (lda >= K, lda % 16 == 0)
 *   sA    fp32 [K/128][ld_sa] (ld_sa >= M, ld_sa % 4 == 0), as written by fp8_quantize_1x128
 *   B     e4m3 [N, K], row stride ldb bytes (ldb >= K, ldb % 16 == 0)
 *   sB    fp32 [ceil(N/128)][K/128], contiguous
 *   D     bf16 [M, N], row stride ldd elements (ldd >= N, ldd % 8 == 0)
 *   M >= 0 (M == 0: no-op), N > 0, N % 16 == 0, K > 0, K % 128 == 0.
 */
int fp8_gemm_nt(const void* A, int64_t lda, const float* sA, int64_t ld_sa, const void* B,
                int64_t ldb, const float* sB, void* D, int64_t ldd, int64_t M, int64_t N,
                int64_t K, void* stream);

/*
 * fp8_gemm_nt_noalloc -- fp8_gemm_nt that never allocates device memory.  The
 * pages have no counterpart of this call: it exists because of the library's own
 * stream-K workspace (see "GEMM workspace" above).
 *
 * Some callers cannot let a library allocate while they run: an allocation can
 * synchronise the device, or fail, in the middle of latency-critical work, and a
 * framework that owns a fixed memory budget or serves allocations from its own
 * pool expects every device buffer to come from it.  fp8_gemm_nt allocates its
 * workspace on the first call on each stream that splits tiles; this call uses a
 * fixed buffer that is part of the library's device image instead: 160 stream-K
 * slots of 128 KiB plus 1 KiB of flags (20 MiB + 1 KiB).  The buffer sits in a module
 * of its own: under lazy module loading (the CUDA default) a device holds it only
 * once this call has run there, until the process exits; with eager loading every
 * device that loads the library holds it.  It does clear the flags with a memset on
 * `stream` before each launch.
 *
 * Same arguments, results and errors as fp8_gemm_nt, plus:
 *  - a device with more than 160 SMs is out of the buffer's range and gets
 *    FP8G_ERR_INVALID_ARG (nothing launched);
 *  - there is one buffer per device, shared by every call of this function on
 *    that device: calls that overlap in time (on different streams, without an
 *    ordering between them) race on it and corrupt each other's results, so the
 *    caller must order them (one stream, or events);
 *  - the first call on each device looks up the buffer's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call before
 *    capturing any stream.  A lookup that fails returns FP8G_ERR_CUDA and is tried
 *    again on the next call.
 */
int fp8_gemm_nt_noalloc(const void* A, int64_t lda, const float* sA, int64_t ld_sa, const void* B,
                        int64_t ldb, const float* sB, void* D, int64_t ldd, int64_t M, int64_t N,
                        int64_t K, void* stream);

/*
 * fp8_grouped_gemm_contiguous -- MoE grouped GEMM, contiguous layout
 * ("DeepGEMM explainer" sec. 3.2 and 4.2; "DeepGEMM FP8 walk-through" sec. 5.3:
 * pass each group's id and token offset; keep each expert's rows contiguous and
 * block-loadable).  Expert e owns rows group_offsets[e] .. group_offsets[e+1]-1
 * of A and D:
 *     D[rows of e] = gemm_nt(A[rows of e], B[e])
 * Rows that belong to no group are left untouched.  Padding rows inside a
 * group are computed like any other row (all-zero rows give zeros).
 *
 *   A             e4m3 [M_total, K], contiguous
 *   sA            fp32 [K/128][ld_sa] (ld_sa >= M_total, ld_sa % 4 == 0)
 *   B             e4m3 [E, N, K], contiguous
 *   sB            fp32 [E][ceil(N/128)][K/128], contiguous
 *   D             bf16 [M_total, N], contiguous
 *   group_offsets int32 [E+1], DEVICE memory, read only by the kernel (the host
 *                 never reads it, so routing can stay on the GPU): non-decreasing,
 *                 each a multiple of 128, group_offsets[E] <= M_total.  Violations
 *                 make the kernel write nothing and set FP8G_ERR_DEVICE_ASSERT.
 *   1 <= E <= 2048, M_total >= 0 and M_total % 128 == 0, N % 16 == 0, K % 128 == 0.
 */
int fp8_grouped_gemm_contiguous(const void* A, const float* sA, int64_t ld_sa, const void* B,
                                const float* sB, void* D, const int32_t* group_offsets,
                                int32_t E, int64_t M_total, int64_t N, int64_t K, void* stream);

/*
 * fp8_grouped_gemm_masked -- MoE grouped GEMM, masked layout: every expert has
 * a fixed capacity of rows and a device-side count of valid rows.  (The pages
 * describe the grouped GEMM but not this layout; it is the decode-time form in
 * which the per-expert token counts stay on the GPU.)
 *     D[e, m, :] = gemm_nt(A[e, m, :], B[e])   for m < masked_m[e]
 * Rows m >= masked_m[e] of D are never written.
 *
 *   A         e4m3 [E, cap, K], contiguous
 *   sA        fp32 [K/128][ld_sa] with row index e*cap + m (ld_sa >= E*cap, ld_sa % 4 == 0)
 *   B         e4m3 [E, N, K], contiguous
 *   sB        fp32 [E][ceil(N/128)][K/128], contiguous
 *   D         bf16 [E, cap, N], contiguous
 *   masked_m  int32 [E], DEVICE memory, 0 <= masked_m[e] <= cap; values outside are
 *             clamped into range and set FP8G_ERR_DEVICE_ASSERT.
 *   1 <= E <= 2048, cap >= 0 and cap % 16 == 0, N % 16 == 0, K % 128 == 0.
 */
int fp8_grouped_gemm_masked(const void* A, const float* sA, int64_t ld_sa, const void* B,
                            const float* sB, void* D, const int32_t* masked_m, int32_t E,
                            int64_t cap, int64_t N, int64_t K, void* stream);

/*
 * Per-tensor / per-token / per-channel scales ("DeepGEMM FP8 walk-through" sec. 2.2:
 * one scale for a whole tensor, or one per token of A and one per output channel of B;
 * "Production FP8 GEMM alignment and Tensor Core peak tuning", the Triton listing's
 * fused epilogue: the FP32 accumulator of the whole K is multiplied once by
 * scale_a * scale_b, then converted to BF16).  Same scale and code rule as the block
 * forms, with the group a whole row or the whole tensor:
 *     amax = max |x|;  s = fp32(amax / 448);  q = e4m3(fp32(x / s));  amax == 0: s = 0, codes 0.
 */

/*
 * fp8_quantize_per_row -- one scale per row over the whole K (per-token for
 * activations, per-channel for weights [N, K] or [E*N, K]).
 *
 *   x   bf16 [M, K], row stride ldx elements (ldx >= K, ldx % 8 == 0)
 *   q   e4m3 [M, K], row stride ldq bytes (ldq >= K, ldq % 16 == 0)
 *   s   fp32 [M]
 *   M >= 0 (M == 0: no-op), K > 0, K % 128 == 0.  x, q 16-byte aligned, s 4-byte aligned.
 */
int fp8_quantize_per_row(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                         float* s, void* stream);

/*
 * fp8_quantize_per_tensor -- one scale per tensor, for E tensors of M rows each (E = 1 for
 * activations; E experts' weights).  Tensor e is rows e*M .. e*M+M-1 of x and q.
 *
 *   x   bf16 [E*M, K], row stride ldx elements (ldx >= K, ldx % 8 == 0)
 *   q   e4m3 [E*M, K], row stride ldq bytes (ldq >= K, ldq % 16 == 0)
 *   s   fp32 [E], output (an empty tensor, M == 0, gets s = 0)
 *   1 <= E <= 65535, M >= 0, K % 128 == 0, M * K / 8 < 2^31.  x, q 16-byte aligned, s 4-byte
 *   aligned.  Two passes over x (the second mostly from L2 when a tensor fits it) and a
 *   memset of s, all on `stream`.
 */
int fp8_quantize_per_tensor(const void* x, int64_t E, int64_t M, int64_t K, int64_t ldx, void* q,
                            int64_t ldq, float* s, void* stream);

/*
 * fp8_gemm_nt_scaled -- dense D = bf16(fp32(acc) * fp32(sA[m] * sB[n])), acc[m, n] the FP32
 * sum over the whole K of A[m, k] * B[n, k].
 *
 *   A, lda, B, ldb, D, ldd, M, N, K   as fp8_gemm_nt
 *   sA   sa_per_row = 1: fp32 [M], one scale per row of A; 0: fp32 [1], one for all of A
 *   sB   sb_per_col = 1: fp32 [N], one scale per row of B (column of D), 16-byte aligned;
 *        0: fp32 [1]
 *   sa_per_row, sb_per_col in {0, 1}.  sA (and sB when sb_per_col == 0) 4-byte aligned.
 * Uses the stream-K workspace of "GEMM workspace" above.
 */
int fp8_gemm_nt_scaled(const void* A, int64_t lda, const float* sA, int32_t sa_per_row,
                       const void* B, int64_t ldb, const float* sB, int32_t sb_per_col, void* D,
                       int64_t ldd, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * fp8_grouped_gemm_contiguous_scaled -- fp8_grouped_gemm_contiguous with epilogue scales:
 *   sA   sa_per_row = 1: fp32 [M_total] (row of A); 0: fp32 [1]
 *   sB   sb_per_col = 1: fp32 [E][N] (16-byte aligned); 0: fp32 [E], one per expert
 * Other arguments, layout and errors as fp8_grouped_gemm_contiguous.
 */
int fp8_grouped_gemm_contiguous_scaled(const void* A, const float* sA, int32_t sa_per_row,
                                       const void* B, const float* sB, int32_t sb_per_col,
                                       void* D, const int32_t* group_offsets, int32_t E,
                                       int64_t M_total, int64_t N, int64_t K, void* stream);

/*
 * fp8_grouped_gemm_masked_scaled -- fp8_grouped_gemm_masked with epilogue scales:
 *   sA   sa_per_row = 1: fp32 [E*cap], row index e*cap + m; 0: fp32 [1]
 *   sB   sb_per_col = 1: fp32 [E][N] (16-byte aligned); 0: fp32 [E]
 * Other arguments, layout and errors as fp8_grouped_gemm_masked.
 */
int fp8_grouped_gemm_masked_scaled(const void* A, const float* sA, int32_t sa_per_row,
                                   const void* B, const float* sB, int32_t sb_per_col, void* D,
                                   const int32_t* masked_m, int32_t E, int64_t cap, int64_t N,
                                   int64_t K, void* stream);

/*
 * Backward GEMMs with e5m2 gradients ("DeepGEMM FP8 walk-through" sec. 2.1 and "Production FP8
 * GEMM alignment and Tensor Core peak tuning", "E4M3 vs E5M2": gradients use e5m2, 1-5-2 bits,
 * range to 57344; OCP "E5M2", with infinities and NaN in the top exponent).
 */

/*
 * fp8_quantize_1x128_e5m2 -- fp8_quantize_1x128 for gradients: s = fp32(amax / 57344), codes
 * e5m2 (round-to-nearest-even, saturating to +-57344).  Same arguments, layout and errors.
 */
int fp8_quantize_1x128_e5m2(const void* x, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                            float* sA, int64_t ld_sa, void* stream);

/*
 * fp8_gemm_nt_dgrad -- the data gradient dX = dY * W as fp8_gemm_nt: A = dY holds e5m2 codes
 * (1x128 scales from fp8_quantize_1x128_e5m2), B = W^T [K_in, N] holds e4m3 codes with 128x128
 * block scales.  Arguments, layout and errors as fp8_gemm_nt.
 */
int fp8_gemm_nt_dgrad(const void* A, int64_t lda, const float* sA, int64_t ld_sa, const void* B,
                      int64_t ldb, const float* sB, void* D, int64_t ldd, int64_t M, int64_t N,
                      int64_t K, void* stream);

/*
 * fp8_grouped_gemm_contiguous_dgrad -- the data gradient of a grouped MoE layer: as
 * fp8_grouped_gemm_contiguous with A = dY in e5m2 (1x128 scales) and B [E, K_in, N] = each
 * expert's W^T in e4m3 (128x128 block scales).  Arguments, layout and errors as
 * fp8_grouped_gemm_contiguous.
 */
int fp8_grouped_gemm_contiguous_dgrad(const void* A, const float* sA, int64_t ld_sa, const void* B,
                                      const float* sB, void* D, const int32_t* group_offsets,
                                      int32_t E, int64_t M_total, int64_t N, int64_t K, void* stream);

/*
 * fp8_grouped_gemm_wgrad -- the weight gradient of a grouped MoE layer, one matrix per expert,
 * contracting over that expert's tokens ("K-grouped"):
 *     D[e] = sum over tokens t of expert e of  A[:, t] (x) B[:, t]      (dW[e] = dY_e^T * X_e)
 * with the block promotion acc += P_kb * (sA[kb][m] * sB[kb][n]) over the expert's 128-token
 * blocks, FP32 accumulation, BF16 output.  An expert with no tokens gets D[e] = 0.
 *
 *   A        e5m2 [M, T] (dY^T: output channels x tokens), row stride lda bytes (lda >= T, % 16)
 *   sA       fp32 [T/128][ld_sa] (ld_sa >= M, % 4), as fp8_quantize_1x128_e5m2 writes it for A
 *   B        e4m3 [N, T] (X^T: input channels x tokens), row stride ldb bytes (ldb >= T, % 16)
 *   sB       fp32 [T/128][ld_sb] (ld_sb >= N, % 4), as fp8_quantize_1x128 writes it for B
 *   D        bf16 [E, M, N], contiguous
 *   offsets  int32 [E+1], DEVICE memory: expert e owns tokens offsets[e] .. offsets[e+1]-1;
 *            non-decreasing multiples of 128, offsets[E] <= T (tokens past it belong to no
 *            expert).  Violations make the kernel write nothing and set FP8G_ERR_DEVICE_ASSERT.
 *   1 <= E <= 2048, M >= 0 and M % 16 == 0 (M == 0: no-op), E*M < 2^31, N % 16 == 0,
 *   T % 128 == 0.  Pointers 16-byte aligned.
 */
int fp8_grouped_gemm_wgrad(const void* A, int64_t lda, const float* sA, int64_t ld_sa, const void* B,
                           int64_t ldb, const float* sB, int64_t ld_sb, void* D, const int32_t* offsets,
                           int32_t E, int64_t M, int64_t N, int64_t T, void* stream);

/*
 * fp8g_get_status -- synchronise `stream`, then return and clear the current
 * device's status word (FP8G_OK if no kernel recorded an error since the last
 * call).  Returns FP8G_ERR_CUDA if the synchronisation itself fails.
 */
int fp8g_get_status(void* stream);

/* fp8g_status_string -- a static, human-readable name for a status code. */
const char* fp8g_status_string(int code);

/*
 * fp8g_selftest_bounded_waits -- runs, on `stream`, the bounded waits every GEMM role uses against
 * an mbarrier phase that nothing completes and a flag that nothing raises (one thread, nothing in
 * flight), each with a budget of `budget_cycles` clock cycles.  Both must run out: out[0] and out[1]
 * are set to 1 when the mbarrier and the flag wait gave up, out[2] to 1 when both raised the abort
 * flag, and the status word records FP8G_ERR_TIMEOUT (read it with fp8g_get_status).  The CUDA
 * context stays usable.  out: uint32 [3], device memory.  0 < budget_cycles <= 2^40.
 */
int fp8g_selftest_bounded_waits(int64_t budget_cycles, uint32_t* out, void* stream);

/*
 * fp8g_last_config -- the tile configuration the last GEMM call on this thread
 * launched: block N (columns per tile), pipeline stages and grid size.
 * Diagnostic only; returns FP8G_OK, or FP8G_ERR_INVALID_ARG for null pointers.
 */
int fp8g_last_config(int* block_n, int* stages, int* grid);

/*
 * fp8g_last_split -- 1 when the last GEMM call on this thread split the K blocks of its
 * last round of tiles over every SM (the stream-K tail, which uses the GEMM workspace or,
 * for fp8_gemm_nt_noalloc, the fixed scratch), else 0.  The masked form decides on the
 * device: 1 there means the launch could split.  Diagnostic only; returns FP8G_OK, or
 * FP8G_ERR_INVALID_ARG for a null pointer.
 */
int fp8g_last_split(int* split);

/*
 * fp8g_last_swap_ab -- 1 when the last GEMM call on this thread ran swapped decode tiles: a
 * block-scaled dense GEMM (fp8_gemm_nt, fp8_gemm_nt_noalloc, fp8_gemm_nt_dgrad) with M <= 64
 * computed as D^T = B A^T, the weight rows taking the MMA's 128 rows and the tokens its 64
 * columns ("DeepGEMM FP8 walk-through" sec. 4.2: small M kept efficient; sec. 3.2: work spread
 * over the SMs from the shape), else 0.  Same results as the unswapped tiles up to FP32
 * summation order.  Opt-in: FP8G_SWAP_AB=1 (and no tile width forced with FP8G_BLOCK_N); the
 * default 64-wide tiles measured faster on the decode shape.  Diagnostic only; returns FP8G_OK, or
 * FP8G_ERR_INVALID_ARG for a null pointer.
 */
int fp8g_last_swap_ab(int* swapped);

/*
 * fp8g_last_cluster_k -- the cluster size c when the last GEMM call on this thread split each
 * 256-wide tile's K blocks over a cluster of c CTAs, else 0.  A block-scaled dense GEMM
 * (fp8_gemm_nt, fp8_gemm_nt_dgrad) with few tiles: rank r of a cluster promotes K blocks
 * [r KB / c, (r+1) KB / c) and rank 0 adds the other ranks' FP32 partials before rounding once
 * ("DeepGEMM FP8 walk-through" sec. 2.3: FP32 accumulation over the whole K, one rounding on
 * write; sec. 3.2: work spread over the SMs from the shape).  Same results up to FP32 summation
 * order.  Taken by default when M > 64, K has 128 blocks or more and the 256-wide tiles fill at
 * most half the SMs (the largest c of 8, 4, 2 whose tiles fit the SMs, dividing the K blocks and
 * leaving each rank 16 or more); FP8G_CLUSTER_K=c (2 .. 8) forces c where the tiles times c fit the
 * SMs and c divides the K blocks (at least two a rank), FP8G_CLUSTER_K=0 turns it off.
 * Diagnostic only; returns FP8G_OK, or FP8G_ERR_INVALID_ARG for a null pointer.
 */
int fp8g_last_cluster_k(int* ck);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H_ */
