/*
 * qfp4.h -- C ABI of libqfp4.so: block-scaled FP4 (MXFP4 / NVFP4) quantiser,
 * scale-factor interleave and tensor-core GEMM for GB300 (sm_103a).
 *
 * Pages this library follows (cited by title and section):
 *   "Packed MXFP4 & NVFP4 GEMM + mega-MoE (SM100, true 2-CTA multicast)"
 *     (DeepGEMM pull request), "Summary" and "Key technical details": the GEMM
 *     [M,K] @ [N,K]^T -> [M,N] in BF16, both operands packed E2M1 two per
 *     byte, MXFP4 = UE8M0 scale per 32 K-elements, NVFP4 = UE4M3 scale per 16
 *     K-elements and per-tensor fp32 global scales applied as
 *     acc * gs_act * gs_weight; the MMA kinds mxf4 (block32) and mxf4nvf4
 *     (block16); per-expert global scales are listed there as missing.
 *   "fp4_quantization" (Mojo kernel module API), "Functions": dynamic
 *     BF16 -> NVFP4/MXFP4 quantisation with per-block scale factors, the
 *     re-interleave of rank-2 scale factors into the 5D TCGEN layout, and the
 *     grouped per-expert quantiser and matmul.
 *   "quadbit" README, "End-to-end serving": the decode GEMM at small M (the
 *     page fills the GPU with split-K; here the weights' CTA pairs are split
 *     over K when that pays, see qfp4_gemm_nt) and the one-launch segmented
 *     MoE kernel.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronises inside these calls (except
 *     qfp4_poll_device_status, which synchronises the given stream).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Work is enqueued asynchronously on `stream`.  Argument errors are
 *     detected on the host before anything is launched and returned as a
 *     negative status; nothing is written in that case.
 *   - Device-side failures (a bounded wait that ran out) are recorded in a
 *     device status word and reported by qfp4_poll_device_status.
 *   - Element k of a packed row lives in byte k/2: even k in bits [3:0], odd
 *     k in bits [7:4].
 *   - Row-major scale factors SF[rows, cols] hold one byte per block of g
 *     elements along K (g = 32 for MXFP4, 16 for NVFP4), cols = K / g.
 *   - The tensor-core ("MMA") scale-factor layout is the 5D layout
 *     [ceil(rows/128)][ceil(cols/4)][32][4][4]: 512-byte tiles of 128 rows x
 *     4 columns, row r and column c of a tile at byte
 *     (r % 32) * 16 + (r / 32) * 4 + c, padded with zero bytes.  Its size is
 *     qfp4_sf_mma_bytes(rows, cols).
 */
#ifndef QFP4_H
#define QFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Formats.  QFP4_NVFP4_B32 is NVFP4 with one UE4M3 scale per 32 elements
 * (plus the fp32 global scale): the format of both operands of the 2:4
 * sparse GEMM (quadbit README, "Accuracy (real models)": the deployed sparse
 * kernel is trained "per-32 matched"; the tensor core's sparse MMA applies
 * one scale per 16 stored elements, i.e. per 32 dense positions).  The
 * quantiser (qfp4_quantize, qfp4_quantize_rows) and the global scales serve
 * it like NVFP4; the dense GEMMs take QFP4_MXFP4 and QFP4_NVFP4 only. */
enum { QFP4_MXFP4 = 0, QFP4_NVFP4 = 1, QFP4_NVFP4_B32 = 2 };

/* Scale-factor layouts. */
enum { QFP4_SF_ROWMAJOR = 0, QFP4_SF_MMA = 1 };

/* Status codes. */
enum {
    QFP4_OK = 0,
    QFP4_ERR_INVALID_ARG = -1,  /* null pointer, bad format/layout, negative size */
    QFP4_ERR_UNSUPPORTED = -2,  /* shape outside what the kernels handle */
    QFP4_ERR_MISALIGNED = -3,   /* pointer not 16-byte aligned */
    QFP4_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
    QFP4_ERR_TIMEOUT = -5,      /* a device-side bounded wait ran out */
    QFP4_ERR_ARCH = -6,         /* current device is not sm_103 */
    QFP4_ERR_WORKSPACE = -7     /* workspace missing or too small */
};

/* Library version (major*10000 + minor*100 + patch). */
int qfp4_version(void);

/* Human-readable text for a status code.  Never NULL. */
const char *qfp4_status_string(int status);

/* QFP4_OK if the current CUDA device is a compute-capability 10.3 GPU
 * (GB300), QFP4_ERR_ARCH otherwise, QFP4_ERR_CUDA if no device is usable. */
int qfp4_device_check(void);

/* Synchronise `stream`, then return and clear the device status word:
 * QFP4_OK; QFP4_ERR_TIMEOUT if any kernel of this library gave up on a
 * bounded wait since the last poll (its outputs are then undefined); or
 * QFP4_ERR_INVALID_ARG if a grouped call found its device row_offsets
 * unusable (see qfp4_global_scale_grouped) and wrote nothing. */
int qfp4_poll_device_status(void *stream);

/* ---------------------------------------------------------------------- */
/* Sizes                                                                    */
/* ---------------------------------------------------------------------- */

/* Elements per scale block: 32 (MXFP4, NVFP4_B32) or 16 (NVFP4); 0 for a bad fmt. */
int qfp4_block_size(int fmt);

/* Bytes of the MMA scale-factor layout for a [rows, cols] scale matrix. */
size_t qfp4_sf_mma_bytes(int64_t rows, int64_t cols);

/* Bytes of the per-group MMA scale-factor layout used by the grouped calls:
 * every group starts on a 128-row tile, so this is the size for
 * sum_e ceil(rows_e / 128) <= ceil(total_rows / 128) + groups tiles. */
size_t qfp4_sf_mma_grouped_bytes(int64_t total_rows, int64_t groups, int64_t cols);

/* ---------------------------------------------------------------------- */
/* Global scale (NVFP4)                                                     */
/* ---------------------------------------------------------------------- */

/* gs_out[0] = amax(|X|) / (6 * 448) in fp32 (one IEEE division), where X is
 * BF16 [rows, cols] row-major.  The block whose |x| reaches amax then gets
 * the largest UE4M3 scale, 448.  DeepGEMM pull request "Summary" (per-tensor
 * fp32 global scales).  Requirements: rows, cols >= 0, X 16-byte aligned,
 * cols % 8 == 0.  An empty X (rows or cols 0; X may then be NULL) gives
 * gs = 0.
 * One launch: the CTAs reduce through one of 1024 slots in the library's
 * device memory, handed out in turn by the host and left at zero by every
 * launch.  So at most 1024 calls may be in flight at once (over all
 * streams), and a CUDA graph that captured a call reuses that slot on every
 * replay: one graph must not be replayed concurrently with itself.  The
 * grouped forms below have 64 slots. */
int qfp4_global_scale(const void *X_bf16, int64_t rows, int64_t cols, float *gs_out,
                      void *stream);

/* Per-group version: group e covers rows [row_offsets[e], row_offsets[e+1])
 * of X (row_offsets is a DEVICE int32 array of groups+1 non-decreasing
 * entries, row_offsets[0] = 0, row_offsets[groups] = total_rows).
 * gs_out[e] = amax over group e / (6 * 448).  Same requirements, and
 * 1 <= groups <= 256.
 * Every grouped call of this library checks its row_offsets on the device
 * (row_offsets[0] == 0, non-decreasing, row_offsets[groups] == the row count
 * passed on the host, and for the GEMMs no group above max_group_rows).
 * Offsets that fail make the kernels skip all work and make the next
 * qfp4_poll_device_status return QFP4_ERR_INVALID_ARG: the GEMMs and the
 * quantiser's codes are left untouched, the grouped quantiser's scale buffer
 * keeps the zeros it is cleared to, and the global scales read 0. */
int qfp4_global_scale_grouped(const void *X_bf16, int64_t total_rows, int64_t cols,
                              int64_t groups, const int32_t *row_offsets, float *gs_out,
                              void *stream);

/* The same per-group global scales with the row count taken from the device:
 * X has row_offsets[groups] rows of K BF16 elements, a value the host need not
 * know (MoE routing writes the offsets on the device).  Launches a full grid
 * of row-walking warps.  DeepGEMM pull request "Known limitations /
 * follow-ups": per-expert global scales as device tensors.  Requirements:
 * 1 <= groups <= 256, K % 8 == 0, X 16-byte aligned; the offsets are checked
 * on the device as for qfp4_global_scale_grouped. */
int qfp4_absmax_gs(int64_t groups, const int32_t *row_offsets, const void *X_bf16, int64_t K,
                   float *gs_out, void *stream);

/* Per-row global scales (two-level NVFP4; quadbit README, "Accuracy (real
 * models)": per-16 UE4M3 local scales under a per-row fp32 global scale):
 * gs_out[r] = amax(|X[r, :]|) / (6 * 448), the rule of qfp4_global_scale on
 * each row alone.  gs_out is a DEVICE fp32 [rows].  Requirements as
 * qfp4_global_scale; rows == 0 launches nothing, cols == 0 writes zeros. */
int qfp4_global_scale_rows(const void *X_bf16, int64_t rows, int64_t cols, float *gs_out,
                           void *stream);

/* ---------------------------------------------------------------------- */
/* Quantiser                                                                */
/* ---------------------------------------------------------------------- */

/* BF16 X [M, K] -> packed E2M1 Q [M, K/2] and scale bytes SF.
 * Per block of g elements along K, in IEEE fp32 with round-to-nearest-even:
 *   amax = max |x|;  t = (amax / 6) / gs;  sf = round-to-format(t)
 *   (UE8M0: nearest power of two, ties to even code, clamp 254;
 *    UE4M3: nearest, ties to even, saturate at 448);
 *   s = decode(sf) * gs;  nibble = E2M1-round(x / s) (nearest even,
 *   saturate at 6, sign kept); if s == 0 the block encodes as zeros.
 * Mojo page "fp4_quantization" (quantize_dynamic_scaled_fp4fp8); DeepGEMM
 * pull request "Summary" (formats).  The output is bit-exact to that rule.
 *   fmt        QFP4_MXFP4 (gs ignored, 1.0), QFP4_NVFP4 or QFP4_NVFP4_B32
 *              (gs required; g = 16 or 32, UE4M3 scales)
 *   gs         DEVICE pointer to one fp32 global scale (NULL allowed for MXFP4)
 *   sf_layout  QFP4_SF_ROWMAJOR: SF is [M, K/g] row-major;
 *              QFP4_SF_MMA: SF is written directly in the MMA layout
 *              (buffer of qfp4_sf_mma_bytes(M, K/g) bytes, padding zeroed).
 * Requirements: M >= 0, K % 128 == 0, X/Q 16-byte aligned, SF 4-byte aligned,
 * and (M + 128) * (K / 16) < 2^32 - 4096 (block indices and scale-byte offsets
 * are 32-bit: up to about 2^36 elements); QFP4_ERR_UNSUPPORTED otherwise. */
int qfp4_quantize(int fmt, const void *X_bf16, int64_t M, int64_t K, const float *gs,
                  void *Q_packed, void *SF, int sf_layout, void *stream);

/* Quantiser with a per-row global scale (two-level NVFP4): row m is
 * quantised exactly as qfp4_quantize quantises it alone with
 * gs = gs_rows[m] (bit-exact to that rule).  gs_rows is a DEVICE fp32 [M]
 * (required for NVFP4; MXFP4 ignores it and runs qfp4_quantize).  Other
 * arguments and requirements as qfp4_quantize. */
int qfp4_quantize_rows(int fmt, const void *X_bf16, int64_t M, int64_t K, const float *gs_rows,
                       void *Q_packed, void *SF, int sf_layout, void *stream);

/* Per-group quantiser for MoE-shaped batches (Mojo page "fp4_quantization",
 * grouped_quantize_dynamic_scaled_fp4_async): rows of group e use gs[e]; the
 * scale factors are written in the per-group MMA layout, group e starting at
 * 128-row tile sum_{e' < e} ceil(rows_e' / 128).  Q is [total_rows, K/2].
 * row_offsets as in qfp4_global_scale_grouped.  SF_mma must hold
 * qfp4_sf_mma_grouped_bytes(total_rows, groups, K/g) bytes; it is zeroed
 * by this call before the scale bytes are written.  Requirements as
 * qfp4_quantize, with 1 <= groups <= 256 and
 * (total_rows + 128 * (groups + 1)) * (K / 16) < 2^32 - 4096. */
int qfp4_quantize_grouped(int fmt, const void *X_bf16, int64_t total_rows, int64_t K,
                          int64_t groups, const int32_t *row_offsets, const float *gs,
                          void *Q_packed, void *SF_mma, void *stream);

/* Grouped quantiser with one global scale per row (two-level NVFP4 for MoE
 * batches): row m is quantised exactly as qfp4_quantize quantises it alone
 * with gs_rows[m], and the scales go to the per-group MMA layout of
 * qfp4_quantize_grouped.  gs_rows is a DEVICE fp32 [total_rows] (NVFP4;
 * MXFP4 ignores it and runs qfp4_quantize_grouped).  Other arguments and
 * requirements as qfp4_quantize_grouped. */
int qfp4_quantize_grouped_rows(int fmt, const void *X_bf16, int64_t total_rows, int64_t K,
                               int64_t groups, const int32_t *row_offsets, const float *gs_rows,
                               void *Q_packed, void *SF_mma, void *stream);

/* Residual add, RMSNorm and quantisation in one pass (quadbit README,
 * "Accuracy (real models)": the fused RMSNorm and residual-add quantisers
 * around the GEMMs, with NVFP4's per-row fp32 global scales; "The stack": the
 * fused block-glue kernels).  Per row m, in fp32:
 *   y = bf16_rne(x + r)                           (r == NULL: y = x)
 *   z = (y * (1 / sqrt(sum(y^2) / K + eps))) * gamma
 *   gs_rows[m] = amax(|z|) / (6 * 448)            (NVFP4 only)
 * and z is quantised by the rule of qfp4_quantize with gs_rows[m] (MXFP4:
 * no global scale), so Q, SF and gs_rows go straight into
 * qfp4_gemm_nt_scaled (row_scale = gs_rows).
 *   X_bf16, R_bf16  [M, K] BF16 (R may be NULL); gamma_bf16 [K] BF16
 *   Y_bf16     [M, K] BF16 output, the new residual stream (NULL: not written)
 *   gs_rows    DEVICE fp32 [M] output (NVFP4; MXFP4 ignores it)
 *   Q_packed   [M, K/2];  SF  [M, K/g] row-major or MMA layout (padding zeroed)
 * y is exact to that rule.  The sum of squares, 1/sqrt and z come from fp32
 * arithmetic whose relative error is at most ((L + 2)/2 + 4) * 2^-24, where
 * L = EPT + 10 is the longest chain of additions in the sum (EPT = 16, 32 or
 * 64 elements per thread: the smallest multiple of g with K / EPT <= 1024);
 * the codes and scale bytes are the rule's output for the kernel's z and
 * gs_rows.  Requirements: K % 128 == 0, K <= 65536, M <= 2^31 - 1, eps >= 0
 * and finite, X/R/gamma/Y/Q 16-byte aligned, SF and gs_rows 4-byte aligned. */
int qfp4_residual_rmsnorm_quantize(int fmt, const void *X_bf16, const void *R_bf16, const void *gamma_bf16,
                                   int64_t M, int64_t K, float eps, void *Y_bf16, float *gs_rows,
                                   void *Q_packed, void *SF, int sf_layout, void *stream);

/* ---------------------------------------------------------------------- */
/* Scale-factor interleave                                                  */
/* ---------------------------------------------------------------------- */

/* Permute scale bytes between the row-major [rows, cols] layout and the MMA
 * layout (Mojo page "fp4_quantization", block_scales_interleave: rank-2 scale
 * factors -> 5D TCGEN layout).
 *   layout == QFP4_SF_MMA:      SF_in row-major -> SF_out MMA layout
 *                               (qfp4_sf_mma_bytes bytes, padding zeroed)
 *   layout == QFP4_SF_ROWMAJOR: SF_in MMA layout -> SF_out row-major
 * SF_in and SF_out must not overlap.  rows, cols >= 0. */
int qfp4_sf_interleave(const void *SF_in, int64_t rows, int64_t cols, void *SF_out,
                       int layout, void *stream);

/* ---------------------------------------------------------------------- */
/* GEMM                                                                     */
/* ---------------------------------------------------------------------- */

/* Workspace bytes qfp4_gemm_nt and qfp4_gemm_nt_scaled use for this shape
 * on the current device: 0 unless M <= 128 and the decode kernel splits K
 * (quadbit README, "End-to-end serving": split-K fills the GPU at decode).
 * It splits K over S = 2, 4 or 8 CTA pairs per 256 weight rows when
 * ceil(N/256) * S pairs fit on the GPU at once and each pair then streams
 * at least 16 fewer 256-K blocks; the workspace then holds an arrival count
 * and a generation word per 128 weight rows (first 256-byte block) and the
 * fp32 partial sums, ceil(N/256) * S * 2 * 128 * ceil32(M) floats. */
size_t qfp4_gemm_workspace_bytes(int fmt, int64_t M, int64_t N, int64_t K);

/* D[M,N] (BF16, row-major) = bf16_rne(gs_a * gs_b * sum_k a[m,k] * b[n,k]),
 * a = E2M1(A) * SF_A, b = E2M1(B) * SF_B (DeepGEMM pull request "Summary":
 * [M,K] @ [N,K]^T -> [M,N], dequant acc * gs_act * gs_weight).
 *   A_packed  [M, K/2] bytes, K-major;  A_sf  MMA layout for [M, K/g]
 *   B_packed  [N, K/2] bytes, K-major;  B_sf  MMA layout for [N, K/g]
 *   gs_a, gs_b DEVICE pointers to one fp32 each (NULL = 1.0; MXFP4 ignores)
 *   workspace  DEVICE scratch, 16-byte aligned, of ws_bytes >=
 *              qfp4_gemm_workspace_bytes(...), ZERO-FILLED before its first
 *              use; every call leaves its arrival counts at zero again, so
 *              it is reused as it is (re-zero it after a reported timeout).
 *              One call at a time per workspace: calls that overlap on the
 *              GPU race on it.  NULL or a smaller one makes the decode
 *              kernel run without split-K (same result bounds, slower).
 * Tensor cores: tcgen05.mma kind::mxf4 (MXFP4) / kind::mxf4nvf4 scale_vec::4X
 * (NVFP4), fp32 accumulation in tensor memory.  Kernels: M <= 128: CTA
 * pairs with A and B swapped (256 weight rows per pair in the MMA's M slot,
 * the tokens in its N slot), each pair over all of K or, with split-K, over
 * its K range, the partials summed in a fixed order (results repeat bit for
 * bit; the split CTAs wait on each other, so the call expects the GPU's SMs
 * to be free for it at once, as other work on the stream leaves them);
 * M > 128 and N % 256 == 0: CTA pairs (cta_group::2) on 256 x 256 tiles;
 * otherwise single-CTA 128 x 128 tiles.
 * Requirements: N % 128 == 0, K % 128 == 0, all pointers 16-byte aligned.
 * Degenerate shapes: M == 0 or N == 0 returns QFP4_OK with nothing launched
 * (no pointer is read); K == 0 is an empty sum and writes D = 0.
 * Accuracy: |D - exact| <= 2^-8 |exact| + 1e-6 sum_k |a_k b_k|. */
int qfp4_gemm_nt(int fmt, int64_t M, int64_t N, int64_t K,
                 const void *A_packed, const void *A_sf,
                 const void *B_packed, const void *B_sf,
                 const float *gs_a, const float *gs_b,
                 void *D_bf16, void *workspace, size_t ws_bytes, void *stream);

/* qfp4_gemm_nt for callers that cannot allocate device memory: code that runs
 * under a fixed device-memory budget planned ahead of time, or inside a host
 * framework whose allocator must own every allocation, and so can neither
 * call cudaMalloc nor hand over a workspace.  (It has no counterpart in the
 * pages: it only changes where the decode split-K keeps its scratch.)
 * Same arguments, result and accuracy as qfp4_gemm_nt without the workspace
 * pair.  The scratch is a static device array of 8 MiB + 4 KiB inside this
 * library, which every GPU that loads the library holds until the process
 * exits: room for the partial sums of 64 CTA pairs at 128 tokens.  A shape
 * whose split-K needs more (qfp4_gemm_workspace_bytes(...) above that size)
 * is rejected with QFP4_ERR_WORKSPACE before anything is launched; shapes
 * that need no scratch run as in qfp4_gemm_nt.  The call allocates and frees
 * nothing.  Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Each call that splits K clears the array's
 * arrival counts on `stream` first.  All calls share the one array, so two
 * calls whose kernels overlap on the GPU (different streams, no ordering
 * between them) race on it: order them on one stream. */
int qfp4_gemm_nt_noalloc(int fmt, int64_t M, int64_t N, int64_t K,
                         const void *A_packed, const void *A_sf,
                         const void *B_packed, const void *B_sf,
                         const float *gs_a, const float *gs_b,
                         void *D_bf16, void *stream);

/* Two-level epilogue (quadbit README, "Accuracy (real models)": a per-row and
 * per-column fp32 global rescale in the MMA epilogue, the deploy path of
 * NVFP4 with per-row global scales):
 *   D[m,n] = bf16_rne( (acc[m,n] * (gs_a*gs_b * row_scale[m])) * col_scale[n] )
 * in fp32, with acc the same sum as in qfp4_gemm_nt (MXFP4 ignores gs_a and
 * gs_b, not the row and column scales).
 *   row_scale  DEVICE fp32 [M] or NULL (ones), e.g. the activations' per-row
 *              global scales from qfp4_global_scale_rows
 *   col_scale  DEVICE fp32 [N] or NULL (ones), e.g. the weights' per-row
 *              (output-channel) global scales
 * With both NULL the result is bit-identical to qfp4_gemm_nt.  Same kernels,
 * requirements and accuracy bound (with the scales in the exact product);
 * the scale pointers must be 4-byte aligned. */
int qfp4_gemm_nt_scaled(int fmt, int64_t M, int64_t N, int64_t K,
                        const void *A_packed, const void *A_sf,
                        const void *B_packed, const void *B_sf,
                        const float *gs_a, const float *gs_b,
                        const float *row_scale, const float *col_scale,
                        void *D_bf16, void *workspace, size_t ws_bytes, void *stream);

/* Grouped per-expert GEMM in one launch (quadbit README "End-to-end
 * serving": one-launch segmented MoE kernel; Mojo page: grouped per-expert
 * block-scaled matmul).  For every group e with rows
 * [row_offsets[e], row_offsets[e+1]):
 *   D[rows_e, :] = bf16(gs_a[e] * gs_b[e] * A[rows_e] @ B[e]^T)
 *   A_packed   [total_rows, K/2];  A_sf  per-group MMA layout (as written by
 *              qfp4_quantize_grouped)
 *   B_packed   [groups, N, K/2];   B_sf  [groups] x MMA layout for [N, K/g]
 *   gs_a, gs_b DEVICE fp32 [groups] (NULL = all 1.0)
 *   row_offsets DEVICE int32 [groups + 1], checked on the device (see
 *              qfp4_global_scale_grouped)
 *   total_rows the rows of A and D; the host needs it for the tensor maps
 *   max_group_rows  upper bound on any group's rows, or 0 for none.  It
 *              bounds the grid (groups * ceil(max_group_rows / tile rows)
 *              when that is below the bound from total_rows); a group above
 *              it is reported like any other bad offsets.
 *   workspace, ws_bytes  DEVICE scratch; the grouped kernels use none
 *              (qfp4_gemm_workspace_bytes is 0 for them), NULL is fine.
 * Requirements as qfp4_gemm_nt, with 1 <= groups <= 256. */
int qfp4_gemm_nt_grouped(int fmt, int64_t groups, const int32_t *row_offsets,
                         int64_t total_rows, int64_t max_group_rows, int64_t N, int64_t K,
                         const void *A_packed, const void *A_sf,
                         const void *B_packed, const void *B_sf,
                         const float *gs_a, const float *gs_b,
                         void *D_bf16, void *workspace, size_t ws_bytes, void *stream);

/* Grouped GEMM with the two-level epilogue of qfp4_gemm_nt_scaled:
 *   D[m,n] = bf16_rne( (acc[m,n] * (gs_a[e]*gs_b[e] * row_scale[m])) * col_scale[e*N + n] )
 * for row m of group e.  row_scale is a DEVICE fp32 [total_rows] (e.g. per-row
 * global scales of the concatenated activations) or NULL; col_scale is a
 * DEVICE fp32 [groups * N] (each expert's per-row weight scales) or NULL.
 * With both NULL the result is bit-identical to qfp4_gemm_nt_grouped.  Other
 * arguments and requirements as qfp4_gemm_nt_grouped. */
int qfp4_gemm_nt_grouped_scaled(int fmt, int64_t groups, const int32_t *row_offsets,
                                int64_t total_rows, int64_t max_group_rows, int64_t N, int64_t K,
                                const void *A_packed, const void *A_sf,
                                const void *B_packed, const void *B_sf,
                                const float *gs_a, const float *gs_b,
                                const float *row_scale, const float *col_scale,
                                void *D_bf16, void *workspace, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------- */
/* 2:4 pair-sparse GEMM                                                     */
/* ---------------------------------------------------------------------- */

/* Bytes of the metadata qfp4_sparse24_compress writes for a [rows, K] operand:
 * QFP4_SF_ROWMAJOR [rows][K/16] (two groups per byte, even group low) or
 * QFP4_SF_MMA, the tiled layout the sparse GEMM reads:
 * [ceil(rows/128)][K/512][128][32] (rows padded to 128 with valid codes). */
size_t qfp4_sparse24_meta_bytes(int64_t rows, int64_t K, int meta_layout);

/* Compress a 2:4 pair-sparse packed operand (quadbit README, "Accuracy (real
 * models)": Blackwell FP4 2:4 sparsity is pair-granular, the MMA keeps 2 of
 * every 4 FP4 pairs; "The stack": the weight packer).  W_packed [rows, K/2]
 * holds at most two non-zero bytes (pairs of E2M1 elements; a pair whose
 * elements both decode to 0, codes 0 and 8, is zero) in every group of four
 * along K.  Per group the kept pairs i0 < i1 (the non-zero ones, padded with
 * the lowest zero ones) go to W_comp [rows, K/4] in that order and the code
 * i0 | i1 << 2 to the metadata.  A group with three or four non-zero pairs
 * is not 2:4: the next qfp4_poll_device_status returns QFP4_ERR_INVALID_ARG
 * (that group's outputs are then undefined).  Requirements: K % 64 == 0
 * (K % 512 == 0 for QFP4_SF_MMA), W_packed / W_comp 16-byte aligned,
 * W_meta 4-byte aligned, of qfp4_sparse24_meta_bytes bytes. */
int qfp4_sparse24_compress(const void *W_packed, int64_t rows, int64_t K, void *W_comp, void *W_meta,
                           int meta_layout, void *stream);

/* D[M,N] (BF16) = X @ W^T with W 2:4 pair-sparse, on the tensor cores'
 * sparse MMA (tcgen05.mma.sp; quadbit README, "Headline result": the sparse
 * FP4 GEMM; "Accuracy (real models)": the two-level sparse kernel with a
 * per-row and per-column fp32 rescale in the epilogue):
 *   D[m,n] = bf16_rne( (acc[m,n] * (gs_x*gs_w * row_scale[m])) * col_scale[n] )
 * with acc = sum_k x[m,k] w[n,k] over the dense K, w the decompressed W.
 *   fmt       QFP4_NVFP4_B32 (one UE4M3 scale per 32 elements for both
 *             operands, the format the sparse MMA applies; others return
 *             QFP4_ERR_UNSUPPORTED)
 *   X_packed  [M, K/2] activations, X_sf MMA layout for [M, K/32]
 *   W_comp    [N, K/4], W_meta tiled (QFP4_SF_MMA) metadata of
 *             qfp4_sparse24_compress; W_sf MMA layout for [N, K/32] (the
 *             scales of the dense W)
 *   gs_x, gs_w DEVICE fp32 scalars (NULL = 1.0); row_scale [M], col_scale
 *             [N] DEVICE fp32 or NULL (ones)
 * Kernel: CTA pairs on 256 weight rows x 256 tokens, stages of 512 K.
 * Requirements: N % 256 == 0, K % 512 == 0, pointers 16-byte aligned (the
 * scale vectors 4-byte); M any (M == 0 or N == 0 launches nothing, K == 0
 * writes D = 0).  Accuracy as qfp4_gemm_nt, with T over the kept products. */
int qfp4_gemm_nt_sparse24(int fmt, int64_t M, int64_t N, int64_t K,
                          const void *X_packed, const void *X_sf,
                          const void *W_comp, const void *W_meta, const void *W_sf,
                          const float *gs_x, const float *gs_w,
                          const float *row_scale, const float *col_scale,
                          void *D_bf16, void *stream);

/* ---------------------------------------------------------------------- */
/* Up-projection with SwiGLU and requantisation                             */
/* ---------------------------------------------------------------------- */

/* The MoE / MLP up-projection fused with its SwiGLU and with the
 * quantisation of the result for the next GEMM (DeepGEMM pull request
 * "Summary": the L1 output is requantised with the L2 activations' global
 * scale; quadbit README "Accuracy (real models)": fused SwiGLU quantiser):
 *   G[m,j] = gs_a*gs_w * sum_k a[m,k] * w_gate[j,k]
 *   U[m,j] = gs_a*gs_w * sum_k a[m,k] * w_up[j,k]          (fp32 accumulation)
 *   H[m,j] = silu(G) * U = G / (1 + exp(-G)) * U            (fp32)
 * and H [M, I] is quantised by the rule of qfp4_quantize with the global
 * scale gs_out (NVFP4) or none (MXFP4), straight from the accumulator: no
 * BF16 output is written.
 *   A_packed  [M, K/2], A_sf MMA layout for [M, K/g] (as for qfp4_gemm_nt)
 *   W_packed  [2I, K/2]: the gate and up rows INTERLEAVED in groups of g
 *             (g = 16 NVFP4, 32 MXFP4): rows 2g b .. 2g b + g - 1 are gate
 *             rows g b .. g b + g - 1, the next g rows the up rows of the same
 *             outputs.  W_sf is the MMA layout for those [2I, K/g] rows.
 *             (Quantise gate and up with one global scale, then permute rows.)
 *   gs_a, gs_w DEVICE fp32 (NULL = 1.0; MXFP4 ignores them)
 *   gs_out    DEVICE fp32, the global scale of H (required for NVFP4; MXFP4
 *             ignores it).  It is an input, e.g. a calibrated value: an amax
 *             of H over the batch would need a pass over H first.
 *   Q_out     [M, I/2] packed codes of H, 16-byte aligned
 *   SF_out    MMA layout for [M, I/g] (qfp4_sf_mma_bytes(M, I/g) bytes,
 *             4-byte aligned); this call zeroes it first, so padding is 0.
 * Requirements: I % 128 == 0, K % 128 == 0; M == 0 or I == 0 launches
 * nothing; K == 0 gives H = 0 (all scale bytes and codes 0).  Kernel: the
 * CTA-pair GEMM on 256 x 256 tiles of [M, 2I] for every M.
 * Accuracy: each block of H is what the rule gives for some fp32 input
 * within the accumulation error of G and U propagated through silu, plus a
 * few fp32 roundings; a code can therefore differ from one computed from
 * the exact H only where that value lies within this error of a rounding
 * boundary. */
int qfp4_gemm_swiglu_quantize(int fmt, int64_t M, int64_t I, int64_t K,
                              const void *A_packed, const void *A_sf,
                              const void *W_packed, const void *W_sf,
                              const float *gs_a, const float *gs_w, const float *gs_out,
                              void *Q_out, void *SF_out, void *stream);

/* Grouped (per-expert) version for MoE batches: rows of group e (row_offsets
 * as in qfp4_gemm_nt_grouped) use expert e's interleaved weights
 * W_packed[e] ([groups, 2I, K/2], W_sf [groups] x MMA layout for [2I, K/g])
 * and gs_a[e], gs_w[e], gs_out[e] (DEVICE fp32 [groups]).  A_sf and SF_out
 * are per-group MMA layouts (as written by qfp4_quantize_grouped; SF_out
 * holds qfp4_sf_mma_grouped_bytes(total_rows, groups, I/g) bytes), so H goes
 * straight into the grouped down-projection.  1 <= groups <= 256; other
 * requirements as qfp4_gemm_swiglu_quantize. */
int qfp4_gemm_swiglu_quantize_grouped(int fmt, int64_t groups, const int32_t *row_offsets,
                                      int64_t total_rows, int64_t I, int64_t K,
                                      const void *A_packed, const void *A_sf,
                                      const void *W_packed, const void *W_sf,
                                      const float *gs_a, const float *gs_w, const float *gs_out,
                                      void *Q_out, void *SF_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QFP4_H */
