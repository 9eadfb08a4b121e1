// qfp4_gemm_internal.cuh -- what the GEMM translation units share (not ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace qfp4 {

// Kernel parameters common to the GEMM kernels.
struct GemmParams {
    const uint8_t *A_sf;        // MMA-layout scale bytes of A (per-group layout when grouped)
    const uint8_t *B_sf;        // MMA-layout scale bytes of B ([groups] x layout when grouped)
    const float *gs_a;          // NVFP4 global scales (device; [groups] when grouped) or NULL
    const float *gs_b;
    __nv_bfloat16 *D;           // [M, N] row-major
    int32_t M, N, K;
    int32_t groups;             // grouped launches only
    const int32_t *row_offsets; // grouped launches only (device, groups + 1)
    // two-level epilogue (dense launches only): D[m,n] =
    // bf16((acc * (gs_a*gs_b * row_scale[m])) * col_scale[n]); NULL = ones
    const float *row_scale;     // [M] or NULL
    const float *col_scale;     // [N] or NULL
    // SwiGLU + requantisation epilogue (launch_gemm_pair_swiglu): the B rows
    // are gate and up rows interleaved in groups of g (block size), N = 2 I;
    // H = silu(gate) * up is quantised with gs_out into Q_out [M, I/2] and
    // SF_out (MMA layout for [M, I/g]; per-group layout when grouped)
    const float *gs_out;        // NVFP4: [1], or [groups] when grouped
    uint8_t *Q_out;
    uint8_t *SF_out;
    int32_t I;                  // columns of H
    int32_t kc_out;             // 512-byte SF atoms per 128 rows of H: I / (4 g)
    // grouped launches: upper bound on any group's rows (0 = no bound); the
    // kernels check the offsets against it and against M (= total rows)
    int32_t max_group_rows;
    // decode split-K (launch_gemm_decode with splits > 1): K is cut into
    // `splits` ranges, one per CTA pair of a weight tile; the fp32 partial
    // sums go to ws_partial and ws_count holds an arrival count (zero
    // between calls) and a generation word per (weight tile pair, CTA rank)
    int32_t splits;
    uint32_t *ws_count;
    float *ws_partial;
};

// 2D byte matrix [rows, inner] tensor map with 128-byte swizzle and a box of
// box_inner bytes x box_rows rows (zero fill out of bounds).
int make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
             uint32_t box_rows);

// Packed FP4 matrix [rows, K/2 bytes] viewed as {128 bytes, rows, K/256 blocks}
// (strides K/2 and 128 bytes), 128-byte swizzle, box {128, 128, 2}: one
// request brings two consecutive 256-K blocks of 128 rows, laid out as two
// 16 KB swizzled tiles one after the other.  K % 512 == 0.
int make_map_kpairs(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows);

// CTA-pair (cta_group::2) GEMM over 256 x 256 tiles; N % 256 == 0.  ma and mb
// have 128-row boxes (2-D, 128 bytes of K; or, when gemm_pair_double_stages
// says so, 3-D {128 bytes, rows, 256-K blocks} boxes of two K-blocks, see
// make_map_kpairs); md is D (BF16) with 32-row x 16-column boxes.
bool gemm_pair_double_stages(int fmt, bool grouped, int64_t K);
int launch_gemm_pair(int fmt, bool grouped, const CUtensorMap &ma, const CUtensorMap &mb,
                     const CUtensorMap &md, const GemmParams &prm, int64_t pair_tiles, cudaStream_t s);

// The same CTA-pair GEMM with the SwiGLU + requantisation epilogue instead
// of a D store: ma and mb as for launch_gemm_pair (2-D, 128-row boxes), the
// output described by prm.Q_out, prm.SF_out, prm.gs_out, prm.I, prm.kc_out.
int launch_gemm_pair_swiglu(int fmt, bool grouped, const CUtensorMap &ma, const CUtensorMap &mb,
                            const GemmParams &prm, int64_t pair_tiles, cudaStream_t s);

int read_clear_status_gemm_pair(cudaStream_t s, uint32_t *out);

// Decode GEMM for M <= 128 (N % 128 == 0), swap AB on CTA pairs: the
// weights (B, map mw with 128-row boxes) fill the MMA's M slot, the tokens
// (A, map mt with 64-row boxes) its N slot; D is written through md (BF16,
// 128 x 128 boxes, no swizzle), or directly from registers with split-K.
// g.splits > 1 selects split-K (g.ws_count and g.ws_partial set, sized by
// decode_workspace_bytes).
int launch_gemm_decode(int fmt, const CUtensorMap &mw, const CUtensorMap &mt, const CUtensorMap &md,
                       const GemmParams &g, cudaStream_t s);
// Split count the decode kernel uses for this shape on the current device
// (1, 2, 4 or 8; 1 = no split-K and no workspace), and the workspace bytes
// it then needs: an arrival count and a generation word (32-bit) per (pair
// tile, CTA) in the first 256-byte aligned block, then the fp32 partials [pairs][splits][2][ceil32(M)][128].
int decode_splits(int64_t M, int64_t N, int64_t K);
size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits);
size_t decode_counter_bytes(int64_t N);
// 2D BF16 matrix [rows, cols] (row stride cols * 2 bytes), box of
// box_cols x box_rows elements, no swizzle: the TMA store map of D.
int make_map_bf16(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                  uint32_t box_rows);
int read_clear_status_gemm_decode(cudaStream_t s, uint32_t *out);

}  // namespace qfp4
