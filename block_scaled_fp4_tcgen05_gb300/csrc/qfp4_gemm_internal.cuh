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
};

// 2D byte matrix [rows, inner] tensor map with 128-byte swizzle and a box of
// box_inner bytes x box_rows rows (zero fill out of bounds).
int make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
             uint32_t box_rows);

// CTA-pair (cta_group::2) GEMM over 256 x 256 tiles; N % 256 == 0.
int launch_gemm_pair(int fmt, bool grouped, const CUtensorMap &ma, const CUtensorMap &mb,
                     const GemmParams &prm, int64_t pair_tiles, cudaStream_t s);

int read_clear_status_gemm_pair(cudaStream_t s, uint32_t *out);

// Decode GEMM for M <= 128 (N % 128 == 0): one CTA per (128-column tile, K
// share), K shares of a tile reduced over a thread-block cluster.
int decode_split(int64_t N, int64_t K);
int launch_gemm_decode(int fmt, const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &g,
                       cudaStream_t s);
int read_clear_status_gemm_decode(cudaStream_t s, uint32_t *out);

}  // namespace qfp4
