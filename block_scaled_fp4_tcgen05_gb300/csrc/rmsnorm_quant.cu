// rmsnorm_quant.cu -- residual add + RMSNorm + BF16 -> NVFP4 / MXFP4
// quantisation in one pass over the activations (HBM-bound, no tensor cores).
//
// Pages: quadbit README, "Accuracy (real models)" (fused RMSNorm, residual-add
// and SwiGLU quantisers around the GEMMs; per-row fp32 global scales under
// the per-16 UE4M3 scales for NVFP4) and "The stack" (the fused block-glue
// kernels).  Per row m, in fp32:
//   y = bf16(x + r)                       the new residual stream (r optional)
//   z = (y * 1/sqrt(mean(y^2) + eps)) * gamma
//   gs[m] = amax(|z|) / (6 * 448)         NVFP4: the row's global scale
// and z is quantised by the rule of qfp4_quantize with gs[m] (MXFP4: none).
//
// One CTA per row; thread t owns elements [t*EPT, (t+1)*EPT), EPT a multiple
// of the block size g, so every scale block lives in one thread's registers:
// the row is read once, y is written once, and only two CTA-wide reductions
// (the sum of squares, then the row's amax of z) stand between the loads and
// the codes.  gamma [K] is read through L1 (every row reuses it).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qfp4_common.cuh"
#include "qfp4_fp4_codes.cuh"

namespace qfp4 {

namespace {

constexpr int kMaxThreads = 1024;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// x + r in fp32, rounded to bf16 (nearest even), for both halves of a word
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t x, uint32_t r)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(__fadd_rn(bf16_lo(x), bf16_lo(r)), __fadd_rn(bf16_hi(x), bf16_hi(r)));
    return *reinterpret_cast<uint32_t *>(&v);
}

// Sum over the CTA: a shuffle tree in every warp, then one over the warps'
// partials in warp 0 (padded with zeros); every thread gets the result.
// Along any path a value meets at most 10 additions here.
__device__ __forceinline__ float cta_sum(float v, float *sred)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sred[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < nw ? sred[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) sred[32] = v;
    }
    __syncthreads();
    return sred[32];
}

__device__ __forceinline__ float cta_max(float v, float *sred)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sred[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < nw ? sred[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) sred[32] = v;
    }
    __syncthreads();
    return sred[32];
}

template <int FMT, int EPT>
__global__ void __launch_bounds__(kMaxThreads)
rmsnorm_quant_kernel(const uint4 *__restrict__ X, const uint4 *__restrict__ R, const uint4 *__restrict__ gamma,
                     int64_t M, int32_t K, float eps, uint4 *__restrict__ Y, float *__restrict__ gs_rows,
                     uint8_t *__restrict__ Q, uint8_t *__restrict__ SF, int sf_layout)
{
    constexpr int G = FMT == QFP4_MXFP4 ? 32 : 16;
    constexpr int BPT = EPT / G;                 // scale blocks per thread: 1, 2 or 4
    constexpr int V = EPT / 8;                   // 16-byte vectors (8 bf16) per thread
    static_assert(EPT % G == 0 && BPT <= 4, "a thread owns whole scale blocks");
    __shared__ float s_sum[33], s_max[33];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t m = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31;
    const bool active = t * EPT < K;             // threads past the row's end only join the reductions
    const uint32_t kg = static_cast<uint32_t>(K / G), kc = kg / 4;
    if (m >= M) {
        // MMA layout: rows [M, ceil128(M)) are padding and read as zero scales
        for (uint32_t w = t; w < kc; w += blockDim.x)
            *reinterpret_cast<uint32_t *>(SF + sf_mma_offset(static_cast<uint32_t>(m / 128),
                                                             static_cast<uint32_t>(m % 128), 4 * w, kc)) = 0u;
        return;
    }
    const size_t row_vec = static_cast<size_t>(m) * (K / 8) + static_cast<size_t>(t) * V;
    uint32_t y[EPT / 2];                          // bf16 pairs
    float ss = 0.0f;
    if (active) {
        uint4 xv[V], rv[V];
#pragma unroll
        for (int v = 0; v < V; ++v) xv[v] = ld_stream(X + row_vec + v);
        if (R) {
#pragma unroll
            for (int v = 0; v < V; ++v) rv[v] = ld_stream(R + row_vec + v);
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const uint32_t xw[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
            const uint32_t rw[4] = {R ? rv[v].x : 0u, R ? rv[v].y : 0u, R ? rv[v].z : 0u, R ? rv[v].w : 0u};
#pragma unroll
            for (int i = 0; i < 4; ++i) y[4 * v + i] = R ? add_bf16x2(xw[i], rw[i]) : xw[i];
        }
        if (Y) {
#pragma unroll
            for (int v = 0; v < V; ++v) Y[row_vec + v] = make_uint4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
        }
        // y is bf16, so y*y is exact in fp32: each step rounds the sum once
#pragma unroll
        for (int i = 0; i < EPT / 2; ++i) {
            ss = __fmaf_rn(bf16_lo(y[i]), bf16_lo(y[i]), ss);
            ss = __fmaf_rn(bf16_hi(y[i]), bf16_hi(y[i]), ss);
        }
    }
    ss = cta_sum(ss, s_sum);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps)));
    float z[EPT];
    float amax = 0.0f;
    if (active) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const uint4 gv = __ldg(gamma + static_cast<size_t>(t) * V + v);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                z[8 * v + 2 * i] = __fmul_rn(__fmul_rn(bf16_lo(y[4 * v + i]), inv), bf16_lo(gw[i]));
                z[8 * v + 2 * i + 1] = __fmul_rn(__fmul_rn(bf16_hi(y[4 * v + i]), inv), bf16_hi(gw[i]));
            }
        }
#pragma unroll
        for (int i = 0; i < EPT; ++i) amax = fmaxf(amax, fabsf(z[i]));
    }
    float gs = 1.0f;
    if (FMT == QFP4_NVFP4) {
        gs = __fdiv_rn(cta_max(amax, s_max), 2688.0f);
        if (t == 0) gs_rows[m] = gs;
    }
    const float inv_gs = __frcp_rn(gs);
    uint32_t codes = 0;                          // this thread's BPT scale bytes, block b in byte b
    if (active) {
        uint32_t packed[EPT / 8];
#pragma unroll
        for (int b = 0; b < BPT; ++b) {
            float bmax = 0.0f;
#pragma unroll
            for (int i = 0; i < G; ++i) bmax = fmaxf(bmax, fabsf(z[b * G + i]));
            const BlockScale bs = block_scale<FMT>(bmax, gs, inv_gs);
            codes |= bs.code << (8 * b);
#pragma unroll
            for (int j = 0; j < G / 8; ++j) packed[b * (G / 8) + j] = encode8_f32<FMT>(&z[b * G + 8 * j], bs);
        }
        uint8_t *qrow = Q + static_cast<size_t>(m) * (K / 2) + static_cast<size_t>(t) * (EPT / 2);
#pragma unroll
        for (int j = 0; j < EPT / 32; ++j)
            reinterpret_cast<uint4 *>(qrow)[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                                                            packed[4 * j + 3]);
        if (EPT == 16) *reinterpret_cast<uint2 *>(qrow) = make_uint2(packed[0], packed[1]);
    }
    // four consecutive scale bytes make one 32-bit word of either layout:
    // gather them from the 4 / BPT neighbouring lanes that own them
    uint32_t word = codes;
    if (BPT == 1) {
        word |= __shfl_down_sync(0xffffffffu, codes, 1) << 8;
        word |= __shfl_down_sync(0xffffffffu, codes, 2) << 16;
        word |= __shfl_down_sync(0xffffffffu, codes, 3) << 24;
    } else if (BPT == 2) {
        word |= __shfl_down_sync(0xffffffffu, codes, 1) << 16;
    }
    if (active && (lane % (4 / BPT)) == 0) {
        const uint32_t c0 = static_cast<uint32_t>(t) * BPT;          // first scale column of the word
        const size_t off = sf_layout == QFP4_SF_MMA
                               ? sf_mma_offset(static_cast<uint32_t>(m / 128), static_cast<uint32_t>(m % 128), c0, kc)
                               : static_cast<size_t>(m) * kg + c0;
        *reinterpret_cast<uint32_t *>(SF + off) = word;
    }
}

template <int FMT, int EPT>
cudaError_t launch(const void *X, const void *R, const void *gamma, int64_t M, int64_t K, float eps, void *Y,
                   float *gs_rows, void *Q, void *SF, int sf_layout, cudaStream_t s)
{
    const int threads = static_cast<int>(((K / EPT) + 31) / 32 * 32);
    const int64_t rows = sf_layout == QFP4_SF_MMA ? (M + 127) / 128 * 128 : M;
    return launch_pdl(rmsnorm_quant_kernel<FMT, EPT>, dim3(static_cast<unsigned>(rows)), dim3(threads), 0, s,
                      static_cast<const uint4 *>(X), static_cast<const uint4 *>(R),
                      static_cast<const uint4 *>(gamma), M, static_cast<int32_t>(K), eps, static_cast<uint4 *>(Y),
                      gs_rows, static_cast<uint8_t *>(Q), static_cast<uint8_t *>(SF), sf_layout);
}

}  // namespace
}  // namespace qfp4

using namespace qfp4;

extern "C" int qfp4_residual_rmsnorm_quantize(int fmt, const void *X_bf16, const void *R_bf16,
                                              const void *gamma_bf16, int64_t M, int64_t K, float eps,
                                              void *Y_bf16, float *gs_rows, void *Q_packed, void *SF,
                                              int sf_layout, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (sf_layout != QFP4_SF_ROWMAJOR && sf_layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || K < 0 || !(eps >= 0.0f) || !(eps < 3.0e38f)) return QFP4_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > 64 * kMaxThreads || M > INT32_MAX) return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return QFP4_OK;
    if (!X_bf16 || !gamma_bf16 || !Q_packed || !SF || (fmt == QFP4_NVFP4 && !gs_rows)) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || (R_bf16 && !aligned16(R_bf16)) || !aligned16(gamma_bf16) ||
        (Y_bf16 && !aligned16(Y_bf16)) || !aligned16(Q_packed) || !aligned4(SF) || (gs_rows && !aligned4(gs_rows)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int g = block_elems(fmt);
    // elements per thread: the smallest multiple of g (at most 4 g) that keeps
    // the CTA within 1024 threads
    int ept = g;
    while (K / ept > kMaxThreads) ept *= 2;
    cudaError_t e;
    if (fmt == QFP4_NVFP4)
        e = ept == 16 ? launch<QFP4_NVFP4, 16>(X_bf16, R_bf16, gamma_bf16, M, K, eps, Y_bf16, gs_rows, Q_packed, SF,
                                               sf_layout, s)
          : ept == 32 ? launch<QFP4_NVFP4, 32>(X_bf16, R_bf16, gamma_bf16, M, K, eps, Y_bf16, gs_rows, Q_packed, SF,
                                               sf_layout, s)
                      : launch<QFP4_NVFP4, 64>(X_bf16, R_bf16, gamma_bf16, M, K, eps, Y_bf16, gs_rows, Q_packed, SF,
                                               sf_layout, s);
    else
        e = ept == 32 ? launch<QFP4_MXFP4, 32>(X_bf16, R_bf16, gamma_bf16, M, K, eps, Y_bf16, nullptr, Q_packed, SF,
                                               sf_layout, s)
                      : launch<QFP4_MXFP4, 64>(X_bf16, R_bf16, gamma_bf16, M, K, eps, Y_bf16, nullptr, Q_packed, SF,
                                               sf_layout, s);
    return launch_status(e);
}
