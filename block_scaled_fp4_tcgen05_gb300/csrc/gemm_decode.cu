// gemm_decode.cu -- block-scaled FP4 GEMM for decode-shaped batches (M <= 128).
//
// Pages: quadbit README, "End-to-end serving": at decode the weights are
// streamed from DRAM, and a kernel that launches too few CTAs leaves the GPU
// idle; splitting K over more CTAs with an fp32 reduction fills the machine.
// DeepGEMM pull request "Summary" for the operation itself.
//
// All M (<= 128) rows fit one MMA tile, so a CTA owns a 128-column tile of N
// and a contiguous share of K: (N / 128) tiles x S splits CTAs, with S the
// largest power of two <= 8 that keeps the grid within one wave of SMs (S = 1
// for N = 14336, where 112 CTAs already outrun HBM; S = 4 for N = 4096).
// The S CTAs of a tile form one thread-block cluster: each accumulates its
// K share in tensor memory, writes the fp32 partial tile into its own shared
// memory, and after a cluster barrier every CTA reduces 128/S rows of the
// tile by reading all S partials over distributed shared memory, in rank
// order (deterministic), scales by gs_a * gs_b and stores BF16.  Nothing goes
// through global memory but the operands and D, and no workspace is needed.
//
// Roles (192 threads): warp 0 TMA producer (A, B and scale tiles of each
// 256-K block into a 6-deep ring); warp 1 tensor-memory owner and MMA issuer
// (scale tiles copied to tensor memory with tcgen05.cp, four K=64 MMAs per
// block); warps 2..5 drain the accumulator.  All waits are bounded.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qfp4_common.cuh"
#include "qfp4_gemm_internal.cuh"
#include "sm103_ptx.cuh"

namespace qfp4 {

__device__ uint32_t g_status_gemm_decode = 0;

int read_clear_status_gemm_decode(cudaStream_t s, uint32_t *out)
{
    uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(out, g_status_gemm_decode, sizeof(uint32_t), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_status_gemm_decode, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 6;
constexpr int kBN = 128;
constexpr int kMaxSplit = 8;

template <int FMT>
struct DecCfg {
    static constexpr int G = FMT == QFP4_MXFP4 ? 32 : 16;
    static constexpr int CPS = (256 / G) / 4;           // 512-B SF tiles per 128 rows per K-block
    static constexpr int A_BYTES = 128 * 128;
    static constexpr int B_BYTES = kBN * 128;
    static constexpr int SF_BYTES = 2 * CPS * 512;      // A then B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int PART_BYTES = 128 * kBN * 4;    // fp32 partial tile (reuses the ring)
    static constexpr int OFF_BAR = kStages * STAGE_BYTES;
    static constexpr int NBAR = 2 * kStages + 1;        // full, empty, acc_full
    static constexpr int SMEM = OFF_BAR + NBAR * 8 + 32 + 1024;
    static constexpr int SF_COLS = 2 * CPS * 4;         // per stage: A then B
    static constexpr int COL_SF = kBN;
    static constexpr int TMEM_COLS = 512;
    static_assert(PART_BYTES <= OFF_BAR, "partial tile must fit in the ring");
    static_assert(COL_SF + kStages * SF_COLS <= TMEM_COLS, "tensor memory overflow");
    static_assert(SMEM <= 232448, "shared memory overflow");
};

__device__ __forceinline__ void record_timeout()
{
    atomicOr(&g_status_gemm_decode, static_cast<uint32_t>(kStatusTimeout));
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// Partial tile layout in shared memory: row r, 16-byte chunk j (columns
// 4j..4j+3) at chunk index r * 32 + (j ^ (r & 31)); the XOR spreads the rows
// a warp writes at the same chunk over all banks.
__device__ __forceinline__ uint32_t part_offset(int r, int j)
{
    return static_cast<uint32_t>((r * 32 + (j ^ (r & 31))) * 16);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p)
{
    using C = DecCfg<FMT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + kStages;
    uint64_t *acc_full = bars + 2 * kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = p.K;
    const int kc = (K / C::G) / 4;
    const int kblocks = (K + 255) / 256;
    const uint32_t S = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int32_t tile = blockIdx.x / S;
    const int per = (kblocks + static_cast<int>(S) - 1) / static_cast<int>(S);
    const int kb0 = min(kblocks, static_cast<int>(rank) * per);
    const int kb1 = min(kblocks, kb0 + per);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(acc_full), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t s = 0, phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&empty[s]), phase ^ 1)) { ok = false; break; }
                const int chunks = min(C::CPS, kc - kb * C::CPS);
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES + 2 * chunks * 512);
                const uint32_t dst = smem_u32(smem + s * C::STAGE_BYTES);
                tma_load_2d(dst, &tmA, fb, kb * 128, 0);
                tma_load_2d(dst + C::A_BYTES, &tmB, fb, kb * 128, tile * kBN);
                const size_t koff = static_cast<size_t>(kb) * C::CPS * 512;
                bulk_load(dst + C::A_BYTES + C::B_BYTES, p.A_sf + koff, chunks * 512, fb);
                bulk_load(dst + C::A_BYTES + C::B_BYTES + C::CPS * 512,
                          p.B_sf + static_cast<size_t>(tile) * kc * 512 + koff, chunks * 512, fb);
                if (++s == kStages) { s = 0; phase ^= 1; }
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t s = 0, phase = 0;
            bool ok = true;
            bool first = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&full[s]), phase)) { ok = false; break; }
                tc_fence_after();
                const int chunks = min(C::CPS, kc - kb * C::CPS);
                const uint32_t sf_t = tmem_base + C::COL_SF + s * C::SF_COLS;
                const uint32_t stage = smem_u32(smem + s * C::STAGE_BYTES);
                const uint32_t sf_s = stage + C::A_BYTES + C::B_BYTES;
                for (int c = 0; c < chunks; ++c) {
                    tc_cp_32x128b_warpx4(sf_t + c * 4, smem_desc(sf_s + c * 512, 128, 128, kSwizzleNone));
                    tc_cp_32x128b_warpx4(sf_t + C::CPS * 4 + c * 4,
                                         smem_desc(sf_s + (C::CPS + c) * 512, 128, 128, kSwizzleNone));
                }
                const int ksteps = min(4, (K - kb * 256) / 64);
                const uint64_t ad0 = smem_desc(stage, 16, 1024, kSwizzle128B);
                const uint64_t bd0 = smem_desc(stage + C::A_BYTES, 16, 1024, kSwizzle128B);
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t accum = first ? 0u : 1u;
                    first = false;
                    if (FMT == QFP4_NVFP4) {
                        constexpr uint32_t id = idesc_block_scaled(128, kBN, false, 0, 0);
                        tc_mma_nvf4(tmem_base, ad0 + 2 * kk, bd0 + 2 * kk, id, sf_t + kk * 4,
                                    sf_t + C::CPS * 4 + kk * 4, accum);
                    } else {
                        constexpr uint32_t id0 = idesc_block_scaled(128, kBN, true, 0, 0);
                        constexpr uint32_t id1 = idesc_block_scaled(128, kBN, true, 2, 2);
                        tc_mma_mxf4(tmem_base, ad0 + 2 * kk, bd0 + 2 * kk, (kk & 1) ? id1 : id0,
                                    sf_t + (kk >> 1) * 4, sf_t + C::CPS * 4 + (kk >> 1) * 4, accum);
                    }
                }
                tc_commit(smem_u32(&empty[s]));
                if (++s == kStages) { s = 0; phase ^= 1; }
            }
            // an empty K share issues no MMA; the commit still arrives
            if (ok) tc_commit(smem_u32(acc_full));
            else { record_timeout(); *abort_flag = 1; }
        }
    } else {
        // ------------------------------------------------ accumulator drain (warps 2..5)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int got = __shfl_sync(0xffffffffu, lane == 0 ? (mbar_wait(smem_u32(acc_full), 0) ? 1 : 0) : 0, 0);
        if (got) {
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(taddr + j * 32, v[j]);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_regs_after_wait(v[j]);
            if (kb1 <= kb0) {
                // empty K share (more splits than K-blocks): contributes zeros
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[j][i] = 0u;
            }
            if (S == 1) {
                float gs = 1.0f;
                if (FMT == QFP4_NVFP4) gs = (p.gs_a ? *p.gs_a : 1.0f) * (p.gs_b ? *p.gs_b : 1.0f);
                if (row < p.M) {
                    __nv_bfloat16 *drow = p.D + static_cast<size_t>(row) * p.N + tile * kBN;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t packed[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(v[j][2 * i]) * gs,
                                                                      __uint_as_float(v[j][2 * i + 1]) * gs);
                            packed[i] = *reinterpret_cast<uint32_t *>(&pr);
                        }
                        st_global_v8(drow + j * 32, *reinterpret_cast<const uint32_t(*)[8]>(&packed[0]));
                        st_global_v8(drow + j * 32 + 16, *reinterpret_cast<const uint32_t(*)[8]>(&packed[8]));
                    }
                }
            } else {
                // the ring is idle now (every load was consumed): keep the
                // fp32 partial tile in shared memory for the cluster reduction
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(smem + part_offset(row, j * 8 + c)) =
                            make_uint4(v[j][4 * c], v[j][4 * c + 1], v[j][4 * c + 2], v[j][4 * c + 3]);
            }
        } else if (lane == 0) {
            record_timeout();
            *abort_flag = 1;
        }
    }

    // ---- all roles done.  Reconverge each warp first: lanes that skipped a
    // single-lane role must not reach the block barrier ahead of their warp's
    // working lane.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) { }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (S > 1) {
        // every CTA of the cluster holds its partial tile in shared memory
        cluster_sync_all();
        float gs = 1.0f;
        if (FMT == QFP4_NVFP4) gs = (p.gs_a ? *p.gs_a : 1.0f) * (p.gs_b ? *p.gs_b : 1.0f);
        const int rows = 128 / static_cast<int>(S);
        const int r0 = static_cast<int>(rank) * rows;
        const uint32_t base = smem_u32(smem);
        // one 16-byte chunk (4 columns) of one row per thread and step; the
        // partials are added in cluster-rank order whichever CTA reads them
        for (int idx = threadIdx.x; idx < rows * 32; idx += kThreads) {
            const int r = r0 + idx / 32, j = idx % 32;
            const uint32_t off = part_offset(r, j);
            float4 a = ld_dsmem_v4(mapa_shared(base + off, 0));
            for (uint32_t q = 1; q < S; ++q) {
                const float4 b = ld_dsmem_v4(mapa_shared(base + off, q));
                a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
            }
            if (r < p.M) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * gs, a.y * gs);
                __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * gs, a.w * gs);
                uint2 w;
                w.x = *reinterpret_cast<uint32_t *>(&lo);
                w.y = *reinterpret_cast<uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(p.D + static_cast<size_t>(r) * p.N + tile * kBN + j * 4) = w;
            }
        }
        // keep this CTA's shared memory alive until every peer has read it
        cluster_sync_all();
    }
}

template <int FMT>
int launch_decode(const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &g, int tiles, int split,
                  cudaStream_t s)
{
    using C = DecCfg<FMT>;
    auto kern = gemm_decode_kernel<FMT>;
    static int configured_device = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QFP4_ERR_CUDA;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return QFP4_ERR_CUDA;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * split));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, ma, mb, g));
}

}  // namespace

// K splits per 128-column tile: the largest power of two <= 8 (and <= the
// number of 256-K blocks) for which the grid still fits one wave of SMs.
int decode_split(int64_t N, int64_t K)
{
    const int64_t tiles = N / kBN, kblocks = (K + 255) / 256;
    int sms = sm_count();
    if (sms <= 0) sms = 148;
    int split = 1;
    while (split * 2 <= kMaxSplit && split * 2 <= kblocks && tiles * split * 2 <= sms) split *= 2;
    return split;
}

int launch_gemm_decode(int fmt, const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &g,
                       cudaStream_t s)
{
    const int tiles = g.N / kBN;
    const int split = decode_split(g.N, g.K);
    return fmt == QFP4_NVFP4 ? launch_decode<QFP4_NVFP4>(ma, mb, g, tiles, split, s)
                             : launch_decode<QFP4_MXFP4>(ma, mb, g, tiles, split, s);
}

}  // namespace qfp4
