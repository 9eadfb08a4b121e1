// gemm_sparse.cu -- 2:4 pair-sparse FP4 GEMM on CTA pairs (tcgen05.mma.sp,
// cta_group::2) and the weight compressor that feeds it.
//
// Pages: quadbit README, "Accuracy (real models)": Blackwell FP4 2:4 sparsity
// is pair-granular (the MMA keeps 2 of every 4 FP4 pairs along K), the
// deployed sparse kernel is two-level (per-row and per-column fp32 rescale in
// the epilogue) and trained "per-32 matched"; "Headline result": the sparse
// GEMM at the Llama-3-8B shapes and square 8192; "The stack": the weight
// packer and cuda/matmul_sp_* kernels.
//
// Operands (format QFP4_NVFP4_B32: E2M1, one UE4M3 scale per 32 elements,
// fp32 global scales):
//   W  the weights [N, K], 2:4 pair-sparse: per group of four bytes along K
//      two are kept; compressed to Wc [N, K/4] with 4-bit metadata per group
//      (kept pair indices i0 < i1 as i0 | i1 << 2).  The tensor core takes the
//      sparse operand in its A (M) slot, so W is A and D^T = W X^T is formed.
//   X  the activations [M, K/2] packed, dense (the MMA's B slot).
// A CTA pair computes 256 weight rows x 256 tokens; each CTA holds its 128
// weight rows and 128 of the tokens.  Per stage (512 dense K, four
// M=256 N=256 K=128 sparse MMAs) each CTA receives 16 KB of compressed
// weights, 32 KB of tokens, 4 KB of metadata and 6 KB of scale bytes.
// Roles (20 warps): warps 0 and 3 weight and token TMA producers; warp 2
// the side-data producer (metadata and scales, bulk copies into a ring of
// their own); warp 1 tensor-memory owner and, in the leader, the MMA issuer;
// warps 4..11, two sets of four taking alternate stages, move metadata and
// scales into the tensor-memory slot of the stage with tcgen05.st; warps
// 12..19 the epilogue: drain D^T, scale, round to BF16, transpose through
// staging boxes and store D with TMA.
//
// Tensor-memory placement (pinned on GB300 by one-hot probes of the
// instruction): the metadata of weight row r sits in lane r, eight group
// nibbles per 32-bit column in group order (two columns per K=128 MMA); the
// scales are laid out as for the dense kernels (A: lane r's word in every
// column of its 4-column atom; B: all 256 token rows, lane n % 32 of column
// n / 32), and each of a row's four scale bytes covers 32 dense K positions.
// Every wait is bounded and reports QFP4_ERR_TIMEOUT.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qfp4_common.cuh"
#include "qfp4_gemm_internal.cuh"
#include "sm103_ptx.cuh"

namespace qfp4 {

__device__ uint32_t g_status_gemm_sparse = 0;

int read_clear_status_gemm_sparse(cudaStream_t s, uint32_t *out)
{
    uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(out, g_status_gemm_sparse, sizeof(uint32_t), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_status_gemm_sparse, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

namespace {

constexpr int kThreads = 640;          // 20 warps
constexpr int kStageK = 512;           // dense K per stage

struct SpCfg {
    static constexpr int W_BYTES = 128 * 128;          // this CTA's 128 weight rows, 512 K compressed
    static constexpr int X_BYTES = 2 * 128 * 128;      // this CTA's 128 tokens, 512 K (two 128-byte tiles)
    static constexpr int AB_BYTES = W_BYTES + X_BYTES;
    static constexpr int AB_STAGES = 3;
    static constexpr int META_BYTES = 128 * 32;        // 64 groups x 4 bits per weight row
    static constexpr int SFW_BYTES = 4 * 512;          // 4 atoms: 128 rows x 16 scales
    static constexpr int SFX_BYTES = 8 * 512;          // 4 atoms for each of the pair's two token tiles
    static constexpr int SIDE_BYTES = META_BYTES + SFW_BYTES + SFX_BYTES;
    static constexpr int SIDE_STAGES = 4;
    static constexpr int D_BOX = 32 * 32 * 2;          // 32 tokens x 32 weight columns, BF16
    static constexpr int D_BUFS = 2;
    static constexpr int OFF_SIDE = AB_STAGES * AB_BYTES;
    static constexpr int OFF_D = OFF_SIDE + SIDE_STAGES * SIDE_BYTES;
    static constexpr int OFF_BAR = OFF_D + 8 * D_BUFS * D_BOX;
    // full/empty[AB], side_full/side_empty[SIDE], acc_full, acc_empty
    static constexpr int NBAR = 2 * AB_STAGES + 2 * SIDE_STAGES + 2;
    static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
    // tensor memory: the accumulator (256 columns), then one slot per
    // operand stage: 16 columns of weight scales, 32 of token scales and
    // 8 of metadata
    static constexpr int COL_SLOT0 = 256;
    static constexpr int SFW_COLS = 16, SFX_COLS = 32, META_COLS = 8;
    static constexpr int SLOT_COLS = SFW_COLS + SFX_COLS + META_COLS;
    static_assert(COL_SLOT0 + AB_STAGES * SLOT_COLS <= 512, "tensor memory overflow");
    static_assert(SMEM <= 232448, "shared memory overflow");
    static_assert(SIDE_STAGES % 2 == 0, "side warps alternate stages");
};

__device__ __forceinline__ void record_timeout()
{
    atomicOr(&g_status_gemm_sparse, static_cast<uint32_t>(kStatusTimeout));
}

__device__ __forceinline__ void mma_sparse_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t meta_tmem, uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred P;\nsetp.ne.b32 P, %7, 0;\n"
        "tcgen05.mma.sp.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, [%3], %4, [%5], [%6], P;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&pr);
}

struct SpParams {
    const uint8_t *X_sf;        // MMA layout for [M, K/32]
    const uint8_t *W_sf;        // MMA layout for [N, K/32]
    const uint8_t *W_meta;      // tiled: [N/128][K/512][128][32 bytes]
    const float *gs_x, *gs_w;   // device scalars or NULL (1.0)
    const float *row_scale;     // [M] (tokens) or NULL
    const float *col_scale;     // [N] (weight rows) or NULL
    int32_t M, N, K;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_sparse_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmD, const SpParams p)
{
    using C = SpCfg;
    constexpr int SAB = C::AB_STAGES, SSD = C::SIDE_STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars;                      // leader: operand bytes of both CTAs + 8 side warps
    uint64_t *empty = full + SAB;               // stage and its tensor-memory slot free (MMA commit)
    uint64_t *side_full = empty + SAB;          // local: metadata and scale bytes landed
    uint64_t *side_empty = side_full + SSD;     // local: side warps done with the slot
    uint64_t *acc_full = side_empty + SSD;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int K = p.K;
    const int nstages = K / kStageK;
    const int kc = (K / 32) / 4;                   // 512-byte scale atoms per 128 rows
    const int wtiles = p.N / 256;
    const int ttiles = (p.M + 255) / 256;
    const int32_t total_tiles = wtiles * ttiles;
    const int32_t pair_id = blockIdx.x >> 1;
    const int32_t npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SAB; ++s) {
            mbar_init(smem_u32(&full[s]), 1 + 8);      // weight producer (with the bytes) + 4 side warps x 2 CTAs
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < SSD; ++s) {
            mbar_init(smem_u32(&side_full[s]), 1);
            mbar_init(smem_u32(&side_empty[s]), 4);
        }
        mbar_init(smem_u32(acc_full), 1);
        mbar_init(smem_u32(acc_empty), 2);             // one release per CTA
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmD);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    // tile t -> (token tile pair tt, weight tile pair wt): groups of 8 token
    // tiles sweep the weight tiles together so that a wave shares them in L2
    auto tile_of = [&](int32_t t, int32_t &tt, int32_t &wt) {
        constexpr int32_t GM = 8;
        const int32_t per_group = GM * wtiles;
        const int32_t grp = t / per_group;
        const int32_t first = grp * GM;
        const int32_t rows_here = min(GM, ttiles - first);
        const int32_t idx = t % per_group;
        tt = first + idx % rows_here;
        wt = idx / rows_here;
    };

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------ weight (warp 0) / token (warp 3) TMA producers
        if (lane == 0) {
            const bool is_w = warp == 0;
            const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), 0);
            uint32_t j = 0;
            bool ok = true;
            for (int32_t t = pair_id; t < total_tiles && ok; t += npairs) {
                int32_t tt, wt;
                tile_of(t, tt, wt);
                const int32_t wrow = wt * 256 + 128 * static_cast<int32_t>(rank);
                const int32_t trow = tt * 256 + 128 * static_cast<int32_t>(rank);
                for (int st = 0; st < nstages; ++st, ++j) {
                    const uint32_t s = j % SAB;
                    if (!mbar_wait(smem_u32(&empty[s]), ((j / SAB) & 1) ^ 1)) { ok = false; break; }
                    const uint32_t dst = smem_u32(smem + s * C::AB_BYTES);
                    const uint32_t fb = full0_leader + s * 8;
                    if (is_w) {
                        if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * C::AB_BYTES);
                        tma_load_2d_pair(dst, &tmW, fb, st * 128, wrow);
                    } else {
                        tma_load_3d_pair(dst + C::W_BYTES, &tmX, fb, 0, trow, 2 * st);
                    }
                }
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ metadata and scales producer (both CTAs)
        if (lane == 0) {
            uint32_t j = 0;
            bool ok = true;
            const int32_t ttiles128 = (p.M + 127) / 128;
            for (int32_t t = pair_id; t < total_tiles && ok; t += npairs) {
                int32_t tt, wt;
                tile_of(t, tt, wt);
                const int32_t wtile128 = 2 * wt + static_cast<int32_t>(rank);
                const int32_t t0 = 2 * tt, t1 = 2 * tt + 1 < ttiles128 ? 2 * tt + 1 : 2 * tt;
                const uint8_t *meta_g = p.W_meta + static_cast<size_t>(wtile128) * nstages * C::META_BYTES;
                const uint8_t *sfw_g = p.W_sf + static_cast<size_t>(wtile128) * kc * 512;
                const uint8_t *sfx0_g = p.X_sf + static_cast<size_t>(t0) * kc * 512;
                const uint8_t *sfx1_g = p.X_sf + static_cast<size_t>(t1) * kc * 512;
                for (int st = 0; st < nstages; ++st, ++j) {
                    const uint32_t s = j % SSD;
                    if (!mbar_wait(smem_u32(&side_empty[s]), ((j / SSD) & 1) ^ 1)) { ok = false; break; }
                    const uint32_t bar = smem_u32(&side_full[s]);
                    mbar_arrive_expect_tx(bar, C::SIDE_BYTES);
                    const uint32_t dst = smem_u32(smem + C::OFF_SIDE + s * C::SIDE_BYTES);
                    const size_t koff = static_cast<size_t>(st) * 4 * 512;
                    bulk_load(dst, meta_g + static_cast<size_t>(st) * C::META_BYTES, C::META_BYTES, bar);
                    bulk_load(dst + C::META_BYTES, sfw_g + koff, C::SFW_BYTES, bar);
                    // a token tile past M repeats the first one's scales: its
                    // rows are zero-filled, so any finite scale gives zeros
                    bulk_load(dst + C::META_BYTES + C::SFW_BYTES, sfx0_g + koff, 4 * 512, bar);
                    bulk_load(dst + C::META_BYTES + C::SFW_BYTES + 4 * 512, sfx1_g + koff, 4 * 512, bar);
                }
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            const uint64_t w_desc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
            const uint64_t x_desc0 = smem_desc(smem_u32(smem) + C::W_BYTES, 16, 1024, kSwizzle128B);
            constexpr uint64_t kStageDesc = static_cast<uint64_t>(C::AB_BYTES >> 4);
            // M = 256 weight rows, N = 256 tokens, UE4M3 scales, sparse A
            constexpr uint32_t idesc = idesc_block_scaled(256, 256, false, 0, 0) | (1u << 2);
            uint32_t s = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            for (int32_t t = pair_id; t < total_tiles && ok; t += npairs) {
                if (!mbar_wait(smem_u32(acc_empty), acc_phase ^ 1)) { ok = false; break; }
                tc_fence_after();
                for (int st = 0; st < nstages; ++st) {
                    if (!mbar_wait(smem_u32(&full[s]), phase)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t wd = w_desc0 + s * kStageDesc;
                    const uint64_t xd = x_desc0 + s * kStageDesc;
                    const uint32_t slot = tmem_base + C::COL_SLOT0 + s * C::SLOT_COLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // weights: 32 compressed bytes per K = 128 along the
                        // 128-byte row; tokens: 64 bytes, in two 16 KB tiles
                        const uint64_t ad = wd + 2 * kk;
                        const uint64_t bd = xd + (kk >> 1) * (16384 >> 4) + (kk & 1) * 4;
                        mma_sparse_pair(tmem_base, ad, bd, slot + C::SFW_COLS + C::SFX_COLS + 2 * kk, idesc,
                                        slot + 4 * kk, slot + C::SFW_COLS + 8 * kk, (st > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit_pair(smem_u32(&empty[s]), 0x3);
                    if (++s == SAB) { s = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(smem_u32(acc_full), 0x3);
                acc_phase ^= 1;
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------ side warps: metadata and scales -> tensor memory
        const int quad = warp & 3;
        const uint32_t set = static_cast<uint32_t>((warp - 4) >> 2);
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t ready0_leader = mapa_shared(smem_u32(&full[0]), 0);
        uint32_t j = 0;
        bool ok = true;
        for (int32_t t = pair_id; t < total_tiles && ok; t += npairs) {
            for (int st = 0; st < nstages; ++st, ++j) {
                if ((j & 1) != set) continue;
                const uint32_t s = j % SSD, slot = j % SAB;
                int got = __shfl_sync(0xffffffffu,
                                      lane == 0 ? (mbar_wait(smem_u32(&side_full[s]), (j / SSD) & 1) ? 1 : 0) : 0, 0);
                if (!got) { ok = false; break; }
                const uint8_t *sd = smem + C::OFF_SIDE + s * C::SIDE_BYTES;
                // metadata of this lane's weight row (32 bytes: 8 words, groups in order)
                uint32_t vm[C::META_COLS];
                const uint4 *mrow = reinterpret_cast<const uint4 *>(sd + (quad * 32 + lane) * 32);
                const uint4 m0 = mrow[0], m1 = mrow[1];
                vm[0] = m0.x; vm[1] = m0.y; vm[2] = m0.z; vm[3] = m0.w;
                vm[4] = m1.x; vm[5] = m1.y; vm[6] = m1.z; vm[7] = m1.w;
                // weight scales: word `quad` of the lane's 16-byte atom row, stored only in column
                // 4 c + quad of atom c, the one this lane quarter's MMA rows read
                uint32_t vw[4];
                // token scales: both token tiles' atoms, 8 columns per K = 128
                uint32_t vx[C::SFX_COLS];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 a4 = *reinterpret_cast<const uint4 *>(sd + C::META_BYTES + c * 512 + lane * 16);
                    vw[c] = quad == 0 ? a4.x : quad == 1 ? a4.y : quad == 2 ? a4.z : a4.w;
                    const uint8_t *xs = sd + C::META_BYTES + C::SFW_BYTES;
                    const uint4 b0 = *reinterpret_cast<const uint4 *>(xs + c * 512 + lane * 16);
                    const uint4 b1 = *reinterpret_cast<const uint4 *>(xs + (4 + c) * 512 + lane * 16);
                    vx[8 * c + 0] = b0.x; vx[8 * c + 1] = b0.y; vx[8 * c + 2] = b0.z; vx[8 * c + 3] = b0.w;
                    vx[8 * c + 4] = b1.x; vx[8 * c + 5] = b1.y; vx[8 * c + 6] = b1.z; vx[8 * c + 7] = b1.w;
                }
                // the tensor-memory slot is free once the MMAs of stage j - SAB completed
                if (j >= static_cast<uint32_t>(SAB)) {
                    const uint32_t js = j - SAB;
                    got = __shfl_sync(0xffffffffu,
                                      lane == 0 ? (mbar_wait(smem_u32(&empty[js % SAB]), (js / SAB) & 1) ? 1 : 0) : 0,
                                      0);
                    if (!got) { ok = false; break; }
                }
                tc_fence_after();
                const uint32_t col = tmem_base + C::COL_SLOT0 + slot * C::SLOT_COLS;
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_st_32x32b_x1(lane_base + col + 4 * c + quad, vw[c]);
                tmem_st_32x32b<C::SFX_COLS>(lane_base + col + C::SFW_COLS, vx);
                tmem_st_32x32b<C::META_COLS>(lane_base + col + C::SFW_COLS + C::SFX_COLS, vm);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&side_empty[s]));
                    mbar_arrive_cluster_relaxed(ready0_leader + slot * 8);
                }
            }
        }
        if (!ok && lane == 0) { record_timeout(); *abort_flag = 1; }
    } else if (warp >= 12) {
        // ------------------------------------------------ epilogue
        // Lane 32q + i of tensor memory is weight row w (a column of D),
        // column c a token (a row of D).  The warp drains its 32 weight rows
        // x 128 tokens into BF16 pairs of neighbouring tokens, releases the
        // accumulator, then writes D through staging boxes of 32 tokens x 32
        // weight columns: neighbouring lanes swap one value per token pair so
        // that each writes two adjacent columns of one token row.
        const int quad = warp & 3;
        const int half = (warp - 12) >> 2;
        const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
        uint8_t *d_stage = smem + C::OFF_D + (warp - 12) * C::D_BUFS * C::D_BOX;
        float gs = (p.gs_x ? p.gs_x[0] : 1.0f) * (p.gs_w ? p.gs_w[0] : 1.0f);
        const bool odd = lane & 1;
        uint32_t acc_phase = 0, nstore = 0;
        bool ok = true;
        for (int32_t t = pair_id; t < total_tiles; t += npairs) {
            int32_t tt, wt;
            tile_of(t, tt, wt);
            const int32_t w = wt * 256 + 128 * static_cast<int32_t>(rank) + quad * 32 + lane;
            const int32_t tok0 = tt * 256 + half * 128;
            const float cs = p.col_scale ? p.col_scale[w] : 1.0f;
            float rsv[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int32_t tk = tok0 + jj * 32 + lane;
                rsv[jj] = p.row_scale && tk < p.M ? p.row_scale[tk] : 1.0f;
            }
            const int got = __shfl_sync(0xffffffffu,
                                        lane == 0 ? (mbar_wait(smem_u32(acc_full), acc_phase) ? 1 : 0) : 0, 0);
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
            uint32_t pk[4][16];                     // BF16 pairs (token 2c, 2c + 1) of this lane's weight row
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + jj * 32, v);
                tmem_ld_wait();
                tmem_regs_after_wait(v);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float g0 = gs, g1 = gs;
                    if (p.row_scale) {
                        g0 = gs * __shfl_sync(0xffffffffu, rsv[jj], 2 * c);
                        g1 = gs * __shfl_sync(0xffffffffu, rsv[jj], 2 * c + 1);
                    }
                    float a = __uint_as_float(v[2 * c]) * g0, b = __uint_as_float(v[2 * c + 1]) * g1;
                    if (p.col_scale) {
                        a = a * cs;
                        b = b * cs;
                    }
                    pk[jj][c] = pack_bf16x2(a, b);
                }
            }
            tc_fence_before();
            if (!named_barrier_and(1, 256, got != 0 && *abort_flag == 0)) { ok = got != 0; break; }
            if (warp == 12 && lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader);
            const int32_t wcol0 = wt * 256 + 128 * static_cast<int32_t>(rank) + quad * 32;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                if (tok0 + jj * 32 >= p.M) break;            // rows past M: nothing to store
                uint8_t *box = d_stage + (nstore % C::D_BUFS) * C::D_BOX;
                if (lane == 0) bulk_wait_group_read<C::D_BUFS - 1>();
                __syncwarp();
                uint32_t *b32 = reinterpret_cast<uint32_t *>(box);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    // lane i holds (D[2c][w_i], D[2c + 1][w_i]); the even lane
                    // writes row 2c, columns (i, i + 1); the odd lane row 2c + 1
                    const uint32_t mine = pk[jj][c];
                    const uint32_t give = odd ? (mine & 0xFFFFu) : (mine >> 16);
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, give, 1);
                    const uint32_t word = odd ? (other | (mine & 0xFFFF0000u)) : ((mine & 0xFFFFu) | (other << 16));
                    b32[(2 * c + (odd ? 1 : 0)) * 16 + (lane >> 1)] = word;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmD, smem_u32(box), wcol0, tok0 + jj * 32);
                    bulk_commit_group();
                }
                ++nstore;
            }
            acc_phase ^= 1;
        }
        if (!ok && lane == 0) { record_timeout(); *abort_flag = 1; }
        if (lane == 0) bulk_wait_group_read<0>();
    }

    // ---- teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) { }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ compressor

// One thread per 32 bytes of a dense packed row (eight groups of four pair
// bytes): keeps the non-zero pairs of every group in order, pads with the
// lowest zero pairs to two, writes the 16 kept bytes and the eight 4-bit
// group codes i0 | i1 << 2 (one 32-bit word).  A pair is zero when both of
// its elements decode to 0 (codes 0 and 8).  A group with more than two
// non-zero pairs is not 2:4: the status word records it.
__global__ void __launch_bounds__(256)
sparse24_compress_kernel(const uint4 *__restrict__ W, int64_t rows, int64_t K, uint4 *__restrict__ Wc,
                         uint8_t *__restrict__ meta, int meta_layout, int64_t padded_rows)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t words_per_row = K / 64;                 // 32-byte pieces per row
    const int64_t total = padded_rows * words_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / words_per_row, w = i - r * words_per_row;
        uint32_t code = 0x44444444u;                      // padding rows: pairs 0 and 1 of zeros
        if (r < rows) {
            const uint4 a = W[2 * i], b = W[2 * i + 1];
            const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t out[4] = {0, 0, 0, 0};
            code = 0;
            bool bad = false;
#pragma unroll
            for (int gi = 0; gi < 8; ++gi) {
                int idx[2] = {-1, -1};
                int n = 0;
#pragma unroll
                for (int pi = 0; pi < 4; ++pi) {
                    const uint32_t byte = (in[gi] >> (8 * pi)) & 0xFFu;
                    const bool zero = (byte & 7u) == 0 && ((byte >> 4) & 7u) == 0;
                    if (!zero) {
                        if (n < 2) idx[n] = pi;
                        ++n;
                    }
                }
                bad |= n > 2;
                // pad with the lowest zero pairs, keeping i0 < i1
                if (n < 2) {
                    for (int pi = 0; pi < 4 && n < 2; ++pi) {
                        const uint32_t byte = (in[gi] >> (8 * pi)) & 0xFFu;
                        const bool zero = (byte & 7u) == 0 && ((byte >> 4) & 7u) == 0;
                        if (zero) {
                            if (n == 1 && pi < idx[0]) { idx[1] = idx[0]; idx[0] = pi; }
                            else idx[n] = pi;
                            ++n;
                        }
                    }
                }
                const uint32_t k0 = (in[gi] >> (8 * idx[0])) & 0xFFu, k1 = (in[gi] >> (8 * idx[1])) & 0xFFu;
                out[gi >> 1] |= (k0 | (k1 << 8)) << (16 * (gi & 1));
                code |= static_cast<uint32_t>(idx[0] | (idx[1] << 2)) << (4 * gi);
            }
            if (bad) atomicOr(&g_status_gemm_sparse, static_cast<uint32_t>(kStatusBadSparsity));
            Wc[i] = make_uint4(out[0], out[1], out[2], out[3]);
        }
        size_t off;
        if (meta_layout == QFP4_SF_MMA) {
            // [rows/128][K/512][128][32 bytes]: a 512-K stage of a 128-row tile is 4 KB
            const int64_t st = w / 8, within = w % 8;
            off = ((static_cast<size_t>(r / 128) * (K / kStageK) + st) * 128 + (r % 128)) * 32 + within * 4;
        } else {
            off = static_cast<size_t>(r) * (K / 16) + w * 4;
        }
        *reinterpret_cast<uint32_t *>(meta + off) = code;
    }
}

}  // namespace
}  // namespace qfp4

using namespace qfp4;

extern "C" size_t qfp4_sparse24_meta_bytes(int64_t rows, int64_t K, int meta_layout)
{
    if (rows < 0 || K < 0) return 0;
    if (meta_layout == QFP4_SF_MMA) return static_cast<size_t>((rows + 127) / 128) * 128 * static_cast<size_t>(K / 16);
    return static_cast<size_t>(rows) * static_cast<size_t>(K / 16);
}

extern "C" int qfp4_sparse24_compress(const void *W_packed, int64_t rows, int64_t K, void *W_comp, void *W_meta,
                                      int meta_layout, void *stream)
{
    if (meta_layout != QFP4_SF_ROWMAJOR && meta_layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (rows < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (K % 64 != 0 || (meta_layout == QFP4_SF_MMA && K % kStageK != 0)) return QFP4_ERR_UNSUPPORTED;
    if (rows == 0 || K == 0) return QFP4_OK;
    if (!W_packed || !W_comp || !W_meta) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(W_packed) || !aligned16(W_comp) || !aligned4(W_meta)) return QFP4_ERR_MISALIGNED;
    const int64_t padded = meta_layout == QFP4_SF_MMA ? (rows + 127) / 128 * 128 : rows;
    const int64_t work = padded * (K / 64);
    const int sms = sm_count();
    int64_t grid = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
    if (grid > cap) grid = cap;
    return launch_status(launch_pdl(sparse24_compress_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                                    static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(W_packed), rows, K,
                                    static_cast<uint4 *>(W_comp), static_cast<uint8_t *>(W_meta), meta_layout,
                                    padded));
}

extern "C" int qfp4_gemm_nt_sparse24(int fmt, int64_t M, int64_t N, int64_t K, const void *X_packed,
                                     const void *X_sf, const void *W_comp, const void *W_meta, const void *W_sf,
                                     const float *gs_x, const float *gs_w, const float *row_scale,
                                     const float *col_scale, void *D_bf16, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4 && fmt != QFP4_NVFP4_B32) return QFP4_ERR_INVALID_ARG;
    if (fmt != QFP4_NVFP4_B32) return QFP4_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (N % 256 != 0 || K % kStageK != 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QFP4_OK;
    if (!D_bf16) return QFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return cudaMemsetAsync(D_bf16, 0, static_cast<size_t>(M) * N * 2, s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
    if (!X_packed || !X_sf || !W_comp || !W_meta || !W_sf) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_packed) || !aligned16(X_sf) || !aligned16(W_comp) || !aligned16(W_meta) || !aligned16(W_sf) ||
        !aligned16(D_bf16) || (gs_x && !aligned4(gs_x)) || (gs_w && !aligned4(gs_w)) ||
        (row_scale && !aligned4(row_scale)) || (col_scale && !aligned4(col_scale)))
        return QFP4_ERR_MISALIGNED;
    CUtensorMap mw, mx, md;
    int rc = make_map(&mw, W_comp, K / 4, N, 128, 128);
    if (rc == QFP4_OK) rc = make_map_kpairs(&mx, X_packed, K, M);
    if (rc == QFP4_OK) rc = make_map_bf16(&md, D_bf16, N, M, 32, 32);
    if (rc != QFP4_OK) return rc;
    SpParams prm{static_cast<const uint8_t *>(X_sf), static_cast<const uint8_t *>(W_sf),
                 static_cast<const uint8_t *>(W_meta), gs_x, gs_w, row_scale, col_scale,
                 static_cast<int32_t>(M), static_cast<int32_t>(N), static_cast<int32_t>(K)};
    rc = ensure_smem_attr(reinterpret_cast<const void *>(gemm_sparse_kernel), SpCfg::SMEM);
    if (rc != QFP4_OK) return rc;
    const int sms = sm_count();
    if (sms < 2) return QFP4_ERR_CUDA;
    const int64_t tiles = ((M + 255) / 256) * (N / 256);
    int64_t pairs = sms / 2;
    if (tiles < pairs) pairs = tiles;
    return launch_status(launch_pdl(gemm_sparse_kernel, dim3(static_cast<unsigned>(2 * pairs)), dim3(kThreads),
                                    SpCfg::SMEM, s, mw, mx, md, prm));
}
