// gemm_decode.cu -- block-scaled FP4 GEMM for decode-shaped batches (M <= 128).
//
// Pages: quadbit README, "End-to-end serving": at decode the weights stream
// from DRAM and the kernel must keep enough SMs busy to do that at full
// bandwidth; DeepGEMM pull request "Key technical details" (swap-AB epilogue,
// 2-CTA cta_group::2 MMAs with per-CTA scale-factor loads).
//
// Swap AB: the weights B [N, K] take the MMA's M slot and the <= 128 tokens
// of A take its N slot, so the tensor core computes D^T.  A CTA pair owns 256
// weight rows (128 per CTA) and, by default, all of K: ceil(N / 256) pairs
// and no cross-CTA reduction (N = 14336: 56 pairs on 112 SMs).  When that
// leaves the GPU short of pairs and K is long enough for it to pay (see
// decode_splits), SPLITK gives each weight tile S pairs with contiguous K
// ranges: fp32 partials go to the caller's workspace, and after a counted
// barrier the S CTAs of a rank each reduce a slice of the columns in split
// order (deterministic) and write D.  Per 256-K block the
// leader issues four M=256 N=128 K=64 MMAs (each CTA's tensor memory
// receives its 128 weight rows x 128 tokens); each CTA streams 16 KB of
// weights, 8 KB of tokens (its half of N) and 4 KB of scale factors.
//
// Roles (384 threads per CTA): warps 0 and 3 weight and token TMA producers
// (both CTAs, completion on the leader's barrier); warp 2 scale-factor producer (bulk
// copies into a local ring); warp 1 tensor-memory owner and, in the leader,
// the MMA issuer; warps 4..11, two sets of four taking alternate K-blocks,
// move the scale bytes into tensor memory with tcgen05.st (the tensor pipe
// then runs MMAs only; one set alone, waiting for each store to complete,
// would take about a K-block's streaming time per K-block); at the end both
// sets drain the accumulator, each half of the tokens: scale by gs_a * gs_b,
// round to BF16, transpose through shared memory and write D with one TMA
// store per CTA.  All waits are bounded.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <mutex>

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

constexpr int kThreads = 384;          // 12 warps
constexpr int kTok = 128;              // MMA N: token rows, 64 per CTA

template <int FMT>
struct DecCfg {
    static constexpr int G = FMT == QFP4_MXFP4 ? 32 : 16;
    static constexpr int CPS = (256 / G) / 4;          // 512-B SF tiles per 128 rows per 256-K block
    static constexpr int W_BYTES = 128 * 128;          // this CTA's 128 weight rows
    static constexpr int T_BYTES = (kTok / 2) * 128;   // this CTA's 64 token rows
    static constexpr int AB_BYTES = W_BYTES + T_BYTES;
    static constexpr int AB_STAGES = 7;
    static constexpr int SFW_BYTES = CPS * 512;         // weight rows' scales (MMA A)
    static constexpr int SFT_BYTES = CPS * 512;         // all 128 token rows' scales (MMA B)
    static constexpr int SF_BYTES = SFW_BYTES + SFT_BYTES;
    static constexpr int SF_STAGES = 8;
    static constexpr int OFF_SF = AB_STAGES * AB_BYTES;
    static constexpr int OFF_BAR = OFF_SF + SF_STAGES * SF_BYTES;
    // full/empty[AB], sf_full/sf_empty[SF], acc_full
    static constexpr int NBAR = 2 * AB_STAGES + 2 * SF_STAGES + 1;
    static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
    static constexpr int SFW_COLS = CPS * 4;            // weight words: quarter q uses column 4 c + q of atom c
    static constexpr int SFT_COLS = CPS * 4;            // all 128 token rows in every quarter
    static constexpr int SLOT_COLS = SFW_COLS + SFT_COLS;
    static constexpr int COL_SF = kTok;                 // accumulator: 128 columns
    static constexpr int TMEM_COLS = 512;
    static constexpr int D_BYTES = kTok * 128 * 2;      // BF16 staging of D^T -> D (reuses the ring)
    static_assert(COL_SF + AB_STAGES * SLOT_COLS <= TMEM_COLS, "tensor memory overflow");
    static_assert(D_BYTES <= OFF_SF, "output staging must fit in the operand ring");
    static_assert(SMEM <= 232448, "shared memory overflow");
};

__device__ __forceinline__ void record_timeout()
{
    atomicOr(&g_status_gemm_decode, static_cast<uint32_t>(kStatusTimeout));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&pr);
}

// Split-K reduction of one weight tile's 128 rows (this CTA's rank) over
// the S CTAs that computed its K ranges: this CTA (split `split`) sums
// columns [split * 128/S, +128/S) of all S fp32 partials in split order
// 0..S-1 (the same order whichever CTA runs it, so results repeat bit for
// bit), applies the epilogue scales, rounds to BF16 and writes them to D,
// where they are columns col0.. of token rows 0..M-1.  A partial is
// [mpad tokens][128 weight rows] fp32, written by other SMs, so the loads
// bypass L1; each thread takes four neighbouring weight rows of one token
// and writes them as one 8-byte piece of a D row.
template <int S>
__device__ __forceinline__ void decode_reduce_slice(const float *part0, size_t part_stride, int split, int M,
                                                    float gs, const float *row_scale, const float *col_scale,
                                                    int col0, __nv_bfloat16 *D, int ldd)
{
    constexpr int R = 128 / S;               // weight rows (D columns) of the slice
    constexpr int V = R / 4;                 // float4 per token in the slice
    constexpr int U = 16 / S;                // float4 positions per thread per round (16 loads in flight)
    const int nvec = M * V;
    const float *src0 = part0 + split * R;
    for (int f0 = threadIdx.x; f0 < nvec; f0 += U * kThreads) {
        float4 v[S][U];
#pragma unroll
        for (int q = 0; q < S; ++q)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * kThreads;
                const int t = f / V, c = f - t * V;
                v[q][u] = f < nvec ? __ldcg(reinterpret_cast<const float4 *>(src0 + q * part_stride + t * 128) + c)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int f = f0 + u * kThreads;
            if (f >= nvec) break;
            float4 a = v[0][u];
#pragma unroll
            for (int q = 1; q < S; ++q) {
                a.x = __fadd_rn(a.x, v[q][u].x);
                a.y = __fadd_rn(a.y, v[q][u].y);
                a.z = __fadd_rn(a.z, v[q][u].z);
                a.w = __fadd_rn(a.w, v[q][u].w);
            }
            const int t = f / V, n = col0 + 4 * (f - t * V);     // token row of D, first D column
            const float g = row_scale ? gs * row_scale[t] : gs;
            float o[4] = {a.x * g, a.y * g, a.z * g, a.w * g};
            if (col_scale) {
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] = o[i] * col_scale[n + i];
            }
            *reinterpret_cast<uint2 *>(D + static_cast<size_t>(t) * ldd + n) =
                make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
        }
    }
}

template <int FMT, bool SPLITK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmT,
                   const __grid_constant__ CUtensorMap tmD, const GemmParams p)
{
    using C = DecCfg<FMT>;
    constexpr int SAB = C::AB_STAGES, SSF = C::SF_STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars;                 // leader: operand bytes of both CTAs + 8 scale warps
    uint64_t *empty = full + SAB;          // stage and its tensor-memory scale slot free (MMA commit)
    uint64_t *sf_full = empty + SAB;       // local: scale bytes landed
    uint64_t *sf_empty = sf_full + SSF;    // local: scale warps done with the slot
    uint64_t *acc_full = sf_empty + SSF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int K = p.K;
    const int kc = (K / C::G) / 4;
    const int kblocks = (K + 255) / 256;
    // split-K: pair = split * pair_tiles + pair tile; split s owns K-blocks
    // [s * kblocks / S, (s + 1) * kblocks / S) (at least one: S <= kblocks)
    const int32_t pair_tiles = (p.N + 255) / 256;
    const int32_t pair = blockIdx.x >> 1;
    const int32_t ptile = SPLITK ? pair % pair_tiles : pair;
    const int split = SPLITK ? pair / pair_tiles : 0;
    const int nsplit = SPLITK ? p.splits : 1;
    const int kb_begin = SPLITK ? (split * kblocks) / nsplit : 0;
    const int nkb = SPLITK ? ((split + 1) * kblocks) / nsplit - kb_begin : kblocks;
    const int32_t wtile = 2 * ptile + static_cast<int32_t>(rank);   // this CTA's 128-row weight tile
    const bool w_valid = wtile < p.N / 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SAB; ++s) {
            mbar_init(smem_u32(&full[s]), 1 + 8);     // leader producer (with the bytes) + 4 scale warps x 2 CTAs
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < SSF; ++s) {
            mbar_init(smem_u32(&sf_full[s]), 1);
            mbar_init(smem_u32(&sf_empty[s]), 4);     // the four warps of one set
        }
        mbar_init(smem_u32(acc_full), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmT);
        prefetch_tensormap(&tmD);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // everything above overlaps the previous kernel's tail; global memory
    // is touched only from here on
    pdl_wait();
    // (the next kernel launches only once every CTA of this grid has passed
    // this point, so all of them are resident before any waits on another
    // in the split-K reduction)
    pdl_launch_dependents();

    // j counts this CTA's K-blocks (ring slots and phases), kb = kb_begin + j
    // is the K-block's position in K
    if (warp == 0 || warp == 3) {
        // ------------------------------------------------ weight (warp 0) / token (warp 3) TMA producers
        // (two issuing warps: the copy engine serves one issuing thread's
        // requests one after another)
        if (lane == 0) {
            const bool is_w = warp == 0;
            const uint32_t full0_leader = mapa_shared(smem_u32(&full[0]), 0);
            bool ok = true;
            for (int j = 0; j < nkb; ++j) {
                const int kb = kb_begin + j;
                const uint32_t s = j % SAB;
                if (!mbar_wait(smem_u32(&empty[s]), ((j / SAB) & 1) ^ 1)) { ok = false; break; }
                const uint32_t dst = smem_u32(smem + s * C::AB_BYTES);
                const uint32_t fb = full0_leader + s * 8;
                if (is_w) {
                    // the leader's weight thread posts the byte count of both CTAs' loads
                    if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * C::AB_BYTES);
                    tma_load_2d_pair(dst, &tmW, fb, kb * 128, wtile * 128);
                } else {
                    tma_load_2d_pair(dst + C::W_BYTES, &tmT, fb, kb * 128, static_cast<int32_t>(rank) * (kTok / 2));
                }
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ scale-factor producer (both CTAs)
        if (lane == 0) {
            const uint8_t *sfw_g = p.B_sf + static_cast<size_t>(wtile) * kc * 512;
            bool ok = true;
            for (int j = 0; j < nkb; ++j) {
                const int kb = kb_begin + j;
                const uint32_t s = j % SSF;
                if (!mbar_wait(smem_u32(&sf_empty[s]), ((j / SSF) & 1) ^ 1)) { ok = false; break; }
                const int chunks = min(C::CPS, kc - kb * C::CPS);
                const uint32_t bar = smem_u32(&sf_full[s]);
                mbar_arrive_expect_tx(bar, (w_valid ? 2 : 1) * chunks * 512);
                const uint32_t dst = smem_u32(smem + C::OFF_SF + s * C::SF_BYTES);
                const size_t koff = static_cast<size_t>(kb) * C::CPS * 512;
                if (w_valid) bulk_load(dst, sfw_g + koff, chunks * 512, bar);
                bulk_load(dst + C::SFW_BYTES, p.A_sf + koff, chunks * 512, bar);
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            const uint64_t w_desc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
            const uint64_t t_desc0 = smem_desc(smem_u32(smem) + C::W_BYTES, 16, 1024, kSwizzle128B);
            constexpr uint64_t kStageDesc = static_cast<uint64_t>(C::AB_BYTES >> 4);
            bool ok = true;
            uint32_t s = 0, phase = 0;
            for (int j = 0; j < nkb; ++j) {
                const int kb = kb_begin + j;
                if (!mbar_wait(smem_u32(&full[s]), phase)) { ok = false; break; }
                tc_fence_after();
                const uint64_t wd = w_desc0 + s * kStageDesc;
                const uint64_t td = t_desc0 + s * kStageDesc;
                const uint32_t sfw_t = tmem_base + C::COL_SF + s * C::SLOT_COLS;
                const uint32_t sft_t = sfw_t + C::SFW_COLS;
                const int ksteps = min(4, (K - kb * 256) / 64);
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                    if (FMT == QFP4_NVFP4) {
                        constexpr uint32_t id = idesc_block_scaled(256, kTok, false, 0, 0);
                        tc_mma_nvf4_pair(tmem_base, wd + 2 * kk, td + 2 * kk, id, sfw_t + kk * 4, sft_t + kk * 4,
                                         acc);
                    } else {
                        constexpr uint32_t id0 = idesc_block_scaled(256, kTok, true, 0, 0);
                        constexpr uint32_t id1 = idesc_block_scaled(256, kTok, true, 2, 2);
                        tc_mma_mxf4_pair(tmem_base, wd + 2 * kk, td + 2 * kk, (kk & 1) ? id1 : id0,
                                         sfw_t + (kk >> 1) * 4, sft_t + (kk >> 1) * 4, acc);
                    }
                }
                tc_commit_pair(smem_u32(&empty[s]), 0x3);
                if (++s == SAB) { s = 0; phase ^= 1; }
            }
            if (ok) tc_commit_pair(smem_u32(acc_full), 0x3);
            else { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp >= 4) {
        const int quad = warp & 3;
        const int set = (warp - 4) >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t ready0_leader = mapa_shared(smem_u32(&full[0]), 0);
        bool ok = true;
        // -------------------------------------------- scale factors -> tensor memory
        // Tensor-memory layout of one 512-byte tile at columns [c, c+4):
        // lane 32q + i, column c + j holds the four scale bytes of row
        // i + 32 j.  Quarter q of the MMA reads its weight rows' scales from
        // column c + q only, but needs all 128 token rows, so the token
        // tile is written in full and the weight word q only into column
        // c + q (fewer columns written: ~0.8% faster at 128x4096x4096).
        // The shared-memory slot is handed back only after the values
        // reached tensor memory.
        for (int j = set; j < nkb; j += 2) {
            const uint32_t s = j % SSF, slot = j % SAB;
            int got = __shfl_sync(0xffffffffu,
                                  lane == 0 ? (mbar_wait(smem_u32(&sf_full[s]), (j / SSF) & 1) ? 1 : 0) : 0, 0);
            if (!got) { ok = false; break; }
            const uint8_t *sf_s = smem + C::OFF_SF + s * C::SF_BYTES;
            uint32_t vw[C::CPS];
            uint32_t vt[C::SFT_COLS];
#pragma unroll
            for (int c = 0; c < C::CPS; ++c) {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(sf_s + c * 512 + lane * 16);
                vw[c] = quad == 0 ? w4.x : quad == 1 ? w4.y : quad == 2 ? w4.z : w4.w;
                const uint4 t4 = *reinterpret_cast<const uint4 *>(sf_s + C::SFW_BYTES + c * 512 + lane * 16);
                vt[4 * c + 0] = t4.x; vt[4 * c + 1] = t4.y; vt[4 * c + 2] = t4.z; vt[4 * c + 3] = t4.w;
            }
            got = __shfl_sync(0xffffffffu,
                              lane == 0 ? (mbar_wait(smem_u32(&empty[slot]), ((j / SAB) & 1) ^ 1) ? 1 : 0) : 0, 0);
            if (!got) { ok = false; break; }
            tc_fence_after();
            const uint32_t col = tmem_base + C::COL_SF + slot * C::SLOT_COLS;
#pragma unroll
            for (int c = 0; c < C::CPS; ++c) tmem_st_32x32b_x1(lane_base + col + 4 * c + quad, vw[c]);
            tmem_st_32x32b<C::SFT_COLS>(lane_base + col + C::SFW_COLS, vt);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&sf_empty[s]));
                mbar_arrive_cluster_relaxed(ready0_leader + slot * 8);
            }
        }
        if (SPLITK && set == 0) {
        // -------------------------------------------- split-K: partial sums out
        // Lane 32q + i is weight row n = 32q + i of this CTA and holds tokens
        // 32j .. 32j+31 of chunk j; partial[t][n] is stored token by token,
        // so each warp store fills one 128-byte line.
        const int got = ok ? __shfl_sync(0xffffffffu,
                                         lane == 0 ? (mbar_wait(smem_u32(acc_full), 0) ? 1 : 0) : 0, 0)
                           : 0;
        if (got && w_valid) {
            tc_fence_after();
            const int nchunks = (p.M + 31) / 32;
            const int mpad = nchunks * 32;
            const int n = quad * 32 + lane;
            float *dst = p.ws_partial +
                         ((static_cast<size_t>(ptile) * nsplit + split) * 2 + rank) * (128u * mpad) + n;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
            for (int j = 0; j < nchunks; ++j) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + j * 32, v);
                tmem_ld_wait();
                tmem_regs_after_wait(v);
#pragma unroll
                for (int i = 0; i < 32; ++i) dst[(j * 32 + i) * 128] = __uint_as_float(v[i]);
            }
        } else if (!got && lane == 0) {
            record_timeout();
            *abort_flag = 1;
        }
        }
        if (!SPLITK) {
        // -------------------------------------------- accumulator drain
        // Both scale sets drain, set s the tokens 64s .. 64s + 63.  Lane
        // 32q + i of tensor memory is weight row n = 32q + i of this CTA;
        // column m is token m.  Each thread writes D[m][n] for its n
        // into a row-major [128 tokens][128 columns] BF16 tile in shared
        // memory (a warp writes 64 consecutive bytes per token), and one
        // TMA store moves the tile to D; rows m >= M are clipped by it.
        // two-level epilogue: D[m][n] = bf16((acc * (gs * row_scale[m])) *
        // col_scale[n]); here n is this lane's weight row and the tokens m
        // are the columns, so the column scale is per lane and lane i holds
        // the row scale of token 32 j + i, shared out by shuffles.  Read
        // before the accumulator wait.
        const int n_lane = quad * 32 + lane;
        const float cs_lane = (p.col_scale && w_valid) ? p.col_scale[wtile * 128 + n_lane] : 1.0f;
        float rsv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            rsv[j] = (p.row_scale && j * 32 + lane < p.M) ? p.row_scale[j * 32 + lane] : 1.0f;
        const bool rscale = p.row_scale != nullptr, cscale = p.col_scale != nullptr;
        const int got = ok ? __shfl_sync(0xffffffffu,
                                         lane == 0 ? (mbar_wait(smem_u32(acc_full), 0) ? 1 : 0) : 0, 0)
                           : 0;
        if (got) {
            tc_fence_after();
            float gs = 1.0f;
            if (FMT == QFP4_NVFP4) gs = (p.gs_a ? *p.gs_a : 1.0f) * (p.gs_b ? *p.gs_b : 1.0f);
            const int n = quad * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
            // Neighbouring lanes (rows n, n^1) swap one value per pair of
            // tokens so that each writes two adjacent columns of one token
            // row as a 4-byte word: the even lane token m, the odd lane m+1.
            uint32_t *stage = reinterpret_cast<uint32_t *>(smem);
            const bool odd = lane & 1;
            const int n0 = n & ~1;
            const int nchunks = (p.M + 31) / 32;
            for (int j = 2 * set; j < nchunks && j < 2 * set + 2; ++j) {   // set s: tokens 64s..64s+63
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + j * 32, v);
                tmem_ld_wait();
                tmem_regs_after_wait(v);
                const float rs_j = j == 0 ? rsv[0] : j == 1 ? rsv[1] : j == 2 ? rsv[2] : rsv[3];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float ga = gs, gb = gs;
                    if (rscale) {
                        ga = gs * __shfl_sync(0xffffffffu, rs_j, i);
                        gb = gs * __shfl_sync(0xffffffffu, rs_j, i + 1);
                    }
                    float a = __uint_as_float(v[i]) * ga, b = __uint_as_float(v[i + 1]) * gb;
                    if (cscale) {
                        a = a * cs_lane;
                        b = b * cs_lane;
                    }
                    const float other = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
                    const int m = j * 32 + i + (odd ? 1 : 0);
                    // columns n0 (low half) and n0 + 1 (high half) of token row m
                    stage[(m * 128 + n0) >> 1] = odd ? pack_bf16x2(other, b) : pack_bf16x2(a, other);
                }
            }
            fence_proxy_async_smem();
        } else if (lane == 0) {
            record_timeout();
            *abort_flag = 1;
        }
        __syncwarp();
        named_barrier_sync(1, 8 * 32);
        if (warp == 4 && lane == 0 && !*abort_flag && w_valid) {
            tma_store_2d(&tmD, smem_u32(smem), wtile * 128, 0);
            bulk_commit_group();
            // the staging tile must outlive the copy engine's reads of it;
            // the writes themselves complete with the grid
            bulk_wait_group_read<0>();
        }
        }
    }

    if constexpr (SPLITK) {
        // ---- split-K reduction.  The S CTAs holding this CTA's rank of the
        // same weight tile meet at a sense-reversing barrier in the
        // workspace: an arrival count and a generation word.  Each reads the
        // generation, adds 1 to the count once its partial is out (release);
        // the last arrival sets the count back to 0 and advances the
        // generation, and the others wait (acquire, bounded) for that.  Every
        // call thus leaves the counts at 0, whatever S the next call uses.
        // All S CTAs are resident: the launch is sized to fit the GPU's
        // clusters at once, and nothing after this kernel can take an SM
        // before all of them started.
        __shared__ int s_go;
        __syncwarp();
        __syncthreads();
        uint32_t *cnt = p.ws_count + 2 * (2 * ptile + rank);
        uint32_t *gen = cnt + 1;
        if (threadIdx.x == 0) {
            int go = (!*abort_flag && w_valid) ? 1 : 0;
            if (go) {
                const uint32_t g = ld_acquire_gpu(gen);
                if (atom_add_acq_rel_gpu(cnt, 1u) == static_cast<uint32_t>(nsplit) - 1u) {
                    st_relaxed_gpu(cnt, 0u);
                    st_release_gpu(gen, g + 1u);
                } else {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(gen) == g) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            go = 0;
                            record_timeout();
                            *abort_flag = 1;
                            break;
                        }
                    }
                }
            }
            s_go = go;
        }
        __syncthreads();
        if (s_go) {
            const int mpad = ((p.M + 31) / 32) * 32;
            const size_t part_stride = 2u * 128u * mpad;                  // floats from split q to q + 1
            const float *part0 = p.ws_partial + (static_cast<size_t>(ptile) * nsplit * 2 + rank) * (128u * mpad);
            float gs = 1.0f;
            if (FMT == QFP4_NVFP4) gs = (p.gs_a ? *p.gs_a : 1.0f) * (p.gs_b ? *p.gs_b : 1.0f);
            const int col0 = wtile * 128 + split * (128 / nsplit);
            switch (nsplit) {
            case 2: decode_reduce_slice<2>(part0, part_stride, split, p.M, gs, p.row_scale, p.col_scale, col0,
                                           p.D, p.N); break;
            case 4: decode_reduce_slice<4>(part0, part_stride, split, p.M, gs, p.row_scale, p.col_scale, col0,
                                           p.D, p.N); break;
            default: decode_reduce_slice<8>(part0, part_stride, split, p.M, gs, p.row_scale, p.col_scale, col0,
                                            p.D, p.N); break;
            }
        }
    }

    // ---- teardown.  Reconverge each warp first: lanes that skipped a
    // single-lane role must not reach the block barrier ahead of their warp's
    // working lane.
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
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

template <int FMT, bool SPLITK>
int launch_decode(const CUtensorMap &mw, const CUtensorMap &mt, const CUtensorMap &md, const GemmParams &g,
                  cudaStream_t s)
{
    using C = DecCfg<FMT>;
    auto kern = gemm_decode_kernel<FMT, SPLITK>;
    {
        const int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM);
        if (rc != QFP4_OK) return rc;
    }
    const int pairs = ((g.N + 255) / 256) * (SPLITK ? g.splits : 1);
    return launch_status(launch_pdl(kern, dim3(2 * pairs), dim3(kThreads), C::SMEM, s, mw, mt, md, g));
}

}  // namespace

int launch_gemm_decode(int fmt, const CUtensorMap &mw, const CUtensorMap &mt, const CUtensorMap &md,
                       const GemmParams &g, cudaStream_t s)
{
    if (g.splits > 1)
        return fmt == QFP4_NVFP4 ? launch_decode<QFP4_NVFP4, true>(mw, mt, md, g, s)
                                 : launch_decode<QFP4_MXFP4, true>(mw, mt, md, g, s);
    return fmt == QFP4_NVFP4 ? launch_decode<QFP4_NVFP4, false>(mw, mt, md, g, s)
                             : launch_decode<QFP4_MXFP4, false>(mw, mt, md, g, s);
}

// Clusters of this kernel the current device holds at once (queried once
// per device; the split-K grid must fit, since its CTAs wait on each other).
static int decode_max_clusters()
{
    static std::mutex mu;
    static int cached[64];
    static bool have[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        using C = DecCfg<QFP4_NVFP4>;
        static_assert(DecCfg<QFP4_MXFP4>::SMEM <= C::SMEM, "the NVFP4 kernel bounds both");
        auto kern = gemm_decode_kernel<QFP4_NVFP4, true>;
        int n = 0;
        if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM) == QFP4_OK) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = C::SMEM;
            if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(kern), &cfg) != cudaSuccess) {
                n = 0;
                cudaGetLastError();
            }
        }
        cached[dev] = n;
        have[dev] = true;
    }
    return cached[dev];
}

// Split-K pays only when it removes enough K-blocks from each pair: the
// partials' trip through L2 (write, the barrier, the reduction) costs about
// as much as streaming 12-13 K-blocks (traced on GB300: ~4.5 us against
// ~0.36 us per 256-K block), so a split must save at least 16 of them.
constexpr int kSplitMinSavedKBlocks = 16;

int decode_splits(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || M > 128 || N < 128 || K < 256) return 1;
    const int64_t pair_tiles = (N + 255) / 256, kblocks = (K + 255) / 256;
    const int sms = sm_count();
    int64_t cap = sms / 2;
    const int clusters = decode_max_clusters();
    if (clusters > 0 && clusters < cap) cap = clusters;
    for (int s : {8, 4, 2})
        if (pair_tiles * s <= cap && s <= kblocks && kblocks - (kblocks + s - 1) / s >= kSplitMinSavedKBlocks)
            return s;
    return 1;
}

size_t decode_counter_bytes(int64_t N)
{
    // an arrival count and a generation word per (pair tile, CTA rank)
    const size_t pair_tiles = static_cast<size_t>((N + 255) / 256);
    return (pair_tiles * 2 * 2 * sizeof(uint32_t) + 255) / 256 * 256;
}

size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits)
{
    (void)K;
    if (splits <= 1) return 0;
    const size_t pair_tiles = static_cast<size_t>((N + 255) / 256);
    const size_t mpad = static_cast<size_t>((M + 31) / 32) * 32;
    return decode_counter_bytes(N) + pair_tiles * splits * 2 * 128 * mpad * sizeof(float);
}

}  // namespace qfp4
