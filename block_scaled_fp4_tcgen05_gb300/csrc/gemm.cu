// gemm.cu -- block-scaled FP4 GEMM D = A . B^T on the sm_103a tensor cores.
//
// Pages: DeepGEMM pull request "Packed MXFP4 & NVFP4 GEMM + mega-MoE (SM100,
// true 2-CTA multicast)", sections "Summary" ([M,K] @ [N,K]^T -> [M,N] BF16,
// packed E2M1 operands, UE8M0 / UE4M3 scales, acc * gs_act * gs_weight) and
// "Key technical details" (MMA kinds mxf4 / mxf4nvf4 scale_vec::4X, scale
// factors copied to tensor memory, NVFP4 carrying twice the scale columns
// per K-block, the scale-factor id selecting a byte inside a 32-bit column
// while whole columns are selected by tensor-memory address); quadbit README
// "End-to-end serving" (one-launch segmented MoE kernel).
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A/B tiles (128-byte swizzle, 128 B of K per
//               row = 256 FP4 per stage) and the stage's scale-factor tiles
//               (plain bulk copies of 512-byte MMA-layout tiles) into a ring
//               of STAGES shared-memory slots, signalled by mbarriers.
//   warp 1      tensor memory owner + MMA issuer: one elected lane copies
//               the stage's scale factors into tensor memory (tcgen05.cp) and
//               issues four K=64 block-scaled MMAs into the fp32 accumulator
//               held in tensor memory; tcgen05.commit frees the slot.
//   warps 2..9  epilogue: tcgen05.ld the accumulator into registers, release
//               it to the MMA warp at once, then scale by gs_a * gs_b, round
//               to BF16 and store, overlapping the next tile's main loop.
// Every wait is bounded; a wait that runs out records QFP4_ERR_TIMEOUT in
// the device status word and the kernel winds down.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "qfp4_common.cuh"
#include "qfp4_gemm_internal.cuh"
#include "sm103_ptx.cuh"

namespace qfp4 {

__device__ uint32_t g_status_gemm = 0;

int read_clear_status_gemm(cudaStream_t s, uint32_t *out)
{
    uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(out, g_status_gemm, sizeof(uint32_t), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_status_gemm, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

namespace {

constexpr int kBM = 128;             // rows of A per tile (MMA M)
constexpr int kBKBytes = 128;        // bytes of K per row per stage (256 FP4)
constexpr int kKStep = 64;           // FP4 elements per MMA instruction
constexpr int kThreads = 320;        // 10 warps
constexpr int kEpiWarps = 8;
constexpr int kMaxGroupsGemm = 256;

template <int FMT, int BN, int STAGES>
struct Cfg {
    static constexpr int G = FMT == QFP4_MXFP4 ? 32 : 16;          // elements per scale
    static constexpr int CPS = (2 * kBKBytes / G) / 4;             // 512-B SF tiles per stage per 128 rows
    static constexpr int NRC = BN / 128;                           // 128-row chunks of B
    static constexpr int A_BYTES = kBM * kBKBytes;
    static constexpr int B_BYTES = BN * kBKBytes;
    static constexpr int SFA_BYTES = CPS * 512;
    static constexpr int SFB_BYTES = NRC * CPS * 512;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 2) * 8 + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;        // + alignment slack
    // tensor memory columns: accumulator, then per-stage scale factors
    static constexpr int SFA_COLS = CPS * 4;
    static constexpr int SFB_COLS = NRC * CPS * 4;
    static constexpr int COL_SF = BN;
    static constexpr int COLS_USED = BN + STAGES * (SFA_COLS + SFB_COLS);
    static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                   : COLS_USED <= 256 ? 256 : 512;
    static_assert(COLS_USED <= 512, "tensor memory overflow");
    static_assert(SMEM <= 232448, "shared memory overflow");
};

using GemmArgs = GemmParams;

struct TileInfo {
    int32_t row0;      // first row of A / D
    int32_t row_end;   // rows of this tile's group end here (exclusive)
    int32_t sf_tile;   // 128-row tile index into A_sf
    int32_t n0;        // first column
    int32_t group;
};

__device__ __forceinline__ void record_timeout()
{
    atomicOr(&g_status_gemm, static_cast<uint32_t>(kStatusTimeout));
}

template <int FMT, int BN, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const GemmArgs args)
{
    using C = Cfg<FMT, BN, STAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    // bars[0..S): full, [S..2S): empty, [2S]: accum full, [2S+1]: accum empty
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int32_t s_offs[GROUPED ? kMaxGroupsGemm + 1 : 1];
    __shared__ int32_t s_tile_start[GROUPED ? kMaxGroupsGemm + 1 : 1];   // prefix of tiles per group

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int K = args.K;
    const int kstages = (K + 2 * kBKBytes - 1) / (2 * kBKBytes);
    const int kc = (K / C::G) / 4;                     // 512-B SF tiles per 128 rows
    const int ntiles_n = args.N / BN;

    // ---- tile count and group tables (the group offsets are the first
    // global reads: wait for the previous kernel before them)
    if (GROUPED) pdl_wait();
    int32_t total_tiles;
    if (GROUPED) {
        __shared__ int s_bad;
        for (int i = threadIdx.x; i <= args.groups; i += blockDim.x) s_offs[i] = args.row_offsets[i];
        __syncthreads();
        if (threadIdx.x == 0) {
            // offsets that do not describe the rows the launch was sized
            // for: no tile is processed and nothing is written
            s_bad = group_offsets_valid(s_offs, args.groups, args.M, args.max_group_rows) ? 0 : 1;
            if (s_bad && blockIdx.x == 0) atomicOr(&g_status_gemm, static_cast<uint32_t>(kStatusBadGroup));
            int32_t acc = 0;
            for (int e = 0; e < args.groups; ++e) {
                s_tile_start[e] = acc;
                const int32_t rows = s_offs[e + 1] - s_offs[e];
                acc += rows > 0 ? (rows + kBM - 1) / kBM : 0;
            }
            s_tile_start[args.groups] = acc;
        }
        __syncthreads();
        total_tiles = s_bad ? 0 : s_tile_start[args.groups] * ntiles_n;
    } else {
        total_tiles = ((args.M + kBM - 1) / kBM) * ntiles_n;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[STAGES + s]), 1);
        }
        mbar_init(smem_u32(&bars[2 * STAGES]), 1);
        mbar_init(smem_u32(&bars[2 * STAGES + 1]), kEpiWarps);
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
    if (!GROUPED) pdl_wait();
    pdl_launch_dependents();

    // Tile t -> coordinates.  Non-grouped: groups of 8 row-tiles sweep the
    // columns together so that a wave of CTAs shares A and B in L2.
    auto tile_info = [&](int32_t t) {
        TileInfo ti;
        if (GROUPED) {
            const int32_t mt_all = t / ntiles_n;      // row-tile over all groups
            ti.n0 = (t % ntiles_n) * BN;
            int lo = 0, hi = args.groups - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_tile_start[mid] <= mt_all) lo = mid; else hi = mid - 1;
            }
            ti.group = lo;
            const int32_t mt = mt_all - s_tile_start[lo];
            ti.row0 = s_offs[lo] + mt * kBM;
            ti.row_end = s_offs[lo + 1];
            ti.sf_tile = mt_all;
        } else {
            const int32_t mtiles = (args.M + kBM - 1) / kBM;
            constexpr int32_t GM = 8;
            const int32_t per_group = GM * ntiles_n;
            const int32_t grp = t / per_group;
            const int32_t first_m = grp * GM;
            const int32_t rows_here = min(GM, mtiles - first_m);
            const int32_t idx = t % per_group;
            const int32_t mt = first_m + idx % rows_here;
            ti.n0 = (idx / rows_here) * BN;
            ti.row0 = mt * kBM;
            ti.row_end = args.M;
            ti.sf_tile = mt;
            ti.group = 0;
        }
        return ti;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(t);
                const uint8_t *sfa = args.A_sf + static_cast<size_t>(ti.sf_tile) * kc * 512;
                const int32_t brow = GROUPED ? ti.group * args.N + ti.n0 : ti.n0;
                const uint8_t *sfb = args.B_sf + static_cast<size_t>(brow / 128) * kc * 512;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(smem_u32(&bars[STAGES + stage]), phase ^ 1)) { ok = false; break; }
                    const int chunks = min(C::CPS, kc - ks * C::CPS);
                    const uint32_t full = smem_u32(&bars[stage]);
                    mbar_arrive_expect_tx(full, C::A_BYTES + C::B_BYTES + (1 + C::NRC) * chunks * 512);
                    tma_load_2d(smem_u32(smem + C::OFF_A + stage * C::A_BYTES), &tmA, full,
                                ks * kBKBytes, ti.row0);
                    tma_load_2d(smem_u32(smem + C::OFF_B + stage * C::B_BYTES), &tmB, full,
                                ks * kBKBytes, brow);
                    bulk_load(smem_u32(smem + C::OFF_SFA + stage * C::SFA_BYTES),
                              sfa + static_cast<size_t>(ks) * C::CPS * 512, chunks * 512, full);
#pragma unroll
                    for (int rc = 0; rc < C::NRC; ++rc)
                        bulk_load(smem_u32(smem + C::OFF_SFB + stage * C::SFB_BYTES + rc * C::CPS * 512),
                                  sfb + (static_cast<size_t>(rc) * kc + ks * C::CPS) * 512,
                                  chunks * 512, full);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t acc_tmem = tmem_base;
            for (int32_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(smem_u32(&bars[2 * STAGES + 1]), acc_phase ^ 1)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(smem_u32(&bars[stage]), phase)) { ok = false; break; }
                    tc_fence_after();
                    const int chunks = min(C::CPS, kc - ks * C::CPS);
                    const uint32_t sfa_t = tmem_base + C::COL_SF + stage * (C::SFA_COLS + C::SFB_COLS);
                    const uint32_t sfb_t = sfa_t + C::SFA_COLS;
                    const uint32_t sfa_s = smem_u32(smem + C::OFF_SFA + stage * C::SFA_BYTES);
                    const uint32_t sfb_s = smem_u32(smem + C::OFF_SFB + stage * C::SFB_BYTES);
                    for (int c = 0; c < chunks; ++c) {
                        tc_cp_32x128b_warpx4(sfa_t + c * 4, smem_desc(sfa_s + c * 512, 128, 128, kSwizzleNone));
#pragma unroll
                        for (int rc = 0; rc < C::NRC; ++rc)
                            tc_cp_32x128b_warpx4(sfb_t + (c * C::NRC + rc) * 4,
                                                 smem_desc(sfb_s + (rc * C::CPS + c) * 512, 128, 128, kSwizzleNone));
                    }
                    const uint32_t a_s = smem_u32(smem + C::OFF_A + stage * C::A_BYTES);
                    const uint32_t b_s = smem_u32(smem + C::OFF_B + stage * C::B_BYTES);
                    const int ksteps = min(4, (K - ks * 2 * kBKBytes) / kKStep);
                    for (int kk = 0; kk < ksteps; ++kk) {
                        const uint64_t ad = smem_desc(a_s + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(b_s + kk * 32, 16, 1024, kSwizzle128B);
                        const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
                        if (FMT == QFP4_NVFP4) {
                            constexpr uint32_t idesc = idesc_block_scaled(kBM, BN, false, 0, 0);
                            tc_mma_nvf4(acc_tmem, ad, bd, idesc, sfa_t + kk * 4,
                                        sfb_t + kk * C::NRC * 4, accum);
                        } else {
                            const int c = kk >> 1;
                            const uint32_t id = (kk & 1) ? idesc_block_scaled(kBM, BN, true, 2, 2)
                                                         : idesc_block_scaled(kBM, BN, true, 0, 0);
                            tc_mma_mxf4(acc_tmem, ad, bd, id, sfa_t + c * 4, sfb_t + c * C::NRC * 4, accum);
                        }
                    }
                    tc_commit(smem_u32(&bars[STAGES + stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&bars[2 * STAGES]));
                acc_phase ^= 1;
            }
            if (!ok) { record_timeout(); *abort_flag = 1; }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
        const int half = (warp - 2) >> 2;          // column half of the tile
        constexpr int COLS = BN / 2;
        constexpr int NCH = COLS / 32;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int32_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
            const TileInfo ti = tile_info(t);
            const int32_t row = ti.row0 + quad * 32 + lane;
            // two-level epilogue: this lane's row scale, and lane i holding
            // the scale of column 32 j + i of each 32-column chunk j (shared
            // out by shuffles); read before the accumulator wait
            const float rsv = (args.row_scale && row < ti.row_end) ? args.row_scale[row] : 1.0f;
            float csv[NCH];
#pragma unroll
            for (int j = 0; j < NCH; ++j)
                csv[j] = args.col_scale
                             ? args.col_scale[(GROUPED ? ti.group * args.N : 0) + ti.n0 + half * COLS + j * 32 + lane]
                             : 1.0f;
            // lane 0 waits; the result is broadcast so the warp stays converged
            // for the warp-wide tensor-memory loads below
            const int got = __shfl_sync(0xffffffffu,
                                        lane == 0 ? (mbar_wait(smem_u32(&bars[2 * STAGES]), acc_phase) ? 1 : 0) : 0, 0);
            if (!got) { ok = false; break; }
            tc_fence_after();
            uint32_t v[NCH][32];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * COLS;
#pragma unroll
            for (int j = 0; j < NCH; ++j) tmem_ld_32x32b_x32(taddr + j * 32, v[j]);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < NCH; ++j) tmem_regs_after_wait(v[j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[2 * STAGES + 1]));
            acc_phase ^= 1;

            float gs = 1.0f;
            if (FMT == QFP4_NVFP4) {
                const int g = GROUPED ? ti.group : 0;
                const float ga = args.gs_a ? args.gs_a[g] : 1.0f;
                const float gb = args.gs_b ? args.gs_b[g] : 1.0f;
                gs = ga * gb;
            }
            if (args.row_scale) gs = gs * rsv;
            const bool cscale = args.col_scale != nullptr;
            if (row < ti.row_end || cscale) {
                __nv_bfloat16 *dst = args.D + static_cast<size_t>(row) * args.N + ti.n0 + half * COLS;
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float lo = __uint_as_float(v[j][2 * i]) * gs;
                        float hi = __uint_as_float(v[j][2 * i + 1]) * gs;
                        if (cscale) {
                            // every lane of the warp takes part in the shuffles
                            lo = lo * __shfl_sync(0xffffffffu, csv[j], 2 * i);
                            hi = hi * __shfl_sync(0xffffffffu, csv[j], 2 * i + 1);
                        }
                        __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
                        packed[i] = *reinterpret_cast<uint32_t *>(&p);
                    }
                    if (row < ti.row_end) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + j * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                               packed[4 * i + 3]);
                    }
                }
            }
        }
        if (!ok && lane == 0) { record_timeout(); *abort_flag = 1; }
    }

    // ---- teardown: all roles done (or timed out); free tensor memory.
    // Reconverge each warp first: lanes that skipped a single-lane role must
    // not reach the block barrier ahead of their warp's working lane.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies and MMAs already in flight drain before the memory goes
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) { }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int encode_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows);
int encode_map_kpairs(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows);
int encode_map_bf16(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows);

// Encoded tensor maps, cached.  A map is a pure function of its encode
// arguments (base address, extents, strides, box, element type, swizzle), so
// an entry keyed by all of them can never be stale: a buffer freed and
// reallocated at the same address with the same shape gets the same map.
// Decode-sized GEMMs run in ~10 us, and encoding two or three maps on the
// host per call is a visible part of that; the cache makes repeated calls on
// the same buffers (the common case: weights, and activations in a reused
// arena) skip the encode.  Fixed size, hash-indexed, replace on collision,
// one mutex (host threads may call the library concurrently).
struct MapKey {
    uint32_t kind;           // 0: make_map, 1: make_map_kpairs, 2: make_map_bf16
    uint32_t box0, box1;
    const void *base;
    uint64_t d0, d1;
    bool operator==(const MapKey &o) const
    {
        return kind == o.kind && box0 == o.box0 && box1 == o.box1 && base == o.base && d0 == o.d0 && d1 == o.d1;
    }
};

constexpr int kMapCacheSize = 256;
struct MapEntry {
    bool used = false;
    MapKey key{};
    CUtensorMap map{};
};

std::mutex g_map_mu;
MapEntry g_map_cache[kMapCacheSize];

size_t map_hash(const MapKey &k)
{
    uint64_t h = 0x9E3779B97F4A7C15ull * (reinterpret_cast<uintptr_t>(k.base) >> 4);
    h ^= (k.d0 * 0xC2B2AE3D27D4EB4Full) + (k.d1 << 17) + (static_cast<uint64_t>(k.box0) << 7) + k.box1 + k.kind;
    h ^= h >> 29;
    return static_cast<size_t>(h % kMapCacheSize);
}

template <typename F>
int cached_map(const MapKey &key, CUtensorMap *out, F encode)
{
    const size_t i = map_hash(key);
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        if (g_map_cache[i].used && g_map_cache[i].key == key) {
            *out = g_map_cache[i].map;
            return QFP4_OK;
        }
    }
    int rc = ensure_thread_context();
    if (rc == QFP4_OK) rc = encode(out);
    if (rc == QFP4_OK) {
        std::lock_guard<std::mutex> lock(g_map_mu);
        g_map_cache[i].used = true;
        g_map_cache[i].key = key;
        g_map_cache[i].map = *out;
    }
    return rc;
}

}  // namespace

// 2D byte matrix [rows, inner] (row stride = inner bytes), box of
// box_inner bytes x box_rows rows, 128-byte swizzle, zero fill out of bounds.
int make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
             uint32_t box_rows)
{
    return cached_map(MapKey{0, box_inner, box_rows, base, inner, rows}, map,
                      [&](CUtensorMap *m) { return encode_map(m, base, inner, rows, box_inner, box_rows); });
}

int make_map_kpairs(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows)
{
    return cached_map(MapKey{1, 0, 0, base, K, rows}, map,
                      [&](CUtensorMap *m) { return encode_map_kpairs(m, base, K, rows); });
}

int make_map_bf16(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                  uint32_t box_rows)
{
    return cached_map(MapKey{2, box_cols, box_rows, base, cols, rows}, map,
                      [&](CUtensorMap *m) { return encode_map_bf16(m, base, cols, rows, box_cols, box_rows); });
}

namespace {

int encode_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows)
{
    auto enc = get_encode_fn();
    if (!enc) return QFP4_ERR_CUDA;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QFP4_OK : QFP4_ERR_CUDA;
}

int encode_map_kpairs(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows)
{
    auto enc = get_encode_fn();
    if (!enc) return QFP4_ERR_CUDA;
    cuuint64_t dims[3] = {128, rows, K / 256};
    cuuint64_t strides[2] = {K / 2, 128};
    cuuint32_t box[3] = {128, 128, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QFP4_OK : QFP4_ERR_CUDA;
}

int encode_map_bf16(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows)
{
    auto enc = get_encode_fn();
    if (!enc) return QFP4_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QFP4_OK : QFP4_ERR_CUDA;
}

}  // namespace

namespace {

template <int FMT, int BN, int STAGES, bool GROUPED>
int launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &a, int32_t tiles,
                cudaStream_t s)
{
    using C = Cfg<FMT, BN, STAGES>;
    auto kern = gemm_kernel<FMT, BN, STAGES, GROUPED>;
    {
        const int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM);
        if (rc != QFP4_OK) return rc;
    }
    const int sms = sm_count();
    if (sms <= 0) return QFP4_ERR_CUDA;
    const int grid = tiles < sms ? (tiles > 0 ? tiles : 1) : sms;
    return launch_status(launch_pdl(kern, dim3(grid), dim3(kThreads), C::SMEM, s, ma, mb, a));
}

}  // namespace
}  // namespace qfp4

using namespace qfp4;

extern "C" size_t qfp4_gemm_workspace_bytes(int fmt, int64_t M, int64_t N, int64_t K)
{
    if ((fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) || M < 1 || M > 128 || N < 1 || K < 1 || N % 128 != 0 ||
        K % 128 != 0 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return 0;   // only the decode kernel splits K; the others keep their sums on chip
    return decode_workspace_bytes(M, N, K, decode_splits(M, N, K));
}

static int gemm_nt_impl(int fmt, int64_t M, int64_t N, int64_t K, const void *A_packed, const void *A_sf,
                        const void *B_packed, const void *B_sf, const float *gs_a, const float *gs_b,
                        const float *row_scale, const float *col_scale, void *D_bf16, void *workspace,
                        size_t ws_bytes, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return QFP4_OK;            // empty D: nothing to do, nothing launched
    if (!D_bf16) return QFP4_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return QFP4_ERR_UNSUPPORTED;
    if (K == 0) {
        // an empty sum: D = 0 (BF16 +0 is all-zero bits)
        if (!aligned16(D_bf16)) return QFP4_ERR_MISALIGNED;
        return cudaMemsetAsync(D_bf16, 0, static_cast<size_t>(M) * static_cast<size_t>(N) * 2,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
                   ? QFP4_OK
                   : QFP4_ERR_CUDA;
    }
    if (!A_packed || !A_sf || !B_packed || !B_sf) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(A_packed) || !aligned16(A_sf) || !aligned16(B_packed) || !aligned16(B_sf) ||
        !aligned16(D_bf16) || (gs_a && !aligned4(gs_a)) || (gs_b && !aligned4(gs_b)) ||
        (row_scale && !aligned4(row_scale)) || (col_scale && !aligned4(col_scale)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmParams a{static_cast<const uint8_t *>(A_sf), static_cast<const uint8_t *>(B_sf), gs_a, gs_b,
                 static_cast<__nv_bfloat16 *>(D_bf16), static_cast<int32_t>(M), static_cast<int32_t>(N),
                 static_cast<int32_t>(K), 0, nullptr, row_scale, col_scale};
    CUtensorMap ma, mb;
    if (M <= 128) {
        // decode shapes: swap AB on CTA pairs, weights in the MMA's M slot;
        // K split over more pairs when the weight tiles alone leave SMs idle
        // and the caller's workspace holds the partial sums
        int splits = decode_splits(M, N, K);
        if (splits > 1 && !(workspace && aligned16(workspace) &&
                            ws_bytes >= decode_workspace_bytes(M, N, K, splits)))
            splits = 1;
        a.splits = splits;
        if (splits > 1) {
            a.ws_count = static_cast<uint32_t *>(workspace);
            a.ws_partial = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + decode_counter_bytes(N));
        }
        CUtensorMap md;
        int rc = make_map(&mb, B_packed, K / 2, N, kBKBytes, 128);
        if (rc == QFP4_OK) rc = make_map(&ma, A_packed, K / 2, M, kBKBytes, 64);
        if (rc == QFP4_OK) rc = make_map_bf16(&md, D_bf16, N, M, 128, 128);   // (split-K stores D directly)
        if (rc != QFP4_OK) return rc;
        return launch_gemm_decode(fmt, mb, ma, md, a, s);
    }
    if (N % 256 == 0 && M > 128) {
        // CTA pairs on 256 x 256 tiles; D leaves in 32-row x 16-column boxes
        CUtensorMap md;
        int rc;
        if (gemm_pair_double_stages(fmt, false, K)) {
            rc = make_map_kpairs(&ma, A_packed, K, M);
            if (rc == QFP4_OK) rc = make_map_kpairs(&mb, B_packed, K, N);
        } else {
            rc = make_map(&ma, A_packed, K / 2, M, kBKBytes, 128);
            if (rc == QFP4_OK) rc = make_map(&mb, B_packed, K / 2, N, kBKBytes, 128);
        }
        if (rc == QFP4_OK) rc = make_map_bf16(&md, D_bf16, N, M, 16, 32);
        if (rc != QFP4_OK) return rc;
        return launch_gemm_pair(fmt, false, ma, mb, md, a, ((M + 255) / 256) * (N / 256), s);
    }
    // single CTAs on 128 x 128 tiles (M > 128, N % 256 == 128)
    int rc = make_map(&ma, A_packed, K / 2, M, kBKBytes, kBM);
    if (rc == QFP4_OK) rc = make_map(&mb, B_packed, K / 2, N, kBKBytes, 128);
    if (rc != QFP4_OK) return rc;
    const int32_t mtiles = static_cast<int32_t>((M + kBM - 1) / kBM);
    if (fmt == QFP4_NVFP4) return launch_gemm<QFP4_NVFP4, 128, 6, false>(ma, mb, a, mtiles * (N / 128), s);
    return launch_gemm<QFP4_MXFP4, 128, 6, false>(ma, mb, a, mtiles * (N / 128), s);
}

extern "C" int qfp4_gemm_nt(int fmt, int64_t M, int64_t N, int64_t K, const void *A_packed,
                            const void *A_sf, const void *B_packed, const void *B_sf,
                            const float *gs_a, const float *gs_b, void *D_bf16, void *workspace,
                            size_t ws_bytes, void *stream)
{
    return gemm_nt_impl(fmt, M, N, K, A_packed, A_sf, B_packed, B_sf, gs_a, gs_b, nullptr, nullptr, D_bf16,
                        workspace, ws_bytes, stream);
}

extern "C" int qfp4_gemm_nt_scaled(int fmt, int64_t M, int64_t N, int64_t K, const void *A_packed,
                                   const void *A_sf, const void *B_packed, const void *B_sf,
                                   const float *gs_a, const float *gs_b, const float *row_scale,
                                   const float *col_scale, void *D_bf16, void *workspace, size_t ws_bytes,
                                   void *stream)
{
    return gemm_nt_impl(fmt, M, N, K, A_packed, A_sf, B_packed, B_sf, gs_a, gs_b, row_scale, col_scale,
                        D_bf16, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// qfp4_gemm_nt_noalloc: qfp4_gemm_nt for callers that cannot allocate device
// memory.  The scratch the decode split-K needs lives in this file-scope
// array instead of a caller-provided workspace.  Every GPU that loads the
// library holds the array until the process exits; every call shares it.
constexpr size_t kNoAllocScratchBytes = (size_t{8} << 20) + 4096;   // 8 MiB of partial sums + 4 KiB of counters
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a stand-in for the symbol, never an address a
// kernel may be given, so the address is asked of the runtime: once per
// device, with that device current, cached behind a mutex.
static int noalloc_scratch_address(void **out)
{
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *addr[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QFP4_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return QFP4_OK;
}

extern "C" int qfp4_gemm_nt_noalloc(int fmt, int64_t M, int64_t N, int64_t K, const void *A_packed,
                                    const void *A_sf, const void *B_packed, const void *B_sf,
                                    const float *gs_a, const float *gs_b, void *D_bf16, void *stream)
{
    const size_t need = qfp4_gemm_workspace_bytes(fmt, M, N, K);
    if (need > kNoAllocScratchBytes) return QFP4_ERR_WORKSPACE;
    if (need == 0)
        return gemm_nt_impl(fmt, M, N, K, A_packed, A_sf, B_packed, B_sf, gs_a, gs_b, nullptr, nullptr, D_bf16,
                            nullptr, 0, stream);
    void *scratch = nullptr;
    const int rc = noalloc_scratch_address(&scratch);
    if (rc != QFP4_OK) return rc;
    // the arrival counts must start at zero; the array keeps whatever the
    // last call (or one that timed out) left there
    if (cudaMemsetAsync(scratch, 0, decode_counter_bytes(N), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return gemm_nt_impl(fmt, M, N, K, A_packed, A_sf, B_packed, B_sf, gs_a, gs_b, nullptr, nullptr, D_bf16,
                        scratch, kNoAllocScratchBytes, stream);
}

static int gemm_nt_grouped_impl(int fmt, int64_t groups, const int32_t *row_offsets, int64_t total_rows,
                                int64_t max_group_rows, int64_t N, int64_t K, const void *A_packed,
                                const void *A_sf, const void *B_packed, const void *B_sf, const float *gs_a,
                                const float *gs_b, const float *row_scale, const float *col_scale, void *D_bf16,
                                void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (groups < 1 || !row_offsets || total_rows < 0 || max_group_rows < 0 || N < 1 || K < 1)
        return QFP4_ERR_INVALID_ARG;
    if (!A_packed || !A_sf || !B_packed || !B_sf || !D_bf16) return QFP4_ERR_INVALID_ARG;
    if (groups > kMaxGroupsGemm || N % 128 != 0 || K % 128 != 0 || total_rows > INT32_MAX / 2 ||
        groups * N > INT32_MAX / 2 || K > INT32_MAX / 2)
        return QFP4_ERR_UNSUPPORTED;
    if (!aligned16(A_packed) || !aligned16(A_sf) || !aligned16(B_packed) || !aligned16(B_sf) ||
        !aligned16(D_bf16) || !aligned4(row_offsets) || (gs_a && !aligned4(gs_a)) ||
        (gs_b && !aligned4(gs_b)) || (row_scale && !aligned4(row_scale)) || (col_scale && !aligned4(col_scale)))
        return QFP4_ERR_MISALIGNED;
    if (total_rows == 0) return QFP4_OK;
    if (max_group_rows > INT32_MAX / 2) max_group_rows = 0;     // no bound worth checking
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmParams a{static_cast<const uint8_t *>(A_sf), static_cast<const uint8_t *>(B_sf), gs_a, gs_b,
                 static_cast<__nv_bfloat16 *>(D_bf16), static_cast<int32_t>(total_rows),
                 static_cast<int32_t>(N), static_cast<int32_t>(K), static_cast<int32_t>(groups),
                 row_offsets, row_scale, col_scale};
    a.max_group_rows = static_cast<int32_t>(max_group_rows);
    // Upper bound on the row tiles of all groups, for the grid: every group
    // may add one partial tile, and no group has more than max_group_rows
    // rows (the kernels check both bounds against the offsets).
    auto tile_bound = [&](int64_t rows_per_tile) {
        const int64_t by_total = (total_rows + rows_per_tile - 1) / rows_per_tile + groups;
        const int64_t by_max = groups * ((max_group_rows + rows_per_tile - 1) / rows_per_tile);
        return max_group_rows > 0 && by_max < by_total ? by_max : by_total;
    };
    CUtensorMap ma, mb;
    if (N % 256 == 0) {
        CUtensorMap md;
        int rc = make_map(&ma, A_packed, K / 2, total_rows, kBKBytes, 128);
        if (rc == QFP4_OK) rc = make_map(&mb, B_packed, K / 2, groups * N, kBKBytes, 128);
        if (rc == QFP4_OK) rc = make_map_bf16(&md, D_bf16, N, total_rows, 16, 32);
        if (rc != QFP4_OK) return rc;
        return launch_gemm_pair(fmt, true, ma, mb, md, a, tile_bound(256) * (N / 256), s);
    }
    int rc = make_map(&ma, A_packed, K / 2, total_rows, kBKBytes, kBM);
    if (rc == QFP4_OK) rc = make_map(&mb, B_packed, K / 2, groups * N, kBKBytes, 128);
    if (rc != QFP4_OK) return rc;
    const int32_t tiles = static_cast<int32_t>(tile_bound(kBM) * (N / 128));
    if (fmt == QFP4_NVFP4) return launch_gemm<QFP4_NVFP4, 128, 6, true>(ma, mb, a, tiles, s);
    return launch_gemm<QFP4_MXFP4, 128, 6, true>(ma, mb, a, tiles, s);
}

extern "C" int qfp4_gemm_nt_grouped(int fmt, int64_t groups, const int32_t *row_offsets,
                                    int64_t total_rows, int64_t max_group_rows, int64_t N, int64_t K,
                                    const void *A_packed, const void *A_sf, const void *B_packed,
                                    const void *B_sf, const float *gs_a, const float *gs_b,
                                    void *D_bf16, void *workspace, size_t ws_bytes, void *stream)
{
    (void)workspace; (void)ws_bytes;    // the grouped kernels need no scratch
    return gemm_nt_grouped_impl(fmt, groups, row_offsets, total_rows, max_group_rows, N, K, A_packed, A_sf,
                                B_packed, B_sf, gs_a, gs_b, nullptr, nullptr, D_bf16, stream);
}

extern "C" int qfp4_gemm_nt_grouped_scaled(int fmt, int64_t groups, const int32_t *row_offsets,
                                           int64_t total_rows, int64_t max_group_rows, int64_t N, int64_t K,
                                           const void *A_packed, const void *A_sf, const void *B_packed,
                                           const void *B_sf, const float *gs_a, const float *gs_b,
                                           const float *row_scale, const float *col_scale, void *D_bf16,
                                           void *workspace, size_t ws_bytes, void *stream)
{
    (void)workspace; (void)ws_bytes;
    return gemm_nt_grouped_impl(fmt, groups, row_offsets, total_rows, max_group_rows, N, K, A_packed, A_sf,
                                B_packed, B_sf, gs_a, gs_b, row_scale, col_scale, D_bf16, stream);
}

// Up-projection with SwiGLU and requantisation: the pair GEMM over the
// interleaved gate/up rows W, its epilogue writing H = silu(gate) * up
// quantised (no D).  Dense (row_offsets NULL) or grouped.
static int gemm_swiglu_impl(int fmt, int64_t groups, const int32_t *row_offsets, int64_t M, int64_t I,
                            int64_t K, const void *A_packed, const void *A_sf, const void *W_packed,
                            const void *W_sf, const float *gs_a, const float *gs_w, const float *gs_out,
                            void *Q_out, void *SF_out, void *stream)
{
    const bool grouped = row_offsets != nullptr;
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || I < 0 || K < 0 || (grouped && groups < 1)) return QFP4_ERR_INVALID_ARG;
    if (grouped && groups > kMaxGroupsGemm) return QFP4_ERR_UNSUPPORTED;
    if (I % 128 != 0 || K % 128 != 0 || M > INT32_MAX / 2 || 2 * I * (grouped ? groups : 1) > INT32_MAX / 2 ||
        K > INT32_MAX / 2)
        return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || I == 0) return QFP4_OK;           // empty H: nothing to do, nothing launched
    const int g = fmt == QFP4_MXFP4 ? 32 : 16;
    if (!Q_out || !SF_out || (fmt == QFP4_NVFP4 && !gs_out)) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(Q_out) || !aligned4(SF_out) || (gs_out && !aligned4(gs_out)) ||
        (grouped && !aligned4(row_offsets)))
        return QFP4_ERR_MISALIGNED;
    if (K > 0) {
        if (!A_packed || !A_sf || !W_packed || !W_sf) return QFP4_ERR_INVALID_ARG;
        if (!aligned16(A_packed) || !aligned16(A_sf) || !aligned16(W_packed) || !aligned16(W_sf) ||
            (gs_a && !aligned4(gs_a)) || (gs_w && !aligned4(gs_w)))
            return QFP4_ERR_MISALIGNED;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sf_bytes = grouped ? qfp4_sf_mma_grouped_bytes(M, groups, I / g) : qfp4_sf_mma_bytes(M, I / g);
    // padding rows of the scale layout must read as zero scales downstream
    if (cudaMemsetAsync(SF_out, 0, sf_bytes, s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (K == 0) {
        // empty sums: G = U = 0, so H = 0, every scale byte 0 and every code +0
        return cudaMemsetAsync(Q_out, 0, static_cast<size_t>(M) * static_cast<size_t>(I / 2), s) == cudaSuccess
                   ? QFP4_OK
                   : QFP4_ERR_CUDA;
    }
    GemmParams a{static_cast<const uint8_t *>(A_sf), static_cast<const uint8_t *>(W_sf), gs_a, gs_w, nullptr,
                 static_cast<int32_t>(M), static_cast<int32_t>(2 * I), static_cast<int32_t>(K),
                 static_cast<int32_t>(grouped ? groups : 0), row_offsets, nullptr, nullptr, gs_out,
                 static_cast<uint8_t *>(Q_out), static_cast<uint8_t *>(SF_out), static_cast<int32_t>(I),
                 static_cast<int32_t>(I / (4 * g))};
    CUtensorMap ma, mb;
    int rc = make_map(&ma, A_packed, K / 2, M, kBKBytes, 128);
    if (rc == QFP4_OK) rc = make_map(&mb, W_packed, K / 2, 2 * I * (grouped ? groups : 1), kBKBytes, 128);
    if (rc != QFP4_OK) return rc;
    const int64_t m_tiles = (M + 255) / 256 + (grouped ? groups : 0);
    return launch_gemm_pair_swiglu(fmt, grouped, ma, mb, a, m_tiles * (2 * I / 256), s);
}

extern "C" int qfp4_gemm_swiglu_quantize(int fmt, int64_t M, int64_t I, int64_t K, const void *A_packed,
                                         const void *A_sf, const void *W_packed, const void *W_sf,
                                         const float *gs_a, const float *gs_w, const float *gs_out, void *Q_out,
                                         void *SF_out, void *stream)
{
    return gemm_swiglu_impl(fmt, 0, nullptr, M, I, K, A_packed, A_sf, W_packed, W_sf, gs_a, gs_w, gs_out, Q_out,
                            SF_out, stream);
}

extern "C" int qfp4_gemm_swiglu_quantize_grouped(int fmt, int64_t groups, const int32_t *row_offsets,
                                                 int64_t total_rows, int64_t I, int64_t K, const void *A_packed,
                                                 const void *A_sf, const void *W_packed, const void *W_sf,
                                                 const float *gs_a, const float *gs_w, const float *gs_out,
                                                 void *Q_out, void *SF_out, void *stream)
{
    if (!row_offsets) return QFP4_ERR_INVALID_ARG;
    return gemm_swiglu_impl(fmt, groups, row_offsets, total_rows, I, K, A_packed, A_sf, W_packed, W_sf, gs_a,
                            gs_w, gs_out, Q_out, SF_out, stream);
}
