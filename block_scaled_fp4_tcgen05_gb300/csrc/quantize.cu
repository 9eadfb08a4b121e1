// quantize.cu -- BF16 -> NVFP4 / MXFP4 quantiser, global scale and the
// scale-factor interleave (HBM-bound kernels, no tensor cores).  The
// quantiser streams its input through shared memory with bulk copies (TMA
// engine) so that enough bytes are in flight per SM to keep HBM busy.
//
// Pages: Mojo "fp4_quantization" module, "Functions"
// (quantize_dynamic_scaled_fp4fp8, grouped_quantize_dynamic_scaled_fp4_async,
// block_scales_interleave); DeepGEMM pull request "Packed MXFP4 & NVFP4 GEMM +
// mega-MoE", "Summary" (formats, per-tensor fp32 global scales).
//
// The quantiser is bit-exact to this rule, in IEEE fp32 round-to-nearest-even:
//   amax = max|x| over a block of g;  t = (amax / 6) / gs;
//   sf = round-to-format(t);  s = decode(sf) * gs;  code_i = E2M1(x_i / s).
// x_i / s must be the correctly rounded quotient.  MXFP4 scales are powers of
// two, so x * 2^-e is that quotient exactly.  For NVFP4 the quotient is
// formed from y = RN(1/s) (CUDA's IEEE reciprocal, once per block) and two
// corrections q' = q + (x - s*q)*y with fused multiply-adds; by Markstein's
// theorem (P. Markstein, IBM J. R&D 34(1), 1990; also Muller et al.,
// "Handbook of Floating-Point Arithmetic", sec. on division with FMA) the
// second correction returns RN(x/s) when y = RN(1/s), the previous quotient
// is within one ulp and nothing underflows or overflows.  Blocks whose scale
// or range could leave that regime take CUDA's IEEE division instead.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "qfp4_common.cuh"
#include "qfp4_fp4_codes.cuh"
#include "sm103_ptx.cuh"

namespace qfp4 {

__device__ uint32_t g_status_quant = 0;

int read_clear_status_quant(cudaStream_t s, uint32_t *out)
{
    uint32_t zero = 0;
    if (cudaMemcpyFromSymbolAsync(out, g_status_quant, sizeof(uint32_t), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_status_quant, &zero, sizeof(uint32_t), 0,
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

namespace {

constexpr int kThreads = 256;
constexpr int kQThreads = kThreads + 32;   // quantiser CTA: 8 consumer warps + 1 producer warp
constexpr int kMaxGroups = 256;

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// bf16 pair in a 32-bit word -> two fp32 (exact).
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float &lo, float &hi)
{
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

// bf16 pair in a 32-bit word -> both values as one fp32 pair (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w)
{
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Largest |x| of a block as fp32 (exact): pairwise max of magnitudes on the
// packed bf16 words (the sign of the result is meaningless and dropped).
template <int W>
__device__ __forceinline__ float block_amax(const uint32_t (&w)[W])
{
    uint32_t m[W];
#pragma unroll
    for (int i = 0; i < W; ++i) m[i] = w[i];
#pragma unroll
    for (int n = W; n > 1; n >>= 1)
#pragma unroll
        for (int i = 0; i < n / 2; ++i)
            asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(m[2 * i]), "r"(m[2 * i + 1]));
    return fmaxf(fabsf(__uint_as_float(m[0] << 16)), fabsf(__uint_as_float(m[0] & 0xFFFF0000u)));
}

// Four bf16 words (8 elements, element 2i in the low half of word i) -> four
// packed E2M1 bytes (element 2i in the low nibble of byte i).
template <int FMT>
__device__ __forceinline__ uint32_t encode8(const uint32_t *w, const BlockScale &b)
{
    float q[8];
    if (FMT == QFP4_MXFP4) {
        const uint64_t inv2 = f2_pack(b.inv, b.inv);       // a power of two: exact
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(bf16x2_to_f2(w[i]), inv2), q[2 * i], q[2 * i + 1]);
        return e2m1x8(q);
    }
    if (b.mode == 1) {
        const uint64_t s2 = f2_pack(b.s, b.s), ny2 = f2_pack(-b.inv, -b.inv);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f2_unpack(f2_neg_quotient(bf16x2_to_f2(w[i]), s2, ny2), q[2 * i], q[2 * i + 1]);
        return e2m1x8(q) ^ kNibbleSigns;
    }
    if (b.mode == 0) return 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[2 * i] = __fdiv_rn(__uint_as_float(w[i] << 16), b.s);
        q[2 * i + 1] = __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), b.s);
    }
    return e2m1x8(q);
}

// Group of a row (row_offsets sorted; offs has groups+1 entries in smem).
__device__ __forceinline__ int find_group(const int32_t *offs, int groups, int64_t row)
{
    int lo = 0, hi = groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

constexpr int kQStages = 2;

// Scale blocks per thread per pipeline stage.  NVFP4 takes two (16 KB
// stages): the per-stage wait, release and refill are then paid once per two
// blocks; MXFP4 blocks are twice as long, one per thread fills 16 KB.
template <int FMT>
__host__ __device__ constexpr int blocks_per_thread() { return FMT == QFP4_NVFP4 ? 2 : 1; }

template <int FMT>
__host__ __device__ constexpr int chunk_bytes()
{
    return kThreads * blocks_per_thread<FMT>() * 2 * (FMT == QFP4_NVFP4 ? 16 : 32);
}

// floor(n / d) for n < 2^32 as the high half of n * m with m = floor(2^64/d) + 1
// (d >= 2): n*m/2^64 = n/d + n*(m - 2^64/d)/2^64, and the second term is below
// 2^-32 <= 1/d, less than the distance from n/d to the next integer.
__host__ __device__ constexpr uint64_t div_magic(uint64_t d) { return ~0ull / d + 1; }

// Persistent quantiser fed by bulk copies: each CTA walks 16 KB chunks of the
// flat BF16 input (rows are contiguous, and a chunk holds whole scale
// blocks), one thread keeps kQStages chunks in flight through mbarriers, and
// every thread encodes whole scale blocks from shared memory.  Consecutive
// threads take consecutive blocks, so the four scale bytes of one 32-bit word
// of the scale layout come from four neighbouring lanes.  GROUPED: per-row
// global scale gs[group] and the per-group MMA scale layout.
// ROWGS (NVFP4): row m has its own global scale gs_ptr[m] (two-level NVFP4).
template <int FMT, int SF_LAYOUT, bool GROUPED, bool ROWGS = false>
__global__ void __launch_bounds__(kQThreads, 5)
quantize_kernel(const uint8_t *__restrict__ X, int64_t total_blocks, int64_t K,
                const float *__restrict__ gs_ptr, uint8_t *__restrict__ Q,
                uint8_t *__restrict__ SF, int64_t M, int groups,
                const int32_t *__restrict__ row_offsets, uint64_t kg_magic)
{
    constexpr int G = FMT == QFP4_NVFP4 ? 16 : 32;
    constexpr int W = G / 2;                            // bf16 words per block
    constexpr int BPT = blocks_per_thread<FMT>();
    constexpr int kChunkBytes = chunk_bytes<FMT>();
    constexpr int BPC = kChunkBytes / (2 * G);          // scale blocks per chunk
    static_assert(BPC == BPT * kThreads, "chunk / thread mismatch");
    const uint32_t kg = static_cast<uint32_t>(K / G), kc = kg / 4;
    extern __shared__ __align__(128) uint8_t qsmem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(qsmem + kQStages * kChunkBytes);
    uint64_t *empty = full + kQStages;
    __shared__ int32_t s_offs[GROUPED ? kMaxGroups + 1 : 1];
    __shared__ int32_t s_tile0[GROUPED ? kMaxGroups : 1];
    // NVFP4 per-group global scales and RN(1/gs), read once per CTA
    constexpr bool GRP_GS = GROUPED && FMT == QFP4_NVFP4 && !ROWGS;
    __shared__ float s_ggs[GRP_GS ? kMaxGroups : 1];
    __shared__ float s_ginv[GRP_GS ? kMaxGroups : 1];
    pdl_wait();                 // first global access below
    pdl_launch_dependents();
    if (GROUPED) {
        for (int i = threadIdx.x; i <= groups; i += blockDim.x) s_offs[i] = row_offsets[i];
    }
    if (GRP_GS) {
        for (int i = threadIdx.x; i < groups; i += blockDim.x) {
            const float g = gs_ptr ? gs_ptr[i] : 1.0f;
            s_ggs[i] = g;
            s_ginv[i] = __frcp_rn(g);
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kThreads / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    __shared__ int s_bad;
    if (GROUPED && threadIdx.x == 0) {
        // offsets that do not cover exactly the M rows of X: nothing is
        // written (the scale buffer keeps the zeros the host wrote)
        s_bad = group_offsets_valid(s_offs, groups, M, 0) ? 0 : 1;
        if (s_bad && blockIdx.x == 0) atomicOr(&g_status_quant, static_cast<uint32_t>(kStatusBadGroup));
        int32_t acc = 0;
        for (int e = 0; e < groups; ++e) {
            s_tile0[e] = acc;
            acc += (s_offs[e + 1] - s_offs[e] + 127) / 128;
        }
    }
    __syncthreads();
    if (GROUPED && s_bad) return;
    const float gs_one = (FMT == QFP4_MXFP4 || GROUPED || ROWGS) ? 1.0f : *gs_ptr;
    const float inv_gs_one = __frcp_rn(gs_one);

    // One NVFP4 global scale for the whole tensor: the scale codes come from
    // a table.  A block's code is a non-decreasing function of its amax (the
    // roundings in t = (amax / 6) / gs and the UE4M3 encoding are monotone),
    // so s_thr[c], the least bf16 magnitude whose code is at least c (found
    // by bisection with nvfp4_scale_code itself), decides it: the estimate
    // c0 = UE4M3(amax * RN(RN(1/6) * RN(1/gs))) is within 2^-21 of t
    // relatively, while UE4M3 rounding boundaries lie at least 2^-4 apart
    // (and both saturate at 448), so c0 is at most one code off and one
    // comparison each way with s_thr[c0] and s_thr[c0 + 1] corrects it.
    // s_sy[c] holds s = decode(c) * gs and RN(1/s).  For gs in
    // [2^-100, 2^100] no factor of the estimate leaves the normal range; other
    // global scales take block_scale for every block.
    constexpr bool TABLE = FMT == QFP4_NVFP4 && !GROUPED && !ROWGS;
    __shared__ float s_thr[TABLE ? 128 : 1];
    __shared__ float2 s_sy[TABLE ? 128 : 1];
    const bool use_table = TABLE && gs_one >= 0x1p-100f && gs_one <= 0x1p100f;
    const float est_k = __fmul_rn(0x1.555556p-3f, inv_gs_one);     // RN(1/6) * RN(1/gs)

    // MMA layout without groups: zero the padding rows [M, ceil128(M)).
    if (SF_LAYOUT == QFP4_SF_MMA && !GROUPED) {
        const int64_t mp = (M + 127) / 128 * 128;
        const int64_t pad = (mp - M) * kc;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pad;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = M + i / kc, c4 = i % kc;
            *reinterpret_cast<uint32_t *>(SF + sf_mma_offset(static_cast<uint32_t>(r / 128),
                                                             static_cast<uint32_t>(r % 128),
                                                             static_cast<uint32_t>(c4 * 4), kc)) = 0u;
        }
    }

    const int64_t total_bytes = total_blocks * (2 * G);
    const int64_t nchunks = (total_bytes + kChunkBytes - 1) / kChunkBytes;
    const int lane = threadIdx.x & 31;
    bool ok = true;

    // producer: the ninth warp's lane 0 keeps kQStages chunks in flight,
    // refilling a stage as soon as the eight consumer warps have released it
    // (a consumer thread doing this would hold up its own warp every chunk)
    auto issue = [&](int64_t c, uint32_t it) {
        const uint32_t st = it % kQStages;
        const int64_t off = c * kChunkBytes;
        const int64_t rem = total_bytes - off;
        const uint32_t bytes = static_cast<uint32_t>(rem < kChunkBytes ? rem : kChunkBytes);
        mbar_arrive_expect_tx(smem_u32(&full[st]), bytes);
        bulk_load(smem_u32(qsmem + st * kChunkBytes), X + off, bytes, smem_u32(&full[st]));
    };
    if (threadIdx.x >= kThreads) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++it) {
                const uint32_t st = it % kQStages;
                // stage st was last filled for iteration it - kQStages
                if (it >= kQStages && !mbar_wait(smem_u32(&empty[st]), ((it / kQStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                issue(c, it);
            }
        }
        if (!ok) {
            atomicOr(&g_status_quant, static_cast<uint32_t>(kStatusTimeout));
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 1000000ull) { }
        }
        return;
    }
    if (TABLE && use_table) {
        // (consumer threads only: the producer warp is already streaming)
        if (threadIdx.x < 128) {
            const uint32_t c = threadIdx.x;
            float th;
            if (c == 0) {
                th = 0.0f;
            } else if (c == 127) {
                th = __uint_as_float(0x7FC00000u);             // NaN: no amax compares >= it
            } else {
                uint32_t lo = 0, hi = 0x7F80u;                 // +inf has code 126 >= c
#pragma unroll 1
                for (int i = 0; i < 16; ++i) {
                    if (lo < hi) {
                        const uint32_t mid = (lo + hi) >> 1;
                        if (nvfp4_scale_code(__uint_as_float(mid << 16), gs_one, inv_gs_one) >= c) hi = mid;
                        else lo = mid + 1;
                    }
                }
                th = __uint_as_float(lo << 16);
            }
            s_thr[c] = th;
            const float sc = __fmul_rn(ue4m3_decode(c < 127 ? c : 126u), gs_one);
            s_sy[c] = make_float2(sc, sc == 0.0f ? 0.0f : __frcp_rn(sc));
        }
        named_barrier_sync(1, kThreads);
    }
    uint32_t it = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++it) {
        const uint32_t st = it % kQStages;
        const uint32_t ph = (it / kQStages) & 1;
        if (!mbar_wait(smem_u32(&full[st]), ph)) { ok = false; break; }
        const uint8_t *chunk = qsmem + st * kChunkBytes;
        // block indices fit 32 bits (checked on the host)
        const uint32_t b0 = static_cast<uint32_t>(c * BPC);
#pragma unroll
        for (int u = 0; u < BPT; ++u) {
            const int local = u * kThreads + threadIdx.x;   // consecutive threads, consecutive blocks
            const uint32_t bu = b0 + static_cast<uint32_t>(local);
            const bool valid = bu < static_cast<uint64_t>(total_blocks);
            uint32_t w[W];
#pragma unroll
            for (int h = 0; h < W / 4; ++h) {
                const uint4 v = *reinterpret_cast<const uint4 *>(chunk + local * (2 * G) + h * 16);
                w[4 * h] = v.x; w[4 * h + 1] = v.y; w[4 * h + 2] = v.z; w[4 * h + 3] = v.w;
            }
            const float amax = block_amax(w);
            const uint32_t row = static_cast<uint32_t>(__umul64hi(bu, kg_magic));
            int grp = 0;
            float gs = gs_one, inv_gs = inv_gs_one;
            if (GROUPED && valid) {
                grp = find_group(s_offs, groups, row);
                if (GRP_GS) {
                    gs = s_ggs[grp];
                    inv_gs = s_ginv[grp];
                }
            }
            if (ROWGS && FMT != QFP4_MXFP4 && valid) {
                gs = gs_ptr[row];
                inv_gs = __frcp_rn(gs);
            }
            BlockScale bs;
            if (TABLE && use_table) {
                const float x = __fmul_rn(amax, est_k);
                const uint32_t c0 = x > 0.0f ? ue4m3_encode(x) : 0u;        // 0..126 (NaN: 0)
                const uint32_t code = c0 + (amax >= s_thr[c0 + 1] ? 1u : 0u) - (amax < s_thr[c0] ? 1u : 0u);
                const float2 sy = s_sy[code];
                bs = nvfp4_block(code, sy.x, sy.y, amax);
            } else {
                bs = block_scale<FMT>(amax, gs, inv_gs);
            }
            uint32_t packed[W / 4];
#pragma unroll
            for (int v = 0; v < W / 4; ++v) packed[v] = encode8<FMT>(&w[4 * v], bs);
            if (valid) {
                if (G == 16) *reinterpret_cast<uint2 *>(Q + static_cast<size_t>(bu) * (G / 2)) = make_uint2(packed[0], packed[1]);
                else *reinterpret_cast<uint4 *>(Q + static_cast<size_t>(bu) * (G / 2)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
            // Scale bytes: lanes 4i..4i+3 hold four consecutive blocks of one
            // row, whose bytes are adjacent in both layouts.  NVFP4 stores one
            // byte per lane (the four stores of a word go out in one warp
            // instruction); MXFP4, with half as many blocks, gathers each word
            // into its first lane (measured faster there).
            const uint32_t c1 = FMT == QFP4_NVFP4 ? 0u : __shfl_down_sync(0xffffffffu, bs.code, 1);
            const uint32_t c2 = FMT == QFP4_NVFP4 ? 0u : __shfl_down_sync(0xffffffffu, bs.code, 2);
            const uint32_t c3 = FMT == QFP4_NVFP4 ? 0u : __shfl_down_sync(0xffffffffu, bs.code, 3);
            if (valid && (FMT == QFP4_NVFP4 || (lane & 3) == 0)) {
                const uint32_t col = bu - row * kg;
                size_t off;
                if (GROUPED) {
                    const uint32_t rr = row - static_cast<uint32_t>(s_offs[grp]);
                    off = sf_mma_offset(static_cast<uint32_t>(s_tile0[grp]) + rr / 128, rr % 128, col, kc);
                } else if (SF_LAYOUT == QFP4_SF_MMA) {
                    off = sf_mma_offset(row / 128, row % 128, col, kc);
                } else {
                    off = bu;
                }
                if (FMT == QFP4_NVFP4) SF[off] = static_cast<uint8_t>(bs.code);
                else *reinterpret_cast<uint32_t *>(SF + off) = bs.code | (c1 << 8) | (c2 << 16) | (c3 << 24);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    if (!ok) atomicOr(&g_status_quant, static_cast<uint32_t>(kStatusTimeout));
    // no bulk copy may be left in flight: every issued chunk was consumed,
    // or (after a timeout) give outstanding copies time to land
    if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) { }
    }
}

// Per-expert amax (the grouped global scales): one warp per row, each row's
// maximum folded into its group's word with atomicMax on the bit pattern
// (non-negative floats order like unsigned integers); a warp keeps a running
// maximum while its rows stay in one group.  One tensor uses amax_flat_kernel.
// rows < 0: the row count is row_offsets[groups], read on the device.
// The group words are those of a reduction slot (groups words, then the
// count of CTAs that have added to them): the CTA that arrives last writes
// gs_out[e] = amax / (6 * 448), 0 for every group when the offsets are bad,
// and puts the slot back to zero.
__global__ void __launch_bounds__(kThreads)
amax_rows_kernel(const uint4 *__restrict__ X, int64_t rows, int64_t chunks_per_row, int groups,
                 const int32_t *__restrict__ row_offsets, uint32_t *__restrict__ amax_bits,
                 float *__restrict__ gs_out)
{
    __shared__ int32_t s_offs[kMaxGroups + 1];
    __shared__ int s_last;
    pdl_wait();
    pdl_launch_dependents();
    __shared__ int s_bad;
    for (int i = threadIdx.x; i <= groups; i += blockDim.x) s_offs[i] = row_offsets[i];
    __syncthreads();
    if (rows < 0) rows = s_offs[groups];
    if (threadIdx.x == 0) {
        s_bad = group_offsets_valid(s_offs, groups, rows, 0) ? 0 : 1;
        if (s_bad && blockIdx.x == 0) atomicOr(&g_status_quant, static_cast<uint32_t>(kStatusBadGroup));
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int cur = -1;
    float run = 0.0f;
    for (int64_t r = s_bad ? rows : warp; r < rows; r += nwarps) {
        const uint4 *p = X + r * chunks_per_row;
        float m = 0.0f;
        int64_t i = lane;
        for (; i + 96 < chunks_per_row; i += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = ld_stream_v4(p + i + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float lo, hi;
                    bf16x2_to_f32(w[j], lo, hi);
                    m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
                }
            }
        }
        for (; i < chunks_per_row; i += 32) {
            const uint4 v = ld_stream_v4(p + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                bf16x2_to_f32(w[j], lo, hi);
                m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int g = find_group(s_offs, groups, r);
        if (g != cur) {
            if (cur >= 0 && lane == 0) atomicMax(amax_bits + cur, __float_as_uint(run));
            cur = g;
            run = 0.0f;
        }
        run = fmaxf(run, m);
    }
    if (cur >= 0 && lane == 0) atomicMax(amax_bits + cur, __float_as_uint(run));
    if (lane == 0) __threadfence();
    __syncthreads();
    uint32_t *count = amax_bits + groups;
    if (threadIdx.x == 0) s_last = atomicAdd(count, 1u) == gridDim.x - 1 ? 1 : 0;
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int e = threadIdx.x; e < groups; e += blockDim.x) {
            const uint32_t bits = atomicExch(amax_bits + e, 0u);
            gs_out[e] = s_bad ? 0.0f : __fdiv_rn(__uint_as_float(bits), 2688.0f);
        }
        if (threadIdx.x == 0) *count = 0u;
    }
}

// Reduction slots of the one-tensor global scale: per slot the running amax
// bit pattern and the count of CTAs that have added to it.  Zero when the
// module loads; every launch leaves its slot at zero again, so a slot can be
// reused by the next launch that draws it.  The host hands the slots out in
// turn, so that launches in flight at the same time (on other streams) use
// different ones as long as fewer than kGsSlots are in flight.
constexpr int kGsSlots = 1024;
__device__ uint32_t g_gs_slots[2 * kGsSlots];
// The same for the per-group form: kMaxGroups group words and a count per slot.
constexpr int kGsGroupSlots = 64;
__device__ uint32_t g_gs_group_slots[kGsGroupSlots * (kMaxGroups + 1)];

// gs = amax(X) / (6 * 448) for all of X (one group), in one launch: the rows
// are contiguous, so X is walked as one flat array of 16-byte vectors, eight
// loads in flight per thread per round (one or two rounds of memory latency
// for a 32 MB tensor instead of one per 2 KB of a row).  Each CTA folds its
// maximum into the slot with one atomic and then counts itself in; the CTA
// that arrives last (all maxima are in by then) divides, writes gs_out and
// puts the slot back to zero.
constexpr int kAmaxUnroll = 8;
__global__ void __launch_bounds__(kThreads)
amax_flat_kernel(const uint4 *__restrict__ X, int64_t nvec, uint32_t *__restrict__ slot, float *__restrict__ gs_out)
{
    __shared__ float s_warp[kThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    float m = 0.0f;
    for (int64_t base = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; base < nvec;
         base += kAmaxUnroll * stride) {
        uint4 v[kAmaxUnroll];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) {
            const int64_t i = base + u * stride;
            v[u] = i < nvec ? ld_stream_v4(X + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                bf16x2_to_f32(w[j], lo, hi);
                m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float cm = 0.0f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) cm = fmaxf(cm, s_warp[w]);
        // non-negative floats order like their bit patterns
        if (cm != 0.0f) atomicMax(slot, __float_as_uint(cm));
        __threadfence();
        if (atomicAdd(slot + 1, 1u) == gridDim.x - 1) {
            __threadfence();
            const uint32_t bits = atomicExch(slot, 0u);
            slot[1] = 0u;
            *gs_out = __fdiv_rn(__uint_as_float(bits), 2688.0f);
        }
    }
}

// Per-row global scales (two-level NVFP4): one warp per row, gs[r] =
// amax(row r) / (6 * 448), written directly (no atomics, no zeroing).
__global__ void __launch_bounds__(kThreads)
gs_rows_kernel(const uint4 *__restrict__ X, int64_t rows, int64_t chunks_per_row, float *__restrict__ gs_out)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const uint4 *p = X + r * chunks_per_row;
        float m = 0.0f;
        int64_t i = lane;
        for (; i + 96 < chunks_per_row; i += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = ld_stream_v4(p + i + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float lo, hi;
                    bf16x2_to_f32(w[j], lo, hi);
                    m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
                }
            }
        }
        for (; i < chunks_per_row; i += 32) {
            const uint4 v = ld_stream_v4(p + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                bf16x2_to_f32(w[j], lo, hi);
                m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) gs_out[r] = __fdiv_rn(m, 2688.0f);
    }
}

// Scale-factor interleave; one thread per 4-byte word of the MMA layout.
template <bool TO_MMA>
__global__ void __launch_bounds__(kThreads)
sf_interleave_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int64_t rows,
                     int64_t cols, int64_t kc, int64_t words)
{
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < words;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = w >> 7, within = w & 127;
        const int64_t i = within >> 2, j = within & 3;
        const int64_t r = (tile / kc) * 128 + j * 32 + i;
        const int64_t c0 = (tile % kc) * 4;
        if (TO_MMA) {
            uint32_t word = 0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int64_t c = c0 + kk;
                if (r < rows && c < cols) word |= static_cast<uint32_t>(in[r * cols + c]) << (8 * kk);
            }
            reinterpret_cast<uint32_t *>(out)[w] = word;
        } else {
            const uint32_t word = reinterpret_cast<const uint32_t *>(in)[w];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int64_t c = c0 + kk;
                if (r < rows && c < cols) out[r * cols + c] = static_cast<uint8_t>(word >> (8 * kk));
            }
        }
    }
}

// Row-major scale bytes [rows, cols] -> MMA layout when cols % 16 == 0 and
// both buffers are 16-byte aligned.  CTA b takes rows [128 R, 128 R + 128)
// and columns [32 C, 32 C + w) (w = 32, or 16 for the last chunk of a row
// whose cols is an odd multiple of 16): w / 4 atoms that lie next to each
// other in the MMA layout.  Thread t reads its row's w bytes (whole 32-byte
// sectors), puts word q (columns 4q .. 4q + 3 of the chunk) into atom q at
// word (t % 32) 4 + t / 32, and the CTA writes the atoms as one contiguous
// run.  Rows past `rows` are the layout's zero padding.
__global__ void __launch_bounds__(128)
sf_to_mma_tiled_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int64_t rows, int64_t cols,
                       int64_t kc, int64_t chunks_per_row)
{
    __shared__ __align__(16) uint32_t atoms[8 * 128];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t R = blockIdx.x / chunks_per_row, C = blockIdx.x % chunks_per_row;
    const int t = threadIdx.x;
    const int64_t c0 = 32 * C;
    const int w = cols - c0 >= 32 ? 32 : 16;
    const int64_t r = 128 * R + t;
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + r * cols + c0);
        v0 = src[0];
        if (w == 32) v1 = src[1];
    }
    const int pos = (t & 31) * 4 + (t >> 5);
    atoms[0 * 128 + pos] = v0.x;
    atoms[1 * 128 + pos] = v0.y;
    atoms[2 * 128 + pos] = v0.z;
    atoms[3 * 128 + pos] = v0.w;
    if (w == 32) {
        atoms[4 * 128 + pos] = v1.x;
        atoms[5 * 128 + pos] = v1.y;
        atoms[6 * 128 + pos] = v1.z;
        atoms[7 * 128 + pos] = v1.w;
    }
    __syncthreads();
    uint4 *dst = reinterpret_cast<uint4 *>(out + (R * kc + 8 * C) * 512);
    const uint4 *srcs = reinterpret_cast<const uint4 *>(atoms);
    dst[t] = srcs[t];
    if (w == 32) dst[t + 128] = srcs[t + 128];
}

// The inverse, MMA layout -> row-major scale bytes, under the same
// conditions: CTA b reads the w / 4 adjacent atoms of rows [128 R, 128 R +
// 128) and columns [32 C, 32 C + w) as one contiguous run into shared
// memory, and thread t writes its row's w bytes (whole 32-byte sectors);
// the layout's padding rows are not written.
__global__ void __launch_bounds__(128)
sf_from_mma_tiled_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int64_t rows,
                         int64_t cols, int64_t kc, int64_t chunks_per_row)
{
    __shared__ __align__(16) uint32_t atoms[8 * 128];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t R = blockIdx.x / chunks_per_row, C = blockIdx.x % chunks_per_row;
    const int t = threadIdx.x;
    const int64_t c0 = 32 * C;
    const int w = cols - c0 >= 32 ? 32 : 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(in + (R * kc + 8 * C) * 512);
    uint4 *stage = reinterpret_cast<uint4 *>(atoms);
    stage[t] = src[t];
    if (w == 32) stage[t + 128] = src[t + 128];
    __syncthreads();
    const int64_t r = 128 * R + t;
    if (r < rows) {
        const int pos = (t & 31) * 4 + (t >> 5);
        uint4 *dst = reinterpret_cast<uint4 *>(out + r * cols + c0);
        dst[0] = make_uint4(atoms[0 * 128 + pos], atoms[1 * 128 + pos], atoms[2 * 128 + pos], atoms[3 * 128 + pos]);
        if (w == 32)
            dst[1] = make_uint4(atoms[4 * 128 + pos], atoms[5 * 128 + pos], atoms[6 * 128 + pos],
                                atoms[7 * 128 + pos]);
    }
}

int grid_for(int64_t work_items, int per_block)
{
    const int sms = sm_count();
    const int64_t want = (work_items + per_block - 1) / per_block;
    int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
    int64_t g = want < cap ? want : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

template <int FMT, int LAYOUT, bool GROUPED, bool ROWGS = false>
cudaError_t launch_quantize(const void *X, int64_t M, int64_t K, const float *gs, void *Q,
                            void *SF, int groups, const int32_t *offs, cudaStream_t s)
{
    constexpr int G = FMT == QFP4_NVFP4 ? 16 : 32;
    const int64_t blocks = M * (K / G);
    constexpr int kChunkBytes = chunk_bytes<FMT>();
    const int64_t chunks = (blocks * 2 * G + kChunkBytes - 1) / kChunkBytes;
    constexpr int smem = kQStages * kChunkBytes + 2 * kQStages * 8;
    auto kern = quantize_kernel<FMT, LAYOUT, GROUPED, ROWGS>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), smem) != QFP4_OK) return cudaErrorUnknown;
    const int sms = sm_count();
    // five CTAs (40 consumer warps) per SM with a two-stage ring each: the
    // per-block scale arithmetic is a dependent chain, and more warps hide
    // it better than deeper rings (measured against 3 x 4, 4 x 3, 4 x 5)
    int64_t grid = static_cast<int64_t>(sms > 0 ? sms : 148) * 5;
    if (chunks < grid) grid = chunks > 0 ? chunks : 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kQThreads), smem, s,
                      static_cast<const uint8_t *>(X), blocks, K, gs, static_cast<uint8_t *>(Q),
                      static_cast<uint8_t *>(SF), M, groups, offs, div_magic(static_cast<uint64_t>(K / G)));
}

}  // namespace
}  // namespace qfp4

using namespace qfp4;

extern "C" int qfp4_block_size(int fmt) { return block_elems(fmt); }

extern "C" size_t qfp4_sf_mma_bytes(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols < 0) return 0;
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((cols + 3) / 4) * 512u;
}

extern "C" size_t qfp4_sf_mma_grouped_bytes(int64_t total_rows, int64_t groups, int64_t cols)
{
    if (total_rows < 0 || groups < 0 || cols < 0) return 0;
    return static_cast<size_t>((total_rows + 127) / 128 + groups) *
           static_cast<size_t>((cols + 3) / 4) * 512u;
}

// Device addresses of the slot pools on the current device (looked up once
// per device): pool 0 one tensor, pool 1 per group.
static uint32_t *gs_slot_pool(int which)
{
    static std::mutex mu;
    static uint32_t *cached[2][64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[which][dev]) {
        void *p = nullptr;
        if ((which == 0 ? cudaGetSymbolAddress(&p, g_gs_slots) : cudaGetSymbolAddress(&p, g_gs_group_slots)) !=
            cudaSuccess)
            return nullptr;
        cached[which][dev] = static_cast<uint32_t *>(p);
    }
    return cached[which][dev];
}

// The next per-group slot (handed out in turn).
static uint32_t *gs_group_slot()
{
    uint32_t *pool = gs_slot_pool(1);
    if (!pool) return nullptr;
    static std::atomic<uint32_t> next_slot{0};
    return pool + (next_slot.fetch_add(1u, std::memory_order_relaxed) % kGsGroupSlots) * (kMaxGroups + 1);
}

extern "C" int qfp4_global_scale(const void *X_bf16, int64_t rows, int64_t cols, float *gs_out,
                                 void *stream)
{
    // X may be NULL when it is empty (nothing is read; gs = 0 is written)
    if (!gs_out || rows < 0 || cols < 0 || (!X_bf16 && rows > 0 && cols > 0)) return QFP4_ERR_INVALID_ARG;
    if (cols % 8 != 0) return QFP4_ERR_UNSUPPORTED;
    if (!aligned16(X_bf16) || !aligned4(gs_out)) return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *slots = gs_slot_pool(0);
    if (!slots) return QFP4_ERR_CUDA;
    static std::atomic<uint32_t> next_slot{0};
    uint32_t *slot = slots + 2 * (next_slot.fetch_add(1u, std::memory_order_relaxed) % kGsSlots);
    const int64_t nvec = rows * (cols / 8);
    const int sms = sm_count();
    int64_t grid = static_cast<int64_t>(sms > 0 ? sms : 148) * 6;
    const int64_t want = (nvec + kThreads - 1) / kThreads;
    if (want < grid) grid = want;
    if (grid < 1) grid = 1;                 // an empty X still writes gs = 0
    return launch_status(launch_pdl(amax_flat_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                                    static_cast<const uint4 *>(X_bf16), nvec, slot, gs_out));
}

extern "C" int qfp4_global_scale_grouped(const void *X_bf16, int64_t total_rows, int64_t cols,
                                         int64_t groups, const int32_t *row_offsets,
                                         float *gs_out, void *stream)
{
    if (!X_bf16 || !gs_out || !row_offsets || total_rows < 0 || cols < 0 || groups < 1)
        return QFP4_ERR_INVALID_ARG;
    if (groups > kMaxGroups || cols % 8 != 0) return QFP4_ERR_UNSUPPORTED;
    if (!aligned16(X_bf16) || !aligned4(gs_out) || !aligned4(row_offsets))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *slot = gs_group_slot();
    if (!slot) return QFP4_ERR_CUDA;
    // one launch; an empty X still runs one CTA, which writes gs = 0
    const int grid = total_rows > 0 && cols > 0 ? grid_for(total_rows, kThreads / 32) : 1;
    return launch_status(launch_pdl(amax_rows_kernel, dim3(grid), dim3(kThreads), 0, s,
                                    static_cast<const uint4 *>(X_bf16), total_rows,
                                    cols / 8, static_cast<int>(groups), row_offsets, slot, gs_out));
}

extern "C" int qfp4_absmax_gs(int64_t groups, const int32_t *row_offsets, const void *X_bf16, int64_t K,
                              float *gs_out, void *stream)
{
    if (!X_bf16 || !gs_out || !row_offsets || K < 0 || groups < 1) return QFP4_ERR_INVALID_ARG;
    if (groups > kMaxGroups || K % 8 != 0) return QFP4_ERR_UNSUPPORTED;
    if (!aligned16(X_bf16) || !aligned4(gs_out) || !aligned4(row_offsets)) return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *slot = gs_group_slot();
    if (!slot) return QFP4_ERR_CUDA;
    // the row count lives on the device: a full grid of row-walking warps
    // (K = 0: one CTA, which walks the rows without reading and writes gs = 0)
    const int sms = sm_count();
    const int grid = K > 0 ? (sms > 0 ? sms : 148) * 8 : 1;
    return launch_status(launch_pdl(amax_rows_kernel, dim3(grid), dim3(kThreads), 0, s,
                                    static_cast<const uint4 *>(X_bf16), int64_t{-1}, K / 8,
                                    static_cast<int>(groups), row_offsets, slot, gs_out));
}

extern "C" int qfp4_global_scale_rows(const void *X_bf16, int64_t rows, int64_t cols, float *gs_out,
                                      void *stream)
{
    if (rows < 0 || cols < 0) return QFP4_ERR_INVALID_ARG;
    if (cols % 8 != 0) return QFP4_ERR_UNSUPPORTED;
    if (rows == 0) return QFP4_OK;
    if (!gs_out) return QFP4_ERR_INVALID_ARG;
    if (!aligned4(gs_out)) return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0)      // empty rows: amax 0, gs 0
        return cudaMemsetAsync(gs_out, 0, sizeof(float) * rows, s) == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
    if (!X_bf16) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16)) return QFP4_ERR_MISALIGNED;
    const int grid = grid_for(rows, kThreads / 32);
    return launch_status(launch_pdl(gs_rows_kernel, dim3(grid), dim3(kThreads), 0, s,
                                    static_cast<const uint4 *>(X_bf16), rows, cols / 8, gs_out));
}

extern "C" int qfp4_quantize_rows(int fmt, const void *X_bf16, int64_t M, int64_t K, const float *gs_rows,
                                  void *Q_packed, void *SF, int sf_layout, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4 && fmt != QFP4_NVFP4_B32) return QFP4_ERR_INVALID_ARG;
    if (sf_layout != QFP4_SF_ROWMAJOR && sf_layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (K % 128 != 0) return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return QFP4_OK;
    if ((M + 128) * (K / 16) >= (int64_t{1} << 32) - 4096) return QFP4_ERR_UNSUPPORTED;
    if (!X_bf16 || !Q_packed || !SF) return QFP4_ERR_INVALID_ARG;
    if (fmt != QFP4_MXFP4 && !gs_rows) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || !aligned16(Q_packed) || !aligned4(SF) || (gs_rows && !aligned4(gs_rows)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fmt == QFP4_NVFP4_B32)
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_NVFP4_B32, QFP4_SF_MMA, false, true>(X_bf16, M, K, gs_rows, Q_packed, SF, 1,
                                                                            nullptr, s)
                : launch_quantize<QFP4_NVFP4_B32, QFP4_SF_ROWMAJOR, false, true>(X_bf16, M, K, gs_rows, Q_packed,
                                                                                 SF, 1, nullptr, s);
    else if (fmt == QFP4_MXFP4)   // MXFP4 has no global scale: the plain quantiser
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_MXFP4, QFP4_SF_MMA, false>(X_bf16, M, K, nullptr, Q_packed, SF, 1, nullptr, s)
                : launch_quantize<QFP4_MXFP4, QFP4_SF_ROWMAJOR, false>(X_bf16, M, K, nullptr, Q_packed, SF, 1,
                                                                       nullptr, s);
    else
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_NVFP4, QFP4_SF_MMA, false, true>(X_bf16, M, K, gs_rows, Q_packed, SF, 1,
                                                                        nullptr, s)
                : launch_quantize<QFP4_NVFP4, QFP4_SF_ROWMAJOR, false, true>(X_bf16, M, K, gs_rows, Q_packed, SF,
                                                                             1, nullptr, s);
    return launch_status(e);
}

extern "C" int qfp4_quantize(int fmt, const void *X_bf16, int64_t M, int64_t K, const float *gs,
                             void *Q_packed, void *SF, int sf_layout, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4 && fmt != QFP4_NVFP4_B32) return QFP4_ERR_INVALID_ARG;
    if (sf_layout != QFP4_SF_ROWMAJOR && sf_layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (K % 128 != 0) return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return QFP4_OK;
    // 32-bit block indices and scale offsets, with room for the last chunk
    // and the padded scale rows
    if ((M + 128) * (K / 16) >= (int64_t{1} << 32) - 4096) return QFP4_ERR_UNSUPPORTED;
    if (!X_bf16 || !Q_packed || !SF) return QFP4_ERR_INVALID_ARG;
    if (fmt != QFP4_MXFP4 && !gs) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || !aligned16(Q_packed) || !aligned4(SF) || (gs && !aligned4(gs)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fmt == QFP4_MXFP4)
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_MXFP4, QFP4_SF_MMA, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s)
                : launch_quantize<QFP4_MXFP4, QFP4_SF_ROWMAJOR, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s);
    else if (fmt == QFP4_NVFP4_B32)
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_NVFP4_B32, QFP4_SF_MMA, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s)
                : launch_quantize<QFP4_NVFP4_B32, QFP4_SF_ROWMAJOR, false>(X_bf16, M, K, gs, Q_packed, SF, 1,
                                                                          nullptr, s);
    else
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_NVFP4, QFP4_SF_MMA, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s)
                : launch_quantize<QFP4_NVFP4, QFP4_SF_ROWMAJOR, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s);
    return launch_status(e);
}

extern "C" int qfp4_quantize_grouped(int fmt, const void *X_bf16, int64_t total_rows, int64_t K,
                                     int64_t groups, const int32_t *row_offsets, const float *gs,
                                     void *Q_packed, void *SF_mma, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (total_rows < 0 || K < 0 || groups < 1 || !row_offsets) return QFP4_ERR_INVALID_ARG;
    if (groups > kMaxGroups || K % 128 != 0) return QFP4_ERR_UNSUPPORTED;
    if ((total_rows + 128 * (groups + 1)) * (K / 16) >= (int64_t{1} << 32) - 4096) return QFP4_ERR_UNSUPPORTED;
    if (fmt == QFP4_NVFP4 && !gs) return QFP4_ERR_INVALID_ARG;
    if (!X_bf16 || !Q_packed || !SF_mma) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || !aligned16(Q_packed) || !aligned4(SF_mma) || !aligned4(row_offsets) ||
        (gs && !aligned4(gs)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sf_bytes = qfp4_sf_mma_grouped_bytes(total_rows, groups, K / block_elems(fmt));
    if (cudaMemsetAsync(SF_mma, 0, sf_bytes, s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (total_rows == 0 || K == 0) return QFP4_OK;
    const int g = static_cast<int>(groups);
    cudaError_t e = fmt == QFP4_MXFP4
        ? launch_quantize<QFP4_MXFP4, QFP4_SF_MMA, true>(X_bf16, total_rows, K, gs, Q_packed, SF_mma, g, row_offsets, s)
        : launch_quantize<QFP4_NVFP4, QFP4_SF_MMA, true>(X_bf16, total_rows, K, gs, Q_packed, SF_mma, g, row_offsets, s);
    return launch_status(e);
}

extern "C" int qfp4_quantize_grouped_rows(int fmt, const void *X_bf16, int64_t total_rows, int64_t K,
                                          int64_t groups, const int32_t *row_offsets, const float *gs_rows,
                                          void *Q_packed, void *SF_mma, void *stream)
{
    if (fmt == QFP4_MXFP4)        // MXFP4 has no global scale: the plain grouped quantiser
        return qfp4_quantize_grouped(fmt, X_bf16, total_rows, K, groups, row_offsets, nullptr, Q_packed, SF_mma,
                                     stream);
    if (fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (total_rows < 0 || K < 0 || groups < 1 || !row_offsets) return QFP4_ERR_INVALID_ARG;
    if (groups > kMaxGroups || K % 128 != 0) return QFP4_ERR_UNSUPPORTED;
    if ((total_rows + 128 * (groups + 1)) * (K / 16) >= (int64_t{1} << 32) - 4096) return QFP4_ERR_UNSUPPORTED;
    if (!gs_rows || !X_bf16 || !Q_packed || !SF_mma) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || !aligned16(Q_packed) || !aligned4(SF_mma) || !aligned4(row_offsets) ||
        !aligned4(gs_rows))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sf_bytes = qfp4_sf_mma_grouped_bytes(total_rows, groups, K / 16);
    if (cudaMemsetAsync(SF_mma, 0, sf_bytes, s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (total_rows == 0 || K == 0) return QFP4_OK;
    return launch_status(launch_quantize<QFP4_NVFP4, QFP4_SF_MMA, true, true>(
        X_bf16, total_rows, K, gs_rows, Q_packed, SF_mma, static_cast<int>(groups), row_offsets, s));
}

extern "C" int qfp4_sf_interleave(const void *SF_in, int64_t rows, int64_t cols, void *SF_out,
                                  int layout, void *stream)
{
    if (layout != QFP4_SF_ROWMAJOR && layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return QFP4_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return QFP4_OK;
    if (!SF_in || !SF_out) return QFP4_ERR_INVALID_ARG;
    const void *mma_side = layout == QFP4_SF_MMA ? SF_out : SF_in;
    if (!aligned4(mma_side)) return QFP4_ERR_MISALIGNED;
    const int64_t kc = (cols + 3) / 4;
    const int64_t words = ((rows + 127) / 128) * kc * 128;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols % 16 == 0 && aligned16(SF_in) && aligned16(SF_out)) {
        const int64_t chunks_per_row = (cols + 31) / 32;
        const int64_t blocks = ((rows + 127) / 128) * chunks_per_row;
        if (blocks <= INT32_MAX)
            return launch_status(launch_pdl(layout == QFP4_SF_MMA ? sf_to_mma_tiled_kernel : sf_from_mma_tiled_kernel,
                                            dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s,
                                            static_cast<const uint8_t *>(SF_in), static_cast<uint8_t *>(SF_out),
                                            rows, cols, kc, chunks_per_row));
    }
    const int grid = grid_for(words, kThreads);
    if (layout == QFP4_SF_MMA)
        return launch_status(launch_pdl(sf_interleave_kernel<true>, dim3(grid), dim3(kThreads), 0, s,
                                        static_cast<const uint8_t *>(SF_in), static_cast<uint8_t *>(SF_out), rows,
                                        cols, kc, words));
    return launch_status(launch_pdl(sf_interleave_kernel<false>, dim3(grid), dim3(kThreads), 0, s,
                                    static_cast<const uint8_t *>(SF_in), static_cast<uint8_t *>(SF_out), rows, cols,
                                    kc, words));
}
