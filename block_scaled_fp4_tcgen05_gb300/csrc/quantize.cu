// quantize.cu -- BF16 -> NVFP4 / MXFP4 quantiser, global scale and the
// scale-factor interleave (HBM-bound kernels, no tensor cores).
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
#include <cstdint>
#include <cuda_runtime.h>

#include "qfp4_common.cuh"

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

// UE4M3 scale byte of t >= 0: round to nearest even, saturate at 448 (0x7E).
__device__ __forceinline__ uint32_t ue4m3_encode(float t)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return static_cast<uint32_t>(r) & 0xFFu;
}

// Value of a UE4M3 byte (0x00..0x7E) as fp32, exact.
__device__ __forceinline__ float ue4m3_decode(uint32_t b)
{
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    return e == 0 ? static_cast<float>(m) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// UE8M0 code of t >= 0: nearest power of two 2^(c-127), ties (1.5 * 2^e) to
// the even code, clamped to [0, 254]; t = 0 gives 0 (the format has no zero).
__device__ __forceinline__ uint32_t ue8m0_encode(float t)
{
    const uint32_t bits = __float_as_uint(t);
    const uint32_t E = bits >> 23, F = bits & 0x7FFFFFu;
    if (E == 0) return F > 0x600000u ? 1u : 0u;   // subnormal: between 2^-127 and 2^-126
    const uint32_t up = (F > 0x400000u) || (F == 0x400000u && (E & 1u));
    const uint32_t c = E + up;
    return c > 254u ? 254u : c;
}

// 2^(127 - c) as fp32 (exact; subnormal for c = 254).
__device__ __forceinline__ float ue8m0_inverse(uint32_t c)
{
    const int e = 127 - static_cast<int>(c);                 // -127 .. 127
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                     : __uint_as_float(0x00400000u);          // 2^-127
}

// Two fp32 -> packed E2M1 byte (first argument in the high nibble), round to
// nearest even, saturating at +-6, sign kept.
__device__ __forceinline__ uint32_t e2m1x2(float hi, float lo)
{
    uint32_t r;
    asm("{\n.reg .b8 t;\ncvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\ncvt.u32.u8 %0, t;\n}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

struct BlockScale {
    float inv;      // MXFP4: exact 2^-e; NVFP4: RN(1/s)
    float s;        // NVFP4 scale s = decode(sf) * gs
    uint32_t code;  // scale byte
    int mode;       // 0: zero block, 1: fast path, 2: IEEE division
};

template <int FMT>
__device__ __forceinline__ BlockScale block_scale(float amax, float gs)
{
    BlockScale b;
    if (FMT == QFP4_MXFP4) {
        const float t = __fdiv_rn(amax, 6.0f);
        b.code = ue8m0_encode(t);
        b.inv = ue8m0_inverse(b.code);
        b.s = 0.0f;
        b.mode = 1;
    } else {
        const float t = __fdiv_rn(__fdiv_rn(amax, 6.0f), gs);
        b.code = ue4m3_encode(t);
        b.s = __fmul_rn(ue4m3_decode(b.code), gs);
        if (b.s == 0.0f) {
            b.mode = 0;
            b.inv = 0.0f;
        } else {
            b.inv = __frcp_rn(b.s);
            const bool fast = b.s >= 0x1p-64f && b.s <= 0x1p64f && amax <= b.s * 0x1p60f;
            b.mode = fast ? 1 : 2;
        }
    }
    return b;
}

template <int FMT>
__device__ __forceinline__ float quotient(float x, const BlockScale &b)
{
    if (FMT == QFP4_MXFP4) return x * b.inv;
    if (b.mode == 1) {
        float q = __fmul_rn(x, b.inv);
        q = __fmaf_rn(__fmaf_rn(-b.s, q, x), b.inv, q);
        q = __fmaf_rn(__fmaf_rn(-b.s, q, x), b.inv, q);
        return copysignf(q, x);
    }
    return __fdiv_rn(x, b.s);
}

// 8 consecutive elements -> 4 packed bytes.
template <int FMT>
__device__ __forceinline__ uint32_t encode8(const float (&x)[8], const BlockScale &b)
{
    if (FMT == QFP4_NVFP4 && b.mode == 0) return 0u;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float q0 = quotient<FMT>(x[2 * i], b);
        const float q1 = quotient<FMT>(x[2 * i + 1], b);
        w |= e2m1x2(q1, q0) << (8 * i);
    }
    return w;
}

__device__ __forceinline__ int64_t sf_mma_offset(int64_t row_tile, int64_t r_in_tile, int64_t c,
                                                 int64_t kc)
{
    return (row_tile * kc + (c >> 2)) * 512 + (r_in_tile & 31) * 16 + (r_in_tile >> 5) * 4 +
           (c & 3);
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

// One pass over X in chunks of 8 elements (16 bytes); TPB = g/8 consecutive
// lanes share one scale block.  GROUPED: per-row global scale gs[group] and
// SF written in the per-group MMA layout.
template <int FMT, int SF_LAYOUT, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const uint4 *__restrict__ X, int64_t total_chunks, int64_t K,
                const float *__restrict__ gs_ptr, uint32_t *__restrict__ Q,
                uint8_t *__restrict__ SF, int64_t M, int groups,
                const int32_t *__restrict__ row_offsets)
{
    constexpr int G = FMT == QFP4_MXFP4 ? 32 : 16;
    constexpr int TPB = G / 8;
    constexpr int U = 4;
    const int64_t kg = K / G, kc = kg / 4;
    const int64_t chunks_per_row = K / 8;
    __shared__ int32_t s_offs[GROUPED ? kMaxGroups + 1 : 1];
    __shared__ int32_t s_tile0[GROUPED ? kMaxGroups : 1];
    if (GROUPED) {
        for (int i = threadIdx.x; i <= groups; i += blockDim.x) s_offs[i] = row_offsets[i];
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int e = 0; e < groups; ++e) {
                s_tile0[e] = acc;
                acc += (s_offs[e + 1] - s_offs[e] + 127) / 128;
            }
        }
        __syncthreads();
    }
    const float gs_one = (FMT == QFP4_MXFP4 || GROUPED) ? 1.0f : *gs_ptr;

    // MMA layout without groups: zero the padding rows [M, ceil128(M)).
    if (SF_LAYOUT == QFP4_SF_MMA && !GROUPED) {
        const int64_t mp = (M + 127) / 128 * 128;
        const int64_t pad = (mp - M) * kc;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pad;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t r = M + i / kc, c4 = i % kc;
            *reinterpret_cast<uint32_t *>(SF + sf_mma_offset(r / 128, r % 128, c4 * 4, kc)) = 0u;
        }
    }

    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    // Loop bounds are warp-uniform so that every lane joins the shuffles.
    const int64_t warp_first = first - lane;
    for (int64_t base = warp_first; base < total_chunks; base += stride * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = base + u * stride + lane;
            v[u] = c < total_chunks ? ld_stream_v4(X + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = base + u * stride + lane;
            const bool valid = c < total_chunks;
            float x[8];
            bf16x2_to_f32(v[u].x, x[0], x[1]);
            bf16x2_to_f32(v[u].y, x[2], x[3]);
            bf16x2_to_f32(v[u].z, x[4], x[5]);
            bf16x2_to_f32(v[u].w, x[6], x[7]);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            if (TPB == 4) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));

            const int64_t row = c / chunks_per_row;
            int grp = 0;
            float gs = gs_one;
            if (GROUPED && valid) {
                grp = find_group(s_offs, groups, row);
                gs = gs_ptr ? gs_ptr[grp] : 1.0f;
                if (FMT == QFP4_MXFP4) gs = 1.0f;
            }
            const BlockScale b = block_scale<FMT>(amax, gs);
            const uint32_t word = encode8<FMT>(x, b);
            if (valid) Q[c] = word;

            // Scale bytes: lanes 0, TPB, 2TPB, 3TPB hold four consecutive
            // blocks of one row; the first of them stores the 4-byte word.
            const uint32_t b1 = __shfl_down_sync(0xffffffffu, b.code, TPB);
            const uint32_t b2 = __shfl_down_sync(0xffffffffu, b.code, 2 * TPB);
            const uint32_t b3 = __shfl_down_sync(0xffffffffu, b.code, 3 * TPB);
            if (valid && (lane % (4 * TPB)) == 0) {
                const uint32_t sfw = b.code | (b1 << 8) | (b2 << 16) | (b3 << 24);
                const int64_t blk = c / TPB;                 // flat block index
                const int64_t col = blk % kg;
                int64_t off;
                if (GROUPED) {
                    const int64_t rr = row - s_offs[grp];
                    off = sf_mma_offset(s_tile0[grp] + rr / 128, rr % 128, col, kc);
                } else if (SF_LAYOUT == QFP4_SF_MMA) {
                    off = sf_mma_offset(row / 128, row % 128, col, kc);
                } else {
                    off = blk;
                }
                *reinterpret_cast<uint32_t *>(SF + off) = sfw;
            }
        }
    }
}

// amax over rows of X, one warp per row; per group via atomicMax on the bit
// pattern (non-negative floats order like unsigned integers).
__global__ void __launch_bounds__(kThreads)
amax_rows_kernel(const uint4 *__restrict__ X, int64_t rows, int64_t chunks_per_row, int groups,
                 const int32_t *__restrict__ row_offsets, uint32_t *__restrict__ amax_bits)
{
    __shared__ int32_t s_offs[kMaxGroups + 1];
    if (row_offsets) {
        for (int i = threadIdx.x; i <= groups; i += blockDim.x) s_offs[i] = row_offsets[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int cur = -1;
    float run = 0.0f;
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
        const int g = row_offsets ? find_group(s_offs, groups, r) : 0;
        if (g != cur) {
            if (cur >= 0 && lane == 0) atomicMax(amax_bits + cur, __float_as_uint(run));
            cur = g;
            run = 0.0f;
        }
        run = fmaxf(run, m);
    }
    if (cur >= 0 && lane == 0) atomicMax(amax_bits + cur, __float_as_uint(run));
}

// gs = amax / (6 * 448), in place over the amax bit patterns.
__global__ void gs_finalize_kernel(uint32_t *bits, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const float amax = __uint_as_float(bits[i]);
        reinterpret_cast<float *>(bits)[i] = __fdiv_rn(amax, 2688.0f);
    }
}

// Scale-factor interleave; one thread per 4-byte word of the MMA layout.
template <bool TO_MMA>
__global__ void __launch_bounds__(kThreads)
sf_interleave_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int64_t rows,
                     int64_t cols, int64_t kc, int64_t words)
{
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

int grid_for(int64_t work_items, int per_block)
{
    const int sms = sm_count();
    const int64_t want = (work_items + per_block - 1) / per_block;
    int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 8;
    int64_t g = want < cap ? want : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

template <int FMT, int LAYOUT, bool GROUPED>
cudaError_t launch_quantize(const void *X, int64_t M, int64_t K, const float *gs, void *Q,
                            void *SF, int groups, const int32_t *offs, cudaStream_t s)
{
    const int64_t chunks = M * (K / 8);
    const int grid = grid_for(chunks, kThreads * 4);
    quantize_kernel<FMT, LAYOUT, GROUPED><<<grid, kThreads, 0, s>>>(
        static_cast<const uint4 *>(X), chunks, K, gs, static_cast<uint32_t *>(Q),
        static_cast<uint8_t *>(SF), M, groups, offs);
    return cudaGetLastError();
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

extern "C" int qfp4_global_scale(const void *X_bf16, int64_t rows, int64_t cols, float *gs_out,
                                 void *stream)
{
    if (!X_bf16 || !gs_out || rows < 0 || cols < 0) return QFP4_ERR_INVALID_ARG;
    if (cols % 8 != 0) return QFP4_ERR_UNSUPPORTED;
    if (!aligned16(X_bf16) || !aligned4(gs_out)) return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(gs_out, 0, sizeof(float), s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (rows > 0 && cols > 0) {
        const int grid = grid_for(rows, kThreads / 32);
        amax_rows_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint4 *>(X_bf16), rows,
                                                   cols / 8, 1, nullptr,
                                                   reinterpret_cast<uint32_t *>(gs_out));
        if (cudaGetLastError() != cudaSuccess) return QFP4_ERR_CUDA;
    }
    gs_finalize_kernel<<<1, 32, 0, s>>>(reinterpret_cast<uint32_t *>(gs_out), 1);
    return launch_status(cudaGetLastError());
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
    if (cudaMemsetAsync(gs_out, 0, sizeof(float) * groups, s) != cudaSuccess) return QFP4_ERR_CUDA;
    if (total_rows > 0 && cols > 0) {
        const int grid = grid_for(total_rows, kThreads / 32);
        amax_rows_kernel<<<grid, kThreads, 0, s>>>(
            static_cast<const uint4 *>(X_bf16), total_rows, cols / 8, static_cast<int>(groups),
            row_offsets, reinterpret_cast<uint32_t *>(gs_out));
        if (cudaGetLastError() != cudaSuccess) return QFP4_ERR_CUDA;
    }
    gs_finalize_kernel<<<(static_cast<int>(groups) + 127) / 128, 128, 0, s>>>(
        reinterpret_cast<uint32_t *>(gs_out), static_cast<int>(groups));
    return launch_status(cudaGetLastError());
}

extern "C" int qfp4_quantize(int fmt, const void *X_bf16, int64_t M, int64_t K, const float *gs,
                             void *Q_packed, void *SF, int sf_layout, void *stream)
{
    if (fmt != QFP4_MXFP4 && fmt != QFP4_NVFP4) return QFP4_ERR_INVALID_ARG;
    if (sf_layout != QFP4_SF_ROWMAJOR && sf_layout != QFP4_SF_MMA) return QFP4_ERR_INVALID_ARG;
    if (M < 0 || K < 0) return QFP4_ERR_INVALID_ARG;
    if (K % 128 != 0) return QFP4_ERR_UNSUPPORTED;
    if (M == 0 || K == 0) return QFP4_OK;
    if (!X_bf16 || !Q_packed || !SF) return QFP4_ERR_INVALID_ARG;
    if (fmt == QFP4_NVFP4 && !gs) return QFP4_ERR_INVALID_ARG;
    if (!aligned16(X_bf16) || !aligned16(Q_packed) || !aligned4(SF) || (gs && !aligned4(gs)))
        return QFP4_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fmt == QFP4_MXFP4)
        e = sf_layout == QFP4_SF_MMA
                ? launch_quantize<QFP4_MXFP4, QFP4_SF_MMA, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s)
                : launch_quantize<QFP4_MXFP4, QFP4_SF_ROWMAJOR, false>(X_bf16, M, K, gs, Q_packed, SF, 1, nullptr, s);
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
    const int grid = grid_for(words, kThreads);
    if (layout == QFP4_SF_MMA)
        sf_interleave_kernel<true><<<grid, kThreads, 0, s>>>(
            static_cast<const uint8_t *>(SF_in), static_cast<uint8_t *>(SF_out), rows, cols, kc, words);
    else
        sf_interleave_kernel<false><<<grid, kThreads, 0, s>>>(
            static_cast<const uint8_t *>(SF_in), static_cast<uint8_t *>(SF_out), rows, cols, kc, words);
    return launch_status(cudaGetLastError());
}
