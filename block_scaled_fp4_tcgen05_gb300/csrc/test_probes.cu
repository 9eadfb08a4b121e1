// test_probes.cu -- encoder probes of the test build (QFP4_FAULT_INJECTION);
// the released library compiles this file to nothing.
//
// The quantisers that take fp32 values (the residual-add + RMSNorm quantiser
// and the SwiGLU epilogue of the up-projection) encode a block with
// block_scale and encode8_f32 from qfp4_fp4_codes.cuh.  These two probes run
// exactly those device functions over a range of fp32 bit patterns, so that a
// test can compare every finite fp32 input with the oracle:
//   qfp4_test_scale_codes:   the scale byte block_scale gives for amax = x_i;
//   qfp4_test_element_codes: the E2M1 code encode8_f32 gives for x_i under a
//                            block scale s (NVFP4: any s > 0, with RN(1/s)
//                            and the fast or IEEE quotient chosen per group of
//                            eight values as the kernels choose it per block;
//                            MXFP4: s = 2^(c - 127), the exact inverse).
// x_i is the float whose bit pattern is first + i (i < n); the caller keeps
// NaN and infinity patterns out.  One code per output byte.
#include <cstdint>
#include <cuda_runtime.h>

#include "qfp4_common.cuh"
#include "qfp4_fp4_codes.cuh"

#ifdef QFP4_FAULT_INJECTION

namespace qfp4 {
namespace {

template <int FMT>
__global__ void __launch_bounds__(256)
scale_codes_kernel(uint32_t first, int64_t n, float gs, uint8_t *__restrict__ codes)
{
    const float inv_gs = __frcp_rn(gs);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float amax = __uint_as_float(first + static_cast<uint32_t>(i));
        codes[i] = static_cast<uint8_t>(block_scale<FMT>(amax, gs, inv_gs).code);
    }
}

// s_or_code: NVFP4 the block scale s; MXFP4 the UE8M0 code c (s = 2^(c-127)).
template <int FMT>
__global__ void __launch_bounds__(256)
element_codes_kernel(uint32_t first, int64_t n, float s_or_code, uint8_t *__restrict__ codes)
{
    const int64_t groups = (n + 7) / 8;
    for (int64_t gi = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; gi < groups;
         gi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i0 = gi * 8;
        float x[8];
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[k] = i0 + k < n ? __uint_as_float(first + static_cast<uint32_t>(i0 + k)) : 0.0f;
            amax = fmaxf(amax, fabsf(x[k]));
        }
        BlockScale b;
        if (FMT == QFP4_NVFP4) {
            const float s = s_or_code;
            b = nvfp4_block(0u, s, s == 0.0f ? 0.0f : __frcp_rn(s), amax);
        } else {
            const uint32_t c = static_cast<uint32_t>(s_or_code);
            b.code = c;
            b.inv = ue8m0_inverse(c);
            b.s = 0.0f;
            b.mode = 1;
        }
        const uint32_t w = encode8_f32<FMT>(x, b);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i0 + k < n) codes[i0 + k] = static_cast<uint8_t>((w >> (4 * k)) & 0xFu);
    }
}

int probe_grid(int64_t work)
{
    const int64_t cap = static_cast<int64_t>(sm_count() > 0 ? sm_count() : 148) * 8;
    const int64_t want = (work + 255) / 256;
    return static_cast<int>(want < 1 ? 1 : want < cap ? want : cap);
}

bool probe_args_ok(int fmt, uint32_t first, int64_t n, const void *codes)
{
    return (fmt == QFP4_MXFP4 || fmt == QFP4_NVFP4) && codes && n >= 0 &&
           static_cast<uint64_t>(first) + static_cast<uint64_t>(n) <= (1ull << 32);
}

}  // namespace
}  // namespace qfp4

using namespace qfp4;

// Scale bytes of amax = float(first + i), i < n, under global scale gs
// (MXFP4 ignores gs), into codes[n] (device).
extern "C" int qfp4_test_scale_codes(int fmt, uint32_t first_bits, int64_t n, float gs, void *codes,
                                     void *stream)
{
    if (!probe_args_ok(fmt, first_bits, n, codes)) return QFP4_ERR_INVALID_ARG;
    if (n == 0) return QFP4_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(codes);
    if (fmt == QFP4_NVFP4) scale_codes_kernel<QFP4_NVFP4><<<probe_grid(n), 256, 0, s>>>(first_bits, n, gs, out);
    else scale_codes_kernel<QFP4_MXFP4><<<probe_grid(n), 256, 0, s>>>(first_bits, n, 1.0f, out);
    return cudaGetLastError() == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

// E2M1 codes of x = float(first + i), i < n, under the block scale s
// (NVFP4, s > 0) or the UE8M0 code c = (int)s (MXFP4, 0..254), into codes[n].
extern "C" int qfp4_test_element_codes(int fmt, uint32_t first_bits, int64_t n, float s_or_code,
                                       void *codes, void *stream)
{
    if (!probe_args_ok(fmt, first_bits, n, codes)) return QFP4_ERR_INVALID_ARG;
    if (fmt == QFP4_NVFP4 ? !(s_or_code > 0.0f) : !(s_or_code >= 0.0f && s_or_code <= 254.0f))
        return QFP4_ERR_INVALID_ARG;
    if (n == 0) return QFP4_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *out = static_cast<uint8_t *>(codes);
    const int grid = probe_grid((n + 7) / 8);
    if (fmt == QFP4_NVFP4) element_codes_kernel<QFP4_NVFP4><<<grid, 256, 0, s>>>(first_bits, n, s_or_code, out);
    else element_codes_kernel<QFP4_MXFP4><<<grid, 256, 0, s>>>(first_bits, n, s_or_code, out);
    return cudaGetLastError() == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

#endif  // QFP4_FAULT_INJECTION
