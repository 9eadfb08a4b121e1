// qfp4_fp4_codes.cuh -- the format encodings shared by the quantiser and by
// the GEMM epilogue that requantises its own output (not ABI).
//
// E2M1 elements and UE8M0 scales follow the OCP Microscaling Formats (MX)
// v1.0 specification; UE4M3 is E4M3 (OCP 8-bit floating point, bias 7) with
// the sign bit fixed at zero.  DeepGEMM pull request "Packed MXFP4 & NVFP4
// GEMM + mega-MoE", section "Summary": MXFP4 = E2M1 with a UE8M0 scale per 32
// elements, NVFP4 = E2M1 with a UE4M3 scale per 16 elements.
#pragma once

#include <cstdint>

namespace qfp4 {

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

// Value 2^(c-127) of a UE8M0 code c (0..254) as fp32, exact (subnormal for c = 0).
__device__ __forceinline__ float ue8m0_decode(uint32_t c)
{
    return c ? __uint_as_float(c << 23) : __uint_as_float(0x00400000u);
}

// Eight fp32 -> four packed bytes: element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8])
{
    uint32_t w;
    asm("{\n.reg .b8 b0, b1, b2, b3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "mov.b32 %0, {b0, b1, b2, b3};\n}"
        : "=r"(w)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return w;
}

}  // namespace qfp4
