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

#include "../../include/qfp4.h"

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

// ---- the quantiser's rule on fp32 values, fast and bit-exact ---------------
// (used by the standalone quantiser, the residual-add + RMSNorm quantiser and
// the GEMM epilogue that requantises its own output)
//
// The rule, in IEEE fp32 round-to-nearest-even:
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

// 2^(127 - c) as fp32 (exact; subnormal for c = 254).
__device__ __forceinline__ float ue8m0_inverse(uint32_t c)
{
    const int e = 127 - static_cast<int>(c);                 // -127 .. 127
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                     : __uint_as_float(0x00400000u);          // 2^-127
}

struct BlockScale {
    float inv;      // MXFP4: exact 2^-e; NVFP4: RN(1/s)
    float s;        // NVFP4 scale s = decode(sf) * gs
    uint32_t code;  // scale byte
    int mode;       // 0: zero block, 1: fast path, 2: IEEE division
};

// RN(a / b) from y = RN(1 / b) with two fused corrections (Markstein); the
// caller guarantees a, b and the quotient stay well inside the normal range.
// The remainder is formed negated, e = b*q - a, and applied as q - e*y: the
// same values, but a = -0 keeps its sign (-0 - (+0) = -0) where the
// a - b*q form would turn it into +0.
__device__ __forceinline__ float div_markstein(float a, float b, float y)
{
    float q = __fmul_rn(a, y);
    q = __fmaf_rn(-__fmaf_rn(b, q, -a), y, q);
    q = __fmaf_rn(-__fmaf_rn(b, q, -a), y, q);
    return q;
}

__device__ __forceinline__ bool normal_range(float v) { return v >= 0x1p-100f && v <= 0x1p100f; }

// t = (amax / 6) / gs, each division correctly rounded.  inv_gs = RN(1/gs).
__device__ __forceinline__ float scale_target(float amax, float gs, float inv_gs)
{
    constexpr float kInv6 = 0x1.555556p-3f;          // RN(1/6)
    if (normal_range(amax)) {
        const float t1 = div_markstein(amax, 6.0f, kInv6);
        if (gs == 1.0f) return t1;
        if (normal_range(t1) && gs >= 0x1p-60f && gs <= 0x1p60f) return div_markstein(t1, gs, inv_gs);
        return __fdiv_rn(t1, gs);
    }
    return gs == 1.0f ? __fdiv_rn(amax, 6.0f) : __fdiv_rn(__fdiv_rn(amax, 6.0f), gs);
}

// UE4M3 scale byte of a block with maximum magnitude amax under global
// scale gs (inv_gs = RN(1/gs)).  t is NaN only when amax and gs are both 0
// (0/0: an all-zero block under a zero global scale) and then takes code 0
// like t = 0; a non-zero block with gs = 0 has t = +inf and saturates to 0x7E
// (s = 448 * 0 = 0 then still encodes it as zeros).
__device__ __forceinline__ uint32_t nvfp4_scale_code(float amax, float gs, float inv_gs)
{
    const float t = scale_target(amax, gs, inv_gs);
    return t > 0.0f ? ue4m3_encode(t) : 0u;
}

// The element-step parameters of an NVFP4 block from its scale s =
// decode(code) * gs and y = RN(1/s) (0 when s is 0).
__device__ __forceinline__ BlockScale nvfp4_block(uint32_t code, float s, float y, float amax)
{
    BlockScale b;
    b.code = code;
    b.s = s;
    b.inv = y;
    const bool fast = s >= 0x1p-64f && s <= 0x1p64f && amax <= s * 0x1p60f;
    b.mode = s == 0.0f ? 0 : fast ? 1 : 2;
    return b;
}

template <int FMT>
__device__ __forceinline__ BlockScale block_scale(float amax, float gs, float inv_gs)
{
    BlockScale b;
    if (FMT == QFP4_MXFP4) {
        const float t = scale_target(amax, 1.0f, 1.0f);
        b.code = ue8m0_encode(t);
        b.inv = ue8m0_inverse(b.code);
        b.s = 0.0f;
        b.mode = 1;
    } else {
        const uint32_t code = nvfp4_scale_code(amax, gs, inv_gs);
        const float s = __fmul_rn(ue4m3_decode(code), gs);
        b = nvfp4_block(code, s, s == 0.0f ? 0.0f : __frcp_rn(s), amax);
    }
    return b;
}

// ---- packed fp32 pairs: one f32x2 instruction works on both halves of a
// 64-bit register pair, halving the arithmetic issue slots of the quotient.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// RN(-x / s) on both halves of x2, from s2 = (s, s) and ny2 = (-y, -y) with
// y = RN(1/s): the two Markstein corrections of div_markstein applied to the
// dividend -x.  q0 = x*(-y) = (-x)*y, e = s*q + x = s*q - (-x) and
// q + e*(-y) = q - e*y are the same roundings as for -x, so the result is
// div_markstein(-x, s, y) = -RN(x/s), and no negation is ever issued.  Signed
// zeros come out right: x = +0 gives -0 and x = -0 gives +0.
__device__ __forceinline__ uint64_t f2_neg_quotient(uint64_t x2, uint64_t s2, uint64_t ny2)
{
    uint64_t q = f2_mul(x2, ny2);
    uint64_t e = f2_fma(s2, q, x2);
    q = f2_fma(e, ny2, q);
    e = f2_fma(s2, q, x2);
    return f2_fma(e, ny2, q);
}

// E2M1 rounding is symmetric (round to nearest even, saturation at +-6), so
// the codes of -q are the codes of q with the sign bit of every nibble set
// the other way.
constexpr uint32_t kNibbleSigns = 0x88888888u;

// Eight fp32 values of one block -> four packed bytes (element 2i in the low
// nibble of byte i): the element step of the rule with the block's scale b.
template <int FMT>
__device__ __forceinline__ uint32_t encode8_f32(const float *x, const BlockScale &b)
{
    float q[8];
    if (FMT == QFP4_MXFP4) {
        // b.inv is a power of two: x * 2^-e is the quotient (a result too
        // small to be exact lies far below the first E2M1 step, 0.25)
        const uint64_t inv2 = f2_pack(b.inv, b.inv);
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_pack(x[2 * i], x[2 * i + 1]), inv2), q[2 * i], q[2 * i + 1]);
        return e2m1x8(q);
    }
    if (b.mode == 1) {
        const uint64_t s2 = f2_pack(b.s, b.s), ny2 = f2_pack(-b.inv, -b.inv);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f2_unpack(f2_neg_quotient(f2_pack(x[2 * i], x[2 * i + 1]), s2, ny2), q[2 * i], q[2 * i + 1]);
        return e2m1x8(q) ^ kNibbleSigns;
    }
    if (b.mode == 0) return 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i], b.s);
    return e2m1x8(q);
}

__device__ __forceinline__ uint32_t sf_mma_offset(uint32_t row_tile, uint32_t r_in_tile, uint32_t c,
                                                  uint32_t kc)
{
    return (row_tile * kc + (c >> 2)) * 512u + (r_in_tile & 31u) * 16u + (r_in_tile >> 5) * 4u + (c & 3u);
}

}  // namespace qfp4
