// codec.cuh -- the e4m3 quantisation arithmetic shared by the quantisers
// (quant.cu) and the GEMM's fused output quantisation (gemm.cu).
//
// Quantisation rule ("DeepSeek-V3" repository overview, section
// "FP8 混合精度训练"): s = amax / 448 over the group or block (fp32, IEEE
// round-to-nearest division), code = e4m3(x / s) with round-to-nearest-even
// and saturation at +-448; an all-zero group has s = 0 and +-0 codes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp8bs {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Packed fp32 pairs (low half = first element): two IEEE round-to-nearest
// operations per instruction, bit-identical to the scalar ones.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Scale-side constants of one group or block.  s = RN32(amax / 448) and
// r = RN32(1 / s).  The quotients use Markstein's correction step
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/b),
// q0 = RN(a y), rem = a - b q0 (exact with one fused multiply-add) and
// q = RN(q0 + rem y) equals RN(a / b).  s itself is formed that way from
// the constant RN32(1/448) = 0x3b124925.  Groups whose amax is below 2^-100
// (where subnormal intermediates could break the argument) use IEEE
// division throughout (`exact_div`).  Bit-exactness of every code and scale
// against RN32 division is checked exhaustively over every bf16 amax and
// every bf16 x with |x| <= amax.
struct GroupScale {
    float s, r;
    bool exact_div;
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
    GroupScale g;
    g.exact_div = !(amax >= 7.888609052210118e-31f);  // 2^-100; also true for amax == 0
    if (g.exact_div) {
        g.s = __fdiv_rn(amax, kE4M3Max);
        g.r = 0.0f;
    } else {
        const float inv448 = __uint_as_float(0x3b124925u);
        const float q0 = __fmul_rn(amax, inv448);
        const float rem = __fmaf_rn(-q0, kE4M3Max, amax);
        g.s = __fmaf_rn(rem, inv448, q0);
        g.r = __frcp_rn(g.s);
    }
    return g;
}

// Power-of-two (UE8M0-style) scale of a group or block, rounded up so that
// nothing saturates: s = 2^e with e the smallest integer such that
// amax <= 448 * 2^e (the scale_fmt reading of the linear() excerpt, "DeepSeek-V3"
// repository overview).  With amax = (1 + f) 2^E (f the 23-bit fraction) and
// 448 = 1.75 * 2^8, e = E - 8 when 1 + f <= 1.75 and E - 7 otherwise; a
// subnormal amax is first scaled by 2^64 (exactly).  x / s is then exact and
// r = 2^-e is its exact reciprocal, so encode8's quotient steps return x * r;
// where 2^-e is not a normal float (e < -126) the codes use IEEE division.
// amax == 0 gives s = 0 (the caller encodes +-0 codes).
__device__ __forceinline__ GroupScale group_scale_pow2(float amax) {
    GroupScale g;
    if (!(amax > 0.0f)) {
        g.s = 0.0f;
        g.r = 0.0f;
        g.exact_div = true;
        return g;
    }
    uint32_t u = __float_as_uint(amax);
    int adj = 0;
    if ((u >> 23) == 0) {  // subnormal amax
        u = __float_as_uint(amax * 18446744073709551616.0f);  // x 2^64, exact
        adj = -64;
    }
    const int ex = static_cast<int>(u >> 23) - 127;
    // (a bf16 amax is at least 2^-133, so e >= -141; the clamp only keeps
    // the shift below defined for any fp32 input)
    const int e = max(ex - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0) + adj, -149);
    g.s = e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(1u << (e + 149));
    g.exact_div = e < -126 || e > 126;
    g.r = g.exact_div ? 0.0f : __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    return g;
}

// Largest |x| over 8 bf16 values held as bit patterns: for non-negative
// IEEE patterns integer order equals value order, so the maximum of
// (bits & 0x7fff) per 16-bit half is the amax's bit pattern.
__device__ __forceinline__ uint32_t absmax_bits8(const uint4& v, uint32_t m) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    return m;
}
__device__ __forceinline__ float bits_to_amax(uint32_t m2) {
    return __uint_as_float((m2 > (m2 << 16) ? m2 & 0xFFFF0000u : m2 << 16));
}

// Encode 8 bf16 values (bit patterns in `raw`, element j in half j of the
// words) into 8 e4m3 codes (little-endian in a uint2): code = e4m3(RN32(x/s)),
// round to nearest-even with saturation (cvt.rn.satfinite).  The sign of
// each code is OR-ed in from the input's sign bit, which keeps -0 as 0x80
// (a nonzero quotient already carries x's sign).  zero_group (amax == 0):
// every code is +-0.
__device__ __forceinline__ uint2 encode8(const uint4& raw, const GroupScale& g, bool zero_group) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    const uint32_t sign0 = __byte_perm(w[0], w[1], 0x7531) & 0x80808080u;
    const uint32_t sign1 = __byte_perm(w[2], w[3], 0x7531) & 0x80808080u;
    if (zero_group) return make_uint2(sign0, sign1);
    uint32_t c[4];
    if (g.exact_div) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[i]), g.s), __fdiv_rn(bf16_hi(w[i]), g.s));
    } else {
        const uint64_t r2 = f2(g.r, g.r);
        const uint64_t ns2 = f2(-g.s, -g.s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t x2 = f2(bf16_lo(w[i]), bf16_hi(w[i]));
            const uint64_t q0 = f2_mul(x2, r2);
            const uint64_t rem = f2_fma(q0, ns2, x2);  // x - s q0, exact
            const uint64_t q = f2_fma(rem, r2, q0);
            c[i] = cvt_e4m3x2(__uint_as_float(static_cast<uint32_t>(q)),
                              __uint_as_float(static_cast<uint32_t>(q >> 32)));
        }
    }
    return make_uint2((c[0] | (c[1] << 16)) | sign0, (c[2] | (c[3] << 16)) | sign1);
}

}  // namespace fp8bs
