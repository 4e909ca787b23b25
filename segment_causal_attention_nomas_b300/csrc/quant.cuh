// quant.cuh -- the INT8 quantisation rule of the K/V cache, shared by the append kernel and the
// projection's fused append so that both produce the same bits.
//
// Per (token, head) row of 128 values x (the BF16 K or V as fp32): a = max |x|; scale =
// fl32(a / 127) by IEEE division; a = 0 gives scale 0 and codes 0; otherwise code =
// clamp(rne(fl32(x / scale)), -127, 127), the quotient correctly rounded (comfyui-wiki news,
// 单张 4090 配置: cached keys and values stored INT8).
#pragma once

#include <cstdint>

namespace nomas {
namespace {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: t + kMagic rounds t to an integer (RNE)

// Packs the low bytes of 16 words (the codes) into 16 bytes.
__device__ __forceinline__ uint4 pack_low_bytes(const uint32_t *yb) {
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo = __byte_perm(yb[4 * q], yb[4 * q + 1], 0x0040);
        const uint32_t hi = __byte_perm(yb[4 * q + 2], yb[4 * q + 3], 0x0040);
        wd[q] = __byte_perm(lo, hi, 0x5410);
    }
    return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t mul2_rn(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2_rn(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

struct Vals16 {
    float v[16];
};

// Codes of 16 values by division, for rows whose scale is below 2^-100 (kept out of line).
__device__ __noinline__ uint4 quant16_divide(Vals16 x, float scale) {
    uint32_t yb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        yb[e] = static_cast<uint32_t>(max(-127, min(127, __float2int_rn(__fdiv_rn(x.v[e], scale)))));
    return pack_low_bytes(yb);
}

// The row's scale fl(a / 127) from its absmax a > 0.  For a >= 2^-100 one correction step from
// the correctly rounded reciprocal of 127 (Markstein's, as for the codes below): t0 = fl(a * r),
// the residual a - 127 t0 exact in one FMA, then fl(t0 + residual * r).  Checked against the
// IEEE quotient with exact rational arithmetic for every BF16 mantissa (every positive BF16 a from
// 2^-100 up); smaller a divide.
__device__ __forceinline__ float quant_scale(float a) {
    if (!(a >= 0x1p-100f)) return __fdiv_rn(a, 127.0f);
    constexpr float r127 = 1.0f / 127.0f;  // fl(1/127)
    const float t0 = __fmul_rn(a, r127);
    const float e = __fmaf_rn(-t0, 127.0f, a);
    return __fmaf_rn(e, r127, t0);
}

// Codes of N (a multiple of 16) values of a row with scale >= 2^-100, by the correction step of
// codes16 below with the reciprocal formed once; the residual's FMA takes -scale as its operand
// (x - t0 * scale exactly as fma(t0, -scale, x)).
template <int N>
__device__ __forceinline__ void codes_fast(const float *x, float scale, uint4 *out) {
    const float rs = __frcp_rn(scale);
    const uint64_t y2 = f2(rs, rs), nb2 = f2(-scale, -scale), m2 = f2(kMagic, kMagic);
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
        uint32_t yb[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const uint64_t x2 = f2(x[16 * c + e], x[16 * c + e + 1]);
            const uint64_t t0 = mul2_rn(x2, y2);
            const uint64_t r = fma2_rn(t0, nb2, x2);  // x - t0 * scale, exact
            const uint64_t t = fma2_rn(r, y2, t0);    // fl(x / scale)
            const uint64_t y = add2_rn(t, m2);
            yb[e] = static_cast<uint32_t>(y);
            yb[e + 1] = static_cast<uint32_t>(y >> 32);
        }
        out[c] = pack_low_bytes(yb);
    }
}

// Codes of 16 values of a row with scale > 0.  The quotient is formed without a division: with
// y = fl(1/scale), t0 = fl(x y), the residual r = x - t0 scale is exact in one FMA, and t0 + r y
// (one more FMA) is the correctly rounded x / scale (Markstein's correction step); rows with a
// scale below 2^-100, where y or the residual could leave the normal range, divide instead.
// t + 1.5 * 2^23 rounds t to an integer whose two's complement is the word's low byte
// (|code| <= 127 since |x| <= absmax).
__device__ __forceinline__ uint4 codes16(const float *x, float scale) {
    if (!(scale >= 0x1p-100f)) {
        Vals16 xv;
#pragma unroll
        for (int e = 0; e < 16; ++e) xv.v[e] = x[e];
        return quant16_divide(xv, scale);
    }
    const float rs = __frcp_rn(scale);
    const uint64_t y2 = f2(rs, rs), b2 = f2(scale, scale), m2 = f2(kMagic, kMagic);
    uint32_t yb[16];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        const uint64_t x2 = f2(x[e], x[e + 1]);
        const uint64_t t0 = mul2_rn(x2, y2);
        const uint64_t r = fma2_rn(t0 ^ 0x8000000080000000ull, b2, x2);  // x - t0 * scale, exact
        const uint64_t t = fma2_rn(r, y2, t0);                            // fl(x / scale)
        const uint64_t y = add2_rn(t, m2);
        yb[e] = static_cast<uint32_t>(y);
        yb[e + 1] = static_cast<uint32_t>(y >> 32);
    }
    return pack_low_bytes(yb);
}

}  // namespace
}  // namespace nomas
