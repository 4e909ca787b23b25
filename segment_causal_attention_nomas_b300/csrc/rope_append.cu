// rope_append.cu -- 3D RoPE (rope3d) and fused RoPE + INT8 append (append_quant).
//
// Both are HBM-bound streaming kernels.  One (token, head) row of 128 BF16 channels is
// handled by 8 consecutive threads, each owning 16 channels (two 16-byte loads).  A thread's
// channels form two groups of 8, and no group of 8 straddles an axis chunk of the
// [16, 56, 56] split, so each group reads one cos/sin row segment of one axis.  Token and
// head indices come from multiply-shift divisions by host-computed magic numbers.
//
// RoPE (comfyui-wiki news, architecture table: 3D RoPE sizes [16, 56, 56], theta 256):
// pair (x0, x1) of an axis chunk -> (x0*c - x1*s, x0*s + x1*c), every product and sum
// rounded to fp32 (__fmul_rn / __fsub_rn / __fadd_rn: no FMA contraction), then BF16 RNE.
//
// Quantisation (comfyui-wiki, "单张 4090 配置": cached K/V stored as INT8): per row,
// a = max|x|, scale = a / 127 (IEEE fp32 division), code = clamp(rne(x / scale), +-127),
// a == 0 -> scale 0 and all codes 0.  The absmax is an 8-lane shuffle reduction.  The code
// of x is the round-half-even of the correctly rounded quotient fl(x / scale); it is taken
// from t = x * fl(1 / scale), which lies within 1.5 * 2^-23 * |x / scale| (< 2^-15 here) of
// fl(x / scale), whenever t is farther than 2^-14 from a half-integer (then both round to the
// same integer; the margin is twice the bound, so a last-bit deviation of the paired fp32
// arithmetic cannot matter).  Lanes with a value closer than that divide exactly (__fdiv_rn).
#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

// n / d for 0 <= n < 2^31 as (umulhi(n, m) + n) >> l (Granlund & Montgomery, "Division by
// invariant integers using multiplication", 1994, with the 32-bit sum safe for n < 2^31).
struct FastDiv {
    uint32_t m, l;
};

FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.l = l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f) { return (__umulhi(n, f.m) + n) >> f.l; }

struct SegPos {
    int32_t t0, n_video, n_tokens, heads, hw, gw;
    FastDiv div_hw, div_gw, div_heads;
};

struct TokPos {
    int t, h, w;
    bool video;
};

__device__ __forceinline__ TokPos token_pos(const SegPos &s, uint32_t k) {
    TokPos p;
    p.video = static_cast<int>(k) < s.n_video;
    const uint32_t tt = fdiv(k, s.div_hw);
    const uint32_t r = k - tt * static_cast<uint32_t>(s.hw);
    const uint32_t hh = fdiv(r, s.div_gw);
    p.t = s.t0 + static_cast<int>(tt);
    p.h = static_cast<int>(hh);
    p.w = static_cast<int>(r - hh * static_cast<uint32_t>(s.gw));
    return p;
}

// Rotates the 8 channels [8*g, 8*g+8) of one head row in place (x as fp32), with scalar
// correctly rounded products and sums (paired f32x2 arithmetic was measured to differ from
// them in the last bit on B300, so the bit-exact rotation does not use it).
__device__ __forceinline__ void rotate8(float *x, int g, const TokPos &p, const RopeDev &rope) {
    // select the axis with conditionals (a dynamic index into the parameter struct would
    // force it into local memory)
    const bool ax_t = g < 2, ax_h = !ax_t && g < 9;
    const int pos = ax_t ? p.t : (ax_h ? p.h : p.w);
    const int half = ax_t ? 8 : 28;
    const int pair0 = ax_t ? 4 * g : (ax_h ? 4 * (g - 2) : 4 * (g - 9));
    const float *ctab = ax_t ? rope.cos[0] : (ax_h ? rope.cos[1] : rope.cos[2]);
    const float *stab = ax_t ? rope.sin[0] : (ax_h ? rope.sin[1] : rope.sin[2]);
    const float4 c = __ldg(reinterpret_cast<const float4 *>(ctab + pos * half + pair0));
    const float4 s = __ldg(reinterpret_cast<const float4 *>(stab + pos * half + pair0));
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = x[2 * i], x1 = x[2 * i + 1];
        x[2 * i] = __fsub_rn(__fmul_rn(x0, cc[i]), __fmul_rn(x1, ss[i]));
        x[2 * i + 1] = __fadd_rn(__fmul_rn(x0, ss[i]), __fmul_rn(x1, cc[i]));
    }
}

__device__ __forceinline__ void unpack8(uint4 w, float *x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8_bf16(const float *x) {
    uint4 r;
    r.x = pack_bf16x2(x[0], x[1]);
    r.y = pack_bf16x2(x[2], x[3]);
    r.z = pack_bf16x2(x[4], x[5]);
    r.w = pack_bf16x2(x[6], x[7]);
    return r;
}

// x and y may be the same buffer (in place): each element is read and written by one thread.
__global__ void __launch_bounds__(256) rope3d_kernel(const uint4 *x, uint4 *y, int64_t row_stride16, SegPos seg,
                                                     RopeDev rope) {
    const int64_t total = static_cast<int64_t>(seg.n_tokens) * seg.heads * 8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int G = static_cast<int>(i & 7);
        const uint32_t row = static_cast<uint32_t>(i >> 3);
        const uint32_t k = fdiv(row, seg.div_heads);
        const int h = static_cast<int>(row - k * static_cast<uint32_t>(seg.heads));
        const int64_t off = static_cast<int64_t>(k) * row_stride16 + h * 16 + 2 * G;
        uint4 w0 = x[off], w1 = x[off + 1];
        const TokPos p = token_pos(seg, k);
        if (p.video) {
            float f[16];
            unpack8(w0, f);
            unpack8(w1, f + 8);
            rotate8(f, 2 * G, p, rope);
            rotate8(f + 8, 2 * G + 1, p, rope);
            w0 = pack8_bf16(f);
            w1 = pack8_bf16(f + 8);
        }
        y[off] = w0;
        y[off + 1] = w1;
    }
}

// absmax over the 8 lanes of a row group (lanes 8q .. 8q+7 of a warp)
__device__ __forceinline__ float group8_max(float a) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    return a;
}

// Quantises this lane's 16 values of a row (8 lanes per row); returns the 16 codes.
// For each value, t = x * fl(1/scale) is rounded to an integer by adding 1.5 * 2^23 (y), whose
// low byte is then the two's-complement code (|code| <= 127 since |x| <= absmax).  If any t of
// the lane lies within 2^-14 of a half-integer, the lane divides exactly instead.
__device__ __forceinline__ uint4 quant16(const float *x, float &scale_out) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
    a = group8_max(a);
    if (a == 0.0f) {
        scale_out = 0.0f;
        return make_uint4(0u, 0u, 0u, 0u);
    }
    const float scale = __fdiv_rn(a, 127.0f);
    const float rs = __frcp_rn(scale);
    scale_out = scale;
    uint32_t yb[16];
    float worst = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        const float2 t = __fmul2_rn(make_float2(x[e], x[e + 1]), make_float2(rs, rs));
        const float2 y = __fadd2_rn(t, make_float2(kMagic, kMagic));
        const float2 n = __fadd2_rn(y, make_float2(-kMagic, -kMagic));
        const float2 f = __fadd2_rn(t, make_float2(-n.x, -n.y));
        worst = fmaxf(worst, fmaxf(fabsf(f.x), fabsf(f.y)));
        yb[e] = __float_as_uint(y.x);
        yb[e + 1] = __float_as_uint(y.y);
    }
    // (fmaxf drops NaN, so a non-finite reciprocal, from a scale below 2^-128, is tested apart)
    if (!(worst < 0.5f - 0x1p-14f) || !(rs < 3.0e38f)) {
        // near a rounding boundary, or no usable reciprocal: exact quotients
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int q = max(-127, min(127, __float2int_rn(__fdiv_rn(x[e], scale))));
            yb[e] = 0x4B400000u + static_cast<uint32_t>(q);
        }
    }
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo = __byte_perm(yb[4 * q], yb[4 * q + 1], 0x0040);
        const uint32_t hi = __byte_perm(yb[4 * q + 2], yb[4 * q + 3], 0x0040);
        wd[q] = __byte_perm(lo, hi, 0x5410);
    }
    return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

// One thread: 16 channels of one (token, head) row of K and of V.  8 lanes per row.
__global__ void __launch_bounds__(256) append_quant_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           int64_t row_stride16, SegPos seg, RopeDev rope,
                                                           uint4 *__restrict__ ck, uint4 *__restrict__ cv,
                                                           float *__restrict__ cks, float *__restrict__ cvs,
                                                           int64_t cap, int64_t length) {
    const int64_t total = static_cast<int64_t>(seg.n_tokens) * seg.heads * 8;
    // the loop condition is uniform over a warp (the shuffles below need all 32 lanes);
    // lanes past the end run with `live` false
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i - (threadIdx.x & 31) < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool live = i < total;
        const int G = static_cast<int>(i & 7);
        const uint32_t row = live ? static_cast<uint32_t>(i >> 3) : 0u;
        const uint32_t tok = fdiv(row, seg.div_heads);
        const int h = static_cast<int>(row - tok * static_cast<uint32_t>(seg.heads));
        const int64_t off = static_cast<int64_t>(tok) * row_stride16 + h * 16 + 2 * G;
        uint4 wk0 = make_uint4(0, 0, 0, 0), wk1 = wk0, wv0 = wk0, wv1 = wk0;
        if (live) {
            wk0 = k[off];
            wk1 = k[off + 1];
            wv0 = v[off];
            wv1 = v[off + 1];
        }
        float fk[16], fv[16];
        unpack8(wk0, fk);
        unpack8(wk1, fk + 8);
        unpack8(wv0, fv);
        unpack8(wv1, fv + 8);
        const TokPos p = token_pos(seg, tok);
        if (live && p.video) {
            rotate8(fk, 2 * G, p, rope);
            rotate8(fk + 8, 2 * G + 1, p, rope);
            // quantise the BF16-rounded rotated K
            unpack8(pack8_bf16(fk), fk);
            unpack8(pack8_bf16(fk + 8), fk + 8);
        }
        float sk, sv;
        const uint4 qk = quant16(fk, sk);
        const uint4 qv = quant16(fv, sv);
        if (live) {
            const int64_t dst = static_cast<int64_t>(h) * cap + length + tok;
            ck[dst * 8 + G] = qk;
            cv[dst * 8 + G] = qv;
            if (G == 0) {
                cks[dst] = sk;
                cvs[dst] = sv;
            }
        }
    }
}

int grid_for(int64_t threads) {
    const int64_t blocks = (threads + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8 * 4;  // a few waves, grid-stride beyond
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

SegPos seg_pos(const SegDesc &s, int32_t heads) {
    SegPos p;
    p.t0 = s.t0;
    p.n_video = s.n_video;
    p.n_tokens = s.n_tokens;
    p.heads = heads;
    p.hw = s.gh * s.gw > 0 ? s.gh * s.gw : 1;
    p.gw = s.gw > 0 ? s.gw : 1;
    p.div_hw = make_fastdiv(static_cast<uint32_t>(p.hw));
    p.div_gw = make_fastdiv(static_cast<uint32_t>(p.gw));
    p.div_heads = make_fastdiv(static_cast<uint32_t>(heads));
    return p;
}

}  // namespace

cudaError_t launch_rope3d(const void *x, void *y, int64_t row_stride, const SegDesc &seg, int32_t heads,
                          const RopeDev &rope, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(seg.n_tokens) * heads * 8;
    if (threads == 0) return cudaSuccess;
    rope3d_kernel<<<grid_for(threads), 256, 0, stream>>>(static_cast<const uint4 *>(x), static_cast<uint4 *>(y),
                                                         row_stride / 8, seg_pos(seg, heads), rope);
    return cudaGetLastError();
}

cudaError_t launch_append_quant(const void *k, const void *v, int64_t row_stride, const SegDesc &seg,
                                int32_t heads, const RopeDev &rope, int8_t *ck, int8_t *cv, float *cks,
                                float *cvs, int64_t cap, int64_t length, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(seg.n_tokens) * heads * 8;
    if (threads == 0) return cudaSuccess;
    append_quant_kernel<<<grid_for(threads), 256, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), row_stride / 8, seg_pos(seg, heads), rope,
        reinterpret_cast<uint4 *>(ck), reinterpret_cast<uint4 *>(cv), cks, cvs, cap, length);
    return cudaGetLastError();
}

}  // namespace nomas
