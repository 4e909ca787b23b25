// rope_append.cu -- 3D RoPE (rope3d) and fused RoPE + INT8 append (append_quant).
//
// Both are HBM-bound streaming kernels.  One (token, head) row of 128 BF16 channels is
// handled by 8 consecutive threads, each owning 16 channels (two 16-byte loads).  A thread's
// channels form two groups of 8, and no group of 8 straddles an axis chunk of the
// [16, 56, 56] split, so each group reads one cos/sin row segment of one axis.  The grid
// stride is a multiple of 8, so a thread always handles the same 16 channels (append_quant sets
// their axes and table columns up once).  Token and head indices come from multiply-shift
// divisions by host-computed magic numbers.
//
// RoPE (comfyui-wiki news, architecture table: 3D RoPE sizes [16, 56, 56], theta 256):
// pair (x0, x1) of an axis chunk -> (x0*c - x1*s, x0*s + x1*c), every product and sum
// rounded to fp32 (__fmul_rn / __fsub_rn / __fadd_rn: no FMA contraction), then BF16 RNE.
// (A paired f32x2 product feeding a paired f32x2 sum, even written as mul.rn / sub.rn.f32x2 in
// PTX, was measured on B300 to differ from these scalar results in the last bit of a few values
// in 100, as if the two had been fused, so the bit-exact rotation does not use paired
// arithmetic.)
//
// Quantisation (comfyui-wiki, "单张 4090 配置": cached K/V stored as INT8): per row,
// a = max|x|, scale = a / 127 (IEEE fp32 division), code = clamp(rne(x / scale), +-127),
// a == 0 -> scale 0 and all codes 0.  The absmax is an 8-lane shuffle reduction.  The code is
// the round-half-even of the correctly rounded quotient fl(x / scale), which is formed without a
// division: t0 = fl(x * y) with y = fl(1 / scale), then t = fl(t0 + y * (x - t0 * scale)), the
// residual and the correction each one FMA (Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990: from the correctly rounded
// reciprocal, this step gives the correctly rounded quotient).  On B300 t equals the IEEE
// quotient for every BF16 x with |x| <= a and every BF16 mantissa of a (all of them checked;
// powers of two scale the rest of the normal range), and the tests compare the codes with the
// oracle's division exhaustively over BF16 values.  Scales below 2^-100, where the residual could
// underflow, divide instead.  The paired fp32 instructions used here are IEEE-exact in each lane
// (checked against the scalar ones on B300); no product in this chain can be fused into a sum.
#include "common.cuh"
#include "quant.cuh"
#include "internal.h"

namespace nomas {
namespace {

// ------------------------------------------------------------------------ rotation
// Where a group of 8 channels [8g, 8g + 8) reads its cos/sin: the table of its axis chunk of
// the [16, 56, 56] split from the column of its first pair, the table's row length, and which
// of the token's (t, h, w) positions selects the row.
struct RopeGroup {
    const float *cos, *sin;
    int half, axis;
};

__device__ __forceinline__ RopeGroup rope_group(int g, const RopeDev &rope) {
    // select with conditionals (a dynamic index into the parameter struct would force it into
    // local memory)
    const bool ax_t = g < 2, ax_h = !ax_t && g < 9;
    const int pair0 = ax_t ? 4 * g : (ax_h ? 4 * (g - 2) : 4 * (g - 9));
    RopeGroup r;
    r.cos = (ax_t ? rope.cos[0] : (ax_h ? rope.cos[1] : rope.cos[2])) + pair0;
    r.sin = (ax_t ? rope.sin[0] : (ax_h ? rope.sin[1] : rope.sin[2])) + pair0;
    r.half = ax_t ? 8 : 28;
    r.axis = ax_t ? 0 : (ax_h ? 1 : 2);
    return r;
}

// Rotates the 8 BF16 channels of one group (4 pairs, one per 32-bit word: x0 in the low half,
// x1 in the high half) and returns them rounded to BF16.
__device__ __forceinline__ uint4 rotate_group(uint4 w, const RopeGroup &g, const TokPos &p) {
    const int pos = g.axis == 0 ? p.t : (g.axis == 1 ? p.h : p.w);
    const float4 c = __ldg(reinterpret_cast<const float4 *>(g.cos + pos * g.half));
    const float4 s = __ldg(reinterpret_cast<const float4 *>(g.sin + pos * g.half));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float x0 = __uint_as_float(u[q] << 16), x1 = __uint_as_float(u[q] & 0xFFFF0000u);
        o[q] = pack_bf16x2(__fsub_rn(__fmul_rn(x0, cc[q]), __fmul_rn(x1, ss[q])),
                           __fadd_rn(__fmul_rn(x0, ss[q]), __fmul_rn(x1, cc[q])));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Rotates the 8 channels [8*g, 8*g+8) of one head row in place (x as fp32), with scalar
// correctly rounded products and sums.  rope3d uses this form (it keeps the kernel's register
// count low); append_quant uses rotate_group.
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

// -------------------------------------------------------------------- quantisation
// max(|a|, |b|) per BF16 half (the sign of each half is the XOR of the operands' signs, which
// the final absolute value discards)
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest |x| of the 16 BF16 values in two 16-byte words, as fp32 (exact).
__device__ __forceinline__ float absmax16(uint4 w0, uint4 w1) {
    const uint32_t t = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(w0.x, w0.y), bf16x2_absmax(w0.z, w0.w)),
                                     bf16x2_absmax(bf16x2_absmax(w1.x, w1.y), bf16x2_absmax(w1.z, w1.w)));
    return fmaxf(__uint_as_float((t << 16) & 0x7FFFFFFFu), __uint_as_float(t & 0x7FFF0000u));
}

// absmax over the 8 lanes of a row group (lanes 8q .. 8q+7 of a warp)
__device__ __forceinline__ float group8_max(float a) {
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    return a;
}

// Codes of this lane's 16 values of a row (8 lanes per row) from the BF16 words and the row's
// absmax a (after the lanes' reduction); the row's scale to scale_out.
__device__ __forceinline__ uint4 quant16(uint4 w0, uint4 w1, float a, float &scale_out) {
    if (a == 0.0f) {
        scale_out = 0.0f;
        return make_uint4(0u, 0u, 0u, 0u);
    }
    const float scale = quant_scale(a);
    scale_out = scale;
    float f[16];
    unpack8(w0, f);
    unpack8(w1, f + 8);
    if (scale >= 0x1p-100f) {
        uint4 c;
        codes_fast<16>(f, scale, &c);
        return c;
    }
    return codes16(f, scale);
}

// One thread: 16 channels of one (token, head) row of K and of V.  8 lanes per row.
__global__ void __launch_bounds__(256, 4) append_quant_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                              int64_t row_stride16, SegPos seg, RopeDev rope,
                                                              uint4 *__restrict__ ck, uint4 *__restrict__ cv,
                                                              float *__restrict__ cks, float *__restrict__ cvs,
                                                              int64_t cap, int64_t length) {
    const int64_t total = static_cast<int64_t>(seg.n_tokens) * seg.heads * 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;  // a multiple of 8
    int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int G = static_cast<int>(i & 7);
    const RopeGroup g0 = rope_group(2 * G, rope), g1 = rope_group(2 * G + 1, rope);
    // the loop condition is uniform over a warp (the shuffles below need all 32 lanes);
    // lanes past the end run with `live` false
    for (; i - (threadIdx.x & 31) < total; i += stride) {
        const bool live = i < total;
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
        const TokPos p = token_pos(seg, tok);
        if (live && p.video) {
            // quantise the BF16-rounded rotated K
            wk0 = rotate_group(wk0, g0, p);
            wk1 = rotate_group(wk1, g1, p);
        }
        const float ak = group8_max(absmax16(wk0, wk1));
        const float av = group8_max(absmax16(wv0, wv1));
        float sk, sv;
        const uint4 qk = quant16(wk0, wk1, ak, sk);
        const uint4 qv = quant16(wv0, wv1, av, sv);
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
    return make_seg_pos(s.t0, s.n_video, s.n_tokens, heads, s.gh, s.gw);
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
