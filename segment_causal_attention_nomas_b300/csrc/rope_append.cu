// rope_append.cu -- 3D RoPE (rope3d) and fused RoPE + INT8 append (append_quant).
//
// Both are HBM-bound streaming kernels.  One (token, head) row of 128 BF16 channels is
// handled by 16 consecutive threads, each owning 8 channels (one 16-byte load): 16
// channel groups of 8 never straddle an axis chunk of the [16, 56, 56] split, so a thread
// reads one cos/sin row segment of one axis.
//
// RoPE (comfyui-wiki news, architecture table: 3D RoPE sizes [16, 56, 56], theta 256):
// pair (x0, x1) of an axis chunk -> (x0*c - x1*s, x0*s + x1*c), every product and sum
// rounded to fp32 (__fmul_rn / __fsub_rn / __fadd_rn: no FMA contraction), then BF16 RNE.
//
// Quantisation (comfyui-wiki, "单张 4090 配置": cached K/V stored as INT8): per row,
// a = max|x|, scale = a / 127 (IEEE fp32 division), code = clamp(rne(x / scale), +-127),
// a == 0 -> scale 0 and all codes 0.  The absmax is a 16-lane shuffle reduction.
#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

struct TokPos {
    int t, h, w;
    bool video;
};

__device__ __forceinline__ TokPos token_pos(const SegDesc &s, int64_t k) {
    TokPos p;
    p.video = k < s.n_video;
    if (p.video) {
        const int hw = s.gh * s.gw;
        const int kk = static_cast<int>(k);
        p.t = s.t0 + kk / hw;
        const int r = kk - (kk / hw) * hw;
        p.h = r / s.gw;
        p.w = r - p.h * s.gw;
    } else {
        p.t = p.h = p.w = -1;
    }
    return p;
}

// Rotates the 8 channels [8*g, 8*g+8) of one head row in place (x as fp32 pairs).
__device__ __forceinline__ void rotate8(float (&x)[8], int g, const TokPos &p, const RopeDev &rope) {
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

__device__ __forceinline__ void unpack8(uint4 w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
    uint4 r;
    r.x = pack_bf16x2(x[0], x[1]);
    r.y = pack_bf16x2(x[2], x[3]);
    r.z = pack_bf16x2(x[4], x[5]);
    r.w = pack_bf16x2(x[6], x[7]);
    return r;
}

// x and y may be the same buffer (in place): each element is read and written by one thread.
__global__ void __launch_bounds__(256) rope3d_kernel(const uint4 *x, uint4 *y,
                                                     int64_t row_stride16, SegDesc seg, int heads, RopeDev rope) {
    const int64_t total = static_cast<int64_t>(seg.n_tokens) * heads * 16;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int g = static_cast<int>(i & 15);
        const int64_t row = i >> 4;
        const int64_t k = row / heads;
        const int h = static_cast<int>(row - k * heads);
        const int64_t off = k * row_stride16 + h * 16 + g;
        uint4 w = x[off];
        const TokPos p = token_pos(seg, k);
        if (p.video) {
            float f[8];
            unpack8(w, f);
            rotate8(f, g, p, rope);
            w = pack8_bf16(f);
        }
        y[off] = w;
    }
}

// absmax over the 16 lanes of a row group (lanes 16q .. 16q+15 of a warp)
__device__ __forceinline__ float group16_max(float a) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    return a;
}

// Quantises this lane's 8 values of a row; returns the 8 codes as two words.
__device__ __forceinline__ uint2 quant8(const float (&x)[8], float &scale_out) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
    a = group16_max(a);
    uint2 r = make_uint2(0u, 0u);
    if (a == 0.0f) {
        scale_out = 0.0f;
        return r;
    }
    const float scale = __fdiv_rn(a, 127.0f);
    scale_out = scale;
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = __float2int_rn(__fdiv_rn(x[i], scale));
        q = max(-127, min(127, q));
        b[i] = static_cast<uint32_t>(q) & 0xFFu;
    }
    r.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
    r.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    return r;
}

// One thread: 8 channels of one (token, head) row of K and of V.  16 lanes per row.
__global__ void __launch_bounds__(256) append_quant_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                           int64_t row_stride16, SegDesc seg, int heads, RopeDev rope,
                                                           uint2 *__restrict__ ck, uint2 *__restrict__ cv,
                                                           float *__restrict__ cks, float *__restrict__ cvs,
                                                           int64_t cap, int64_t length) {
    const int64_t total = static_cast<int64_t>(seg.n_tokens) * heads * 16;
    // the loop condition is uniform over a warp (the shuffles below need all 32 lanes);
    // lanes past the end run with `live` false
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i - (threadIdx.x & 31) < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool live = i < total;
        const int g = static_cast<int>(i & 15);
        const int64_t row = live ? (i >> 4) : 0;
        const int64_t tok = row / heads;
        const int h = static_cast<int>(row - tok * heads);
        const int64_t off = tok * row_stride16 + h * 16 + g;
        uint4 wk = live ? k[off] : make_uint4(0, 0, 0, 0);
        uint4 wv = live ? v[off] : make_uint4(0, 0, 0, 0);
        float fk[8], fv[8];
        unpack8(wk, fk);
        unpack8(wv, fv);
        const TokPos p = token_pos(seg, tok);
        if (live && p.video) {
            rotate8(fk, g, p, rope);
            // quantise the BF16-rounded rotated K
            uint4 r = pack8_bf16(fk);
            unpack8(r, fk);
        }
        float sk, sv;
        const uint2 qk = quant8(fk, sk);
        const uint2 qv = quant8(fv, sv);
        if (live) {
            const int64_t dst = static_cast<int64_t>(h) * cap + length + tok;
            ck[dst * 16 + g] = qk;
            cv[dst * 16 + g] = qv;
            if (g == 0) {
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

}  // namespace

cudaError_t launch_rope3d(const void *x, void *y, int64_t row_stride, const SegDesc &seg, int32_t heads,
                          const RopeDev &rope, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(seg.n_tokens) * heads * 16;
    if (threads == 0) return cudaSuccess;
    rope3d_kernel<<<grid_for(threads), 256, 0, stream>>>(static_cast<const uint4 *>(x), static_cast<uint4 *>(y),
                                                         row_stride / 8, seg, heads, rope);
    return cudaGetLastError();
}

cudaError_t launch_append_quant(const void *k, const void *v, int64_t row_stride, const SegDesc &seg,
                                int32_t heads, const RopeDev &rope, int8_t *ck, int8_t *cv, float *cks,
                                float *cvs, int64_t cap, int64_t length, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(seg.n_tokens) * heads * 16;
    if (threads == 0) return cudaSuccess;
    append_quant_kernel<<<grid_for(threads), 256, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), row_stride / 8, seg, heads, rope,
        reinterpret_cast<uint2 *>(ck), reinterpret_cast<uint2 *>(cv), cks, cvs, cap, length);
    return cudaGetLastError();
}

}  // namespace nomas
