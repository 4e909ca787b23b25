// qkv_proj.cu -- W8A16 QKV projection with the 3D RoPE fused into its epilogue (tcgen05, sm_103a).
//
// The linear layer in front of every attention of a dual-stream block (comfyui-wiki news,
// 模型内部: hidden size 2,048 = 16 heads x 128; 单张 4090 配置: DiT weights stored INT8, linear
// layers computed in BF16): qkv[l, n] = scale[n] * sum_k x[l, k] * code[n, k], output channels
// [0, H*128) = Q, [H*128, 2H*128) = K, [2H*128, 3H*128) = V (head-major inside each), then Q and
// K rotated by the 3D RoPE of the token's (t, h, w) exactly as nomas_rope3d does it (the rotation
// starts from the BF16-rounded projection), V left as projected.
//
// Two kernels:
//   codes_to_bf16_kernel  the INT8 codes as BF16 (exact: |code| <= 127 needs 7 bits), once per
//                         call, into the caller's workspace; the scales stay fp32 for the epilogue.
//   qkv_proj_kernel       one CTA per 128 x 256 output tile (192 threads), two CTAs per SM (97 KB
//                         of shared memory and 256 TMEM columns each), so one CTA's epilogue
//                         overlaps the other's main loop (measured: 25 % faster than one CTA
//                         per SM with a 4-deep ring):
//     warp 0   TMA producer: x and code tiles, 64 hidden channels per stage (one 128-byte
//              swizzle row), in a 2-deep ring (48 KB a stage).
//     warp 1   MMA issuer: D[128 x 256] += X[128 x 16] . C[256 x 16]^T, kind::f16 with BF16 operands
//              (M = 128, N = 256), fp32 accumulator in TMEM (256 columns).
//     warps 2-5 epilogue, one thread per token row (TMEM lane = row): D * scale rounded to BF16,
//              RoPE on Q/K video tokens (scalar correctly rounded products and sums, as in
//              rope3d), BF16 stored to the fused [L][3][H][128] output.
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "quant.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr int PM = 128;             // token rows per tile
constexpr int PN = 256;             // output channels per tile
constexpr int PK = 64;              // hidden channels per stage
constexpr int kStages = 2;
constexpr int kProjThreads = 192;
constexpr uint32_t P_A = 0;                           // kStages x [128 rows][128 B]
constexpr uint32_t P_B = P_A + kStages * 16384;       // kStages x [256 rows][128 B]
constexpr uint32_t P_BAR = P_B + kStages * 32768;
constexpr uint32_t P_MISC = P_BAR + 128;
constexpr uint32_t P_TOTAL = P_MISC + 64;
static_assert(P_TOTAL <= 232448, "shared memory map exceeds 227 KB");

enum { PB_FULL = 0, PB_FREE = PB_FULL + kStages, PB_DONE = PB_FREE + kStages, PB_COUNT = PB_DONE + 1 };
static_assert(PB_COUNT * 8 <= 128, "barrier area");
// PB_FULL[s] is waited by the MMA thread only and PB_FREE[s] by the producer only, each one
// phase per use of stage s; a stage is refilled only after its MMAs completed.

struct ProjParams {
    int32_t lq, hidden, heads;
    int64_t out_stride;   // elements between consecutive tokens of the output
    uint16_t *out;
    const float *scale;   // [3 * heads * 128]
    SegPos seg;
    RopeDev rope;
    int *status;
    // fused append (kAppend): K and V of token l go to cache row length + l of every head
    uint4 *ck, *cv;       // int8 [heads][cap][128]
    float *cks, *cvs;     // [heads][cap]
    int64_t cap, length;
};

// One 32-channel chunk of a token's projection, channels n .. n + 31: the accumulator times the
// channel scales rounded to BF16, then (Q and K video tokens) the 3D RoPE in scalar correctly
// rounded arithmetic exactly as rope3d does it.  o[j] holds channels n + 2j, n + 2j + 1.
__device__ __forceinline__ void proj_chunk(const uint32_t (&r)[32], int n, bool rotate, const TokPos &tp,
                                           const ProjParams &p, uint32_t (&o)[16]) {
    const int d0 = n % kHeadDim;  // first channel of this chunk within its head
    const float4 *sc4 = reinterpret_cast<const float4 *>(p.scale + n);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float4 s4 = __ldg(sc4 + (i >> 1));
        const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int j = i + h2;  // pair j: chunk columns 2j, 2j + 1
            // the BF16-rounded projection, as fp32
            const uint32_t pw =
                pack_bf16x2(__uint_as_float(r[2 * j]) * sc[2 * h2], __uint_as_float(r[2 * j + 1]) * sc[2 * h2 + 1]);
            float x0 = __uint_as_float(pw << 16), x1 = __uint_as_float(pw & 0xFFFF0000u);
            if (rotate) {
                const int d = d0 + 2 * j;
                const int axis = d < 16 ? 0 : (d < 72 ? 1 : 2);
                const int pair = (d - (axis == 0 ? 0 : (axis == 1 ? 16 : 72))) >> 1;
                const int half = axis == 0 ? 8 : 28;
                const int pos = axis == 0 ? tp.t : (axis == 1 ? tp.h : tp.w);
                const float *ct = axis == 0 ? p.rope.cos[0] : (axis == 1 ? p.rope.cos[1] : p.rope.cos[2]);
                const float *st = axis == 0 ? p.rope.sin[0] : (axis == 1 ? p.rope.sin[1] : p.rope.sin[2]);
                const float cv = __ldg(ct + pos * half + pair), sv = __ldg(st + pos * half + pair);
                const float y0 = __fsub_rn(__fmul_rn(x0, cv), __fmul_rn(x1, sv));
                const float y1 = __fadd_rn(__fmul_rn(x0, sv), __fmul_rn(x1, cv));
                x0 = y0;
                x1 = y1;
            }
            o[j] = pack_bf16x2(x0, x1);
        }
    }
}

__device__ __forceinline__ void store_chunk(const ProjParams &p, int tok, int n, const uint32_t (&o)[16]) {
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(tok) * p.out_stride + n);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    dst[2] = make_uint4(o[8], o[9], o[10], o[11]);
    dst[3] = make_uint4(o[12], o[13], o[14], o[15]);
}

// The cache row of one (token, head) from its 128 BF16 values (64 words, channel pairs): the
// same absmax, scale and quotient as append_quant_kernel.
__device__ __forceinline__ void quantise_row(const uint32_t (&hw)[64], uint4 *codes, float *scale_out) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < 64; ++w)
        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(hw[w] << 16)), fabsf(__uint_as_float(hw[w] & 0xFFFF0000u))));
    if (a == 0.0f) {
#pragma unroll
        for (int g = 0; g < 8; ++g) codes[g] = make_uint4(0u, 0u, 0u, 0u);
        *scale_out = 0.0f;
        return;
    }
    const float scale = quant_scale(a);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        float x[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            x[2 * e] = __uint_as_float(hw[8 * g + e] << 16);
            x[2 * e + 1] = __uint_as_float(hw[8 * g + e] & 0xFFFF0000u);
        }
        codes[g] = codes16(x, scale);
    }
    *scale_out = scale;
}

__device__ __noinline__ void proj_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_test(addr, parity)) return;
        if ((spin & 255u) == 255u && globaltimer_ns() - t0 > 50000000ull) return;
    }
}

template <bool kAppend>
__global__ void __launch_bounds__(kProjThreads, 2)
qkv_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                const __grid_constant__ ProjParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * PM;
    const int n0 = blockIdx.y * PN;
    const int n_k = p.hidden / PK;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) record_status(p.status, kStatusTimeout, 950);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P_MISC + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[PB_FULL + s], 1);
            mbar_init(&bars[PB_FREE + s], 1);
        }
        mbar_init(&bars[PB_DONE], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================================== producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_c);
            uint32_t armed = 0, armed_par = 0;
            for (int kt = 0; kt < n_k; ++kt) {
                const int s = kt % kStages;
                const uint32_t u = static_cast<uint32_t>(kt / kStages) & 1u;
                if (!mbar_wait(&bars[PB_FREE + s], u ^ 1u, p.status, abort_flag, 501)) break;
                mbar_arrive_expect_tx(&bars[PB_FULL + s], 16384 + 32768);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (u << s);
                tma_load_2d(smem + P_A + s * 16384, &tm_x, &bars[PB_FULL + s], kt * PK, m0);
                tma_load_2d(smem + P_B + s * 32768, &tm_c, &bars[PB_FULL + s], kt * PK, n0);
            }
            for (int s = 0; s < kStages; ++s)
                if (armed & (1u << s)) proj_drain(&bars[PB_FULL + s], (armed_par >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ======================================================================= MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(true, false, PM, PN);  // BF16 x BF16, both K-major
            for (int kt = 0; kt < n_k; ++kt) {
                const int s = kt % kStages;
                const uint32_t u = static_cast<uint32_t>(kt / kStages) & 1u;
                if (!mbar_wait(&bars[PB_FULL + s], u, p.status, abort_flag, 502)) break;
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + P_A + s * 16384), sb = smem_u32(smem + P_B + s * 32768);
#pragma unroll
                for (int kk = 0; kk < PK / 16; ++kk)
                    mma_ss(tmem, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024), idesc,
                           (kt > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&bars[PB_FREE + s]);
            }
            tc_commit(&bars[PB_DONE]);
            proj_drain(&bars[PB_DONE], 0);  // no MMA may still run when TMEM is freed
        }
        __syncwarp();
    } else {
        // ================================================================== epilogue
        const int q = warp & 3;  // TMEM lane quarter
        const int row = q * 32 + lane;
        const int tok = m0 + row;
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_DONE], 0, p.status, abort_flag, 503));
        if (ok) {
            tc_fence_after();
            const int per = p.heads * kHeadDim;  // channels of each of Q, K, V
            const int which = n0 / per;          // a tile lies inside one of Q, K, V (per is a multiple of 256)
            const bool live = tok < p.lq;
            const TokPos tp = token_pos(p.seg, static_cast<uint32_t>(live ? tok : 0));
            const bool rotate = live && which < 2 && tp.video;
            const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
            if (kAppend && which > 0) {
                // K or V tile (two heads): each head's 128 values also go to the cache
#pragma unroll 1
                for (int hb = 0; hb < 2; ++hb) {
                    uint32_t hw[64];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = hb * 4 + cc;
                        uint32_t r[32];
                        tmem_ld32(trow + c * 32, r);
                        tmem_wait_ld(r);
                        uint32_t o[16];
                        proj_chunk(r, n0 + c * 32, rotate, tp, p, o);
                        if (live) store_chunk(p, tok, n0 + c * 32, o);
#pragma unroll
                        for (int j = 0; j < 16; ++j) hw[cc * 16 + j] = o[j];
                    }
                    if (live) {
                        const int head = (n0 % per) / kHeadDim + hb;
                        const int64_t dst = static_cast<int64_t>(head) * p.cap + p.length + tok;
                        quantise_row(hw, (which == 1 ? p.ck : p.cv) + dst * 8, (which == 1 ? p.cks : p.cvs) + dst);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < PN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(trow + c * 32, r);
                    tmem_wait_ld(r);
                    if (!live) continue;
                    uint32_t o[16];
                    proj_chunk(r, n0 + c * 32, rotate, tp, p, o);
                    store_chunk(p, tok, n0 + c * 32, o);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// The INT8 codes as BF16 (exact), 16 codes per item.
__global__ void __launch_bounds__(256) codes_to_bf16_kernel(const int8_t *__restrict__ codes, int64_t n,
                                                            uint16_t *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(codes) + i);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
        uint32_t h[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float f[4];
            s8x4_to_f32(words[q], f);
            h[2 * q] = pack_bf16x2(f[0], f[1]);
            h[2 * q + 1] = pack_bf16x2(f[2], f[3]);
        }
        uint4 *d = reinterpret_cast<uint4 *>(out) + 2 * i;
        d[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

bool encode2d(CUtensorMap *m, void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_outer,
              char *err, size_t err_len, const char *what) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) {
        snprintf(err, err_len, "cuTensorMapEncodeTiled unavailable");
        return false;
    }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {PK, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(err, err_len, "tensor map for %s rejected (CUresult %d)", what, static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace

size_t qkv_project_workspace_bytes(int32_t heads, int32_t hidden) {
    return static_cast<size_t>(3) * heads * kHeadDim * hidden * 2;
}

nomas_status launch_qkv_project(const QkvLaunch &a, cudaStream_t stream, char *err, size_t err_len) {
    const bool append = a.cache != nullptr;
    static bool attr_set[2][64] = {{false}};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[append][dev]) {
        cudaError_t e =
            append ? cudaFuncSetAttribute(qkv_proj_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_TOTAL)
                   : cudaFuncSetAttribute(qkv_proj_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_TOTAL);
        if (e != cudaSuccess) {
            snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
        if (dev >= 0 && dev < 64) attr_set[append][dev] = true;
    }
    const int64_t n_out = 3ll * a.heads * kHeadDim;
    uint16_t *cb = static_cast<uint16_t *>(a.workspace);  // codes as BF16, [n_out][hidden]
    CUtensorMap tx, tc;
    if (!encode2d(&tx, const_cast<void *>(a.x), a.hidden, a.lq, a.x_row_stride * 2, PM, err, err_len, "x") ||
        !encode2d(&tc, cb, a.hidden, n_out, static_cast<uint64_t>(a.hidden) * 2, PN, err, err_len, "weights"))
        return NOMAS_EINVAL;
    const int sms = device_sm_count();
    const int64_t items = n_out * a.hidden / 16;
    int64_t blocks = (items + 255) / 256;
    if (blocks > sms * 8) blocks = sms * 8;
    codes_to_bf16_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(a.w_codes, items, cb);
    ProjParams p;
    memset(&p, 0, sizeof(p));
    p.lq = a.lq;
    p.hidden = a.hidden;
    p.heads = a.heads;
    p.out_stride = a.out_row_stride;
    p.out = static_cast<uint16_t *>(a.out);
    p.scale = a.w_scale;
    p.seg = make_seg_pos(a.seg.t0, a.seg.n_video, a.seg.n_tokens, a.heads, a.seg.gh, a.seg.gw);
    p.rope = a.rope;
    p.status = device_status_word();
    const dim3 grid(static_cast<unsigned>((a.lq + PM - 1) / PM), static_cast<unsigned>(n_out / PN));
    if (append) {
        p.ck = reinterpret_cast<uint4 *>(a.cache->k);
        p.cv = reinterpret_cast<uint4 *>(a.cache->v);
        p.cks = a.cache->k_scale;
        p.cvs = a.cache->v_scale;
        p.cap = a.cache->capacity;
        p.length = a.cache->length;
        qkv_proj_kernel<true><<<grid, kProjThreads, P_TOTAL, stream>>>(tx, tc, p);
    } else {
        qkv_proj_kernel<false><<<grid, kProjThreads, P_TOTAL, stream>>>(tx, tc, p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "qkv_project launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    return NOMAS_OK;
}

}  // namespace nomas
