// camera.cu -- camera conditioning: camera tokens and the camera cross-attention (sm_103a).
//
// comfyui-wiki news, 相机控制作为一等输入: a trajectory gives camera-to-world matrices c2ws
// [N, 4, 4]; the extrinsics are normalised, grouped by four video frames and each group is
// flattened to a 64-value input, which the video tokens query through a cross-attention in every
// dual-stream block (模型内部 table, 相机条件 row); trajectory_translation_scale defaults to 1.0
// and trajectory_rotation_scale to 2.5.
//
// Two kernels:
//   camera_tokens_kernel  one thread per video frame i: E_i = inverse(c2w[0]) . c2w[i] with the
//                         rigid inverse [R0^T | -R0^T t0]; the rotation block times
//                         rotation_scale, the translation column times translation_scale, the
//                         bottom row (0, 0, 0, 1); the 16 values row-major at token i / 4,
//                         columns 16 (i % 4) .. 16 (i % 4) + 15.  fp32.
//   camera_xattn_kernel   one CTA (128 threads) per (128 video tokens, head), O = softmax(q k^T *
//                         scale) v over all camera tokens of the segment:
//     TMA   the Q tile [128 tokens][128] BF16 and the head's camera K, V [NC][128] BF16 (NC = the
//           camera-token count rounded up to 32; rows past the last token arrive as zeros), in
//           128-byte-swizzled boxes of 64 channels.
//     MMA   S[128 x NC] = Q . K^T  (kind::f16 with BF16 operands, M = 128, N = NC, fp32 in TMEM).
//     all   one thread per query row (TMEM lane = row): the row maximum over the real camera
//           tokens, p = 2^(s * c - max * c) (c = scale * log2 e) rounded to FP16, l = the sum of
//           the rounded p, P written K-major and swizzled over the Q tile (Q is dead once S is
//           complete); the tile's V converted in place from BF16 to FP16 (exact for |v| in FP16's
//           normal range, as for the staged operands of the segment attention).
//     MMA   O[128 x 128] = P . V  (kind::f16 with FP16 operands, V MN-major), fp32 in the TMEM
//           columns S occupied (every row of S is in registers before this MMA is issued).
//     all   O / l rounded to BF16, written swizzled over the tile buffer; one thread stores the
//           two 64-channel boxes with TMA (rows past the last token are not written).
//   Shared memory: 32 KB for the tile plus 512 B per padded camera token (four CTAs per SM at up
//   to 32 camera tokens); TMEM: 128 columns.  The kernel moves 512 B per (token, head) from and
//   to HBM plus the camera K and V from L2: it is bound by HBM bandwidth.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr int CM = 128;          // query rows per tile
constexpr int kCamThreads = 128;
constexpr uint32_t C_Q = 0;      // [2][128 rows][128 B]: Q, then P, then O
constexpr uint32_t C_K = 32768;  // [2][NC rows][128 B], then V the same
enum { CB_LOAD = 0, CB_S, CB_O, CB_COUNT };

uint32_t cam_smem_bytes(int nc) { return C_K + static_cast<uint32_t>(nc) * 512u + 64u; }

struct CamParams {
    int32_t lq, heads, n_cam, nc;
    float scale_log2;  // softmax scale * log2(e)
    int *status;
};

// Bounded wait that ignores the abort flag: an operation this CTA issued must finish before its
// shared memory or TMEM is released.
__device__ __noinline__ void cam_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_test(addr, parity)) return;
        if ((spin & 255u) == 255u && globaltimer_ns() - t0 > 50000000ull) return;
    }
}

// Writes 32 consecutive 16-bit columns (16 words) of row `row` into a K-major, 128-byte-swizzled
// [128 rows][64 columns] block pair: columns 32c .. 32c + 31 lie in block c / 2, 16-byte chunks
// 4 (c % 2) .. 4 (c % 2) + 3 of the row, each chunk index XORed with row % 8.
__device__ __forceinline__ void store_row_chunk32(uint8_t *tile, int row, int c, const uint32_t (&w)[16]) {
    uint8_t *base = tile + (c >> 1) * 16384 + row * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int chunk = ((c & 1) * 4 + i) ^ (row & 7);
        *reinterpret_cast<uint4 *>(base + chunk * 16) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

__global__ void __launch_bounds__(kCamThreads, 4)
camera_xattn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CamParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int row = tid;  // query row of this thread = TMEM lane
    const int head = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.heads));
    const int tok0 = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.heads)) * CM;
    const int nc = p.nc;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0) record_status(p.status, kStatusTimeout, 960);
        return;
    }
    uint8_t *sq = smem + C_Q;
    uint8_t *sk = smem + C_K;
    uint8_t *sv = sk + nc * 256;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sv + nc * 256);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + CB_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    if (tid == 0) {
        for (int b = 0; b < CB_COUNT; ++b) mbar_init(&bars[b], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);

    bool issued_s = false, issued_o = false;
    if (tid == 0) {
        tma_prefetch_desc(&tm_q);
        mbar_arrive_expect_tx(&bars[CB_LOAD], 32768u + static_cast<uint32_t>(nc) * 512u);
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(sq + half * 16384, &tm_q, &bars[CB_LOAD], half * 64, head, tok0);
            tma_load_3d(sk + half * nc * 128, &tm_k, &bars[CB_LOAD], half * 64, head, 0);
            tma_load_3d(sv + half * nc * 128, &tm_v, &bars[CB_LOAD], half * 64, head, 0);
        }
        if (mbar_wait(&bars[CB_LOAD], 0, p.status, abort_flag, 601)) {
            tc_fence_after();
            const uint32_t idesc = idesc_f16(true, false, CM, nc);  // BF16 x BF16, both K-major
            const uint32_t aq = smem_u32(sq), ak = smem_u32(sk);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem, sdesc_sw128(aq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                       sdesc_sw128(ak + (kk >> 2) * nc * 128 + (kk & 3) * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
            tc_commit(&bars[CB_S]);
            issued_s = true;
        }
    }

    // ---------------------------------------------------------------- softmax, P and V to FP16
    float l = 0.0f;
    bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bars[CB_S], 0, p.status, abort_flag, 602));
    // this thread's own observation of the load, so that the copied V is visible to it
    ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(&bars[CB_LOAD], 0, p.status, abort_flag, 603));
    if (ok) {
        tc_fence_after();
        const float c = p.scale_log2;
        float m = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < nc / 32; ++ch) {
            uint32_t r[32];
            tmem_ld32(trow + ch * 32, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (ch * 32 + j < p.n_cam) m = fmaxf(m, __uint_as_float(r[j]));
        }
        const float mc = m * c;
#pragma unroll 1
        for (int ch = 0; ch < nc / 32; ++ch) {
            uint32_t r[32];
            tmem_ld32(trow + ch * 32, r);
            tmem_wait_ld(r);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = ch * 32 + 2 * j;
                const float p0 = col < p.n_cam ? ex2_approx(fmaf(__uint_as_float(r[2 * j]), c, -mc)) : 0.0f;
                const float p1 = col + 1 < p.n_cam ? ex2_approx(fmaf(__uint_as_float(r[2 * j + 1]), c, -mc)) : 0.0f;
                w[j] = pack_f16x2_sat(p0, p1);
                const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
                l += __low2float(h) + __high2float(h);
            }
            store_row_chunk32(sq, row, ch, w);
        }
        uint4 *v4 = reinterpret_cast<uint4 *>(sv);
        for (int i = tid; i < nc * 16; i += kCamThreads) v4[i] = bf16x8_to_f16x8(v4[i]);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok && !*abort_flag) {
        tc_fence_after();
        const uint32_t idesc = idesc_f16(false, true, CM, kHeadDim);  // FP16, V MN-major
        const uint32_t ap = smem_u32(sq), av = smem_u32(sv);
#pragma unroll 1
        for (int kk = 0; kk < nc / 16; ++kk)
            mma_ss(tmem, sdesc_sw128(ap + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(av + kk * 2048, nc * 128, 1024), idesc, kk > 0 ? 1u : 0u);
        tc_commit(&bars[CB_O]);
        issued_o = true;
    }

    // ------------------------------------------------------------------------------ epilogue
    ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(&bars[CB_O], 0, p.status, abort_flag, 604));
    if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;  // l >= 1: the row maximum contributes 2^0
#pragma unroll 1
        for (int ch = 0; ch < kHeadDim / 32; ++ch) {
            uint32_t r[32];
            tmem_ld32(trow + ch * 32, r);
            tmem_wait_ld(r);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                w[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv_l, __uint_as_float(r[2 * j + 1]) * inv_l);
            store_row_chunk32(sq, row, ch, w);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        if (ok && !*abort_flag) {
            for (int half = 0; half < 2; ++half) tma_store_3d(&tm_o, sq + half * 16384, half * 64, head, tok0);
            bulk_commit_group();
            bulk_wait_group_read0();
        }
        // nothing this CTA issued may still run when its shared memory and TMEM are released
        cam_drain(&bars[CB_LOAD], 0);
        if (issued_s) cam_drain(&bars[CB_S], 0);
        if (issued_o) cam_drain(&bars[CB_O], 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

__global__ void camera_tokens_kernel(const float *__restrict__ c2w, int32_t n_frames, float ts, float rs,
                                     float *__restrict__ tokens) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_frames) return;
    float a[12], b[12];  // first three rows of c2w[0] and c2w[i]
    const float4 *a4 = reinterpret_cast<const float4 *>(c2w);
    const float4 *b4 = reinterpret_cast<const float4 *>(c2w + 16ll * i);
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const float4 x = __ldg(a4 + r), y = __ldg(b4 + r);
        a[4 * r] = x.x, a[4 * r + 1] = x.y, a[4 * r + 2] = x.z, a[4 * r + 3] = x.w;
        b[4 * r] = y.x, b[4 * r + 1] = y.y, b[4 * r + 2] = y.z, b[4 * r + 3] = y.w;
    }
    float e[16];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        // row r of R0^T R_i and of R0^T (t_i - t0): sums over k of R0[k][r] * (.)[k]
#pragma unroll
        for (int c = 0; c < 3; ++c) e[4 * r + c] = rs * (a[r] * b[c] + a[4 + r] * b[4 + c] + a[8 + r] * b[8 + c]);
        e[4 * r + 3] = ts * (a[r] * (b[3] - a[3]) + a[4 + r] * (b[7] - a[7]) + a[8 + r] * (b[11] - a[11]));
    }
    e[12] = 0.0f, e[13] = 0.0f, e[14] = 0.0f, e[15] = 1.0f;
    float4 *o = reinterpret_cast<float4 *>(tokens + 64ll * (i / 4) + 16 * (i % 4));
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] = make_float4(e[4 * r], e[4 * r + 1], e[4 * r + 2], e[4 * r + 3]);
}

// 3D map {128 channels, heads, tokens} over a [tokens][heads][128] BF16 tensor, box {64, 1, rows}.
bool encode_rows(CUtensorMap *m, const void *base, int32_t heads, int64_t tokens, int64_t row_stride,
                 uint32_t box_rows, char *err, size_t err_len, const char *what) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) {
        snprintf(err, err_len, "cuTensorMapEncodeTiled unavailable");
        return false;
    }
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, static_cast<cuuint64_t>(row_stride) * 2};
    const cuuint32_t box[3] = {64, 1, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(err, err_len, "tensor map for %s rejected (CUresult %d)", what, static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace

cudaError_t launch_camera_tokens(const float *c2w, int32_t n_frames, float translation_scale,
                                 float rotation_scale, float *tokens, cudaStream_t stream) {
    const int threads = 128;
    camera_tokens_kernel<<<(n_frames + threads - 1) / threads, threads, 0, stream>>>(c2w, n_frames, translation_scale,
                                                                                    rotation_scale, tokens);
    return cudaGetLastError();
}

nomas_status launch_camera_xattn(const CamLaunch &a, cudaStream_t stream, char *err, size_t err_len) {
    const int nc = (a.n_cam + 31) / 32 * 32;
    const uint32_t smem = cam_smem_bytes(nc);
    static uint32_t attr_bytes[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || attr_bytes[dev] < smem) {
        cudaError_t e =
            cudaFuncSetAttribute(camera_xattn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cam_smem_bytes(128));
        if (e != cudaSuccess) {
            snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
        if (dev >= 0 && dev < 64) attr_bytes[dev] = cam_smem_bytes(128);
    }
    CUtensorMap tq, tk, tv, to;
    if (!encode_rows(&tq, a.q, a.heads, a.lq, a.q_row_stride, CM, err, err_len, "q") ||
        !encode_rows(&tk, a.k, a.heads, a.n_cam, a.cam_row_stride, nc, err, err_len, "camera k") ||
        !encode_rows(&tv, a.v, a.heads, a.n_cam, a.cam_row_stride, nc, err, err_len, "camera v") ||
        !encode_rows(&to, a.out, a.heads, a.lq, a.out_row_stride, CM, err, err_len, "out"))
        return NOMAS_EINVAL;
    CamParams p;
    memset(&p, 0, sizeof(p));
    p.lq = a.lq;
    p.heads = a.heads;
    p.n_cam = a.n_cam;
    p.nc = nc;
    const float scale = a.softmax_scale != 0.0f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(kHeadDim));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = device_status_word();
    const int64_t ctas = (static_cast<int64_t>(a.lq) + CM - 1) / CM * a.heads;
    camera_xattn_kernel<<<static_cast<unsigned>(ctas), kCamThreads, smem, stream>>>(tq, tk, tv, to, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "camera_xattn launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    return NOMAS_OK;
}

}  // namespace nomas
