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
//   qkv_proj_pair_kernel  a persistent CTA-pair GEMM (cta_group::2, 256 x 256 tiles) whose epilogue
//                         (one thread per token row: D * scale rounded to BF16, RoPE on Q/K video
//                         tokens in scalar correctly rounded products and sums as in rope3d, BF16
//                         stored to the fused [L][3][H][128] output) overlaps the next tile's MMAs;
//                         its layout is described above the kernel.
#include <algorithm>
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
// rounded arithmetic exactly as rope3d does it.  o[j] holds channels n + 2j, n + 2j + 1.  The
// chunk is four groups of 8 channels; no group straddles an axis chunk of the [16, 56, 56] split,
// so each group's 4 cos and 4 sin values are one 16-byte load each.
__device__ __forceinline__ void proj_chunk(const uint32_t (&r)[32], int n, bool rotate, const TokPos &tp,
                                           const ProjParams &p, uint32_t (&o)[16]) {
    const int d0 = n % kHeadDim;  // first channel of this chunk within its head
    const float4 *sc4 = reinterpret_cast<const float4 *>(p.scale + n);
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
        const float4 sa = __ldg(sc4 + 2 * gi), sb = __ldg(sc4 + 2 * gi + 1);
        const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
        float cs[4] = {1.0f, 1.0f, 1.0f, 1.0f}, sn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (rotate) {
            const int d = d0 + 8 * gi;
            const int axis = d < 16 ? 0 : (d < 72 ? 1 : 2);
            const int pair0 = (d - (axis == 0 ? 0 : (axis == 1 ? 16 : 72))) >> 1;
            const int half = axis == 0 ? 8 : 28;
            const int pos = axis == 0 ? tp.t : (axis == 1 ? tp.h : tp.w);
            const float *ct = axis == 0 ? p.rope.cos[0] : (axis == 1 ? p.rope.cos[1] : p.rope.cos[2]);
            const float *st = axis == 0 ? p.rope.sin[0] : (axis == 1 ? p.rope.sin[1] : p.rope.sin[2]);
            const float4 c4 = __ldg(reinterpret_cast<const float4 *>(ct + pos * half + pair0));
            const float4 s4 = __ldg(reinterpret_cast<const float4 *>(st + pos * half + pair0));
            cs[0] = c4.x, cs[1] = c4.y, cs[2] = c4.z, cs[3] = c4.w;
            sn[0] = s4.x, sn[1] = s4.y, sn[2] = s4.z, sn[3] = s4.w;
        }
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
            const int j = 4 * gi + h2;  // pair j: chunk columns 2j, 2j + 1
            // the BF16-rounded projection, as fp32
            const uint32_t pw =
                pack_bf16x2(__uint_as_float(r[2 * j]) * sc[2 * h2], __uint_as_float(r[2 * j + 1]) * sc[2 * h2 + 1]);
            float x0 = __uint_as_float(pw << 16), x1 = __uint_as_float(pw & 0xFFFF0000u);
            if (rotate) {
                const float y0 = __fsub_rn(__fmul_rn(x0, cs[h2]), __fmul_rn(x1, sn[h2]));
                const float y1 = __fadd_rn(__fmul_rn(x0, sn[h2]), __fmul_rn(x1, cs[h2]));
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

// Largest |x| of the 32 BF16 values of one chunk (16 words of channel pairs), as fp32 (exact).
__device__ __forceinline__ float chunk_absmax(const uint32_t (&o)[16]) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < 16; ++w)
        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(o[w] << 16)), fabsf(__uint_as_float(o[w] & 0xFFFF0000u))));
    return a;
}

// The 32 codes of one chunk (16 words of channel pairs) of a cache row whose scale is `scale`
// (> 0), with the append kernel's rule: two 16-byte words.
__device__ __forceinline__ void chunk_codes(const uint32_t (&o)[16], float scale, uint4 *codes) {
    float x[32];
#pragma unroll
    for (int w = 0; w < 16; ++w) {
        x[2 * w] = __uint_as_float(o[w] << 16);
        x[2 * w + 1] = __uint_as_float(o[w] & 0xFFFF0000u);
    }
    if (scale >= 0x1p-100f) {
        codes_fast<32>(x, scale, codes);
    } else {
        codes[0] = codes16(x, scale);
        codes[1] = codes16(x + 16, scale);
    }
}

__device__ __noinline__ void proj_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_test(addr, parity)) return;
        if ((spin & 255u) == 255u && globaltimer_ns() - t0 > 50000000ull) return;
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
// A cluster of two CTAs (one per SM of a pair) computes 256 x 256 output tiles with cta_group::2
// MMAs (M = 256, N = 256): CTA r of the pair loads its own 128 token rows of x and weight rows
// n0 + 128 r .. + 127 (half of the tile's N) each stage, so per SM the bytes loaded per FLOP are
// two thirds of a single-CTA 128 x 256 tile's.  The kernel is persistent: each cluster walks the
// tiles t = cluster, cluster + clusters, ... (the N tiles of one 256-row band of x consecutively,
// so the band stays in L2 while the weight tiles stream past it), one cluster per pair of SMs, with
//   warp 0    TMA producer (both CTAs): a ring of stages (PairCfg) that runs on across tiles;
//             each stage's copies complete on the leader's full barrier, which both CTAs arm
//             with their own bytes;
//   warp 1    MMA issuer (the leader only): a tile's stages (hidden / (64 kBoxes): 16 or 32 at
//             hidden 2,048) into one of two TMEM accumulators (256 columns each); every commit
//             arrives on the barrier of both CTAs (multicast);
//   warps 2-9 epilogue (both CTAs): warp w takes TMEM lane quarter w % 4 and one of the tile's two
//             heads; it processes tile i from accumulator i % 2 while the MMAs of tile i + 1 fill
//             the other, and hands the accumulator back to the leader (a remote arrive).
// The accumulator rows of CTA r (128 x 256 fp32) are in CTA r's tensor memory.
constexpr int kPairAccs = 2;       // TMEM accumulators per CTA (256 columns each)
constexpr int kPairThreads = 320;  // producer, MMA issuer, eight epilogue warps
constexpr int kEpiWarps = 8;
// The ring of each instance: a stage holds kBoxes blocks of PK hidden channels of both operands
// ([128 rows][128 B] each, 128-byte swizzled).  The projection takes three stages of 128 channels
// (252 against 260 us on 16,096 tokens: half the stage hand-overs); the fused-append instance,
// whose longer epilogue wants deeper buffering, four of 64 (302 against 312 us).
template <bool kAppend>
struct PairCfg {
    static constexpr int kBoxes = kAppend ? 1 : 2;   // 64-channel blocks per stage
    static constexpr int kStages = kAppend ? 4 : 3;
    static constexpr uint32_t kStageBytes = kBoxes * 16384u;  // of one operand
    static constexpr uint32_t Q_A = 0;                        // kStages x kBoxes x [128 rows][128 B]
    static constexpr uint32_t Q_B = Q_A + kStages * kStageBytes;
    static constexpr uint32_t Q_BAR = Q_B + kStages * kStageBytes;
    static constexpr uint32_t Q_MISC = Q_BAR + 256;
    static constexpr uint32_t Q_TOTAL = Q_MISC + 64;
    // QB_FULL[s]   the leader's, armed by both CTAs, completed by both CTAs' copies -> MMA
    // QB_FREE[s]   each CTA's, multicast commit after the stage's MMAs              -> producer
    // QB_ACC_FULL[a]  each CTA's, multicast commit after a tile's last MMA           -> epilogue
    // QB_ACC_EMPTY[a] the leader's, one arrive per epilogue warp of both CTAs        -> MMA
    // QB_DRAIN     the leader's, commit after the last MMA                          -> teardown
    static constexpr int QB_FULL = 0;
    static constexpr int QB_FREE = QB_FULL + kStages;
    static constexpr int QB_ACC_FULL = QB_FREE + kStages;
    static constexpr int QB_ACC_EMPTY = QB_ACC_FULL + kPairAccs;
    static constexpr int QB_DRAIN = QB_ACC_EMPTY + kPairAccs;
    static constexpr int QB_COUNT = QB_DRAIN + 1;
    static_assert(Q_TOTAL + 1024 <= 232448, "one pair CTA per SM");
    static_assert(QB_COUNT * 8 <= 256, "barrier area");
};

template <bool kAppend>
__global__ void __launch_bounds__(kPairThreads, 1)
qkv_proj_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
                     const __grid_constant__ ProjParams p, int32_t n_tiles_n, int32_t n_tiles) {
    using C = PairCfg<kAppend>;
    constexpr int kPairStages = C::kStages;
    constexpr int QB_FULL = C::QB_FULL, QB_FREE = C::QB_FREE, QB_ACC_FULL = C::QB_ACC_FULL,
                  QB_ACC_EMPTY = C::QB_ACC_EMPTY, QB_DRAIN = C::QB_DRAIN;
    constexpr uint32_t Q_A = C::Q_A, Q_B = C::Q_B, Q_BAR = C::Q_BAR, Q_MISC = C::Q_MISC;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the map starts at the first 1024-byte boundary (the launch reserves 1024 bytes for it); both
    // CTAs of a pair run the same layout, so their buffers sit at the same offsets
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the leader
    const int cluster = static_cast<int>(blockIdx.x >> 1);
    const int n_clusters = static_cast<int>(gridDim.x >> 1);
    const int n_k = (p.hidden + C::kBoxes * PK - 1) / (C::kBoxes * PK);  // stages per tile (the last may
                                                                           // reach past hidden: zero-filled)
    // this cluster's tiles: t = cluster + j * n_clusters, j < my_tiles
    const int my_tiles = cluster < n_tiles ? (n_tiles - 1 - cluster) / n_clusters + 1 : 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Q_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Q_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Q_MISC + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&bars[QB_FULL + s], 2);  // both CTAs arm the leader's with their bytes
            mbar_init(&bars[QB_FREE + s], 1);
        }
        for (int a = 0; a < kPairAccs; ++a) {
            mbar_init(&bars[QB_ACC_FULL + a], 1);
            mbar_init(&bars[QB_ACC_EMPTY + a], 2 * kEpiWarps);
        }
        mbar_init(&bars[QB_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kPairAccs * PN);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // barriers initialised and tensor memory allocated in both CTAs before any remote traffic
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tile_mn = [&](int j, int &m_pair, int &n_tile) {
        const int t = cluster + j * n_clusters;
        m_pair = t / n_tiles_n;
        n_tile = t - m_pair * n_tiles_n;
    };

    if (warp == 0) {
        // ================================================================== producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_c);
            int g = 0;  // stage sequence number across tiles
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                int mp, nt;
                tile_mn(j, mp, nt);
                const int m0 = (mp * 2 + static_cast<int>(rank)) * PM;
                const int nb = nt * PN + PM * static_cast<int>(rank);
                for (int kt = 0; kt < n_k; ++kt, ++g) {
                    const int s = g % kPairStages;
                    const uint32_t u = static_cast<uint32_t>(g / kPairStages) & 1u;
                    if (!mbar_wait(&bars[QB_FREE + s], u ^ 1u, p.status, abort_flag, 511)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = mapa_shared(smem_u32(&bars[QB_FULL + s]), 0);
                    mbar_arrive_expect_tx_cluster(full, 2 * C::kStageBytes);
                    for (int hb = 0; hb < C::kBoxes; ++hb) {
                        const int k0 = (kt * C::kBoxes + hb) * PK;
                        tma_load_2d_pair(smem + Q_A + s * C::kStageBytes + hb * 16384, &tm_x, full, k0, m0);
                        tma_load_2d_pair(smem + Q_B + s * C::kStageBytes + hb * 16384, &tm_c, full, k0, nb);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ======================================================= MMA (the leader only)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_f16(true, false, 2 * PM, PN);  // BF16 x BF16, M = 256 over the pair
            int g = 0;
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const int a = j % kPairAccs;
                if (j >= kPairAccs &&
                    !mbar_wait(&bars[QB_ACC_EMPTY + a], static_cast<uint32_t>((j - kPairAccs) / kPairAccs) & 1u,
                               p.status, abort_flag, 514))
                    break;
                tc_fence_after();
                const uint32_t acc = tmem + static_cast<uint32_t>(a * PN);
                for (int kt = 0; kt < n_k; ++kt, ++g) {
                    const int s = g % kPairStages;
                    const uint32_t u = static_cast<uint32_t>(g / kPairStages) & 1u;
                    if (!mbar_wait(&bars[QB_FULL + s], u, p.status, abort_flag, 512)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + Q_A + s * C::kStageBytes);
                    const uint32_t sb = smem_u32(smem + Q_B + s * C::kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < C::kBoxes * PK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;  // block kk / 4, k-step kk % 4
                        mma_ss_pair(acc, sdesc_sw128(sa + off, 16, 1024), sdesc_sw128(sb + off, 16, 1024), idesc,
                                    (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit_pair_mc(&bars[QB_FREE + s], 0x3);
                }
                if (ok) tc_commit_pair_mc(&bars[QB_ACC_FULL + a], 0x3);
            }
            // nothing the leader issued may still run when the pair's tensor memory is freed
            tc_commit_pair_mc(&bars[QB_DRAIN], 0x1);
            proj_drain(&bars[QB_DRAIN], 0);
        }
        __syncwarp();
    } else {
        // ================================================================== epilogue
        const int q = warp & 3;          // TMEM lane quarter
        const int hb = (warp - 2) >> 2;  // which of the tile's two heads
        const int row = q * 32 + lane;
        const int per = p.heads * kHeadDim;  // channels of each of Q, K, V
        const uint32_t empty = mapa_shared(smem_u32(&bars[QB_ACC_EMPTY]), 0);  // the leader's
        for (int j = 0; j < my_tiles; ++j) {
            const int a = j % kPairAccs;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[QB_ACC_FULL + a], static_cast<uint32_t>(j / kPairAccs) & 1u,
                                                   p.status, abort_flag, 513)))
                break;
            tc_fence_after();
            int mp, nt;
            tile_mn(j, mp, nt);
            const int tok = (mp * 2 + static_cast<int>(rank)) * PM + row;
            const int n0 = nt * PN;
            const int which = n0 / per;  // a tile lies inside one of Q, K, V (per is a multiple of 256)
            const bool live = tok < p.lq;
            const TokPos tp = token_pos(p.seg, static_cast<uint32_t>(live ? tok : 0));
            const bool rotate = live && which < 2 && tp.video;
            const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * PN + hb * kHeadDim;
            const int nh = n0 + hb * kHeadDim;  // this warp's head's first channel
            // K or V of the fused-append variant: the head row also goes to the cache, in two
            // passes over the accumulator (its absmax first, then the codes with the row's scale),
            // so that no thread holds the row's 128 values
            const bool to_cache = kAppend && which > 0;
            float scale = 0.0f;
            if (to_cache) {
                float amax = 0.0f;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(trow + cc * 32, r);
                    tmem_wait_ld(r);
                    uint32_t o[16];
                    proj_chunk(r, nh + cc * 32, rotate, tp, p, o);
                    amax = fmaxf(amax, chunk_absmax(o));
                }
                scale = amax == 0.0f ? 0.0f : quant_scale(amax);
            }
            const int head = (n0 % per) / kHeadDim + hb;
            const int64_t dst = static_cast<int64_t>(head) * p.cap + p.length + tok;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t r[32];
                tmem_ld32(trow + cc * 32, r);
                tmem_wait_ld(r);
                if (cc == 3) {
                    // the accumulator's last columns are in registers: hand it back to the MMA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(empty + 8u * static_cast<uint32_t>(a));
                }
                uint32_t o[16];
                proj_chunk(r, nh + cc * 32, rotate, tp, p, o);
                if (live) store_chunk(p, tok, nh + cc * 32, o);
                if (to_cache && live) {
                    uint4 *codes = (which == 1 ? p.ck : p.cv) + dst * 8 + 2 * cc;
                    if (scale > 0.0f) {
                        chunk_codes(o, scale, codes);
                    } else {
                        codes[0] = codes[1] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            if (to_cache && live) (which == 1 ? p.cks : p.cvs)[dst] = scale;
        }
    }
    if (warp == 0 && lane == 0 && rank == 0) {
        // the copies of every stage armed must land before the pair may exit: the leader's MMA
        // thread waited each full phase it consumed; after an early stop, wait for the last phases
        const int total = my_tiles * n_k;
        for (int s = 0; s < kPairStages; ++s) {
            const int uses = total > s ? (total - 1 - s) / kPairStages + 1 : 0;  // phases of stage s
            if (uses > 0) proj_drain(&bars[QB_FULL + s], static_cast<uint32_t>(uses - 1) & 1u);
        }
    }
    tc_fence_before();
    // no remote arrive, copy or MMA of the pair may still target either CTA past this point
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPairAccs * PN);
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
            append ? cudaFuncSetAttribute(qkv_proj_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          PairCfg<true>::Q_TOTAL + 1024)
                   : cudaFuncSetAttribute(qkv_proj_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          PairCfg<false>::Q_TOTAL + 1024);
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
        !encode2d(&tc, cb, a.hidden, n_out, static_cast<uint64_t>(a.hidden) * 2, PM, err, err_len, "weights"))
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
    if (append) {
        p.ck = reinterpret_cast<uint4 *>(a.cache->k);
        p.cv = reinterpret_cast<uint4 *>(a.cache->v);
        p.cks = a.cache->k_scale;
        p.cvs = a.cache->v_scale;
        p.cap = a.cache->capacity;
        p.length = a.cache->length;
    }
    // persistent CTA pairs over 256-row x 256-channel tiles, one cluster per pair of SMs
    const int64_t pairs_m = (a.lq + 2 * PM - 1) / (2 * PM);
    const int32_t n_tiles_n = static_cast<int32_t>(n_out / PN);
    const int64_t n_tiles = pairs_m * n_tiles_n;
    if (n_tiles >= (1ll << 30)) {
        snprintf(err, err_len, "%d tokens exceed the projection's tile count", a.lq);
        return NOMAS_EUNSUPPORTED;
    }
    // one cluster per pair of SMs: each CTA's epilogue of tile i overlaps the MMAs of tile i + 1 in
    // its second accumulator (two clusters per SM pair with one accumulator each measured 304 us
    // against 259 us on 16,096 tokens)
    const int64_t clusters = std::min<int64_t>(n_tiles, std::max(1, device_sm_count() / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = (append ? PairCfg<true>::Q_TOTAL : PairCfg<false>::Q_TOTAL) + 1024;  // room to align
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int32_t nt32 = static_cast<int32_t>(n_tiles);
    cudaError_t e = append ? cudaLaunchKernelEx(&cfg, qkv_proj_pair_kernel<true>, tx, tc, p, n_tiles_n, nt32)
                           : cudaLaunchKernelEx(&cfg, qkv_proj_pair_kernel<false>, tx, tc, p, n_tiles_n, nt32);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "qkv_project launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    return NOMAS_OK;
}

}  // namespace nomas
