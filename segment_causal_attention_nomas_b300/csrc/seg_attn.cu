// seg_attn.cu -- segment-causal attention over the INT8 lifelong KV cache (tcgen05, sm_103a).
//
// Method (Hy-Nomas, comfyui-wiki news, section "一个世界，分段生成"): the segment being
// denoised attends to the K/V cache of every earlier segment and is causal across segments.
// Query i of current segment s sees every history key and the current keys of segments
// 0..s.  History K/V are INT8 codes with per-token-per-head fp32 scales (section
// "单张 4090 配置": cached K/V stored INT8, attention in BF16).
//
// Design (one CTA = one head x 256 query rows = two 128-row Q tiles, over a range of
// 128-key tiles; history tiles first, then current-segment tiles):
//   warp 8      TMA producer: Q once; per history tile the INT8 K and V codes (16 KB each)
//               into a 2-slot staging ring plus the two 512-byte scale rows; per current
//               tile the BF16 K (straight into the MMA operand buffer) and BF16 V.
//   warps 10-13 converters: INT8 K codes -> BF16 (exact) into a 128B-swizzled K-major
//               operand; INT8 V codes -> FP16 (exact) into a 128B-swizzled MN-major
//               operand; current V BF16 -> FP16 in place.
//   warp 9      MMA issuer (one thread): S_t = Q_t K^T (BF16, kind::f16, M=N=128, fp32 in
//               TMEM) for both Q tiles, then O_t += P_t V with P_t read from TMEM (FP16).
//   warps 0-7   softmax, one thread per query row (TMEM lane = row): the K scale is
//               applied to the fp32 scores, online softmax in the exp2 domain with lazy
//               rescaling (O is rescaled only when the row maximum grows by more than 2^8),
//               P' = p * v_scale written back over S as FP16, epilogue O / l.
// TMEM: S0 | S1 | O0 | O1, 128 columns each (512).  P_t aliases the first 64 columns of S_t.
// Several CTAs per head and Q block ("splits") may share one key range; they write fp32
// partials (O/l, natural-log LSE) that combine_kernel merges in a fixed order.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kRowsPerCta = 2 * BM;
constexpr int kThreads = 448;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kConvWarp0 = 10;
constexpr int kConvThreads = 128;
constexpr int kConvBarrier = 1;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_Q = 0;                   // 2 Q tiles x (2 halves x [128 rows][128 B])
constexpr uint32_t SM_KC = SM_Q + 65536;       // BF16 K operand, 2 halves x 16 KB
constexpr uint32_t SM_VC = SM_KC + 32768;      // 2 buffers x FP16 V operand (2 halves x 16 KB)
constexpr uint32_t SM_STG = SM_VC + 65536;     // 2 slots x (INT8 K 16 KB + INT8 V 16 KB)
constexpr uint32_t SM_SC = SM_STG + 65536;     // 2 slots x (k_scale[128] + v_scale[128])
constexpr uint32_t SM_BAR = SM_SC + 2048;      // mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 256;     // TMEM base address, abort flag
constexpr uint32_t SM_TOTAL = SM_MISC + 64;

enum {
    B_Q = 0,
    B_STG_FULL = 1,   // 2
    B_STG_FREE = 3,   // 2
    B_SC_FULL = 5,    // 2
    B_SC_FREE = 7,    // 2
    B_KC_FULL = 9,
    B_KC_FREE = 10,
    B_VTMA = 11,      // 2
    B_VC_FULL = 13,   // 2
    B_VC_FREE = 15,   // 2
    B_S_FULL = 17,    // 2
    B_P_FULL = 19,    // 2
    B_O_DONE = 21,    // 2
    B_DRAIN = 23,
    B_GRANT = 24,     // converter -> producer: the operand buffers of a current tile are free
    B_COUNT = 25
};
// Every barrier is waited, phase after phase, by exactly one role (the softmax warps of a
// Q tile count as one role), and no barrier can complete twice before that role has seen
// the earlier completion.  That keeps every parity wait unambiguous.  The converter warps
// are the only role that waits for the K/V operand buffers to be free; for a
// current-segment tile they pass the buffers on to the producer through B_GRANT.

struct AttnParams {
    int32_t heads, lq, lh, n_seg;
    int32_t seg_off[NOMAS_MAX_SEGMENTS + 1];
    int64_t hcap;
    float scale_log2;  // softmax_scale * log2(e)
    int32_t q_blocks, n_splits, n_hist_tiles;
    uint16_t *out;
    float *lse;
    float *part_o;    // [n_splits][lq][heads][128]
    float *part_lse;  // [n_splits][heads][lq]
    int *status;
    int32_t fault;    // 1: the producer withholds the Q load (test hook)
};

__device__ __forceinline__ bool bar_red_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kConvBarrier), "n"(kConvThreads)
        : "memory");
    return r != 0;
}

// Bounded wait used while draining after an abort: ignores the abort flag, gives up
// after ~50 ms (it only guards copies that were already issued).
__device__ __noinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_test(addr, parity)) return;
        if ((spin & 255u) == 255u && globaltimer_ns() - t0 > 50000000ull) return;
    }
}

__device__ __forceinline__ int seg_end_of_row(const AttnParams &p, int row) {
    if (row >= p.lq) return 0;
    int s = 0;
    while (s + 1 < p.n_seg && p.seg_off[s + 1] <= row) ++s;
    return p.seg_off[s + 1];
}

__global__ void __launch_bounds__(kThreads, 1)
seg_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_hk,
                const __grid_constant__ CUtensorMap tm_hv, const __grid_constant__ CUtensorMap tm_hks,
                const __grid_constant__ CUtensorMap tm_hvs, const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item
    const int qb = blockIdx.x % p.q_blocks;
    const int rest = blockIdx.x / p.q_blocks;
    const int head = rest % p.heads;
    const int split = rest / p.heads;
    const int q0 = qb * kRowsPerCta;
    const int last_row = min(q0 + kRowsPerCta, p.lq) - 1;
    const int n_cur_tiles = (seg_end_of_row(p, last_row) + BN - 1) / BN;
    const int n_hist = p.n_hist_tiles;
    const int n_all = n_hist + n_cur_tiles;
    const int g_begin = static_cast<int>((static_cast<int64_t>(n_all) * split) / p.n_splits);
    const int g_end = static_cast<int>((static_cast<int64_t>(n_all) * (split + 1)) / p.n_splits);
    const int n_loc = g_end - g_begin;
    const int n_hist_loc = max(0, min(g_end, n_hist) - g_begin);

    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) record_status(p.status, kStatusTimeout, 900);
        return;
    }
    if (n_loc <= 0) {
        // empty key range: an empty partial (only with several splits)
        for (int i = threadIdx.x; i < kRowsPerCta; i += kThreads) {
            const int row = q0 + i;
            if (row >= p.lq) continue;
            p.part_lse[(static_cast<int64_t>(split) * p.heads + head) * p.lq + row] = -INFINITY;
            float4 *o = reinterpret_cast<float4 *>(
                p.part_o + ((static_cast<int64_t>(split) * p.lq + row) * p.heads + head) * kHeadDim);
            for (int c = 0; c < kHeadDim / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM_MISC + 4);

    if (threadIdx.x == 0) {
        mbar_init(&bars[B_Q], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_STG_FULL + i], 1);
            mbar_init(&bars[B_STG_FREE + i], 1);
            mbar_init(&bars[B_SC_FULL + i], 1);
            mbar_init(&bars[B_SC_FREE + i], 8);
            mbar_init(&bars[B_VTMA + i], 1);
            mbar_init(&bars[B_VC_FULL + i], 1);
            mbar_init(&bars[B_VC_FREE + i], 1);
            mbar_init(&bars[B_S_FULL + i], 1);
            mbar_init(&bars[B_P_FULL + i], 4);
            mbar_init(&bars[B_O_DONE + i], 1);
        }
        mbar_init(&bars[B_KC_FULL], 1);
        mbar_init(&bars[B_KC_FREE], 1);
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_GRANT], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto is_hist = [&](int j) { return g_begin + j < n_hist; };
    auto key0_of = [&](int j) { return is_hist(j) ? (g_begin + j) * BN : (g_begin + j - n_hist) * BN; };

    if (warp == kProducerWarp) {
        // =================================================================== producer
        if (lane == 0) {
            uint32_t armed = 0, armed_par = 0;  // bit per barrier index: armed / parity armed
            auto arm = [&](int b, uint32_t bytes, uint32_t par) {
                mbar_arrive_expect_tx(&bars[b], bytes);
                armed |= 1u << b;
                armed_par = (armed_par & ~(1u << b)) | (par << b);
            };
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (n_hist_loc > 0) {
                tma_prefetch_desc(&tm_hk);
                tma_prefetch_desc(&tm_hv);
                tma_prefetch_desc(&tm_hks);
                tma_prefetch_desc(&tm_hvs);
            }
            arm(B_Q, 2 * 32768, 0);
            if (p.fault != 1) {
                for (int t = 0; t < 2; ++t)
                    for (int half = 0; half < 2; ++half)
                        tma_load_3d(smem + SM_Q + t * 32768 + half * 16384, &tm_q, &bars[B_Q], half * 64, head,
                                    q0 + t * BM);
            }
            for (int j = 0; j < n_loc; ++j) {
                const int key0 = key0_of(j);
                if (is_hist(j)) {
                    const int s = j & 1;
                    const uint32_t u = static_cast<uint32_t>(j >> 1) & 1u;
                    if (!mbar_wait(&bars[B_STG_FREE + s], u ^ 1u, p.status, abort_flag, 101)) break;
                    arm(B_STG_FULL + s, 32768, u);
                    const int y = static_cast<int>(static_cast<int64_t>(head) * p.hcap + key0);
                    tma_load_2d(smem + SM_STG + s * 32768, &tm_hk, &bars[B_STG_FULL + s], 0, y);
                    tma_load_2d(smem + SM_STG + s * 32768 + 16384, &tm_hv, &bars[B_STG_FULL + s], 0, y);
                    if (!mbar_wait(&bars[B_SC_FREE + s], u ^ 1u, p.status, abort_flag, 102)) break;
                    arm(B_SC_FULL + s, 1024, u);
                    tma_load_2d(smem + SM_SC + s * 1024, &tm_hks, &bars[B_SC_FULL + s], key0, head);
                    tma_load_2d(smem + SM_SC + s * 1024 + 512, &tm_hvs, &bars[B_SC_FULL + s], key0, head);
                } else {
                    const int jc = j - n_hist_loc;
                    const int b = j & 1;
                    if (!mbar_wait(&bars[B_GRANT], static_cast<uint32_t>(jc) & 1u, p.status, abort_flag, 103)) break;
                    arm(B_KC_FULL, 32768, static_cast<uint32_t>(j) & 1u);
                    tma_load_3d(smem + SM_KC, &tm_k, &bars[B_KC_FULL], 0, head, key0);
                    tma_load_3d(smem + SM_KC + 16384, &tm_k, &bars[B_KC_FULL], 64, head, key0);
                    arm(B_VTMA + (jc & 1), 32768, (static_cast<uint32_t>(jc) >> 1) & 1u);
                    tma_load_3d(smem + SM_VC + b * 32768, &tm_v, &bars[B_VTMA + (jc & 1)], 0, head, key0);
                    tma_load_3d(smem + SM_VC + b * 32768 + 16384, &tm_v, &bars[B_VTMA + (jc & 1)], 64, head, key0);
                }
            }
            // every copy this thread issued must have landed before the CTA may exit
            for (int b = 0; b < B_COUNT; ++b)
                if (armed & (1u << b)) mbar_drain(&bars[b], (armed_par >> b) & 1u);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ======================================================================= MMA
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(true, false, BM, BN);   // BF16 x BF16, K-major both
            constexpr uint32_t idesc_pv = idesc_f16(false, true, BM, kHeadDim);  // FP16, B MN-major
            const uint32_t sq = smem_u32(smem + SM_Q);
            const uint32_t skc = smem_u32(smem + SM_KC);
            const uint32_t svc = smem_u32(smem + SM_VC);
            auto issue_qk = [&](int t) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + t * 128, sdesc_sw128(sq + t * 32768 + off, 16, 1024),
                           sdesc_sw128(skc + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int b, bool acc) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                           sdesc_sw128(svc + b * 32768 + kk * 2048, 16384, 1024), idesc_pv,
                           (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(&bars[B_Q], 0, p.status, abort_flag, 201);
            ok = ok && mbar_wait(&bars[B_KC_FULL], 0, p.status, abort_flag, 202);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
                tc_commit(&bars[B_S_FULL + 0]);
                issue_qk(1);
                tc_commit(&bars[B_S_FULL + 1]);
                tc_commit(&bars[B_KC_FREE]);
                for (int j = 0; j < n_loc; ++j) {
                    const int b = j & 1;
                    const uint32_t pj = static_cast<uint32_t>(j) & 1u;
                    if (!mbar_wait(&bars[B_VC_FULL + b], (static_cast<uint32_t>(j) >> 1) & 1u, p.status, abort_flag,
                                   203))
                        break;
                    if (!mbar_wait(&bars[B_P_FULL + 0], pj, p.status, abort_flag, 204)) break;
                    tc_fence_after();
                    issue_pv(0, b, j > 0);
                    tc_commit(&bars[B_O_DONE + 0]);
                    const bool more = j + 1 < n_loc;
                    if (more) {
                        if (!mbar_wait(&bars[B_KC_FULL], pj ^ 1u, p.status, abort_flag, 205)) break;
                        tc_fence_after();
                        issue_qk(0);
                        tc_commit(&bars[B_S_FULL + 0]);
                    }
                    if (!mbar_wait(&bars[B_P_FULL + 1], pj, p.status, abort_flag, 206)) break;
                    tc_fence_after();
                    issue_pv(1, b, j > 0);
                    tc_commit(&bars[B_O_DONE + 1]);
                    tc_commit(&bars[B_VC_FREE + b]);
                    if (more) {
                        issue_qk(1);
                        tc_commit(&bars[B_S_FULL + 1]);
                        tc_commit(&bars[B_KC_FREE]);
                    }
                }
            }
            // no MMA may still be running when TMEM is freed
            tc_commit(&bars[B_DRAIN]);
            mbar_drain(&bars[B_DRAIN], 0);
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // ================================================================ converters
        const int ct = threadIdx.x - kConvWarp0 * 32;
        uint8_t *kc = smem + SM_KC;
        for (int j = 0; j < n_loc; ++j) {
            const int b = j & 1;
            uint8_t *vc = smem + SM_VC + b * 32768;
            const uint32_t u = (static_cast<uint32_t>(j) >> 1) & 1u;
            if (is_hist(j)) {
                const uint8_t *stg = smem + SM_STG + b * 32768;
                bool ok = mbar_wait(&bars[B_STG_FULL + b], u, p.status, abort_flag, 301);
                ok = ok && mbar_wait(&bars[B_KC_FREE], (static_cast<uint32_t>(j) & 1u) ^ 1u, p.status, abort_flag, 302);
                if (!bar_red_and(ok)) break;
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int idx = ct + kConvThreads * i;
                    const int row = idx >> 4, ch = idx & 15;
                    const uint2 w = *reinterpret_cast<const uint2 *>(stg + row * 128 + ch * 8);
                    *reinterpret_cast<uint4 *>(kc + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) =
                        s8x8_to_bf16x8(w);
                }
                fence_proxy_async_smem();
                ok = mbar_wait(&bars[B_VC_FREE + b], u ^ 1u, p.status, abort_flag, 303);
                if (!bar_red_and(ok)) break;
                if (ct == 0) mbar_arrive(&bars[B_KC_FULL]);
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int idx = ct + kConvThreads * i;
                    const int row = idx >> 4, ch = idx & 15;
                    const uint2 w = *reinterpret_cast<const uint2 *>(stg + 16384 + row * 128 + ch * 8);
                    *reinterpret_cast<uint4 *>(vc + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) =
                        s8x8_to_f16x8(w);
                }
                fence_proxy_async_smem();
                bar_red_and(true);
                if (ct == 0) {
                    mbar_arrive(&bars[B_VC_FULL + b]);
                    mbar_arrive(&bars[B_STG_FREE + b]);
                }
            } else {
                const int jc = j - n_hist_loc;
                bool ok = mbar_wait(&bars[B_KC_FREE], (static_cast<uint32_t>(j) & 1u) ^ 1u, p.status, abort_flag, 304);
                ok = ok && mbar_wait(&bars[B_VC_FREE + b], u ^ 1u, p.status, abort_flag, 305);
                if (!bar_red_and(ok)) break;
                if (ct == 0) mbar_arrive(&bars[B_GRANT]);
                ok = mbar_wait(&bars[B_VTMA + (jc & 1)], (static_cast<uint32_t>(jc) >> 1) & 1u, p.status, abort_flag,
                               306);
                if (!bar_red_and(ok)) break;
                uint4 *v4 = reinterpret_cast<uint4 *>(vc);
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int idx = ct + kConvThreads * i;
                    v4[idx] = bf16x8_to_f16x8(v4[idx]);
                }
                fence_proxy_async_smem();
                bar_red_and(true);
                if (ct == 0) mbar_arrive(&bars[B_VC_FULL + b]);
            }
        }
    } else {
        // =================================================================== softmax
        const int t = warp >> 2;          // Q tile
        const int wq = warp & 3;          // TMEM lane quarter
        const int row_in_tile = wq * 32 + lane;
        const int grow = q0 + t * BM + row_in_tile;
        const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_bits + t * 128;
        const uint32_t tO = tmem + lane_bits + 256 + t * 128;
        const int seg_end = seg_end_of_row(p, grow);
        const float c = p.scale_log2;
        float m2 = -INFINITY;  // running reference maximum, log2 domain
        float l = 0.0f;
        bool ok = true;
        for (int j = 0; j < n_loc; ++j) {
            const bool hist = is_hist(j);
            const int b = j & 1;
            const uint32_t pj = static_cast<uint32_t>(j) & 1u;
            ok = mbar_wait(&bars[B_S_FULL + t], pj, p.status, abort_flag, 401);
            if (hist) ok = ok && mbar_wait(&bars[B_SC_FULL + b], (static_cast<uint32_t>(j) >> 1) & 1u, p.status,
                                           abort_flag, 402);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key0 = key0_of(j);
            const int limit = hist ? (p.lh - key0) : (seg_end - key0);  // columns < limit are visible
            const float *ks = reinterpret_cast<const float *>(smem + SM_SC + b * 1024);
            const float *vs = ks + 128;

            // pass 1: row maximum of the (K-scaled) scores
            float mx = -INFINITY;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tS + ch * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int col = ch * 32 + k;
                    float x = __uint_as_float(r[k]);
                    if (hist) x *= ks[col];
                    if (col >= limit) x = -INFINITY;
                    mx = fmaxf(mx, x);
                }
            }
            const float mnew = mx * c;
            // lazy rescale: move the reference only when the maximum grew by more than 8 (x256)
            const bool grow_ref = mnew > m2 + 8.0f;
            if (__any_sync(0xFFFFFFFFu, grow_ref)) {
                const float alpha = grow_ref ? ex2_approx(m2 - mnew) : 1.0f;  // m2 = -inf -> 0
                if (grow_ref) {
                    l *= alpha;
                    m2 = mnew;
                }
                if (j > 0) {
                    // O already holds earlier tiles: wait for the last PV, then scale it
                    bool okw = mbar_wait(&bars[B_O_DONE + t], (static_cast<uint32_t>(j) - 1u) & 1u, p.status,
                                         abort_flag, 403);
                    okw = __all_sync(0xFFFFFFFFu, okw);
                    if (!okw) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t r[32];
                        tmem_ld32(tO + ch * 32, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                        tmem_st32(tO + ch * 32, r);
                    }
                    tmem_st_wait();
                }
            }
            // pass 2: p = 2^(x*c - m2); l += p; P' = p * v_scale -> FP16 over S
            const float mref = (m2 == -INFINITY) ? 0.0f : m2;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tS + ch * 32, r);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    float pv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = ch * 32 + k + e;
                        float x = __uint_as_float(r[k + e]);
                        if (hist) x *= ks[col];
                        float pe = ex2_approx(fmaf(x, c, -mref));
                        float pw = hist ? pe * vs[col] : pe;
                        if (col >= limit) {
                            pe = 0.0f;
                            pw = 0.0f;
                        }
                        l += pe;
                        pv[e] = pw;
                    }
                    pk[k >> 1] = pack_f16x2_sat(pv[0], pv[1]);
                }
                tmem_st16(tS + ch * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_P_FULL + t]);
                if (hist) mbar_arrive(&bars[B_SC_FREE + b]);
            }
        }
        // ---- epilogue
        if (ok) {
            bool okw = mbar_wait(&bars[B_O_DONE + t], (static_cast<uint32_t>(n_loc) - 1u) & 1u, p.status, abort_flag,
                                 404);
            ok = __all_sync(0xFFFFFFFFu, okw);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            const float lse_row = l > 0.0f ? (m2 + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            const bool live = grow < p.lq;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tO + ch * 32, r);
                tmem_ld_wait();
                if (!live) continue;
                if (p.n_splits == 1) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(grow) * p.heads + head) *
                                                                        kHeadDim + ch * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * inv_l, __uint_as_float(r[8 * q + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv_l, __uint_as_float(r[8 * q + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv_l, __uint_as_float(r[8 * q + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv_l, __uint_as_float(r[8 * q + 7]) * inv_l);
                        dst[q] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(
                        p.part_o + ((static_cast<int64_t>(split) * p.lq + grow) * p.heads + head) * kHeadDim + ch * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv_l, __uint_as_float(r[4 * q + 1]) * inv_l,
                                             __uint_as_float(r[4 * q + 2]) * inv_l,
                                             __uint_as_float(r[4 * q + 3]) * inv_l);
                }
            }
            if (live) {
                if (p.n_splits == 1) {
                    if (p.lse) p.lse[static_cast<int64_t>(head) * p.lq + grow] = lse_row;
                } else {
                    p.part_lse[(static_cast<int64_t>(split) * p.heads + head) * p.lq + grow] = lse_row;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Split-KV merge: O = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max lse), fixed order.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                                                      int n_splits, int lq, int heads, uint16_t *__restrict__ out,
                                                      float *__restrict__ lse) {
    const int64_t total = static_cast<int64_t>(lq) * heads * 32;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int g = static_cast<int>(i & 31);
        const int64_t rh = i >> 5;
        const int row = static_cast<int>(rh / heads);
        const int h = static_cast<int>(rh - static_cast<int64_t>(row) * heads);
        float mmax = -INFINITY;
        for (int s = 0; s < n_splits; ++s) mmax = fmaxf(mmax, part_lse[(static_cast<int64_t>(s) * heads + h) * lq + row]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.0f;
        if (mmax != -INFINITY) {
            for (int s = 0; s < n_splits; ++s) {
                const float w = __expf(part_lse[(static_cast<int64_t>(s) * heads + h) * lq + row] - mmax);
                const float4 o = reinterpret_cast<const float4 *>(
                    part_o + ((static_cast<int64_t>(s) * lq + row) * heads + h) * kHeadDim)[g];
                acc.x += w * o.x;
                acc.y += w * o.y;
                acc.z += w * o.z;
                acc.w += w * o.w;
                wsum += w;
            }
        }
        const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
        uint2 w2;
        w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        reinterpret_cast<uint2 *>(out + (static_cast<int64_t>(row) * heads + h) * kHeadDim)[g] = w2;
        if (g == 0 && lse != nullptr) lse[static_cast<int64_t>(h) * lq + row] = wsum > 0.0f ? mmax + logf(wsum) : -INFINITY;
    }
}

// ------------------------------------------------------------------ host helpers
bool encode(CUtensorMap *m, CUtensorMapDataType dt, cuuint32_t rank, void *base, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw, char *err, size_t err_len,
            const char *what) {
    const cuuint32_t estr[3] = {1, 1, 1};
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) {
        snprintf(err, err_len, "cuTensorMapEncodeTiled unavailable");
        return false;
    }
    CUresult r = fn(m, dt, rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(err, err_len, "tensor map for %s rejected (CUresult %d)", what, static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace

int32_t attn_num_splits(int64_t lq, int64_t lh, int32_t heads, int num_sms) {
    const int64_t items = ((lq + kRowsPerCta - 1) / kRowsPerCta) * heads;
    const int64_t tiles = (lh + BN - 1) / BN + (lq + BN - 1) / BN;
    if (items <= 0 || num_sms <= 0) return 1;
    int best = 1;
    double best_score = -1.0;
    for (int s = 1; s <= 16; ++s) {
        if (s > 1 && tiles / s < 8) break;  // keep at least 8 key tiles per split
        const int64_t ctas = items * s;
        const int64_t waves = (ctas + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(ctas) / static_cast<double>(waves * num_sms);
        const double score = eff - 0.02 * (s - 1);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = s;
        }
    }
    return best;
}

size_t attn_workspace_bytes(int64_t lq, int32_t heads, int32_t n_splits) {
    if (n_splits <= 1) return 0;
    return static_cast<size_t>(n_splits) * static_cast<size_t>(lq) * heads * (kHeadDim + 1) * sizeof(float);
}

nomas_status launch_seg_attn(const AttnLaunch &a, cudaStream_t stream, char *err, size_t err_len) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(seg_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SM_TOTAL);
        if (e != cudaSuccess) {
            snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
        attr_set[dev] = true;
    }
    AttnParams p;
    memset(&p, 0, sizeof(p));
    p.heads = a.heads;
    p.lq = a.lq;
    p.lh = static_cast<int32_t>(a.lh);
    p.n_seg = a.n_seg;
    for (int i = 0; i <= a.n_seg; ++i) p.seg_off[i] = a.seg_off[i];
    p.hcap = a.hist ? a.hist->capacity : 0;
    const float scale = a.softmax_scale != 0.0f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(kHeadDim));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.q_blocks = (a.lq + kRowsPerCta - 1) / kRowsPerCta;
    p.n_splits = a.n_splits;
    p.n_hist_tiles = static_cast<int32_t>((a.lh + BN - 1) / BN);
    p.out = static_cast<uint16_t *>(a.out);
    p.lse = a.lse;
    if (a.n_splits > 1) {
        p.part_o = static_cast<float *>(a.workspace);
        p.part_lse = p.part_o + static_cast<size_t>(a.n_splits) * a.lq * a.heads * kHeadDim;
    }
    p.status = device_status_word();
    p.fault = a.fault;

    CUtensorMap tq, tk, tv, thk, thv, thks, thvs;
    memset(&thk, 0, sizeof(thk));
    memset(&thv, 0, sizeof(thv));
    memset(&thks, 0, sizeof(thks));
    memset(&thvs, 0, sizeof(thvs));
    {
        const cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(a.heads), static_cast<cuuint64_t>(a.lq)};
        const cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(a.row_stride) * 2};
        const cuuint32_t box[3] = {64, 1, 128};
        if (!encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B, err, err_len, "q") ||
            !encode(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B, err, err_len, "k_cur") ||
            !encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v), dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B, err, err_len, "v_cur"))
            return NOMAS_EINVAL;
    }
    if (a.lh > 0) {
        const nomas_kv_cache &h = *a.hist;
        const cuuint64_t dims[2] = {kHeadDim, static_cast<cuuint64_t>(h.heads) * static_cast<cuuint64_t>(h.capacity)};
        const cuuint64_t strides[1] = {kHeadDim};
        const cuuint32_t box[2] = {128, 128};
        const cuuint64_t sdims[2] = {static_cast<cuuint64_t>(h.capacity), static_cast<cuuint64_t>(h.heads)};
        const cuuint64_t sstrides[1] = {static_cast<cuuint64_t>(h.capacity) * 4};
        const cuuint32_t sbox[2] = {128, 1};
        if (!encode(&thk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, h.k, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, err,
                    err_len, "history k") ||
            !encode(&thv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, h.v, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, err,
                    err_len, "history v") ||
            !encode(&thks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h.k_scale, sdims, sstrides, sbox,
                    CU_TENSOR_MAP_SWIZZLE_NONE, err, err_len, "history k_scale") ||
            !encode(&thvs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h.v_scale, sdims, sstrides, sbox,
                    CU_TENSOR_MAP_SWIZZLE_NONE, err, err_len, "history v_scale"))
            return NOMAS_EINVAL;
    }
    const int64_t grid = static_cast<int64_t>(p.q_blocks) * a.heads * a.n_splits;
    if (grid <= 0) return NOMAS_OK;
    if (grid > 0x7FFFFFFF) {
        snprintf(err, err_len, "grid too large");
        return NOMAS_EUNSUPPORTED;
    }
    seg_attn_kernel<<<static_cast<unsigned>(grid), kThreads, SM_TOTAL, stream>>>(tq, tk, tv, thk, thv, thks, thvs, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "seg_attn launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    if (a.n_splits > 1) {
        const int64_t threads = static_cast<int64_t>(a.lq) * a.heads * 32;
        int64_t blocks = (threads + 255) / 256;
        const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8 * 4;
        if (blocks > cap) blocks = cap;
        combine_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(p.part_o, p.part_lse, a.n_splits, a.lq, a.heads,
                                                                     p.out, a.lse);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(err, err_len, "combine launch: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
    }
    return NOMAS_OK;
}

}  // namespace nomas
