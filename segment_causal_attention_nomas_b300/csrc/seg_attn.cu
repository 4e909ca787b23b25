// seg_attn.cu -- segment-causal attention over the INT8 lifelong KV cache (tcgen05, sm_103a).
//
// Method (Hy-Nomas, comfyui-wiki news, section "一个世界，分段生成"): the segment being
// denoised attends to the K/V cache of every earlier segment and is causal across segments.
// Query i of current segment s sees every history key and the current keys of segments
// 0..s.  History K/V are INT8 codes with per-token-per-head fp32 scales (section
// "单张 4090 配置": cached K/V stored INT8, attention in BF16).
//
// One call runs these kernels on the caller's stream:
//   range_kernel  per-head maxima of |K|, |V| of the current tokens (and, when the call stages the
//       history, of the history's k and v row scales), folded with atomicMax on the bit patterns.
//   stage_cur_kernel, stage_hist_kernel  (HBM-bound) write the tensor-core operands into the
//       workspace, head-major so that every operand tile is one contiguous 32 KB block: Q and the
//       current K/V converted BF16 -> FP16 ([H][Lq][128]), and the history codes times their
//       scales rounded to FP16 ([H][Lh][128]).  Each operand block is multiplied by an exact power
//       of two that puts its maximum in [2^14, 2^15): a Q row by its own (the exponent stored per
//       row), a head's current K, current V, history K and history V by one each.  So every
//       finite BF16 input lands in FP16's normal range, and the attention kernel undoes the
//       factors exactly (in its softmax multipliers and its output).
//       Every history tile is read by every Q block of its head, so expanding it once, rather
//       than inside the attention loop, keeps the SM's shared-memory port and issue slots for the
//       tensor cores; a caller may also stage the history once for several calls.
//   seg_attn_kernel<kPair>  one CTA = one head x 256 query rows (two 128-row Q tiles) over a range
//       of 128-key tiles, history tiles first; in the pair variant a cluster of two CTAs (one per SM
//       of a pair) takes two neighbouring Q blocks of a head and each CTA holds half of every key
//       tile (chosen for long unsplit calls, where the GPU runs at its power cap; see
//       attn_use_pair):
//     warp 8     TMA producer: Q once, then per key tile the FP16 K and V tiles (128B-swizzled)
//                into a 3-deep K ring and a 2-deep V ring of 32 KB buffers (pair: 4-deep rings of
//                16 KB halves, completing on the leader's barriers).
//     warp 9     MMA issuer (one thread; the pair's leader): S_t = Q_t K^T (kind::f16, N = 128,
//                M = 128 or 256 over the pair, fp32 in TMEM) for both Q tiles, then
//                O_t += P_t V with P_t read from TMEM (FP16).
//     warps 0-7  softmax, one thread per query row (TMEM lane = row), exp2 domain: the row's 128
//                scores are loaded with one wait and their maximum taken first.  The row keeps a
//                reference maximum and moves it (rescaling O and the running sum) only when a
//                tile's maximum exceeds it by more than 2^kRescaleLog2, so every P value is at
//                most 256 and fits FP16 with room to spare.  Masking runs on boundary tiles only.
//                History and current tiles get their own softmax multiplier (the K exponents
//                differ); at the first current tile O is rescaled once by the ratio of the
//                current and history V factors.
//   combine_kernel  merges the fp32 partials when several CTAs ("splits") share a head and Q
//       block (short Lq over a long history), in a fixed order.
// TMEM: S0 | S1 | O0 | O1, 128 columns each (512).  P_t aliases the first 64 columns of S_t.
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
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// The reference maximum of a row is kept while the row's scores stay within this many binary
// orders above it, so every P value is at most 2^kRescaleLog2.
constexpr float kRescaleLog2 = 8.0f;

// The two variants of the attention kernel, one CTA per SM either way.  kPair = false: a CTA
// holds whole 128-key K and V tiles.  kPair = true: a cluster of two CTAs (one per SM of a pair)
// takes two neighbouring 256-row Q blocks of a head and issues M = 256 MMAs (cta_group::2); each
// CTA holds half of every K tile (its 64 keys, all 128 dims) and half of every V tile (its 64
// dims, all 128 keys), so an SM loads half the key tiles' bytes and its tensor cores read 6 of
// the 8 KB of operands per Q.K^T step from its own shared memory.
template <bool kPair>
struct AttnCfg {
    static constexpr int NK = kPair ? 4 : 3;                     // K operand buffers
    static constexpr int NV = kPair ? 4 : 2;                     // V operand buffers
    static constexpr uint32_t KVB = kPair ? 16384u : 32768u;     // bytes of one K or V buffer
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr uint32_t SM_Q = 0;                    // 2 Q tiles x (2 halves x [128 rows][128 B])
    static constexpr uint32_t SM_K = SM_Q + 65536;         // NK K buffers (K-major, SW128)
    static constexpr uint32_t SM_V = SM_K + NK * KVB;      // NV V buffers (MN-major, SW128)
    static constexpr uint32_t SM_BAR = SM_V + NV * KVB;    // mbarriers
    static constexpr uint32_t SM_MISC = SM_BAR + 256;      // TMEM base address, abort flag
    static constexpr uint32_t SM_TOTAL = SM_MISC + 64;
    // mbarriers.  In the pair variant B_Q, B_K_FULL, B_V_FULL, B_P_FULL and B_DRAIN are used in
    // the leader, which both CTAs arm or arrive on; B_K_FREE, B_V_FREE, B_S_FULL and B_O_DONE in
    // each CTA, completed by the leader's multicast commits.
    static constexpr int B_Q = 0;                   // Q landed (both CTAs' Q)     -> MMA
    static constexpr int B_K_FULL = 1;              // NK: K tile landed            -> MMA
    static constexpr int B_K_FREE = B_K_FULL + NK;  // NK: both QK^T of the tile done -> producer
    static constexpr int B_V_FULL = B_K_FREE + NK;  // NV: V tile landed            -> MMA
    static constexpr int B_V_FREE = B_V_FULL + NV;  // NV: both PV of the tile done -> producer
    static constexpr int B_S_FULL = B_V_FREE + NV;  // 2: S of Q tile t             -> softmax
    static constexpr int B_P_FULL = B_S_FULL + 2;   // 2: P of Q tile t stored (4 warps per CTA) -> MMA
    static constexpr int B_O_DONE = B_P_FULL + 2;   // 2: the last PV of Q tile t   -> softmax epilogue
    static constexpr int B_DRAIN = B_O_DONE + 2;
    static constexpr int B_COUNT = B_DRAIN + 1;
    static_assert(SM_TOTAL + 1024 <= 232448, "shared memory map exceeds 227 KB");
    static_assert(B_COUNT * 8 <= 256, "barrier area");
    static_assert(B_COUNT <= 32, "producer arms at most 32 barriers");
};
// Every barrier is completed once per use of its buffer or slot and waited, phase after
// phase, by one role that cannot fall two phases behind it: a buffer is refilled (next phase)
// only after the role that waits on its current phase has released it.  That keeps every
// parity wait unambiguous.

struct AttnParams {
    int32_t heads, lq, lh, n_seg;
    int32_t q_pairs;  // pairs of 256-row Q blocks (the pair variant)
    int32_t seg_off[NOMAS_MAX_SEGMENTS + 1];
    float scale_log2;  // softmax_scale * log2(e)
    int32_t q_blocks, n_splits, n_hist_tiles;
    uint16_t *out;
    float *lse;
    float *part_o;    // [n_splits][lq][heads][128]
    float *part_lse;  // [n_splits][heads][lq]
    const int8_t *qexp;        // [heads][lq]: staged Q row = Q * 2^qexp
    const uint32_t *cur_max;   // [2][heads]: max |K|, max |V| of the current tokens (fp32 bits)
    const uint32_t *hist_max;  // [2][heads]: largest history k, v row scale (fp32 bits)
    int *status;
    int32_t fault;    // 1: the producer withholds the Q load (test hook)
};

// Largest softmax multiplier (log2 units per raw FP16-product score) that keeps every score
// finite: raw scores of FP16 operands below 2^15 stay below 128 * 2^30 = 2^37, so x * c stays
// below 2^123.  A larger multiplier means true scores beyond about 1e34 (NOMAS_ERANGE).
constexpr float kMaxSoftmaxMul = 0x1p86f;
// Largest |e_V(current) - e_V(history)| for which rescaling O between the history and the
// current key tiles is exact in fp32 (|O| < 2^15 * 2^8 * 2^30 before the rescale).
constexpr int kMaxVExpShift = 70;

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

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// All 128 raw scores of this thread's row of S (TMEM lane = row): four loads, one wait.
__device__ __forceinline__ void load_s_row(uint32_t tS, uint32_t (&r)[4][32]) {
    tmem_ld32(tS, r[0]);
    tmem_ld32(tS + 32, r[1]);
    tmem_ld32(tS + 64, r[2]);
    tmem_ld32(tS + 96, r[3]);
    tmem_wait_ld(r[0]);
    tmem_tie(r[1]);
    tmem_tie(r[2]);
    tmem_tie(r[3]);
}

// Columns >= limit are not visible to this row: their scores become -inf.
__device__ __forceinline__ void mask_row(uint32_t (&r)[4][32], int limit) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (q * 32 + k >= limit) r[q][k] = 0xFF800000u;
}

// Maximum raw score of the row (-inf if every column is masked); eight independent chains.
__device__ __forceinline__ float row_max(const uint32_t (&r)[4][32]) {
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m[i] = fmaxf(__uint_as_float(r[i >> 1][(i & 1) * 16]), __uint_as_float(r[i >> 1][(i & 1) * 16 + 1]));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t *x = &r[i >> 1][(i & 1) * 16];
#pragma unroll
        for (int k = 2; k < 16; k += 2) m[i] = max3f(m[i], __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
    }
    return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// p = 2^(x * c - mu) over the row, packed to FP16 pairs: columns 2i, 2i + 1 go to w[i / 32][i % 32]
// (TMEM column i of the P block).  Returns the sum of the fp32 p values.
__device__ __forceinline__ float row_probs(const uint32_t (&r)[4][32], float c, float mu, uint32_t (&w)[2][32]) {
    const float2 negm = make_float2(-mu, -mu);
    const float2 cc = make_float2(c, c);
    float2 s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(r[q][k]), __uint_as_float(r[q][k + 1])), cc, negm);
            const float2 pa = make_float2(ex2_approx(a.x), ex2_approx(a.y));
            s[(k >> 1) & 3] = __fadd2_rn(s[(k >> 1) & 3], pa);
            const int i = q * 16 + (k >> 1);
            w[i >> 5][i & 31] = pack_f16x2_sat(pa.x, pa.y);
        }
    }
    const float2 t = __fadd2_rn(__fadd2_rn(s[0], s[1]), __fadd2_rn(s[2], s[3]));
    return t.x + t.y;
}

// Multiplies 128 fp32 TMEM columns (one O row block) by alpha, 16 columns at a time (inline and
// in few registers: the caller keeps a whole S row live across it).
__device__ __forceinline__ void rescale_o_row(uint32_t taddr, float alpha) {
#pragma unroll 1
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t r[16];
        tmem_ld16(taddr + ch * 16, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
        tmem_st16(taddr + ch * 16, r);
    }
    tmem_st_wait();
}

// 320 threads, one CTA per SM (in the pair variant, clusters of two).  Ten warps put three on two
// of the SM's four sub-partitions, whose 64 KB register files then cap a thread at 168 registers.
template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
seg_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_hk,
                const __grid_constant__ CUtensorMap tm_hv, const __grid_constant__ AttnParams p) {
    using C = AttnCfg<kPair>;
    constexpr int NK = C::NK, NV = C::NV;
    constexpr int B_Q = C::B_Q, B_K_FULL = C::B_K_FULL, B_K_FREE = C::B_K_FREE, B_V_FULL = C::B_V_FULL,
                  B_V_FREE = C::B_V_FREE, B_S_FULL = C::B_S_FULL, B_P_FULL = C::B_P_FULL, B_O_DONE = C::B_O_DONE,
                  B_DRAIN = C::B_DRAIN, B_COUNT = C::B_COUNT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the map starts at the first 1024-byte boundary (the launch reserves 1024 bytes for it); both
    // CTAs of a pair run the same layout, so their buffers sit at the same offsets
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item.  Q blocks run last to first: under the segment-causal mask later blocks see
    // more keys, so the heaviest CTAs start first and the lightest fill the last wave.  A pair
    // takes Q blocks 2 pb (the leader, rank 0) and 2 pb + 1 of one head and split, over the key
    // tiles that the later block needs.
    uint32_t rank = 0;
    int qb, rest, tiles_row;
    if constexpr (kPair) {
        rank = cluster_ctarank();
        const int cluster = static_cast<int>(blockIdx.x >> 1);
        const int pb = p.q_pairs - 1 - cluster % p.q_pairs;
        rest = cluster / p.q_pairs;
        qb = 2 * pb + static_cast<int>(rank);
        tiles_row = min((2 * pb + 2) * kRowsPerCta, p.lq) - 1;
    } else {
        qb = p.q_blocks - 1 - static_cast<int>(blockIdx.x % p.q_blocks);
        rest = blockIdx.x / p.q_blocks;
        tiles_row = min((qb + 1) * kRowsPerCta, p.lq) - 1;
    }
    const int head = rest % p.heads;
    const int split = rest / p.heads;
    const int q0 = qb * kRowsPerCta;
    const int n_cur_tiles = (seg_end_of_row(p, tiles_row) + BN - 1) / BN;
    const int n_hist = p.n_hist_tiles;
    const int n_all = n_hist + n_cur_tiles;
    const int g_begin = static_cast<int>((static_cast<int64_t>(n_all) * split) / p.n_splits);
    const int g_end = static_cast<int>((static_cast<int64_t>(n_all) * (split + 1)) / p.n_splits);
    const int n_loc = g_end - g_begin;
    const int n_hist_loc = max(0, min(g_end, n_hist) - g_begin);

    if (n_loc <= 0) {
        // empty key range (for both CTAs of a pair): an empty partial (only with several splits)
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

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::SM_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SM_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SM_MISC + 4);

    if (threadIdx.x == 0) {
        constexpr uint32_t copies = kPair ? 2 : 1;  // a pair's copies land on the leader's barriers
        mbar_init(&bars[B_Q], copies);
        for (int i = 0; i < NK; ++i) {
            mbar_init(&bars[B_K_FULL + i], copies);
            mbar_init(&bars[B_K_FREE + i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&bars[B_V_FULL + i], copies);
            mbar_init(&bars[B_V_FREE + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_S_FULL + i], 1);
            mbar_init(&bars[B_P_FULL + i], kPair ? 8 : 4);  // the softmax warps of the tile (of both CTAs)
            mbar_init(&bars[B_O_DONE + i], 1);
        }
        mbar_init(&bars[B_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_slot, 512);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, 512);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (kPair)
        cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs before any remote traffic
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto is_hist = [&](int j) { return j < n_hist_loc; };
    auto key0_of = [&](int j) { return is_hist(j) ? (g_begin + j) * BN : (g_begin + j - n_hist) * BN; };

    if (warp == kProducerWarp) {
        // =================================================================== producer
        // Q once, then per key tile its K and V.  In a pair each CTA loads its own Q tiles, its
        // 64 keys (key0 + 64 rank ..) of each K tile and its 64 dims (64 rank ..) of each V tile,
        // and every copy completes on the leader's barrier, which each CTA arms with its bytes.
        if (lane == 0) {
            uint32_t armed = 0, armed_par = 0;  // bit per barrier index: armed / parity armed
            auto bar_of = [&](int b) -> uint32_t {
                return kPair ? mapa_shared(smem_u32(&bars[b]), 0) : smem_u32(&bars[b]);
            };
            auto arm = [&](int b, uint32_t bytes, uint32_t par) {
                if constexpr (kPair)
                    mbar_arrive_expect_tx_cluster(bar_of(b), bytes);
                else
                    mbar_arrive_expect_tx(&bars[b], bytes);
                armed |= 1u << b;
                armed_par = (armed_par & ~(1u << b)) | (par << b);
            };
            auto load = [&](void *dst, const CUtensorMap *map, int b, int x, int y, int z) {
                if constexpr (kPair)
                    tma_load_3d_pair(dst, map, bar_of(b), x, y, z);
                else
                    tma_load_3d(dst, map, &bars[b], x, y, z);
            };
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (n_hist_loc > 0) {
                tma_prefetch_desc(&tm_hk);
                tma_prefetch_desc(&tm_hv);
            }
            arm(B_Q, 2 * 32768, 0);
            if (p.fault != 1) {
                for (int t = 0; t < 2; ++t)
                    for (int half = 0; half < 2; ++half)
                        load(smem + C::SM_Q + t * 32768 + half * 16384, &tm_q, B_Q, half * 64, q0 + t * BM, head);
            }
            const int kr = 64 * static_cast<int>(rank);  // the pair CTA's keys (K) and dims (V)
            for (int j = 0; j < n_loc; ++j) {
                const int key0 = key0_of(j);
                const int kb = j % NK, vb = j % NV;
                const uint32_t uk = static_cast<uint32_t>(j / NK) & 1u;
                const uint32_t uv = static_cast<uint32_t>(j / NV) & 1u;
                uint8_t *kbuf = smem + C::SM_K + kb * C::KVB;
                uint8_t *vbuf = smem + C::SM_V + vb * C::KVB;
                const bool hist = is_hist(j);
                if (!mbar_wait(&bars[B_K_FREE + kb], uk ^ 1u, p.status, abort_flag, 101)) break;
                arm(B_K_FULL + kb, C::KVB, uk);
                for (int half = 0; half < 2; ++half)
                    load(kbuf + half * (C::KVB / 2), hist ? &tm_hk : &tm_k, B_K_FULL + kb, half * 64, key0 + kr, head);
                if (!mbar_wait(&bars[B_V_FREE + vb], uv ^ 1u, p.status, abort_flag, 102)) break;
                arm(B_V_FULL + vb, C::KVB, uv);
                if constexpr (kPair) {
                    load(vbuf, hist ? &tm_hv : &tm_v, B_V_FULL + vb, kr, key0, head);
                } else {
                    for (int half = 0; half < 2; ++half)
                        load(vbuf + half * 16384, hist ? &tm_hv : &tm_v, B_V_FULL + vb, half * 64, key0, head);
                }
            }
            // every copy this thread issued must have landed before the CTA may exit.  In a pair the
            // copies complete on the leader's barriers, which the leader drains (the peer leaves
            // only after the cluster barrier at the end, which the leader reaches after this).
            if (!kPair || rank == 0)
                for (int b = 0; b < B_COUNT; ++b)
                    if (armed & (1u << b)) mbar_drain(&bars[b], (armed_par >> b) & 1u);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ======================================================= MMA (in a pair, the leader's)
        if (lane == 0 && rank == 0) {
            constexpr int M = kPair ? 2 * BM : BM;  // a pair's MMA covers both CTAs' 128 rows
            constexpr uint32_t idesc_qk = idesc_f16(false, false, M, BN);       // FP16 x FP16, K-major both
            constexpr uint32_t idesc_pv = idesc_f16(false, true, M, kHeadDim);  // FP16, B MN-major
            const uint32_t sq = smem_u32(smem + C::SM_Q);
            auto mma_smem = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
                if constexpr (kPair)
                    mma_ss_pair(d, a, b, idesc, acc);
                else
                    mma_ss(d, a, b, idesc, acc);
            };
            auto mma_tmem = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
                if constexpr (kPair)
                    mma_ts_pair(d, a, b, idesc, acc);
                else
                    mma_ts(d, a, b, idesc, acc);
            };
            auto commit = [&](int b) {  // in a pair the barrier of both CTAs
                if constexpr (kPair)
                    tc_commit_pair_mc(&bars[b], 0x3);
                else
                    tc_commit(&bars[b]);
            };
            auto issue_qk = [&](int t, int kb) {
                const uint32_t sk = smem_u32(smem + C::SM_K + kb * C::KVB);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_smem(tmem + t * 128, sdesc_sw128(sq + t * 32768 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sk + (kk >> 2) * (C::KVB / 2) + (kk & 3) * 32, 16, 1024), idesc_qk,
                             kk > 0 ? 1u : 0u);
            };
            auto issue_pv = [&](int t, int vb, bool acc) {
                // V, MN-major: 8-key groups 1 KB apart; the two 64-dim halves 16 KB apart (a pair
                // CTA holds one half)
                const uint32_t sv = smem_u32(smem + C::SM_V + vb * C::KVB);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_tmem(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                             sdesc_sw128(sv + kk * 2048, kPair ? 0 : 16384, 1024), idesc_pv, (acc || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&bars[B_Q], 0, p.status, abort_flag, 201);
            ok = ok && mbar_wait(&bars[B_K_FULL + 0], 0, p.status, abort_flag, 202);
            if (ok) {
                tc_fence_after();
                issue_qk(0, 0);
                commit(B_S_FULL + 0);
                issue_qk(1, 0);
                commit(B_S_FULL + 1);
                commit(B_K_FREE + 0);
                for (int j = 0; j < n_loc; ++j) {
                    const int vb = j % NV;
                    const uint32_t pj = static_cast<uint32_t>(j) & 1u;
                    if (!mbar_wait(&bars[B_V_FULL + vb], static_cast<uint32_t>(j / NV) & 1u, p.status, abort_flag,
                                   203))
                        break;
                    if (!mbar_wait(&bars[B_P_FULL + 0], pj, p.status, abort_flag, 204)) break;
                    tc_fence_after();
                    issue_pv(0, vb, j > 0);
                    commit(B_O_DONE + 0);
                    const bool more = j + 1 < n_loc;
                    const int kn = (j + 1) % NK;
                    if (more) {
                        if (!mbar_wait(&bars[B_K_FULL + kn], static_cast<uint32_t>((j + 1) / NK) & 1u, p.status,
                                       abort_flag, 205))
                            break;
                        tc_fence_after();
                        issue_qk(0, kn);
                        commit(B_S_FULL + 0);
                    }
                    if (!mbar_wait(&bars[B_P_FULL + 1], pj, p.status, abort_flag, 206)) break;
                    tc_fence_after();
                    issue_pv(1, vb, j > 0);
                    commit(B_O_DONE + 1);
                    commit(B_V_FREE + vb);
                    if (more) {
                        issue_qk(1, kn);
                        commit(B_S_FULL + 1);
                        commit(B_K_FREE + kn);
                    }
                }
            }
            // no MMA may still be running when TMEM is freed
            if constexpr (kPair)
                tc_commit_pair_mc(&bars[B_DRAIN], 0x1);
            else
                tc_commit(&bars[B_DRAIN]);
            mbar_drain(&bars[B_DRAIN], 0);
        }
        __syncwarp();
    } else {
        // =================================================================== softmax
        const int t = warp >> 2;  // Q tile
        const int wq = warp & 3;  // TMEM lane quarter
        const int row_in_tile = wq * 32 + lane;
        const int grow = q0 + t * BM + row_in_tile;
        const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_bits + t * 128;
        const uint32_t tO = tmem + lane_bits + 256 + t * 128;
        // P of this tile is ready: the leader's barrier in a pair (a remote arrive)
        const uint32_t pfull = kPair ? mapa_shared(smem_u32(&bars[B_P_FULL + t]), 0) : 0u;
        const int seg_end = seg_end_of_row(p, grow);
        // Operand exponents: the staged Q row is Q * c0 * 2^eq (c0 = softmax scale * log2 e), the
        // head's current K and V are K * 2^ek and V * 2^ev, its history K and V are dequantised
        // values * 2^ehk and * 2^ehv.  A raw score of a current key is therefore 2^(eq + ek) times
        // the true score in log2 units, of a history key 2^(eq + ehk) times it: each tile kind gets
        // its own multiplier, an exact power of two (at least the smallest normal float, so that
        // masked -inf scores stay -inf: below it every true score is under 2^-89 and rounds to the
        // same probabilities).  Scaled scores are exact, so the row maximum maps to 2^0 exactly.
        const int eq = grow < p.lq ? static_cast<int>(p.qexp[static_cast<int64_t>(head) * p.lq + grow]) : 0;
        const int ek = operand_exp(__uint_as_float(p.cur_max[head]));
        const int ev = operand_exp(__uint_as_float(p.cur_max[p.heads + head]));
        const int ehk = p.lh > 0 ? history_exp(__uint_as_float(p.hist_max[head])) : 0;
        const int ehv = p.lh > 0 ? history_exp(__uint_as_float(p.hist_max[p.heads + head])) : 0;
        const float c_cur = fmaxf(mul_pow2(1.0f, -(eq + ek)), 0x1p-126f);
        const float c_hist = fmaxf(mul_pow2(1.0f, -(eq + ehk)), 0x1p-126f);
        // O accumulates history values at 2^ehv and current values at 2^ev: at the first current
        // tile after history tiles it is rescaled by 2^(ev - ehv)
        const int dv = ev - ehv;
        const bool v_switch = n_hist_loc > 0 && n_loc > n_hist_loc && dv != 0;
        const float v_switch_fac = pow2i(max(-126, min(127, dv)));
        const int e_out = n_loc > n_hist_loc ? ev : ehv;  // O is in units of 2^e_out at the end
        if (grow < p.lq && (c_cur > kMaxSoftmaxMul || (n_hist_loc > 0 && c_hist > kMaxSoftmaxMul) ||
                            (v_switch && (dv > kMaxVExpShift || dv < -kMaxVExpShift))))
            record_status(p.status, kStatusRange, 410);
        float mref = -INFINITY;        // reference maximum (log2 domain)
        float l = 0.0f;                // running sum of p against the reference
        bool ok = true;
        for (int j = 0; j < n_loc; ++j) {
            const bool hist = is_hist(j);
            const float c = hist ? c_hist : c_cur;  // > 0
            const uint32_t pj = static_cast<uint32_t>(j) & 1u;
            ok = mbar_wait_inline(&bars[B_S_FULL + t], pj, p.status, abort_flag, 401);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key0 = key0_of(j);
            const int limit = hist ? (p.lh - key0) : (seg_end - key0);  // columns < limit are visible
            uint32_t r[4][32];
            load_s_row(tS, r);
            if (limit < BN) mask_row(r, limit);
            const float mnew = fmaxf(mref, row_max(r) * c);
            const bool grow_ref = mnew > mref + kRescaleLog2;  // always on the row's first visible tile
            const bool switch_now = v_switch && j == n_hist_loc;  // uniform over the CTA
            if (__any_sync(0xFFFFFFFFu, grow_ref) || switch_now) {
                const float alpha = grow_ref ? ex2_approx(mref - mnew) : 1.0f;  // mref = -inf -> 0
                if (j > 0) {
                    // O holds earlier tiles; their PV completed before this tile's QK^T did (the
                    // tensor core completes one thread's MMAs in order), so the wait returns at once
                    const bool okw = mbar_wait_inline(&bars[B_O_DONE + t], (static_cast<uint32_t>(j) - 1u) & 1u,
                                                      p.status, abort_flag, 403);
                    if (!__all_sync(0xFFFFFFFFu, okw)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    rescale_o_row(tO, switch_now ? alpha * v_switch_fac : alpha);
                }
                l *= alpha;
                if (grow_ref) mref = mnew;
            }
            uint32_t w[2][32];
            l += row_probs(r, c, mref == -INFINITY ? 0.0f : mref, w);
            tmem_st32(tS, w[0]);
            tmem_st32(tS + 32, w[1]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (kPair)
                    mbar_arrive_cluster(pfull);
                else
                    mbar_arrive(&bars[B_P_FULL + t]);
            }
        }
        // ---- epilogue
        if (ok) {
            bool okw = mbar_wait_inline(&bars[B_O_DONE + t], (static_cast<uint32_t>(n_loc) - 1u) & 1u, p.status,
                                        abort_flag, 404);
            ok = __all_sync(0xFFFFFFFFu, okw);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            const float vf = pow2i(-e_out);  // e_out in [-113, 126]
            const float lse_row = l > 0.0f ? (mref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
            const bool live = grow < p.lq;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tO + ch * 32, r);
                tmem_wait_ld(r);
                if (!live) continue;
                if (p.n_splits == 1) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(grow) * p.heads + head) *
                                                                        kHeadDim + ch * 32);
                    auto o_at = [&](int k) { return __uint_as_float(r[k]) * inv_l * vf; };
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2_sat(o_at(8 * q + 0), o_at(8 * q + 1));
                        w.y = pack_bf16x2_sat(o_at(8 * q + 2), o_at(8 * q + 3));
                        w.z = pack_bf16x2_sat(o_at(8 * q + 4), o_at(8 * q + 5));
                        w.w = pack_bf16x2_sat(o_at(8 * q + 6), o_at(8 * q + 7));
                        dst[q] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(
                        p.part_o + ((static_cast<int64_t>(split) * p.lq + grow) * p.heads + head) * kHeadDim + ch * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv_l * vf,
                                             __uint_as_float(r[4 * q + 1]) * inv_l * vf,
                                             __uint_as_float(r[4 * q + 2]) * inv_l * vf,
                                             __uint_as_float(r[4 * q + 3]) * inv_l * vf);
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
    if constexpr (kPair) {
        // no remote arrive, copy or MMA of the pair may still target either CTA past this point
        cluster_sync_all();
        if (warp == kMmaWarp) {
            tc_fence_after();
            tmem_dealloc_pair(tmem, 512);
        }
    } else {
        __syncthreads();
        if (warp == kMmaWarp) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    }
}

// ------------------------------------------------------------------- operand staging
// Both staging kernels walk one flat index over their outputs, in output order (head-major
// rows, so every warp writes contiguous bytes), and each thread issues kStageUnroll independent
// 16-byte loads before converting any of them, to keep enough bytes in flight for HBM.
constexpr int kStageUnroll = 4;

// Maxima, per head, of the current K and V magnitudes (as fp32 bit patterns) and of the history
// K and V row scales: cur_max[0][h] = max |K|, cur_max[1][h] = max |V| over the current tokens,
// hist_max[0][h] = max k_scale, hist_max[1][h] = max v_scale over the history rows.  Block
// (x, h) folds its share into the maxima with atomicMax on the bit patterns (non-negative floats
// order as unsigned integers), so the result does not depend on the order of the blocks.  The
// targets are zeroed before the launch.
struct RangeParams {
    const uint16_t *k, *v;  // current K, V bf16 [lq][heads][128] (token stride row_stride), or null
    int64_t row_stride;
    int32_t lq, heads;
    const float *ks, *vs;   // history scales [heads][cap], or null
    int64_t cap;
    int32_t lh;
    uint32_t *cur_max;      // [2][heads]
    uint32_t *hist_max;     // [2][heads]
};
constexpr int kRangeCurRows = 256;    // current rows per block (16 per pass of 256 threads)
constexpr int kRangeHistRows = 4096;  // history rows per block (256 per pass)

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t m = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) m = max(m, red[i]);
    return m;
}

__global__ void __launch_bounds__(256) range_kernel(const __grid_constant__ RangeParams p) {
    __shared__ uint32_t red[8];
    const int head = blockIdx.y;
    if (p.k != nullptr) {
        const int r0 = blockIdx.x * kRangeCurRows;
        uint32_t km = 0, vm = 0;
        if (r0 < p.lq) {
            const int r1 = min(p.lq, r0 + kRangeCurRows);
            const int sub = threadIdx.x & 15;
            for (int row = r0 + (threadIdx.x >> 4); row < r1; row += 16) {
                const int64_t off = static_cast<int64_t>(row) * p.row_stride + head * kHeadDim + sub * 8;
                km = max(km, bf16x8_absmax_bits(__ldg(reinterpret_cast<const uint4 *>(p.k + off))));
                vm = max(vm, bf16x8_absmax_bits(__ldg(reinterpret_cast<const uint4 *>(p.v + off))));
            }
        }
        km = block_max_u32(km, red);
        vm = block_max_u32(vm, red);
        if (threadIdx.x == 0 && r0 < p.lq) {
            atomicMax(p.cur_max + head, km << 16);
            atomicMax(p.cur_max + p.heads + head, vm << 16);
        }
    }
    if (p.ks != nullptr) {
        const int r0 = blockIdx.x * kRangeHistRows;
        uint32_t km = 0, vm = 0;
        if (r0 < p.lh) {
            const int r1 = min(p.lh, r0 + kRangeHistRows);
            const float *ks = p.ks + static_cast<int64_t>(head) * p.cap;
            const float *vs = p.vs + static_cast<int64_t>(head) * p.cap;
            for (int row = r0 + threadIdx.x; row < r1; row += 256) {
                km = max(km, __float_as_uint(__ldg(ks + row)) & 0x7FFFFFFFu);
                vm = max(vm, __float_as_uint(__ldg(vs + row)) & 0x7FFFFFFFu);
            }
        }
        km = block_max_u32(km, red);
        vm = block_max_u32(vm, red);
        if (threadIdx.x == 0 && r0 < p.lh) {
            atomicMax(p.hist_max + head, km);
            atomicMax(p.hist_max + p.heads + head, vm);
        }
    }
}

struct StageCur {
    const uint16_t *src[3];  // q, k, v: bf16 [lq][heads][128], token stride row_stride elements
    uint16_t *dst;           // FP16 [3][heads][lq][128] (Q, K, V)
    int8_t *qexp;            // [heads][lq]: the exponent e of each staged Q row (Q * c0 * 2^e)
    const uint32_t *cur_max; // [2][heads]: max |K|, max |V| (fp32 bit patterns)
    float c0;                // softmax scale * log2(e)
    int *status;
    int64_t row_stride;
    int32_t heads, lq;
    FastDiv div_lq, div_heads;
};

// Q, K, V BF16 -> FP16 into the head-major layout.  A Q row is multiplied by c0 = softmax scale *
// log2(e) and by the power of two 2^e that puts its largest product in [2^14, 2^15) (the 16 lanes
// holding the row reduce its maximum); K and V of a head by the power of two from that head's
// maximum.  With the scale inside Q, the attention kernel's score multiplier is an exact power of
// two, so scaled scores are exact and the row maximum's own probability is exactly 2^0 at any
// score magnitude.  Item o is 8 values (16 bytes): output row r = o / 16 =
// (which * heads + head) * lq + token; the 16 items of a row sit in 16 consecutive lanes.
__global__ void __launch_bounds__(256) stage_cur_kernel(const __grid_constant__ StageCur s) {
    const int64_t n = 3ll * s.heads * s.lq * 16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;  // a multiple of 256
    // the loop condition is uniform over a half-warp (n and stride are multiples of 16), so
    // the row reductions below see all 16 lanes of a row
    for (int64_t o0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o0 - (threadIdx.x & 31) < n;
         o0 += kStageUnroll * stride) {
        uint4 w[kStageUnroll];
        uint32_t row[kStageUnroll], which[kStageUnroll], head[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int64_t o = o0 + u * stride;
            w[u] = make_uint4(0u, 0u, 0u, 0u);
            row[u] = 0u, which[u] = 3u, head[u] = 0u;
            if (o < n) {
                const uint32_t r = static_cast<uint32_t>(o >> 4);
                const uint32_t wh = fdiv(r, s.div_lq);  // which * heads + head
                const uint32_t tok = r - wh * static_cast<uint32_t>(s.lq);
                which[u] = fdiv(wh, s.div_heads);
                head[u] = wh - which[u] * static_cast<uint32_t>(s.heads);
                row[u] = tok;
                const uint16_t *src = s.src[which[u] == 0 ? 0 : (which[u] == 1 ? 1 : 2)];
                w[u] = __ldg(reinterpret_cast<const uint4 *>(src + static_cast<int64_t>(tok) * s.row_stride +
                                                             head[u] * kHeadDim + (o & 15) * 8));
            }
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            // the row maximum over the 16 lanes of this row (used for Q rows)
            uint32_t m = bf16x8_absmax_bits(w[u]);
#pragma unroll
            for (int d = 8; d >= 1; d >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
            const int64_t o = o0 + u * stride;
            if (o >= n) continue;
            float f;
            if (which[u] == 0) {
                const float qm = __uint_as_float(m << 16) * s.c0;  // the row's largest |q| * c0
                const int e = operand_exp(qm);
                f = s.c0 * pow2i(e);
                if ((o & 15) == 0) {
                    s.qexp[static_cast<int64_t>(head[u]) * s.lq + row[u]] = static_cast<int8_t>(e);
                    if (!(qm < INFINITY)) record_status(s.status, kStatusRange, 411);  // |q| * scale > 3e38
                }
            } else {
                f = pow2i(operand_exp(__uint_as_float(__ldg(s.cur_max + (which[u] - 1) * s.heads + head[u]))));
            }
            reinterpret_cast<uint4 *>(s.dst)[o] = bf16x8_to_f16x8_scaled(w[u], f);
        }
    }
}

struct StageHist {
    const int8_t *codes[2];   // history k, v: [heads][cap][128]
    const float *scale[2];    // [heads][cap]
    uint16_t *dst;            // FP16 [2][heads][dst_cap][128] (K, V)
    const uint32_t *hist_max; // [2][heads]: the largest k and v row scale (fp32 bit patterns)
    int64_t cap, dst_cap;
    int32_t lh, heads;
    FastDiv div_lh;
};

// History K and V: codes times the row's scale times the head's power of two 2^e, the exact
// integer code multiplied in fp32 by scale * 2^e (itself exact) and the product rounded to FP16.
// Item o is 16 codes (16 bytes in, 32 bytes out): row r = o / 8 = (which * heads + head) * lh +
// token.
__global__ void __launch_bounds__(256) stage_hist_kernel(const __grid_constant__ StageHist s) {
    const int64_t n = 2ll * s.heads * s.lh * 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t o0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o0 < n;
         o0 += kStageUnroll * stride) {
        uint4 w[kStageUnroll];
        float sc[kStageUnroll];
        int64_t drow[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int64_t o = o0 + u * stride;
            if (o < n) {
                const uint32_t r = static_cast<uint32_t>(o >> 3);
                const uint32_t wh = fdiv(r, s.div_lh);  // which * heads + head
                const uint32_t tok = r - wh * static_cast<uint32_t>(s.lh);
                const int which = static_cast<int>(wh) >= s.heads ? 1 : 0;
                const int head = static_cast<int>(wh) - which * s.heads;
                const int64_t srow = static_cast<int64_t>(head) * s.cap + tok;
                drow[u] = static_cast<int64_t>(wh) * s.dst_cap + tok;
                w[u] = __ldg(reinterpret_cast<const uint4 *>(s.codes[which] + srow * kHeadDim) + (o & 7));
                const int e = history_exp(__uint_as_float(__ldg(s.hist_max + which * s.heads + head)));
                sc[u] = __ldg(s.scale[which] + srow) * pow2i(e);
            }
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int64_t o = o0 + u * stride;
            if (o >= n) continue;
            const uint32_t words[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[4];
                s8x4_to_f32(words[q], f);
                h[2 * q] = pack_f16x2_sat(f[0] * sc[u], f[1] * sc[u]);
                h[2 * q + 1] = pack_f16x2_sat(f[2] * sc[u], f[3] * sc[u]);
            }
            uint4 *d = reinterpret_cast<uint4 *>(s.dst + drow[u] * kHeadDim) + 2 * (o & 7);
            d[0] = make_uint4(h[0], h[1], h[2], h[3]);
            d[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

// Split-KV merge: O = sum_s w_s O_s with w_s = exp(lse_s - max lse) / sum_t exp(lse_t - max lse),
// in a fixed order.  The weights are normalised first, so the sum is a convex combination of the
// partials and cannot overflow for outputs near the top of the BF16 range.
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
            for (int s = 0; s < n_splits; ++s) wsum += __expf(part_lse[(static_cast<int64_t>(s) * heads + h) * lq + row] - mmax);
            const float inv = 1.0f / wsum;  // wsum >= 1: the largest partial contributes exp(0)
            for (int s = 0; s < n_splits; ++s) {
                const float w = __expf(part_lse[(static_cast<int64_t>(s) * heads + h) * lq + row] - mmax) * inv;
                const float4 o = reinterpret_cast<const float4 *>(
                    part_o + ((static_cast<int64_t>(s) * lq + row) * heads + h) * kHeadDim)[g];
                acc.x += w * o.x;
                acc.y += w * o.y;
                acc.z += w * o.z;
                acc.w += w * o.w;
            }
        }
        uint2 w2;
        w2.x = pack_bf16x2_sat(acc.x, acc.y);
        w2.y = pack_bf16x2_sat(acc.z, acc.w);
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

int grid_for(int64_t items, int per_block_items, int cap) {
    const int64_t b = (items + per_block_items - 1) / per_block_items;
    return static_cast<int>(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

// Number of CTAs ("splits") sharing the key range of one head and Q block, from a time model:
// waves x (key tiles per CTA x the time of one tile + a CTA's fixed start and finish), plus, for
// several splits, the partials' HBM traffic (each split's fp32 partials written, then read once
// by the merge, which writes the BF16 output).  The constants are B300 measurements of this
// kernel (about 3,250 SM cycles per tile for both Q tiles of a CTA).
int32_t attn_num_splits(int64_t lq, int64_t lh, int32_t heads, int num_sms) {
    constexpr double kTileUs = 1.6;               // one 128-key tile of a CTA, both Q tiles
    constexpr double kCtaUs = 20.0;               // a CTA's start (Q load, pipeline fill) and finish
    constexpr double kMergeBytesPerUs = 5.0e6;    // about 5 TB/s
    constexpr double kMergeLaunchUs = 3.0;
    const int64_t items = ((lq + kRowsPerCta - 1) / kRowsPerCta) * heads;
    const int64_t tiles = (lh + BN - 1) / BN + (lq + BN - 1) / BN;
    if (items <= 0 || num_sms <= 0) return 1;
    int best = 1;
    double best_us = 0.0;
    for (int s = 1; s <= 16; ++s) {
        if (s > 1 && tiles / s < 8) break;  // keep at least 8 key tiles per split
        const int64_t waves = (items * s + num_sms - 1) / num_sms;
        double us = static_cast<double>(waves) * (static_cast<double>((tiles + s - 1) / s) * kTileUs + kCtaUs);
        if (s > 1)
            us += static_cast<double>(2 * s * (kHeadDim + 1) * 4 + kHeadDim * 2) * static_cast<double>(lq) * heads /
                      kMergeBytesPerUs + kMergeLaunchUs;
        if (s == 1 || us < 0.99 * best_us) {  // a split must save at least 1 %
            best_us = us;
            best = s;
        }
    }
    return best;
}

namespace {
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

size_t staged_history_bytes(int64_t cap_rows, int32_t heads) {
    if (cap_rows <= 0 || heads <= 0) return 0;
    return staged_history_header_bytes(heads) + 2 * static_cast<size_t>(cap_rows) * heads * kHeadDim * 2;
}

size_t staged_history_header_bytes(int32_t heads) { return round_up(static_cast<size_t>(heads) * 8, 1024); }

AttnWorkspace attn_workspace_layout(int64_t lq, int64_t lh, int32_t heads, int32_t n_splits, bool with_history) {
    AttnWorkspace w;
    const size_t row = static_cast<size_t>(kHeadDim) * 2;  // one FP16 head row
    w.cur_bytes = static_cast<size_t>(lq) * heads * row;   // each of Q, K, V
    w.hist_off = 3 * w.cur_bytes;
    w.hist_bytes = with_history ? staged_history_bytes(lh, heads) : 0;
    w.part_off = w.hist_off + w.hist_bytes;
    w.part_bytes = n_splits > 1 ? round_up(static_cast<size_t>(n_splits) * static_cast<size_t>(lq) * heads *
                                               (kHeadDim + 1) * sizeof(float), 256)
                                : 0;
    w.qexp_off = w.part_off + w.part_bytes;
    w.qexp_bytes = round_up(static_cast<size_t>(lq) * heads, 256);
    w.max_off = w.qexp_off + w.qexp_bytes;
    w.max_bytes = round_up(static_cast<size_t>(heads) * 8, 256);
    w.total = w.max_off + w.max_bytes;
    return w;
}

nomas_status launch_stage_history(const nomas_kv_cache &h, int64_t lh, void *block, int64_t cap_rows,
                                  cudaStream_t stream, char *err, size_t err_len) {
    if (lh <= 0) return NOMAS_OK;
    if (2ll * h.heads * lh >= (1ll << 31)) {
        snprintf(err, err_len, "staged rows exceed 2^31 (heads x history tokens too large)");
        return NOMAS_EUNSUPPORTED;
    }
    uint8_t *b = static_cast<uint8_t *>(block);
    uint32_t *hist_max = reinterpret_cast<uint32_t *>(b);
    cudaError_t e = cudaMemsetAsync(hist_max, 0, static_cast<size_t>(h.heads) * 8, stream);
    if (e != cudaSuccess) {
        snprintf(err, err_len, "history maxima reset: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    RangeParams rp;
    memset(&rp, 0, sizeof(rp));
    rp.heads = h.heads;
    rp.ks = h.k_scale;
    rp.vs = h.v_scale;
    rp.cap = h.capacity;
    rp.lh = static_cast<int32_t>(lh);
    rp.hist_max = hist_max;
    const dim3 rgrid(static_cast<unsigned>((lh + kRangeHistRows - 1) / kRangeHistRows), static_cast<unsigned>(h.heads));
    range_kernel<<<rgrid, 256, 0, stream>>>(rp);
    StageHist sh;
    sh.codes[0] = h.k;
    sh.codes[1] = h.v;
    sh.scale[0] = h.k_scale;
    sh.scale[1] = h.v_scale;
    sh.dst = reinterpret_cast<uint16_t *>(b + staged_history_header_bytes(h.heads));  // K, then V
    sh.hist_max = hist_max;
    sh.cap = h.capacity;
    sh.dst_cap = cap_rows;
    sh.lh = static_cast<int32_t>(lh);
    sh.heads = h.heads;
    sh.div_lh = make_fastdiv(static_cast<uint32_t>(lh));
    stage_hist_kernel<<<grid_for(2ll * h.heads * lh * 8, 256 * kStageUnroll, device_sm_count() * 8), 256, 0,
                        stream>>>(sh);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "history staging launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    return NOMAS_OK;
}

// Whether a call runs the CTA-pair variant: one that is not split and does at least 1e13 FLOP.
// Such calls run long enough to hold the GPU at its power cap, where the pair's halved key-tile
// loads and operand reads let the clock stay higher (B300, config 3: 1,216 against 1,195 TFLOP/s
// at 1,627 against 1,566 MHz; Lq 63,616 over 300,000 history tokens: 1,235 against 1,202); on
// shorter calls the cross-SM hand-overs cost more than that (Lq 3,776 without history: 725
// against 760 TFLOP/s).  `force` (the test hook): 1 the single-CTA variant, 2 the pair.
bool attn_use_pair(const AttnLaunch &a, int32_t q_blocks, int32_t force) {
    if (force == 1) return false;
    if (force == 2) return true;
    const double flop = 4.0 * kHeadDim * a.heads * static_cast<double>(a.lq) * static_cast<double>(a.lh + a.lq);
    return a.n_splits == 1 && q_blocks >= 2 && flop >= 1e13;
}

nomas_status launch_seg_attn(const AttnLaunch &a, cudaStream_t stream, char *err, size_t err_len) {
    const int32_t q_blocks = (a.lq + kRowsPerCta - 1) / kRowsPerCta;
    const bool pair = attn_use_pair(a, q_blocks, a.variant);
    static bool attr_set[2][64] = {{false}};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[pair][dev]) {
        cudaError_t e = pair ? cudaFuncSetAttribute(seg_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    AttnCfg<true>::SM_TOTAL + 1024)
                             : cudaFuncSetAttribute(seg_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    AttnCfg<false>::SM_TOTAL + 1024);
        if (e != cudaSuccess) {
            snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
        attr_set[pair][dev] = true;
    }
    // the workspace holds the current operands; the history block (header of maxima, then FP16
    // K and V [heads][hist_cap][128]) is either inside it or the caller's staged history
    const AttnWorkspace lay = attn_workspace_layout(a.lq, a.lh, a.heads, a.n_splits, false);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    uint16_t *qh = reinterpret_cast<uint16_t *>(ws);
    uint16_t *kh = reinterpret_cast<uint16_t *>(ws + lay.cur_bytes);
    uint16_t *vh = reinterpret_cast<uint16_t *>(ws + 2 * lay.cur_bytes);
    uint8_t *part = ws + a.part_off;
    int8_t *qexp = reinterpret_cast<int8_t *>(ws + a.qexp_off);
    uint32_t *cur_max = reinterpret_cast<uint32_t *>(ws + a.max_off);
    const uint8_t *hb = static_cast<const uint8_t *>(a.hist_block);
    const uint32_t *hist_max = a.lh > 0 ? reinterpret_cast<const uint32_t *>(hb) : cur_max;
    const uint16_t *hkh =
        a.lh > 0 ? reinterpret_cast<const uint16_t *>(hb + staged_history_header_bytes(a.heads)) : nullptr;
    const uint16_t *hvh = a.lh > 0 ? hkh + static_cast<size_t>(a.hist_cap) * a.heads * kHeadDim : nullptr;

    AttnParams p;
    memset(&p, 0, sizeof(p));
    p.heads = a.heads;
    p.lq = a.lq;
    p.lh = static_cast<int32_t>(a.lh);
    p.n_seg = a.n_seg;
    for (int i = 0; i <= a.n_seg; ++i) p.seg_off[i] = a.seg_off[i];
    const float scale = a.softmax_scale != 0.0f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(kHeadDim));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.q_blocks = q_blocks;
    p.q_pairs = (q_blocks + 1) / 2;
    p.n_splits = a.n_splits;
    p.n_hist_tiles = static_cast<int32_t>((a.lh + BN - 1) / BN);
    p.out = static_cast<uint16_t *>(a.out);
    p.lse = a.lse;
    if (a.n_splits > 1) {
        p.part_o = reinterpret_cast<float *>(part);
        p.part_lse = p.part_o + static_cast<size_t>(a.n_splits) * a.lq * a.heads * kHeadDim;
    }
    p.qexp = qexp;
    p.cur_max = cur_max;
    p.hist_max = hist_max;
    p.status = device_status_word();
    p.fault = a.fault;

    CUtensorMap tq, tk, tv, thk, thv;
    memset(&thk, 0, sizeof(thk));
    memset(&thv, 0, sizeof(thv));
    {
        // staged Q / K / V: FP16 [heads][lq][128]; rows past lq read as zero.  Boxes of 64 dims x
        // 128 rows, K's 64 rows in the pair variant (each CTA loads half of a K tile's keys)
        const cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(a.lq), static_cast<cuuint64_t>(a.heads)};
        const cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(a.lq) * kHeadDim * 2};
        const cuuint32_t box[3] = {64, 128, 1};
        const cuuint32_t kbox[3] = {64, pair ? 64u : 128u, 1};
        if (!encode(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, qh, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, err,
                    err_len, "q") ||
            !encode(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, kh, dims, strides, kbox, CU_TENSOR_MAP_SWIZZLE_128B, err,
                    err_len, "k_cur") ||
            !encode(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vh, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, err,
                    err_len, "v_cur"))
            return NOMAS_EINVAL;
    }
    if (a.lh > 0) {
        // staged history K / V: FP16 [heads][hist_cap][128]; rows past lh read as zero
        const cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(a.lh), static_cast<cuuint64_t>(a.heads)};
        const cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(a.hist_cap) * kHeadDim * 2};
        const cuuint32_t box[3] = {64, 128, 1};
        const cuuint32_t kbox[3] = {64, pair ? 64u : 128u, 1};
        if (!encode(&thk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t *>(hkh), dims, strides, kbox,
                    CU_TENSOR_MAP_SWIZZLE_128B, err, err_len, "history k") ||
            !encode(&thv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t *>(hvh), dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B, err, err_len, "history v"))
            return NOMAS_EINVAL;
    }
    const int64_t grid = (pair ? 2ll * p.q_pairs : static_cast<int64_t>(p.q_blocks)) * a.heads * a.n_splits;
    if (grid <= 0) return NOMAS_OK;
    if (grid > 0x7FFFFFFF) {
        snprintf(err, err_len, "grid too large");
        return NOMAS_EUNSUPPORTED;
    }
    if (3ll * a.heads * a.lq >= (1ll << 31)) {
        snprintf(err, err_len, "staged rows exceed 2^31 (heads x tokens too large)");
        return NOMAS_EUNSUPPORTED;
    }
    const int sms = device_sm_count();
    cudaError_t e = cudaMemsetAsync(cur_max, 0, static_cast<size_t>(a.heads) * 8, stream);
    if (e != cudaSuccess) {
        snprintf(err, err_len, "operand maxima reset: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    {
        RangeParams rp;
        memset(&rp, 0, sizeof(rp));
        rp.k = static_cast<const uint16_t *>(a.k);
        rp.v = static_cast<const uint16_t *>(a.v);
        rp.row_stride = a.row_stride;
        rp.lq = a.lq;
        rp.heads = a.heads;
        rp.cur_max = cur_max;
        const dim3 rgrid(static_cast<unsigned>((a.lq + kRangeCurRows - 1) / kRangeCurRows),
                         static_cast<unsigned>(a.heads));
        range_kernel<<<rgrid, 256, 0, stream>>>(rp);
    }
    {
        StageCur sc;
        sc.src[0] = static_cast<const uint16_t *>(a.q);
        sc.src[1] = static_cast<const uint16_t *>(a.k);
        sc.src[2] = static_cast<const uint16_t *>(a.v);
        sc.dst = qh;  // Q, K, V follow one another
        sc.qexp = qexp;
        sc.cur_max = cur_max;
        sc.c0 = p.scale_log2;
        sc.status = p.status;
        sc.row_stride = a.row_stride;
        sc.heads = a.heads;
        sc.lq = a.lq;
        sc.div_lq = make_fastdiv(static_cast<uint32_t>(a.lq));
        sc.div_heads = make_fastdiv(static_cast<uint32_t>(a.heads));
        stage_cur_kernel<<<grid_for(3ll * a.heads * a.lq * 16, 256 * kStageUnroll, sms * 8), 256, 0, stream>>>(sc);
    }
    if (pair) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = AttnCfg<true>::SM_TOTAL + 1024;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, seg_attn_kernel<true>, tq, tk, tv, thk, thv, p);
    } else {
        seg_attn_kernel<false><<<static_cast<unsigned>(grid), kThreads, AttnCfg<false>::SM_TOTAL + 1024, stream>>>(
            tq, tk, tv, thk, thv, p);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "seg_attn launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    if (a.n_splits > 1) {
        const int64_t threads = static_cast<int64_t>(a.lq) * a.heads * 32;
        int64_t blocks = (threads + 255) / 256;
        const int64_t cap = static_cast<int64_t>(sms) * 8 * 4;
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
