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
//   warp 8      TMA producer: Q once; per key tile the K and V tiles into a 2-deep ring of
//               32 KB operand buffers each.  History tiles arrive as INT8 codes in the upper
//               half of the buffer (plus their K and V scale rows); current tiles as BF16.
//   warps 10-13 converters: Q (once) and current K and V tiles BF16 -> FP16 in place; history
//               tiles, one thread per key row, codes * k_scale and codes * v_scale formed in
//               fp32 and rounded once to FP16, expanded in place into the 128B-swizzled
//               operand layout (each thread reads its whole row before writing over it).
//   warp 9      MMA issuer (one thread): S_t = Q_t K^T (FP16, kind::f16, M=N=128, fp32 in
//               TMEM) for both Q tiles, then O_t += P_t V with P_t read from TMEM (FP16).
//               FP16 operands hold BF16 inputs exactly within FP16's range (|x| <= 65504,
//               beyond which they saturate) and the dequantised history to 11 bits.
//   warps 0-7   softmax, one thread per query row (TMEM lane = row), exp2 domain: one pass
//               over S per tile against the running reference maximum (paired fp32 FMA/ADD,
//               ex2 on the SFU), 32-column chunks; a chunk is redone with a new reference, and
//               the stored P, l and O rescaled, only when its sum would leave the FP16 range of
//               P (always on a row's first tile).  Masking runs on boundary tiles only.
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
constexpr int NK = 2;     // K operand buffers
constexpr int NV = 2;     // V operand buffers
constexpr int NSC = 2;    // history scale slots
// A chunk of P is accepted against the running reference when its probability
// sum stays below this bound: every P value then fits FP16 (max 65504) with room to spare.
constexpr float kChunkSumLimit = 32768.0f;
constexpr int kChunk = 32;              // S columns per softmax step
constexpr int kChunks = BN / kChunk;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_Q = 0;                        // 2 Q tiles x (2 halves x [128 rows][128 B])
constexpr uint32_t SM_K = SM_Q + 65536;             // NK x 32 KB K operand (K-major, SW128)
constexpr uint32_t SM_V = SM_K + NK * 32768;        // NV x 32 KB V operand (MN-major, SW128)
constexpr uint32_t SM_SC = SM_V + NV * 32768;       // NSC x (k_scale[128] + v_scale[128]) fp32
constexpr uint32_t SM_BAR = SM_SC + NSC * 1024;     // mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 512;          // TMEM base address, abort flag
constexpr uint32_t SM_TOTAL = SM_MISC + 64;
static_assert(SM_TOTAL <= 232448, "shared memory map exceeds 227 KB");

enum {
    B_Q = 0,
    B_K_LOADED = 1,                 // NK: INT8 codes or BF16 K landed        -> converters
    B_K_FULL = B_K_LOADED + NK,     // NK: FP16 K operand ready               -> MMA
    B_K_FREE = B_K_FULL + NK,       // NK: both QK^T of the tile done         -> producer
    B_V_LOADED = B_K_FREE + NK,     // NV: INT8 codes or BF16 V landed        -> converters
    B_V_FULL = B_V_LOADED + NV,     // NV: FP16 V operand ready               -> MMA
    B_V_FREE = B_V_FULL + NV,       // NV: both PV of the tile done           -> producer
    B_SC_FULL = B_V_FREE + NV,      // NSC: scale rows landed                 -> converters
    B_SC_FREE = B_SC_FULL + NSC,    // NSC: converters done with the scales   -> producer
    B_Q_READY = B_SC_FREE + NSC,    // Q converted to FP16                    -> MMA
    B_S_FULL = B_Q_READY + 1,       // 2
    B_P_FULL = B_S_FULL + 2,        // 2 (4 warps each)
    B_O_DONE = B_P_FULL + 2,        // 2
    B_DRAIN = B_O_DONE + 2,
    B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT * 8 <= 512, "barrier area");
static_assert(B_COUNT <= 32, "producer arms at most 32 barriers");
// Every barrier is completed once per use of its buffer or slot and waited, phase after
// phase, by roles that cannot fall two phases behind it: a buffer is refilled (next phase)
// only after every role that waits on its current phase has released it.  That keeps every
// parity wait unambiguous.

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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) { return pack_f16x2_sat(lo, hi); }

// One key row of a history K tile: 128 INT8 codes at `in` (the upper half of the buffer)
// -> FP16(code * k_scale) (formed in fp32, rounded once, saturating) into the K-major SW128
// operand (`buf`, row `t`).  Every input chunk is read before any output is written, since
// the row's upper-half output overlays its input.
__device__ __forceinline__ void expand_k_row(uint8_t *buf, int t, float ks) {
    const uint8_t *in = buf + 16384 + t * 128;
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint4 *>(in + (((i + t) & 7) << 4));
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    const float2 sc = make_float2(ks, ks);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int cc = (i + t) & 7;  // input chunk: dims 16cc .. 16cc+15
        const uint32_t words[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t u = words[q] ^ 0x80808080u;
            float2 a = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)));
            float2 b = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)));
            a = __fmul2_rn(__fadd2_rn(a, bias), sc);
            b = __fmul2_rn(__fadd2_rn(b, bias), sc);
            o[2 * q] = pack_f16x2_sat(a.x, a.y);
            o[2 * q + 1] = pack_f16x2_sat(b.x, b.y);
        }
        const int g0 = 2 * cc;  // 8-element output group (16 bytes)
        uint8_t *d0 = buf + (g0 >> 3) * 16384 + t * 128;
        *reinterpret_cast<uint4 *>(d0 + ((((g0 & 7)) ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4 *>(d0 + ((((g0 + 1) & 7) ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// One key row of a history V tile: codes * v_scale rounded once to FP16 (saturating) into
// the MN-major SW128 operand (row = key), in place as for K.
__device__ __forceinline__ void expand_v_row(uint8_t *buf, int t, float vs) {
    const uint8_t *in = buf + 16384 + t * 128;
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint4 *>(in + (((i + t) & 7) << 4));
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
    const float2 sc = make_float2(vs, vs);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int cc = (i + t) & 7;
        const uint32_t words[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t u = words[q] ^ 0x80808080u;
            float2 a = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)));
            float2 b = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                   __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)));
            a = __fmul2_rn(__fadd2_rn(a, bias), sc);
            b = __fmul2_rn(__fadd2_rn(b, bias), sc);
            o[2 * q] = pack_f16x2_sat(a.x, a.y);
            o[2 * q + 1] = pack_f16x2_sat(b.x, b.y);
        }
        const int g0 = 2 * cc;
        uint8_t *d0 = buf + (g0 >> 3) * 16384 + t * 128;
        *reinterpret_cast<uint4 *>(d0 + ((((g0 & 7)) ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4 *>(d0 + ((((g0 + 1) & 7) ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// One key row of a current V tile, BF16 -> FP16 in place (element positions unchanged).
__device__ __forceinline__ void convert_v_row_bf16(uint8_t *buf, int t) {
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
        uint4 *p = reinterpret_cast<uint4 *>(buf + (k >> 3) * 16384 + t * 128 + (((k + t) & 7) << 4));
        *p = bf16x8_to_f16x8(*p);
    }
}

// TMEM <-> registers for one softmax chunk (overloads by chunk width).
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32(taddr, r); }
__device__ __forceinline__ void tmem_st_chunk(uint32_t taddr, const uint32_t (&w)[8]) { tmem_st8(taddr, w); }
__device__ __forceinline__ void tmem_st_chunk(uint32_t taddr, const uint32_t (&w)[16]) { tmem_st16(taddr, w); }

// p = 2^(x * c - mref) for the raw scores r of columns col0 .. col0 + kChunk - 1 (columns >=
// limit give 0), packed to FP16 pairs in w.  Returns the sum of the fp32 p values.
__device__ __forceinline__ float chunk_probs(const uint32_t (&r)[kChunk], float c, int col0, int limit, float mref,
                                             uint32_t (&w)[kChunk / 2]) {
    const float2 negm = make_float2(-mref, -mref);
    const float2 cc = make_float2(c, c);
    const bool masked = col0 + kChunk > limit;
    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kChunk; k += 4) {
        float2 a = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), cc, negm);
        float2 b = __ffma2_rn(make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])), cc, negm);
        if (masked) {
            const int lim = limit - col0;
            if (k >= lim) a.x = -INFINITY;
            if (k + 1 >= lim) a.y = -INFINITY;
            if (k + 2 >= lim) b.x = -INFINITY;
            if (k + 3 >= lim) b.y = -INFINITY;
        }
        const float2 pa = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        const float2 pb = make_float2(ex2_approx(b.x), ex2_approx(b.y));
        s01 = __fadd2_rn(s01, pa);
        s23 = __fadd2_rn(s23, pb);
        w[k >> 1] = pack_f16x2(pa.x, pa.y);
        w[(k >> 1) + 1] = pack_f16x2(pb.x, pb.y);
    }
    const float2 s = __fadd2_rn(s01, s23);
    return s.x + s.y;
}

// Maximum of x * c over the visible columns of one chunk (-inf if none).
__device__ __forceinline__ float chunk_max(const uint32_t (&r)[kChunk], float c, int col0, int limit) {
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
        if (col0 + k < limit) mx = fmaxf(mx, __uint_as_float(r[k]) * c);
    return mx;
}

// Multiplies the FP16 pairs in TMEM columns [taddr, taddr + 8 * n8) by alpha.
__device__ __noinline__ void rescale_f16_cols(uint32_t taddr, int n8, float alpha) {
    for (int q = 0; q < n8; ++q) {
        uint32_t w[8];
        tmem_ld8(taddr + q * 8, w);
        tmem_wait_ld(w);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[k]);
            const float2 f = __half22float2(h);
            w[k] = pack_f16x2(f.x * alpha, f.y * alpha);
        }
        tmem_st8(taddr + q * 8, w);
    }
    tmem_st_wait();
}

// Multiplies 128 fp32 TMEM columns (one O row block) by alpha.
__device__ __noinline__ void rescale_f32_cols(uint32_t taddr, float alpha) {
    for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tmem_ld32(taddr + ch * 32, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
        tmem_st32(taddr + ch * 32, r);
    }
    tmem_st_wait();
}

// Slow path of a softmax tile (warp-uniform):
// chunk `ch` would push P past the FP16 range against the reference `mref`.  The new
// reference is max(mref, maximum of chunks ch..7); the P already stored (columns [0, 8ch))
// and, when earlier tiles were accumulated (`o_done` non-null), O are rescaled to it.
// Returns the new reference, the factor alpha applied, and ok = 0 if the wait for the last
// PV gave up.
struct Recovery {
    float mref, alpha;
    int ok;
};
__device__ __noinline__ Recovery recover_reference(uint32_t tS, uint32_t tO, int ch, int limit, float c,
                                                   float mref, uint64_t *o_done,
                                                   uint32_t o_parity, int *status, volatile int *abort) {
    float mx = -INFINITY;
    for (int c2 = ch; c2 < kChunks; ++c2) {
        uint32_t r[kChunk];
        tmem_ld_chunk(tS + c2 * kChunk, r);
        tmem_wait_ld(r);
        mx = fmaxf(mx, chunk_max(r, c, c2 * kChunk, limit));
    }
    Recovery rec;
    const float mnew = fmaxf(mref, mx);
    const bool grow_ref = mnew > mref;
    rec.alpha = grow_ref ? ex2_approx(mref - mnew) : 1.0f;  // mref = -inf -> 0
    rec.mref = grow_ref ? mnew : mref;
    rec.ok = 1;
    if (__any_sync(0xFFFFFFFFu, grow_ref)) {
        if (ch > 0) {
            tmem_st_wait();  // the P chunks stored so far must have landed
            rescale_f16_cols(tS, ch * (kChunk / 16), rec.alpha);
        }
        if (o_done != nullptr) {
            // O holds earlier tiles: wait for the last PV, then scale it
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(o_done, o_parity, status, abort, 403))) {
                rec.ok = 0;
                return rec;
            }
            tc_fence_after();
            rescale_f32_cols(tO, rec.alpha);
        }
    }
    return rec;
}

// Per-row state of the softmax while it walks one tile.
struct RowTile {
    uint32_t tS, tO;
    int limit;
    float c;
    float mref;      // reference maximum (log2 domain)
    float l;         // running sum of earlier tiles (rescaled with the reference)
    float tsum;      // sum of this tile's chunks so far
    uint64_t *o_done;
    uint32_t o_parity;
    int *status;
    volatile int *abort;
};

// One chunk of kChunk columns: probabilities against the reference, the rare recovery, and
// the FP16 P store to columns [ch * kChunk / 2, (ch + 1) * kChunk / 2) (which overlay only S
// columns already read).  After a recovery the chunk's scores are reloaded from TMEM (its S
// columns are still intact), so no register array stays live across the call.  Returns
// false if a wait gave up.
__device__ __forceinline__ bool softmax_chunk(const uint32_t (&r)[kChunk], int ch, RowTile &st) {
    uint32_t w[kChunk / 2];
    float cs = chunk_probs(r, st.c, ch * kChunk, st.limit, st.mref, w);
    const bool bad = !(cs <= kChunkSumLimit);  // also catches inf / NaN (mref = -inf)
    if (__any_sync(0xFFFFFFFFu, bad)) {
        const Recovery rec = recover_reference(st.tS, st.tO, ch, st.limit, st.c, st.mref, st.o_done, st.o_parity,
                                               st.status, st.abort);
        if (!rec.ok) return false;
        st.mref = rec.mref;
        st.l *= rec.alpha;
        st.tsum *= rec.alpha;
        uint32_t r2[kChunk];
        tmem_ld_chunk(st.tS + ch * kChunk, r2);
        tmem_wait_ld(r2);
        cs = chunk_probs(r2, st.c, ch * kChunk, st.limit, st.mref, w);
        if (st.mref == -INFINITY) {
            // nothing visible in this row so far
#pragma unroll
            for (int k = 0; k < kChunk / 2; ++k) w[k] = 0u;
            cs = 0.0f;
        }
    }
    st.tsum += cs;
    tmem_st_chunk(st.tS + ch * (kChunk / 2), w);
    return true;
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
        for (int i = 0; i < NK; ++i) {
            mbar_init(&bars[B_K_LOADED + i], 1);
            mbar_init(&bars[B_K_FULL + i], 1);
            mbar_init(&bars[B_K_FREE + i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&bars[B_V_LOADED + i], 1);
            mbar_init(&bars[B_V_FULL + i], 1);
            mbar_init(&bars[B_V_FREE + i], 1);
        }
        for (int i = 0; i < NSC; ++i) {
            mbar_init(&bars[B_SC_FULL + i], 1);
            mbar_init(&bars[B_SC_FREE + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_S_FULL + i], 1);
            mbar_init(&bars[B_P_FULL + i], 4);
            mbar_init(&bars[B_O_DONE + i], 1);
        }
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_Q_READY], 1);
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

    auto is_hist = [&](int j) { return j < n_hist_loc; };
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
                const int kb = j % NK, vb = j % NV, sb = j % NSC;
                const uint32_t uk = static_cast<uint32_t>(j / NK) & 1u;
                const uint32_t uv = static_cast<uint32_t>(j / NV) & 1u;
                const uint32_t us = static_cast<uint32_t>(j / NSC) & 1u;
                uint8_t *kbuf = smem + SM_K + kb * 32768;
                uint8_t *vbuf = smem + SM_V + vb * 32768;
                if (!mbar_wait(&bars[B_K_FREE + kb], uk ^ 1u, p.status, abort_flag, 101)) break;
                if (is_hist(j)) {
                    const int y = static_cast<int>(static_cast<int64_t>(head) * p.hcap + key0);
                    arm(B_K_LOADED + kb, 16384, uk);
                    tma_load_2d(kbuf + 16384, &tm_hk, &bars[B_K_LOADED + kb], 0, y);
                    if (!mbar_wait(&bars[B_SC_FREE + sb], us ^ 1u, p.status, abort_flag, 102)) break;
                    arm(B_SC_FULL + sb, 1024, us);
                    tma_load_2d(smem + SM_SC + sb * 1024, &tm_hks, &bars[B_SC_FULL + sb], key0, head);
                    tma_load_2d(smem + SM_SC + sb * 1024 + 512, &tm_hvs, &bars[B_SC_FULL + sb], key0, head);
                    if (!mbar_wait(&bars[B_V_FREE + vb], uv ^ 1u, p.status, abort_flag, 103)) break;
                    arm(B_V_LOADED + vb, 16384, uv);
                    tma_load_2d(vbuf + 16384, &tm_hv, &bars[B_V_LOADED + vb], 0, y);
                } else {
                    arm(B_K_LOADED + kb, 32768, uk);
                    tma_load_3d(kbuf, &tm_k, &bars[B_K_LOADED + kb], 0, head, key0);
                    tma_load_3d(kbuf + 16384, &tm_k, &bars[B_K_LOADED + kb], 64, head, key0);
                    if (!mbar_wait(&bars[B_V_FREE + vb], uv ^ 1u, p.status, abort_flag, 104)) break;
                    arm(B_V_LOADED + vb, 32768, uv);
                    tma_load_3d(vbuf, &tm_v, &bars[B_V_LOADED + vb], 0, head, key0);
                    tma_load_3d(vbuf + 16384, &tm_v, &bars[B_V_LOADED + vb], 64, head, key0);
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
            constexpr uint32_t idesc_qk = idesc_f16(false, false, BM, BN);       // FP16 x FP16, K-major both
            constexpr uint32_t idesc_pv = idesc_f16(false, true, BM, kHeadDim);  // FP16, B MN-major
            const uint32_t sq = smem_u32(smem + SM_Q);
            auto issue_qk = [&](int t, int kb) {
                const uint32_t sk = smem_u32(smem + SM_K + kb * 32768);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + t * 128, sdesc_sw128(sq + t * 32768 + off, 16, 1024), sdesc_sw128(sk + off, 16, 1024),
                           idesc_qk, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int vb, bool acc) {
                const uint32_t sv = smem_u32(smem + SM_V + vb * 32768);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, sdesc_sw128(sv + kk * 2048, 16384, 1024),
                           idesc_pv, (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(&bars[B_Q_READY], 0, p.status, abort_flag, 201);
            ok = ok && mbar_wait(&bars[B_K_FULL + 0], 0, p.status, abort_flag, 202);
            if (ok) {
                tc_fence_after();
                issue_qk(0, 0);
                tc_commit(&bars[B_S_FULL + 0]);
                issue_qk(1, 0);
                tc_commit(&bars[B_S_FULL + 1]);
                tc_commit(&bars[B_K_FREE + 0]);
                for (int j = 0; j < n_loc; ++j) {
                    const int vb = j % NV;
                    const uint32_t pj = static_cast<uint32_t>(j) & 1u;
                    if (!mbar_wait(&bars[B_V_FULL + vb], static_cast<uint32_t>(j / NV) & 1u, p.status, abort_flag,
                                   203))
                        break;
                    if (!mbar_wait(&bars[B_P_FULL + 0], pj, p.status, abort_flag, 204)) break;
                    tc_fence_after();
                    issue_pv(0, vb, j > 0);
                    tc_commit(&bars[B_O_DONE + 0]);
                    const bool more = j + 1 < n_loc;
                    const int kn = (j + 1) % NK;
                    if (more) {
                        if (!mbar_wait(&bars[B_K_FULL + kn], static_cast<uint32_t>((j + 1) / NK) & 1u, p.status,
                                       abort_flag, 205))
                            break;
                        tc_fence_after();
                        issue_qk(0, kn);
                        tc_commit(&bars[B_S_FULL + 0]);
                    }
                    if (!mbar_wait(&bars[B_P_FULL + 1], pj, p.status, abort_flag, 206)) break;
                    tc_fence_after();
                    issue_pv(1, vb, j > 0);
                    tc_commit(&bars[B_O_DONE + 1]);
                    tc_commit(&bars[B_V_FREE + vb]);
                    if (more) {
                        issue_qk(1, kn);
                        tc_commit(&bars[B_S_FULL + 1]);
                        tc_commit(&bars[B_K_FREE + kn]);
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
        const int t = threadIdx.x - kConvWarp0 * 32;  // key row of the tile
        {
            // Q (both tiles, both halves) BF16 -> FP16 in place, row t of each block
            const bool okq = mbar_wait(&bars[B_Q], 0, p.status, abort_flag, 300);
            if (bar_red_and(okq)) {
#pragma unroll 4
                for (int k = 0; k < 32; ++k) {
                    uint4 *q = reinterpret_cast<uint4 *>(smem + SM_Q + (k >> 3) * 16384 + t * 128 + (((k + t) & 7) << 4));
                    *q = bf16x8_to_f16x8(*q);
                }
                fence_proxy_async_smem();
                bar_red_and(true);
                if (t == 0) mbar_arrive(&bars[B_Q_READY]);
            }
        }
        for (int j = 0; j < n_loc; ++j) {
            const int kb = j % NK, vb = j % NV, sb = j % NSC;
            const uint32_t uk = static_cast<uint32_t>(j / NK) & 1u;
            const uint32_t uv = static_cast<uint32_t>(j / NV) & 1u;
            const uint32_t us = static_cast<uint32_t>(j / NSC) & 1u;
            uint8_t *vbuf = smem + SM_V + vb * 32768;
            if (is_hist(j)) {
                uint8_t *kbuf = smem + SM_K + kb * 32768;
                float *sc = reinterpret_cast<float *>(smem + SM_SC + sb * 1024);
                bool ok = mbar_wait(&bars[B_K_LOADED + kb], uk, p.status, abort_flag, 301);
                ok = ok && mbar_wait(&bars[B_SC_FULL + sb], us, p.status, abort_flag, 302);
                if (!bar_red_and(ok)) break;
                const float vs = sc[128 + t];
                expand_k_row(kbuf, t, sc[t]);
                fence_proxy_async_smem();
                bar_red_and(true);
                if (t == 0) mbar_arrive(&bars[B_K_FULL + kb]);
                ok = mbar_wait(&bars[B_V_LOADED + vb], uv, p.status, abort_flag, 303);
                if (!bar_red_and(ok)) break;
                expand_v_row(vbuf, t, vs);
                fence_proxy_async_smem();
                bar_red_and(true);
                if (t == 0) {
                    mbar_arrive(&bars[B_V_FULL + vb]);
                    mbar_arrive(&bars[B_SC_FREE + sb]);
                }
            } else {
                uint8_t *kbuf = smem + SM_K + kb * 32768;
                bool ok = mbar_wait(&bars[B_K_LOADED + kb], uk, p.status, abort_flag, 305);
                if (!bar_red_and(ok)) break;
                convert_v_row_bf16(kbuf, t);  // the same in-place BF16 -> FP16 as for V
                fence_proxy_async_smem();
                bar_red_and(true);
                if (t == 0) mbar_arrive(&bars[B_K_FULL + kb]);
                ok = mbar_wait(&bars[B_V_LOADED + vb], uv, p.status, abort_flag, 304);
                if (!bar_red_and(ok)) break;
                convert_v_row_bf16(vbuf, t);
                fence_proxy_async_smem();
                bar_red_and(true);
                if (t == 0) mbar_arrive(&bars[B_V_FULL + vb]);
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
        RowTile st;
        st.tS = tS;
        st.tO = tO;
        st.c = p.scale_log2;
        st.mref = -INFINITY;
        st.l = 0.0f;
        st.status = p.status;
        st.abort = abort_flag;
        bool ok = true;
        for (int j = 0; j < n_loc; ++j) {
            const bool hist = is_hist(j);
            const uint32_t pj = static_cast<uint32_t>(j) & 1u;
            ok = mbar_wait(&bars[B_S_FULL + t], pj, p.status, abort_flag, 401);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const int key0 = key0_of(j);
            st.limit = hist ? (p.lh - key0) : (seg_end - key0);  // columns < limit are visible
            st.tsum = 0.0f;
            st.o_done = j > 0 ? &bars[B_O_DONE + t] : nullptr;
            st.o_parity = (static_cast<uint32_t>(j) - 1u) & 1u;

            // one pass over S in chunks of kChunk columns
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
                uint32_t r[kChunk];
                tmem_ld_chunk(tS + ch * kChunk, r);
                tmem_wait_ld(r);
                if (!softmax_chunk(r, ch, st)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            st.l += st.tsum;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_P_FULL + t]);
        }
        const float mref = st.mref;
        const float l = st.l;
        // ---- epilogue
        if (ok) {
            bool okw = mbar_wait(&bars[B_O_DONE + t], (static_cast<uint32_t>(n_loc) - 1u) & 1u, p.status, abort_flag,
                                 404);
            ok = __all_sync(0xFFFFFFFFu, okw);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
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
