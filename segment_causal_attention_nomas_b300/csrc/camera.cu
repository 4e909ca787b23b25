// camera.cu -- camera conditioning: camera tokens and the camera cross-attention (sm_103a).
//
// comfyui-wiki news, 相机控制作为一等输入: a trajectory gives camera-to-world matrices c2ws
// [N, 4, 4]; the extrinsics are normalised, grouped by four video frames and each group is
// flattened to a 64-value input, which the video tokens query through a cross-attention in every
// dual-stream block (模型内部 table, 相机条件 row); trajectory_translation_scale defaults to 1.0
// and trajectory_rotation_scale to 2.5.
//
// camera_tokens_kernel   one thread per video frame i: E_i = inverse(c2w[0]) . c2w[i] with the
//                        rigid inverse [R0^T | -R0^T t0]; the rotation block times rotation_scale,
//                        the translation column times translation_scale, the bottom row
//                        (0, 0, 0, 1); the 16 values row-major at token i / 4, columns
//                        16 (i % 4) .. 16 (i % 4) + 15.  fp32.
//
// The cross-attention O = softmax(q k^T * scale) v over all camera tokens of the segment, per
// (128 video tokens, head) item:
//   TMA   the Q tile [128 tokens][128] BF16 and the head's camera K, V [NC][128] BF16 (NC = the
//         camera-token count rounded up to 32; rows past the last token arrive as zeros), in
//         128-byte-swizzled boxes of 64 channels.
//   MMA   S[128 x NC] = Q . K^T  (kind::f16 with BF16 operands, M = 128, N = NC, fp32 in TMEM).
//   rows  one thread per query row (TMEM lane = row): the row maximum over the real camera
//         tokens, p = 2^(fl(s * c) - fl(max * c)) (c = scale * log2 e; product and difference
//         rounded separately, so the maximum's p is exactly 1 at any score magnitude, where a fused
//         multiply-subtract would leave the product's rounding error in the exponent) rounded to
//         FP16, l = the sum of the rounded p; V converted in place from BF16 to FP16 after an
//         exact multiplication by 2^ev, ev chosen per head from max |V| so that it lands in
//         [2^14, 2^15) (as for the staged operands of the segment attention); a non-finite l
//         (scores beyond fp32) is reported as NOMAS_ERANGE.
//   MMA   O[128 x 128] = P . V  (kind::f16 with FP16 operands, V MN-major), fp32 in TMEM.
//   rows  O / l * 2^-ev rounded to BF16, staged 128-byte-swizzled in shared memory, stored by TMA
//         (rows past the last token are not written).
// Each item moves 64 KB to and from HBM (plus the camera K and V, from L2): the work is bound
// by HBM bandwidth, and what decides the speed is how many tiles are in flight per SM.
//
// camera_xattn_persistent_kernel<NC>  (NC = 32, 64, 96, 128) one CTA per SM walking a run of
// items of one head:
//     warp 8    TMA: a ring of 3-4 Q tiles, K and V once per head.
//     warp 9    MMA: S of the next item issued before P.V of the current one; two accumulators
//               of 256 TMEM columns (S, with P over its first columns, then O).  Items, heads and
//               ring stages are walked with running counters: the issuing thread shares its SM
//               sub-partition with two softmax warps, and a 64-bit division per item on its path
//               (it used five) made every P.V wait about 1,700 cycles for it.
//     warps 0-7 two groups of four warps on alternate items: softmax (the row's S read from
//               TMEM in one round trip, P to TMEM), epilogue (O to the group's staging tile, one
//               TMA store per item).  The group that takes a head's first item converts its V and
//               publishes the exponent to the other group.
//     A Q tile is handed back as soon as its Q.K^T completes.  Measured on 16 heads (a copy of
//     the same tiles with no arithmetic takes 84.5 us at 63,360 queries): 28 us at 15,840 queries
//     over 18 camera tokens, 36 us at 21,120 over 24, and 88 / 90 / 90 / 97 us at 63,360 over 64 /
//     72 / 96 / 128, against 34, 42.5 and 188 us (72 tokens) for a kernel with one CTA per item.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr int CM = 128;          // query rows per tile
constexpr uint32_t kTile = 32768;  // one [2][128 rows][128 B] tile of 128 tokens x 128 channels

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

constexpr int kPerThreads = 320;   // warps 0-7 softmax/epilogue (two groups), 8 TMA, 9 MMA
constexpr int kPerTmaWarp = 8, kPerMmaWarp = 9;
constexpr int kPerMaxStages = 6;
enum {
    PB_QFULL = 0,                          // [stages] Q tile landed             -> MMA
    PB_QFREE = PB_QFULL + kPerMaxStages,   // [stages] its Q.K^T completed       -> TMA
    PB_KVFULL = PB_QFREE + kPerMaxStages,  // camera K, V of a head landed       -> MMA, softmax warps
    PB_KVFREE,                             // every MMA of that head completed   -> TMA
    PB_SFULL,                              // [2] S in accumulator a             -> softmax group a
    PB_PFULL = PB_SFULL + 2,               // [2] (4 warps) P in TMEM, V FP16    -> MMA
    PB_OFULL = PB_PFULL + 2,               // [2] O in accumulator a             -> softmax group a
    PB_ACCFREE = PB_OFULL + 2,             // [2] (4 warps) O of accumulator a read (NC <= 64) -> MMA
    PB_OSTAGED = PB_ACCFREE + 2,           // [2] (4 warps) O tile staged        -> the group's storing thread
    PB_OFREE = PB_OSTAGED + 2,             // [2] the group's last store read    -> the group's warps
    PB_VRED = PB_OFREE + 2,                // [2] (4 warps) the group's |V| maxima written -> the group
    PB_KVREADY = PB_VRED + 2,              // (4 warps) a head's V in FP16, its exponent published
    PB_DRAIN,
    PB_COUNT
};
// after the barriers: vred [2 groups][4 warps] and vexp [2 head generations] (uint32 each)
constexpr int kPerMiscWords = 10;
static_assert(PB_COUNT * 8 + kPerMiscWords * 4 <= 280, "barrier area");

// Q ring, then two O staging tiles (one per softmax group), then K, V, then barriers.
int per_stages(int nc) {
    const int s = static_cast<int>((232448u - 2u * kTile - static_cast<uint32_t>(nc) * 512u - 320u) / kTile);
    return s < kPerMaxStages ? s : kPerMaxStages;
}
uint32_t per_smem_bytes(int nc) {
    return static_cast<uint32_t>(per_stages(nc) + 2) * kTile + static_cast<uint32_t>(nc) * 512u + 320u;
}
static_assert(280 + 8 <= 320, "barriers and misc fit the 320-byte tail");

struct PerParams {
    int32_t lq, heads, n_cam, nc, nq;
    int32_t tiles;    // 128-token tiles per head
    int64_t items;    // tiles * heads, item = head * tiles + tile
    float scale_log2; // softmax scale * log2(e)
    int *status;
};

// NC = camera tokens rounded up to 32 (64, 96 or 128): S, P and the P.V steps unroll fully.
template <int NC>
__global__ void __launch_bounds__(kPerThreads, 1)
camera_xattn_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ PerParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int nc = NC;
    const int nq = p.nq, tiles = p.tiles;
    // this CTA's run of items: with at least as many CTAs as heads, CTA b takes head b % heads
    // and the k-th of that head's tile ranges (k = b / heads), so the CTAs working at one time
    // read every head of neighbouring token rows; otherwise contiguous runs of the head-major list
    int64_t it0, it1;
    if (static_cast<int>(gridDim.x) >= p.heads) {
        const int h = static_cast<int>(blockIdx.x) % p.heads, k = static_cast<int>(blockIdx.x) / p.heads;
        const int ch = (static_cast<int>(gridDim.x) - h + p.heads - 1) / p.heads;  // CTAs on head h
        it0 = static_cast<int64_t>(h) * tiles + static_cast<int64_t>(tiles) * k / ch;
        it1 = static_cast<int64_t>(h) * tiles + static_cast<int64_t>(tiles) * (k + 1) / ch;
    } else {
        it0 = p.items * blockIdx.x / gridDim.x;
        it1 = p.items * (blockIdx.x + 1) / gridDim.x;
    }
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0) record_status(p.status, kStatusTimeout, 960);
        return;
    }
    uint8_t *so = smem + nq * kTile;  // [2] O staging tiles
    uint8_t *sk = so + 2 * kTile;
    uint8_t *sv = sk + nc * 256;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sv + nc * 256);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(bars) + 280);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint32_t *vred = reinterpret_cast<uint32_t *>(bars + PB_COUNT);  // [2][4]
    volatile uint32_t *vexp = vred + 8;                                // [2]
    if (tid == 0) {
        for (int s = 0; s < nq; ++s) {
            mbar_init(&bars[PB_QFULL + s], 1);
            mbar_init(&bars[PB_QFREE + s], 1);
        }
        mbar_init(&bars[PB_KVFULL], 1);
        mbar_init(&bars[PB_KVFREE], 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars[PB_SFULL + a], 1);
            mbar_init(&bars[PB_PFULL + a], 4);
            mbar_init(&bars[PB_OFULL + a], 1);
            mbar_init(&bars[PB_ACCFREE + a], 4);
            mbar_init(&bars[PB_OSTAGED + a], 4);
            mbar_init(&bars[PB_OFREE + a], 1);
            mbar_init(&bars[PB_VRED + a], 4);
        }
        mbar_init(&bars[PB_KVREADY], 4);
        mbar_init(&bars[PB_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kPerMmaWarp) {
        tmem_alloc(tmem_slot, 512);  // accumulator a: S (P over its first columns) at 256a, O at 256a + 128
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kPerTmaWarp) {
        // ================================================================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            uint32_t armed = 0, armed_par = 0;  // bit s: Q stage s, bit kPerMaxStages: K/V
            int gen = -1;
            int head = static_cast<int>(it0 / tiles), pos = static_cast<int>(it0 % tiles);  // of item i
            int s = 0;
            uint32_t u = 0;  // Q stage of item i and its use count, mod 2
            const int n = static_cast<int>(it1 - it0);
            for (int i = 0; i < n; ++i) {
                const int tok0 = pos * CM;
                if (i == 0 || pos == 0) {
                    ++gen;
                    if (gen >= 1 && !mbar_wait(&bars[PB_KVFREE], (gen - 1) & 1, p.status, abort_flag, 701)) break;
                    mbar_arrive_expect_tx(&bars[PB_KVFULL], static_cast<uint32_t>(nc) * 512u);
                    armed |= 1u << kPerMaxStages;
                    armed_par = (armed_par & ~(1u << kPerMaxStages)) | ((gen & 1u) << kPerMaxStages);
                    for (int half = 0; half < 2; ++half) {
                        tma_load_3d(sk + half * nc * 128, &tm_k, &bars[PB_KVFULL], half * 64, head, 0);
                        tma_load_3d(sv + half * nc * 128, &tm_v, &bars[PB_KVFULL], half * 64, head, 0);
                    }
                }
                if (!mbar_wait(&bars[PB_QFREE + s], u ^ 1u, p.status, abort_flag, 702)) break;
                mbar_arrive_expect_tx(&bars[PB_QFULL + s], kTile);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (u << s);
                for (int half = 0; half < 2; ++half)
                    tma_load_3d(smem + s * kTile + half * 16384, &tm_q, &bars[PB_QFULL + s], half * 64, head, tok0);
                if (++s == nq) s = 0, u ^= 1u;
                if (++pos == tiles) pos = 0, ++head;
            }
            // every copy this thread issued must have landed before the CTA may exit
            for (int b = 0; b <= kPerMaxStages; ++b)
                if (armed & (1u << b)) cam_drain(&bars[b == kPerMaxStages ? PB_KVFULL : PB_QFULL + b], (armed_par >> b) & 1u);
        }
        __syncwarp();
    } else if (warp == kPerMmaWarp) {
        // ========================================================================== MMA
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_f16(true, false, CM, nc);         // BF16 x BF16, both K-major
            const uint32_t idesc_pv = idesc_f16(false, true, CM, kHeadDim);   // FP16, V MN-major
            const uint32_t ak = smem_u32(sk), av = smem_u32(sv);
            const int n = static_cast<int>(it1 - it0);
            // items are walked with running counters (no division per item): the position of
            // items ns and no within their head's tiles, the Q stage of ns and its use parity
            int pos_s = static_cast<int>(it0 % tiles), pos_o = pos_s;
            int st_s = 0;
            uint32_t ph_s = 0;
            int gen_s = -1;  // K/V generation of the last item whose S was issued
            auto issue_s = [&](int i, bool first) -> bool {
                const int a = i & 1;
                if (first) {
                    ++gen_s;
                    if (!mbar_wait(&bars[PB_KVFULL], gen_s & 1, p.status, abort_flag, 711)) return false;
                }
                // S of item i reuses the S/P columns of item i - 2.  They are free once that
                // item's P.V has completed: its epilogue reads only the O columns, and P.V of item
                // i, which overwrites those, waits for the group's P, stored after the epilogue's
                // loads.  Issuing S that early measured faster for 96 and 128 columns (90 against
                // 96 us, 97 against 106 us at 63,360 queries x 16 heads), waiting for the
                // epilogue's loads as well for 32 and 64 columns (88 against 99 us at 64).
                constexpr int kSGate = NC <= 64 ? PB_ACCFREE : PB_OFULL;
                if (i >= 2 && !mbar_wait(&bars[kSGate + a], ((i >> 1) - 1) & 1, p.status, abort_flag, 712))
                    return false;
                if (!mbar_wait(&bars[PB_QFULL + st_s], ph_s, p.status, abort_flag, 713)) return false;
                tc_fence_after();
                const uint32_t aq = smem_u32(smem + st_s * kTile);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + a * 256, sdesc_sw128(aq + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                           sdesc_sw128(ak + (kk >> 2) * nc * 128 + (kk & 3) * 32, 16, 1024), idesc_qk,
                           kk > 0 ? 1u : 0u);
                tc_commit(&bars[PB_SFULL + a]);
                tc_commit(&bars[PB_QFREE + st_s]);  // the Q tile is dead once S is complete
                return true;
            };
            auto issue_o = [&](int i, bool last) -> bool {
                const int a = i & 1;
                if (!mbar_wait(&bars[PB_PFULL + a], (i >> 1) & 1, p.status, abort_flag, 714)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < nc / 16; ++kk)
                    mma_ts(tmem + a * 256 + 128, tmem + a * 256 + kk * 8, sdesc_sw128(av + kk * 2048, nc * 128, 1024),
                           idesc_pv, kk > 0 ? 1u : 0u);
                tc_commit(&bars[PB_OFULL + a]);
                if (last) tc_commit(&bars[PB_KVFREE]);
                return true;
            };
            // Static order: S of item j is issued at most two items ahead of the P.V issued so
            // far (two accumulators), and the first item of a new head only once every P.V of the
            // previous head is issued (its K and V load after those complete):
            // S0, S1, O0, S2, O1, S3, ... within one head.
            bool ok = true;
            int ns = 0, no = 0;
            while (ok && no < n) {
                const bool s_first = ns == 0 || pos_s == 0;  // item ns begins a head
                if (ns < n && ns <= no + 1 && (!s_first || ns == 0 || no == ns)) {
                    ok = issue_s(ns, s_first);
                    ++ns;
                    if (++pos_s == tiles) pos_s = 0;
                    if (++st_s == nq) st_s = 0, ph_s ^= 1u;
                } else {
                    ok = issue_o(no, no + 1 == n || pos_o + 1 == tiles);
                    ++no;
                    if (++pos_o == tiles) pos_o = 0;
                }
            }
            tc_commit(&bars[PB_DRAIN]);
            cam_drain(&bars[PB_DRAIN], 0);  // no MMA may still run when TMEM is freed
        }
        __syncwarp();
    } else {
        // ======================================= softmax and epilogue: group g = warps 4g .. 4g+3
        // takes the items i with i % 2 == g, accumulator g and TMEM lanes 0-127
        const int grp = warp >> 2;
        const int gtid = tid & 127;
        const int row = gtid;  // query row = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tacc = tmem + lane_off + grp * 256;
        uint8_t *ostage = so + grp * kTile;
        const float c = p.scale_log2;
        const int head0 = static_cast<int>(it0 / tiles);
        const int n = static_cast<int>(it1 - it0);
        int ev = 0, ev_head = -1;  // the V exponent of head ev_head (V in FP16 = V * 2^ev)
        uint32_t n_conv = 0;       // V conversions this group has made (PB_VRED phases)
        // head and tile position of item i, advanced by running counters
        int head = static_cast<int>((it0 + grp) / tiles), pos = static_cast<int>((it0 + grp) % tiles);
        for (int i = grp; i < n; i += 2) {
            const int tok0 = pos * CM;
            const int a = grp;
            const uint32_t ph = (i >> 1) & 1;  // this group's item count, mod 2
            // the first item of a head converts that head's V (generation = head - first head)
            const bool new_kv = i == 0 || pos == 0;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_SFULL + a], ph, p.status, abort_flag, 721))) break;
            tc_fence_after();
            // S of the row in registers, one TMEM round trip
            constexpr int NCH = NC / 32;
            uint32_t r[NCH][32];
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) tmem_ld32(tacc + ch * 32, r[ch]);
            tmem_wait_ld(r[0]);
#pragma unroll
            for (int ch = 1; ch < NCH; ++ch) tmem_tie(r[ch]);
            // the row maximum over the real camera tokens (columns below nc - 32 always are)
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (ch < NCH - 1 || ch * 32 + j < p.n_cam) m4[j & 3] = fmaxf(m4[j & 3], __uint_as_float(r[ch][j]));
            const float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            const float mc = m * c;
            float l4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = ch * 32 + 2 * j;
                    const float s0 = __fsub_rn(__fmul_rn(__uint_as_float(r[ch][2 * j]), c), mc);
                    const float s1 = __fsub_rn(__fmul_rn(__uint_as_float(r[ch][2 * j + 1]), c), mc);
                    const float p0 = (ch < NCH - 1 || col < p.n_cam) ? ex2_approx(s0) : 0.0f;
                    const float p1 = (ch < NCH - 1 || col + 1 < p.n_cam) ? ex2_approx(s1) : 0.0f;
                    w[j] = pack_f16x2_sat(p0, p1);
                    const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
                    l4[j & 3] += __low2float(h) + __high2float(h);
                }
                // P of columns 32ch .. 32ch + 31 as FP16 pairs over TMEM columns 16ch .. 16ch + 15
                tmem_st16(tacc + ch * 16, w);
            }
            const float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            tmem_st_wait();
            if (!(l < INFINITY)) record_status(p.status, kStatusRange, 726);  // scores beyond fp32
            const uint32_t gen = static_cast<uint32_t>(head - head0) & 1u;
            if (new_kv) {
                // this head's V to FP16 in place, times 2^ev from its max |V| (no P.V of the
                // previous head can still read it: the producer reloads K and V only after those
                // MMAs completed, and the MMA thread issues this head's first P.V, which waits for
                // this group, before any other).  The group's four warps combine their maxima
                // through PB_VRED; the exponent goes to vexp[gen] for the other group, published
                // by PB_KVREADY.
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_KVFULL], gen, p.status, abort_flag, 722))) break;
                uint4 *v4 = reinterpret_cast<uint4 *>(sv);
                uint32_t vm = 0;
                for (int k = gtid; k < nc * 16; k += 128) vm = max(vm, bf16x8_absmax_bits(v4[k]));
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) vm = max(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, o));
                if (lane == 0) {
                    vred[grp * 4 + (warp & 3)] = vm;
                    mbar_arrive(&bars[PB_VRED + grp]);
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_VRED + grp], n_conv & 1u, p.status, abort_flag, 727)))
                    break;
                ++n_conv;
                const uint32_t *r4 = vred + grp * 4;
                ev = operand_exp(__uint_as_float(max(max(r4[0], r4[1]), max(r4[2], r4[3])) << 16));
                ev_head = head;
                const float vf = pow2i(ev);
                for (int k = gtid; k < nc * 16; k += 128) v4[k] = bf16x8_to_f16x8_scaled(v4[k], vf);
                fence_proxy_async_smem();
                if ((warp & 3) == 0 && lane == 0) vexp[gen] = static_cast<uint32_t>(ev);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[PB_KVREADY]);
            } else if (head != ev_head) {
                // the other group converted this head's V: its exponent (the barrier's phase for
                // this head cannot be overtaken: the next head's conversion waits for this head's
                // last P.V, which waits for this group's P below)
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_KVREADY], gen, p.status, abort_flag, 728))) break;
                ev = static_cast<int>(vexp[gen]);
                ev_head = head;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[PB_PFULL + a]);

            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_OFULL + a], ph, p.status, abort_flag, 723))) break;
            tc_fence_after();
            // the staging tile is free once this group's previous store has read it
            if ((warp & 3) == 0 && lane == 0) {
                bulk_wait_group_read0();
                mbar_arrive(&bars[PB_OFREE + a]);
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[PB_OFREE + a], ph, p.status, abort_flag, 725))) break;
            const float inv_l = 1.0f / l;  // l >= 1: the row maximum contributes 2^0
            const float vinv = pow2i(-ev);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t o[2][32];
                tmem_ld32(tacc + 128 + hf * 64, o[0]);
                tmem_ld32(tacc + 128 + hf * 64 + 32, o[1]);
                tmem_wait_ld(o[0]);
                tmem_tie(o[1]);
                if (NC <= 64 && hf == 1) {
                    // the accumulator's O is in registers (S of item i + 2 waits for this)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[PB_ACCFREE + a]);
                }
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        w[j] = pack_bf16x2_sat(__uint_as_float(o[c2][2 * j]) * inv_l * vinv,
                                               __uint_as_float(o[c2][2 * j + 1]) * inv_l * vinv);
                    store_row_chunk32(ostage, row, 2 * hf + c2, w);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[PB_OSTAGED + a]);
            if ((warp & 3) == 0) {
                bool st_ok = true;
                if (lane == 0) {
                    st_ok = mbar_wait(&bars[PB_OSTAGED + a], ph, p.status, abort_flag, 724);
                    if (st_ok) {
                        for (int half = 0; half < 2; ++half)
                            tma_store_3d(&tm_o, ostage + half * 16384, half * 64, head, tok0);
                        bulk_commit_group();
                    }
                }
                if (!__shfl_sync(0xFFFFFFFFu, st_ok ? 1 : 0, 0)) break;
            }
            pos += 2;
            while (pos >= tiles) pos -= tiles, ++head;
        }
        if (gtid == 0) bulk_wait_group_read0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPerMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
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

namespace {
// The kernel instance for NC camera-token columns (32, 64, 96 or 128).
using CamKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const PerParams);
CamKernel cam_kernel(int nc) {
    return nc == 32   ? camera_xattn_persistent_kernel<32>
           : nc == 64 ? camera_xattn_persistent_kernel<64>
           : nc == 96 ? camera_xattn_persistent_kernel<96>
                      : camera_xattn_persistent_kernel<128>;
}

}  // namespace

nomas_status launch_camera_xattn(const CamLaunch &a, cudaStream_t stream, char *err, size_t err_len) {
    const int nc = (a.n_cam + 31) / 32 * 32;
    const CamKernel kernel = cam_kernel(nc);
    const uint32_t smem = per_smem_bytes(nc);
    static uint32_t attr_bytes[4][64] = {{0}};  // per kernel instance (NC / 32 - 1) and device
    const int ki = nc / 32 - 1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || attr_bytes[ki][dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            return NOMAS_ECUDA;
        }
        if (dev >= 0 && dev < 64) attr_bytes[ki][dev] = smem;
    }
    CUtensorMap tq, tk, tv, to;
    if (!encode_rows(&tq, a.q, a.heads, a.lq, a.q_row_stride, CM, err, err_len, "q") ||
        !encode_rows(&tk, a.k, a.heads, a.n_cam, a.cam_row_stride, nc, err, err_len, "camera k") ||
        !encode_rows(&tv, a.v, a.heads, a.n_cam, a.cam_row_stride, nc, err, err_len, "camera v") ||
        !encode_rows(&to, a.out, a.heads, a.lq, a.out_row_stride, CM, err, err_len, "out"))
        return NOMAS_EINVAL;
    const float scale = a.softmax_scale != 0.0f ? a.softmax_scale : 1.0f / std::sqrt(static_cast<float>(kHeadDim));
    const int tiles = (a.lq + CM - 1) / CM;
    const int64_t items = static_cast<int64_t>(tiles) * a.heads;
    PerParams p;
    memset(&p, 0, sizeof(p));
    p.lq = a.lq;
    p.heads = a.heads;
    p.n_cam = a.n_cam;
    p.nc = nc;
    p.nq = per_stages(nc);
    p.tiles = tiles;
    p.items = items;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = device_status_word();
    const int sms = device_sm_count();
    const int64_t ctas = items < sms ? items : sms;  // one CTA per SM
    kernel<<<static_cast<unsigned>(ctas), kPerThreads, smem, stream>>>(tq, tk, tv, to, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(err, err_len, "camera_xattn launch: %s", cudaGetErrorString(e));
        return NOMAS_ECUDA;
    }
    return NOMAS_OK;
}

}  // namespace nomas
