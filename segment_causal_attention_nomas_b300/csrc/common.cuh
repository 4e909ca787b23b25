// common.cuh -- device-side building blocks shared by the libnomas kernels (sm_103a).
//
// Inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), and the tcgen05 tensor-core
// path (TMEM allocation, MMA issue/commit, TMEM loads/stores), plus the bounded waits every
// kernel uses: a wait that does not complete within about a second records NOMAS_ETIMEOUT
// and the code point in the library's device status word, raises the CTA's abort flag and
// returns false, so the kernel can drain its in-flight copies, free TMEM and exit.
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nomas {

constexpr int kHeadDim = 128;
constexpr int kStatusTimeout = 5;          // == NOMAS_ETIMEOUT
constexpr int kStatusRange = 6;            // == NOMAS_ERANGE
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s of wall time

// ----------------------------------------------------------------- generic helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Records a device-side failure: status[0] = code (first writer wins), status[1] = where.
__device__ __forceinline__ void record_status(int *status, int code, int where) {
    if (atomicCAS(status, 0, code) == 0) status[1] = where;
}

// n / d for 0 <= n < 2^31 as (umulhi(n, m) + n) >> l (Granlund & Montgomery, "Division by
// invariant integers using multiplication", 1994, with the 32-bit sum safe for n < 2^31).
struct FastDiv {
    uint32_t m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.l = l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f) { return (__umulhi(n, f.m) + n) >> f.l; }

// Token layout of one segment: T*gh*gw video tokens in (t, h, w) row-major order from frame t0,
// then text tokens (no position).
struct SegPos {
    int32_t t0, n_video, n_tokens, heads, hw, gw;
    FastDiv div_hw, div_gw, div_heads;
};

inline SegPos make_seg_pos(int32_t t0, int32_t n_video, int32_t n_tokens, int32_t heads, int32_t gh, int32_t gw) {
    SegPos p;
    p.t0 = t0;
    p.n_video = n_video;
    p.n_tokens = n_tokens;
    p.heads = heads;
    // a segment without video tokens may carry any grid (its positions are never used): the
    // product is formed in 64 bits and only kept when it is a real grid of at most n_video tokens
    const int64_t hw = static_cast<int64_t>(gh) * gw;
    p.hw = n_video > 0 && hw > 0 ? static_cast<int32_t>(hw) : 1;
    p.gw = gw > 0 ? gw : 1;
    p.div_hw = make_fastdiv(static_cast<uint32_t>(p.hw));
    p.div_gw = make_fastdiv(static_cast<uint32_t>(p.gw));
    p.div_heads = make_fastdiv(static_cast<uint32_t>(heads > 0 ? heads : 1));
    return p;
}

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

// ------------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// One test of the phase with parity `parity`, suspending the thread in hardware until the
// phase completes or about kSuspendHintNs have passed (a waiting warp then issues nothing).
constexpr uint32_t kSuspendHintNs = 1000000u;
__device__ __forceinline__ bool mbar_test_sleep(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Slow path of mbar_wait: keeps testing (each test sleeps until completion or the hint)
// until the phase completes, another thread of the CTA raised *abort, or kWaitLimitNs of wall
// time passed (then it records NOMAS_ETIMEOUT at `where` and raises *abort).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t addr, uint32_t parity, int *status, volatile int *abort,
                                                   int where) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_test_sleep(addr, parity)) return true;
        if (*abort) return false;
        if (spin >= 4 && globaltimer_ns() - t0 > kWaitLimitNs) {
            record_status(status, kStatusTimeout, where);
            *abort = 1;
            return false;
        }
    }
}

// Waits until the phase with parity `parity` of `bar` has completed.  Bounded: gives up
// (returns false) after about kWaitLimitNs of wall time, or as soon as another thread of the
// CTA raised *abort.  `where` identifies the wait in the status word.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *abort,
                                          int where) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_test_sleep(addr, parity)) return true;
    return mbar_wait_slow(addr, parity, status, abort, where);
}

// mbar_wait with the slow path inline too, for callers that keep many registers live across
// the wait (a call would have to save them).
__device__ __forceinline__ bool mbar_wait_inline(uint64_t *bar, uint32_t parity, int *status, volatile int *abort,
                                                 int where) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_test_sleep(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_test_sleep(addr, parity)) return true;
        if (*abort) return false;
        if (spin >= 4 && globaltimer_ns() - t0 > kWaitLimitNs) {
            record_status(status, kStatusTimeout, where);
            *abort = 1;
            return false;
        }
    }
}

// -------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Shared -> global tile store (bulk-group completion); rows or columns past the tensor's
// extent are not written.  Coordinates must be non-negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int32_t x, int32_t y,
                                             int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Returns once every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tensor-core operand fetch).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------- CTA pairs (cta_group::2, clusters)
// A cluster of two CTAs on the two SMs of a pair: rank 0 (the leader) issues the pair's MMAs,
// which read the A rows and half of B from each CTA's shared memory at the same offsets and write
// each CTA's accumulator rows into its own tensor memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the object at this CTA's shared address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
// arrive.expect_tx on an mbarrier given by its shared::cluster address (possibly the peer's).  The
// release is at CTA scope: what the barrier guards is either tracked by its transaction count
// (the copies) or complete and fenced before the arrive (tensor-memory reads), and a
// cluster-scope release costs about a thousand cycles per arrive (measured on B300, where it made
// the pair GEMM's producer the bottleneck: 435 against 308 us).
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cluster.b64 _, [%0], %1;" ::"r"(bar_cluster),
                 "r"(bytes)
                 : "memory");
}
// arrive on an mbarrier given by its shared::cluster address (possibly the peer's); release at CTA
// scope, as above.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// Every thread of both CTAs of the cluster meets here (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// TMA 2D load into this CTA's shared memory whose completion is signalled on the mbarrier at the
// shared::cluster address `bar_cluster` (the pair leader's barrier).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
// The same for a 3D tensor map.
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// Tensor memory of a CTA pair: allocated, relinquished and freed collectively by one warp of each
// CTA (the same column address in both).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The pair's D[tmem] (+)= A[smem] * B[smem]^T (issued by the leader only).
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The pair's D[tmem] (+)= A[tmem] * B[smem]^T (issued by the leader only; A is each CTA's own rows
// in its own tensor memory).
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on the mbarrier at this shared offset in every CTA of `cta_mask` when the pair
// MMAs the leader issued so far have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (tcgen05 format):
// start address, leading/stride byte offsets (16-byte units), descriptor version 1
// (bits 46-47), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 (dense): D format bits 4-5 (1 = f32), A format
// bits 7-9 and B format bits 10-12 (0 = f16, 1 = bf16), A major bit 15, B major bit 16
// (0 = K-major, 1 = MN-major), N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(bool ab_bf16, bool b_mn_major, int m, int n) {
    return (1u << 4) | ((ab_bf16 ? 1u : 0u) << 7) | ((ab_bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// TMEM -> registers: 32 lanes x 32 consecutive 32-bit columns (thread i gets lane base+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// TMEM -> registers: 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}
// Waits for this thread's TMEM loads and ties the destination registers to the wait, so the
// compiler cannot move a use of them above it (the load's asm "produces" them early).
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Ties registers filled by a TMEM load to a preceding tmem_wait_ld (emits nothing): asm
// volatile statements keep their order, so no use of r can move above the wait.
__device__ __forceinline__ void tmem_tie(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// registers -> TMEM: 32 lanes x 16 consecutive columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// registers -> TMEM: 32 lanes x 32 consecutive columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ number formats
// 2^x on the SFU (approximate, flushes denormals).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Packs (lo, hi) into an f16x2 word, round-to-nearest, saturating to the finite range.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// Packs (lo, hi) into a bf16x2 word, round-to-nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// Packs (lo, hi) into a bf16x2 word, round-to-nearest-even, saturating to the finite range.
__device__ __forceinline__ uint32_t pack_bf16x2_sat(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ----------------------------------------------------------- power-of-two operand scaling
// The tensor-core operands are FP16 (normal range 2^-14 .. 65,504); the BF16 inputs span
// 2^-133 .. 2^128.  Each operand block (a query row, a head's current K or V, a head's history K
// or V) is therefore multiplied by an exact power of two 2^e chosen from its largest magnitude,
// so that the block's maximum lands in [2^14, 2^15): nothing overflows, and every value within
// 2^28 of the maximum stays a normal FP16 number.  The factor is undone exactly in fp32 (in the
// softmax multiplier for Q and K, in the epilogue for V).  Host and device derive e from the same
// maximum with the functions below, so both sides agree on it bit for bit.

// floor(log2 x) for a finite x > 0, normal or subnormal (from the fp32 bit pattern).
__host__ __device__ __forceinline__ int ilog2_pos(float x) {
#ifdef __CUDA_ARCH__
    const uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu;
    const int lz = __clz(static_cast<int>(b));
#else
    uint32_t b;
    memcpy(&b, &x, 4);
    b &= 0x7FFFFFFFu;
    const int lz = b ? __builtin_clz(b) : 32;
#endif
    const int ef = static_cast<int>(b >> 23);
    return ef != 0 ? ef - 127 : -149 + (31 - lz);
}

// Exponent e for a block of BF16 (or fp32) values of largest magnitude amax >= 0:
// amax * 2^e in [2^14, 2^15); 0 for an all-zero block.  e lies in [-113, 126], so 2^e and 2^-e
// are both normal floats.  (The cap at 126 binds only below amax = 2^-112, where every BF16 value,
// a multiple of 2^-133, times 2^126 is still a normal FP16 number.)
__host__ __device__ __forceinline__ int operand_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    const int e = 14 - ilog2_pos(amax);
    return e > 126 ? 126 : e;
}

// Exponent e for a head's history rows, from the largest row scale smax >= 0: with smax in
// [2^k, 2^(k+1)) and e = 7 - k, every dequantised value |code| * scale * 2^e is below
// 128 * 2^8 = 2^15, and a row at the largest scale with code 127 reaches at least 127 * 2^7.
__host__ __device__ __forceinline__ int history_exp(float smax) {
    if (!(smax > 0.0f)) return 0;
    const int e = 7 - ilog2_pos(smax);
    return e > 126 ? 126 : (e < -126 ? -126 : e);
}

// 2^e as fp32 for e in [-126, 127] (exact).
__host__ __device__ __forceinline__ float pow2i(int e) {
    const uint32_t b = static_cast<uint32_t>(e + 127) << 23;
#ifdef __CUDA_ARCH__
    return __uint_as_float(b);
#else
    float f;
    memcpy(&f, &b, 4);
    return f;
#endif
}

// x * 2^a for any integer a (two exact steps; a result below the fp32 range flushes towards 0).
__host__ __device__ __forceinline__ float mul_pow2(float x, int a) {
    const int a1 = a > 127 ? 127 : (a < -126 ? -126 : a);
    int a2 = a - a1;
    a2 = a2 > 127 ? 127 : (a2 < -126 ? -126 : a2);
    return x * pow2i(a1) * pow2i(a2);
}

// Four signed INT8 codes (one 32-bit word) -> exact values as fp32.
// Each byte b is biased to u = b ^ 0x80 (= b + 128), placed in the mantissa of 2^23
// (0x4B000000 | u = 2^23 + u exactly), and 2^23 + 128 is subtracted.
__device__ __forceinline__ void s8x4_to_f32(uint32_t w, float (&f)[4]) {
    const uint32_t u = w ^ 0x80808080u;
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - 8388736.0f;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - 8388736.0f;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - 8388736.0f;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - 8388736.0f;
}
// Largest magnitude of the 8 BF16 values of a 16-byte word, as the BF16 bit pattern (sign
// cleared; for finite values the integer order of these patterns is the order of magnitudes).
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 w) {
    const uint32_t m = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

// Eight BF16 -> eight FP16 after an exact multiplication by the power of two f (round to
// nearest; the operand exponents keep every product below 2^15, so nothing saturates).
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 w, float f) {
    uint4 r;
    r.x = pack_f16x2_sat(__uint_as_float(w.x << 16) * f, __uint_as_float(w.x & 0xFFFF0000u) * f);
    r.y = pack_f16x2_sat(__uint_as_float(w.y << 16) * f, __uint_as_float(w.y & 0xFFFF0000u) * f);
    r.z = pack_f16x2_sat(__uint_as_float(w.z << 16) * f, __uint_as_float(w.z & 0xFFFF0000u) * f);
    r.w = pack_f16x2_sat(__uint_as_float(w.w << 16) * f, __uint_as_float(w.w & 0xFFFF0000u) * f);
    return r;
}

// Eight BF16 -> eight FP16 (round-to-nearest, saturating).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w) {
    uint4 r;
    r.x = pack_f16x2_sat(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
    r.y = pack_f16x2_sat(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    r.z = pack_f16x2_sat(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
    r.w = pack_f16x2_sat(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
    return r;
}

}  // namespace nomas
