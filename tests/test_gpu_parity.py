"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element.

Bar: bit-exact INT8 codes, fp32 scales, gather indices and RoPE'd BF16; attention within
max |gpu - oracle| <= 1e-2 * max |oracle| and sum |gpu - oracle| / sum |oracle| <= 2e-3.
Inputs are the seeded synthetic tensors of the five workloads (nomas_synth); the largest
ones are compared on sampled query rows (rows are independent, so those rows are exact).
"""
import math

import numpy as np
import pytest
import torch

import nomas_synth as ns
import oracle
import segment_causal_attention_nomas_b300 as nb
from harness import (archive_chunks, assert_attn_close, bf16_to_f64, current_qkv, sample_rows, seg_offsets,
                     segment_kv, workload_outliers)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def tables():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from segment_causal_attention_nomas_b300 import build
    build.build()
    t = nb.nomas_rope_tables_create(256.0, (16, 56, 56), 512, 64, 64)
    yield t
    t.close()


def bits(t: torch.Tensor) -> np.ndarray:
    return ns.bf16_bits(t.detach().cpu())


# ------------------------------------------------------------------------------ builders
def gpu_history(w, tables, cap_extra=0):
    segs = w.history
    cap = sum(s.n_tokens for s in segs) + cap_extra
    cache = nb.KVCache(w.heads, max(cap, 4))
    out = workload_outliers(w)
    for i, s in enumerate(segs):
        k, v = segment_kv(w.config, i, s, w.heads, out)
        nb.nomas_kv_append_quant(cache, k.to(DEV), v.to(DEV), s, tables)
    return cache


def oracle_history(w):
    segs = w.history
    cap = max(sum(s.n_tokens for s in segs), 4)
    cache = oracle.Cache(w.heads, cap)
    out = workload_outliers(w)
    for i, s in enumerate(segs):
        k, v = segment_kv(w.config, i, s, w.heads, out)
        cache.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(s))
    return cache


def current_positions(w):
    return np.concatenate([oracle.segment_positions(s) for s in w.current], 0)


def run_gpu_attention(w, tables, history, step=0, lse=False):
    """rope3d(Q), rope3d(K) per current segment, then seg_attn; returns (out, lse) on host."""
    q, k, v = current_qkv(w, step, workload_outliers(w))
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    offs = seg_offsets(w.current)
    for i, s in enumerate(w.current):
        a, b = int(offs[i]), int(offs[i + 1])
        nb.nomas_rope3d(q[a:b], q[a:b], s, tables)
        nb.nomas_rope3d(k[a:b], k[a:b], s, tables)
    # outputs start as NaN, so an element the call leaves unwritten fails the finiteness check
    # (a recycled allocation could otherwise still hold a previous call's correct values)
    out = torch.full_like(q, float("nan"))
    lse_t = torch.full((w.heads, w.lq), float("nan"), dtype=torch.float32, device=DEV) if lse else None
    nb.nomas_seg_attn(q, k, v, offs, history, out, lse_t)
    nb.nomas_stream_check()
    return out, lse_t


def run_oracle_attention(w, history, rows, step=0):
    q, k, v = current_qkv(w, step, workload_outliers(w))
    pos = current_positions(w)
    qr = oracle.rope_bf16(ns.bf16_bits(q), pos)
    kr = oracle.rope_bf16(ns.bf16_bits(k), pos)
    return oracle.seg_attn(qr, kr, ns.bf16_bits(v), seg_offsets(w.current), history, rows=rows)


def check_attention(w, tables, n_rows=None, step=0, check_lse=True, gpu_hist=None, orc_hist=None):
    gpu_hist = gpu_history(w, tables) if gpu_hist is None and w.history else gpu_hist
    orc_hist = oracle_history(w) if orc_hist is None and w.history else orc_hist
    rows = None if n_rows is None else sample_rows(w.lq, n_rows, w.current)
    out, lse = run_gpu_attention(w, tables, gpu_hist, step, lse=check_lse)
    ref, ref_lse = run_oracle_attention(w, orc_hist, rows, step)
    got = bf16_to_f64(out)
    if rows is not None:
        got = got[rows]
    res = assert_attn_close(got, ref, w.name)
    if check_lse:
        gl = lse.cpu().numpy().astype(np.float64).T          # [Lq][H]
        if rows is not None:
            gl = gl[rows]
        assert np.max(np.abs(gl - ref_lse)) <= 1e-3 * max(1.0, np.max(np.abs(ref_lse))), "lse"
    return res


# ----------------------------------------------------------------------------- RoPE / append
def test_rope_tables_bitwise_equal_to_oracle(tables):
    for axis, d in enumerate((16, 56, 56)):
        c, s = nb.nomas_rope_tables_read(tables, axis)
        oc, os_ = oracle.rope_table(tables.max_pos[axis], d)
        assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
        assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("wl", [ns.config1, ns.config2, ns.config3])
def test_rope3d_bit_exact(tables, wl):
    w = wl()
    seg = w.current[0]
    x = ns.bf16_normal((seg.n_tokens, w.heads, 128), ns.seed_of(w.config, ns.T_Q, 0, 0))
    ref = oracle.rope_bf16(ns.bf16_bits(x), oracle.segment_positions(seg))
    xd = x.to(DEV)
    y = torch.empty_like(xd)
    nb.nomas_rope3d(xd, y, seg, tables)                      # out of place
    nb.nomas_rope3d(xd, xd, seg, tables)                     # in place
    nb.nomas_stream_check()
    assert np.array_equal(bits(y), ref)
    assert np.array_equal(bits(xd), ref)


def test_rope3d_strided_fused_qkv_layout(tables):
    # Q as a view of a fused [L][3][H][128] QKV tensor: token stride 3*H*128
    seg = ns.Segment(5, 3, 7, 9, 13)
    heads = 4
    qkv = ns.bf16_normal((seg.n_tokens, 3, heads, 128), 77)
    ref = oracle.rope_bf16(ns.bf16_bits(qkv[:, 0]), oracle.segment_positions(seg))
    d = qkv.to(DEV)
    nb.nomas_rope3d(d[:, 0], d[:, 0], seg, tables)
    nb.nomas_stream_check()
    assert np.array_equal(bits(d[:, 0]), ref)
    assert torch.equal(d[:, 1:].cpu(), qkv[:, 1:])           # K, V untouched


def test_positions_past_the_tables_rejected_without_int32_wrap(tables):
    # t0 + T past 2^31 must not wrap to a small number that passes the table bound: rope3d,
    # append and the projection refuse the segment before launching anything, and write nothing
    seg = ns.Segment(2 ** 31 - 10, 20, 1, 1, 0)                 # 20 tokens, t up to 2^31 + 9
    heads = 2
    x = torch.full((seg.n_tokens, heads, 128), 3.0, dtype=torch.bfloat16, device=DEV)
    y = torch.full_like(x, 5.0)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_rope3d(x, y, seg, tables)
    assert e.value.status == nb.NOMAS_EINVAL and "RoPE tables" in nb.nomas_last_error()
    cache = nb.KVCache(heads, 64)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_kv_append_quant(cache, x, x, seg, tables)
    assert e.value.status == nb.NOMAS_EINVAL and cache.length == 0
    xh = torch.ones((seg.n_tokens, 64), dtype=torch.bfloat16, device=DEV)
    codes = torch.ones((3 * heads * 128, 64), dtype=torch.int8, device=DEV)
    scale = torch.ones(3 * heads * 128, dtype=torch.float32, device=DEV)
    qkv = torch.full((seg.n_tokens, 3, heads, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    for append_to in (None, cache):
        with pytest.raises(nb.NomasError) as e:
            nb.nomas_qkv_project_rope(xh, codes, scale, seg, tables, qkv, append_to=append_to)
        assert e.value.status == nb.NOMAS_EINVAL
    nb.nomas_stream_check()
    assert torch.all(y == 5.0) and torch.all(qkv == 5.0)
    assert cache.length == 0 and torch.all(cache.k_scale == 0)


@pytest.mark.parametrize("wl", [ns.config1, ns.config2, ns.config3])
def test_append_bit_exact(tables, wl):
    w = wl()
    g = gpu_history(w, tables)
    o = oracle_history(w)
    n = o.length
    assert g.length == n
    assert np.array_equal(g.k[:, :n].cpu().numpy(), o.k[:, :n])
    assert np.array_equal(g.v[:, :n].cpu().numpy(), o.v[:, :n])
    assert np.array_equal(g.k_scale[:, :n].cpu().numpy().view(np.uint32), o.ks[:, :n].view(np.uint32))
    assert np.array_equal(g.v_scale[:, :n].cpu().numpy().view(np.uint32), o.vs[:, :n].view(np.uint32))


def test_append_edge_rows(tables):
    # zero rows, exact ties (absmax 127 -> scale 1), a lone absmax, strided K/V, appended twice
    heads = 3
    seg = ns.Segment(0, 1, 2, 3, 2)                         # 6 video + 2 text
    k = ns.bf16_normal((seg.n_tokens, heads, 128), 91)
    v = ns.bf16_normal((seg.n_tokens, heads, 128), 92)
    k[6] = 0.0                                               # a zero text row: scale 0, codes 0
    v[7, 1] = 0.0
    v[0, 0] = torch.tensor([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5] + [0.0] * 120)
    kv = torch.stack([k, v], 1).to(DEV)                      # [n][2][H][128]: token stride 2*H*128
    cache = nb.KVCache(heads, 2 * seg.n_tokens)
    nb.nomas_kv_append_quant(cache, kv[:, 0], kv[:, 1], seg, tables)
    seg2 = ns.Segment(1, 1, 2, 3, 2)
    nb.nomas_kv_append_quant(cache, kv[:, 0], kv[:, 1], seg2, tables)
    nb.nomas_stream_check()
    o = oracle.Cache(heads, 2 * seg.n_tokens)
    o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(seg))
    o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(seg2))
    assert np.array_equal(cache.k.cpu().numpy()[:, :16], o.k[:, :16])
    assert np.array_equal(cache.v.cpu().numpy()[:, :16], o.v[:, :16])
    assert np.array_equal(cache.k_scale.cpu().numpy()[:, :16], o.ks[:, :16])
    assert np.array_equal(cache.v_scale.cpu().numpy()[:, :16], o.vs[:, :16])
    assert cache.v[0, 0, :8].tolist() == [127, 2, 4, -2, -4, 0, 2, 0]
    assert np.all(cache.k_scale.cpu().numpy()[:, 6] == 0)


def _bf16_from_f32(a: np.ndarray) -> torch.Tensor:
    """float32 values -> BF16 tensor (values chosen to be exactly representable or rounded by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def test_append_quant_rounding_boundaries(tables):
    # Text-only segment (K is not rotated), so the rows reach the quantiser as constructed:
    # exact ties x / scale = k + 1/2 (scale 1), values a few ULPs either side of ties for an
    # awkward scale, rows whose scale is subnormal (no finite reciprocal), tiny and huge rows,
    # and zero rows.  Codes and scale bits must equal the oracle's.
    rng = np.random.default_rng(5)
    rows = []
    ties = np.array([127.0] + [k + 0.5 for k in range(-127, 127)], np.float32)
    for start in range(0, ties.size, 127):
        r = np.zeros(128, np.float32)
        chunk = ties[start:start + 127]
        r[0] = 127.0
        r[1:1 + chunk.size] = chunk
        rows.append(r)
    for a in (100.0, 3.0, 0.7, 1e-3, 1e20):
        s = np.float32(np.float32(a) / np.float32(127.0))
        k = rng.integers(-126, 126, 127).astype(np.float32) + 0.5
        near = (k * s).astype(np.float32)
        r = np.concatenate([[np.float32(a)], near]).astype(np.float32)
        rows.append(r)
        rows.append(np.nextafter(r, np.float32(np.inf)))
        rows.append(np.nextafter(r, np.float32(-np.inf)))
    for e in (-130, -133, -140):                      # subnormal absmax -> subnormal scale
        r = np.zeros(128, np.float32)
        r[:64] = np.ldexp(rng.integers(-127, 128, 64).astype(np.float32), e - 7)
        r[64] = np.ldexp(np.float32(127.0), e - 7)
        rows.append(r)
    rows.append(np.zeros(128, np.float32))
    rows.append(rng.standard_normal(128).astype(np.float32) * 5e37)
    x = np.stack(rows)                                 # [n, 128]
    n = x.shape[0]
    heads = 2
    kk = _bf16_from_f32(np.stack([x, -x[::-1]], 1))   # [n, 2, 128]
    vv = _bf16_from_f32(np.stack([x[::-1] * 0.5, x], 1))
    seg = ns.Segment(0, 0, 0, 0, n)
    cache = nb.KVCache(heads, n)
    nb.nomas_kv_append_quant(cache, kk.to(DEV), vv.to(DEV), seg, tables)
    nb.nomas_stream_check()
    o = oracle.Cache(heads, cache.capacity)
    o.append(ns.bf16_bits(kk), ns.bf16_bits(vv), oracle.segment_positions(seg))
    assert np.array_equal(cache.k.cpu().numpy()[:, :n], o.k[:, :n])
    assert np.array_equal(cache.v.cpu().numpy()[:, :n], o.v[:, :n])
    assert np.array_equal(cache.k_scale.cpu().numpy()[:, :n].view(np.uint32), o.ks[:, :n].view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy()[:, :n].view(np.uint32), o.vs[:, :n].view(np.uint32))


def test_append_quant_exhaustive_bf16(tables):
    # Every BF16 value x with |x| <= a, for every one of the 128 BF16 mantissas of the row
    # absmax a (exponent 0, plus a few other exponents): codes and scales must equal the
    # oracle's division-based rule.  The kernel forms the quotient without a division, so this
    # checks that form against the definition over every input the quantiser can receive (BF16
    # K and V), up to the power-of-two scaling that leaves the quotient unchanged.
    rows = []
    for e, mants in ((0, range(128)), (40, (0, 1, 63, 127)), (-60, (0, 64, 127))):
        for m in mants:
            a_bits = ((127 + e) << 7) | m
            a = np.array([a_bits << 16], np.uint32).view(np.float32)[0]
            mags = (np.arange(a_bits + 1, dtype=np.uint32) << 16).view(np.float32)
            xs = np.concatenate([mags, -mags[1:]])
            for start in range(0, xs.size, 127):
                r = np.zeros(128, np.float32)
                r[0] = a
                chunk = xs[start:start + 127]
                r[1:1 + chunk.size] = chunk
                rows.append(r)
    x = np.stack(rows)
    n = x.shape[0]
    heads = 2
    kk = _bf16_from_f32(np.stack([x, -x], 1))
    vv = _bf16_from_f32(np.stack([-x, x], 1))
    seg = ns.Segment(0, 0, 0, 0, n)
    cache = nb.KVCache(heads, n)
    nb.nomas_kv_append_quant(cache, kk.to(DEV), vv.to(DEV), seg, tables)
    nb.nomas_stream_check()
    o = oracle.Cache(heads, cache.capacity)
    o.append(ns.bf16_bits(kk), ns.bf16_bits(vv), oracle.segment_positions(seg))
    assert np.array_equal(cache.k.cpu().numpy()[:, :n], o.k[:, :n])
    assert np.array_equal(cache.v.cpu().numpy()[:, :n], o.v[:, :n])
    assert np.array_equal(cache.k_scale.cpu().numpy()[:, :n].view(np.uint32), o.ks[:, :n].view(np.uint32))
    assert np.array_equal(cache.v_scale.cpu().numpy()[:, :n].view(np.uint32), o.vs[:, :n].view(np.uint32))


def test_append_capacity_overflow_writes_nothing(tables):
    heads = 2
    seg = ns.Segment(0, 1, 2, 2, 0)
    k = ns.bf16_normal((4, heads, 128), 93).to(DEV)
    cache = nb.KVCache(heads, 4)
    nb.nomas_kv_append_quant(cache, k, k, seg, tables)
    before = cache.k.clone()
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_kv_append_quant(cache, k, k, seg, tables)
    assert e.value.status == nb.NOMAS_ECAPACITY
    nb.nomas_stream_check()
    assert cache.length == 4 and torch.equal(before, cache.k)


# ------------------------------------------------------------------------------- gather
def test_gather_bit_exact_config4(tables):
    w = ns.config4()
    chunks = archive_chunks(w)
    cap = sum(s.n_tokens for s in chunks)
    arch_g = nb.KVCache(w.heads, cap)
    arch_o = oracle.Cache(w.heads, cap)
    for i, s in enumerate(chunks):
        k, v = segment_kv(w.config, i, s, w.heads)
        nb.nomas_kv_append_quant(arch_g, k.to(DEV), v.to(DEV), s, tables)
        arch_o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(s))
    fto = [f * ns.TOKENS_PER_FRAME for f in range(w.archive_frames)]
    dst = nb.KVCache(w.heads, w.lh)
    idx = torch.full((w.lh,), -1, dtype=torch.int32, device=DEV)
    nb.nomas_kv_gather_context(arch_g, fto, ns.TOKENS_PER_FRAME, w.gather, dst, idx)
    nb.nomas_stream_check()
    ref, ref_idx = oracle.gather(arch_o, fto, ns.TOKENS_PER_FRAME, w.gather)
    assert len(w.gather) == 18 and w.gather[-6:] == list(range(234, 240))
    assert dst.length == ref.length == 18 * 880
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    n = ref.length
    assert np.array_equal(dst.k[:, :n].cpu().numpy(), ref.k[:, :n])
    assert np.array_equal(dst.v[:, :n].cpu().numpy(), ref.v[:, :n])
    assert np.array_equal(dst.k_scale[:, :n].cpu().numpy(), ref.ks[:, :n])
    assert np.array_equal(dst.v_scale[:, :n].cpu().numpy(), ref.vs[:, :n])
    # the archive itself matches too (append parity over 211,200 tokens)
    assert np.array_equal(arch_g.k[:, :cap].cpu().numpy(), arch_o.k[:, :cap])


def test_gather_ragged_frames_bit_exact(tables):
    # 37 tokens per frame (not a multiple of the copy piece), frames at irregular offsets, 3
    # heads; one selection of several frames, one of a single frame, one empty
    heads, tpf = 3, 37
    seg = ns.Segment(0, 0, 0, 0, 600)                       # 600 unrotated rows
    k, v = segment_kv(12, 0, seg, heads)
    arch_g = nb.KVCache(heads, 600)
    nb.nomas_kv_append_quant(arch_g, k.to(DEV), v.to(DEV), seg, tables)
    arch_o = oracle.Cache(heads, arch_g.capacity)
    arch_o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(seg))
    fto = [0, 37, 81, 118, 201, 250, 333, 401, 460, 563]     # frame starts (the last ends at 600)
    for frames in ([1, 2, 4, 7, 9], [3], []):
        n = len(frames) * tpf
        dst = nb.KVCache(heads, max(n, 4))
        idx = torch.full((max(n, 1),), -1, dtype=torch.int32, device=DEV)
        nb.nomas_kv_gather_context(arch_g, fto, tpf, frames, dst, idx)
        nb.nomas_stream_check()
        assert dst.length == n
        if n == 0:
            continue
        ref, ref_idx = oracle.gather(arch_o, fto, tpf, frames)
        assert np.array_equal(idx.cpu().numpy()[:n], ref_idx)
        assert np.array_equal(dst.k[:, :n].cpu().numpy(), ref.k[:, :n])
        assert np.array_equal(dst.v[:, :n].cpu().numpy(), ref.v[:, :n])
        assert np.array_equal(dst.k_scale[:, :n].cpu().numpy(), ref.ks[:, :n])
        assert np.array_equal(dst.v_scale[:, :n].cpu().numpy(), ref.vs[:, :n])


def test_gather_host_archive_config4(tables):
    # The config-4 archive copied to pinned host memory, gathered on a side stream while the
    # default stream runs attention: codes, scales and index map equal the oracle's.
    w = ns.config4()
    chunks = archive_chunks(w)
    cap = sum(s.n_tokens for s in chunks)
    arch_g = nb.KVCache(w.heads, cap)
    arch_o = oracle.Cache(w.heads, cap)
    for i, s in enumerate(chunks):
        k, v = segment_kv(w.config, i, s, w.heads)
        nb.nomas_kv_append_quant(arch_g, k.to(DEV), v.to(DEV), s, tables)
        arch_o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(s))
    torch.cuda.synchronize()
    arch_h = nb.HostKVCache.from_device(arch_g)
    fto = [f * ns.TOKENS_PER_FRAME for f in range(w.archive_frames)]
    dst = nb.KVCache(w.heads, w.lh)
    idx = torch.full((w.lh,), -1, dtype=torch.int32, device=DEV)
    # unrelated attention work on the default stream while the copy engines gather
    q = ns.bf16_normal((2048, w.heads, 128), 71).to(DEV)
    out = torch.empty_like(q)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        nb.nomas_kv_gather_context_host(arch_h, fto, ns.TOKENS_PER_FRAME, w.gather, dst, idx, stream=side)
    nb.nomas_seg_attn(q, q, q, [0, 2048], None, out)
    side.synchronize()
    nb.nomas_stream_check()
    ref, ref_idx = oracle.gather(arch_o, fto, ns.TOKENS_PER_FRAME, w.gather)
    n = ref.length
    assert dst.length == n == 18 * 880
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(dst.k[:, :n].cpu().numpy(), ref.k[:, :n])
    assert np.array_equal(dst.v[:, :n].cpu().numpy(), ref.v[:, :n])
    assert np.array_equal(dst.k_scale[:, :n].cpu().numpy(), ref.ks[:, :n])
    assert np.array_equal(dst.v_scale[:, :n].cpu().numpy(), ref.vs[:, :n])


def test_gather_host_archive_ragged_and_checks(tables):
    # Runs of consecutive frames (one copy each) and isolated frames, 37 tokens per frame, 3
    # heads; then a device archive is refused (not pinned host memory) without touching dst.
    heads, tpf = 3, 37
    seg = ns.Segment(0, 0, 0, 0, 600)
    k, v = segment_kv(12, 0, seg, heads)
    arch_g = nb.KVCache(heads, 600)
    nb.nomas_kv_append_quant(arch_g, k.to(DEV), v.to(DEV), seg, tables)
    torch.cuda.synchronize()
    arch_h = nb.HostKVCache.from_device(arch_g)
    arch_o = oracle.Cache(heads, arch_g.capacity)
    arch_o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(seg))
    fto = [0, 37, 74, 118, 201, 238, 275, 401, 460, 563]     # frames 0-2 and 4-6 are consecutive runs
    for frames in ([0, 1, 2, 4, 5, 6, 9], [3], [7, 8]):
        n = len(frames) * tpf
        dst = nb.KVCache(heads, n)
        idx = torch.full((n,), -1, dtype=torch.int32, device=DEV)
        nb.nomas_kv_gather_context_host(arch_h, fto, tpf, frames, dst, idx)
        nb.nomas_stream_check()
        ref, ref_idx = oracle.gather(arch_o, fto, tpf, frames)
        assert dst.length == n
        assert np.array_equal(idx.cpu().numpy()[:n], ref_idx)
        assert np.array_equal(dst.k[:, :n].cpu().numpy(), ref.k[:, :n])
        assert np.array_equal(dst.v[:, :n].cpu().numpy(), ref.v[:, :n])
        assert np.array_equal(dst.k_scale[:, :n].cpu().numpy(), ref.ks[:, :n])
        assert np.array_equal(dst.v_scale[:, :n].cpu().numpy(), ref.vs[:, :n])
    dst = nb.KVCache(heads, tpf)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_kv_gather_context_host(arch_g, fto, tpf, [2], dst)
    assert e.value.status == nb.NOMAS_EINVAL and "pinned" in nb.nomas_last_error()
    assert dst.length == 0 and int(dst.k.abs().sum()) == 0


# ----------------------------------------------------------------------------- attention
def test_attention_config1_full(tables):
    check_attention(ns.config1(), tables)


def test_attention_config1_two_segments_causal(tables):
    check_attention(ns.config1_two_segments(), tables)


def test_attention_config1_causality_on_gpu(tables):
    # appending a later segment to the call leaves the earlier segment's outputs unchanged
    w2 = ns.config1_two_segments()
    out2, _ = run_gpu_attention(w2, tables, None)
    w1 = ns.Workload("seg0 only", 1, 2, [], [w2.current[0]])
    q, k, v = current_qkv(w2)
    n0 = w2.current[0].n_tokens
    qd, kd, vd = q[:n0].to(DEV), k[:n0].to(DEV), v[:n0].to(DEV)
    s0 = w2.current[0]
    nb.nomas_rope3d(qd, qd, s0, tables)
    nb.nomas_rope3d(kd, kd, s0, tables)
    out1 = torch.empty_like(qd)
    nb.nomas_seg_attn(qd, kd, vd, [0, n0], None, out1)
    nb.nomas_stream_check()
    assert torch.equal(out1, out2[:n0])


def test_attention_config2_steps(tables):
    w = ns.config2()
    gh, oh = gpu_history(w, tables), oracle_history(w)
    for step in (0, 7):
        check_attention(w, tables, n_rows=96, step=step, gpu_hist=gh, orc_hist=oh)


def test_attention_config3_sampled(tables):
    check_attention(ns.config3(), tables, n_rows=40)


def test_attention_config4_gather_then_attend(tables):
    w = ns.config4()
    chunks = archive_chunks(w)
    cap = sum(s.n_tokens for s in chunks)
    arch_g = nb.KVCache(w.heads, cap)
    arch_o = oracle.Cache(w.heads, cap)
    for i, s in enumerate(chunks):
        k, v = segment_kv(w.config, i, s, w.heads)
        nb.nomas_kv_append_quant(arch_g, k.to(DEV), v.to(DEV), s, tables)
        arch_o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(s))
    fto = [f * ns.TOKENS_PER_FRAME for f in range(w.archive_frames)]
    hist_g = nb.KVCache(w.heads, w.lh)
    nb.nomas_kv_gather_context(arch_g, fto, ns.TOKENS_PER_FRAME, w.gather, hist_g)
    hist_o, _ = oracle.gather(arch_o, fto, ns.TOKENS_PER_FRAME, w.gather)
    check_attention(w, tables, n_rows=64, gpu_hist=hist_g, orc_hist=hist_o)


@pytest.mark.parametrize("lh,T", [(0, 4), (8_000, 4), (32_000, 24), (100_000, 4), (300_000, 4)])
def test_attention_sweep_points(tables, lh, T):
    check_attention(ns.config5(lh, T), tables, n_rows=24)


@pytest.mark.parametrize("n_seg,T,n_rows", [(5, 2, 60), (5, 72, 20), (12, 3, 48)])
def test_attention_packed_segments(tables, n_seg, T, n_rows):
    # Packed multi-segment forward: n_seg segments in one call with the segment-causal mask
    # (5 x 72 frames = 318,080 tokens), sampled rows in every segment against the oracle.
    check_attention(ns.packed(n_seg, T), tables, n_rows=n_rows)


@pytest.mark.parametrize("segs,hist", [
    ([ns.Segment(0, 1, 1, 1, 0)], []),                                   # Lq = 1, no history: O = v
    ([ns.Segment(3, 1, 5, 26, 0)], [ns.Segment(0, 0, 0, 0, 200)]),       # Lq 130, Lh 200: ragged tails
    ([ns.Segment(3, 1, 3, 3, 4), ns.Segment(4, 2, 5, 7, 1), ns.Segment(6, 1, 11, 13, 100)],
     [ns.Segment(0, 1, 3, 43, 0)]),                                      # 3 segments, Lh 129
    ([ns.Segment(1, 3, 11, 17, 256)], [ns.Segment(0, 0, 0, 0, 1)]),      # one history token
    ([ns.Segment(9, 4, 22, 40, 256)], [ns.Segment(0, 3, 22, 40, 0)]),    # whole frames
])
def test_attention_edge_shapes(tables, segs, hist):
    w = ns.Workload("edge", 9, 3, hist, segs)
    check_attention(w, tables)


def test_attention_history_with_zero_rows(tables):
    # rows with scale 0 (all-zero K or V) in the history
    w = ns.Workload("zero rows", 9, 2, [ns.Segment(0, 1, 10, 30, 0)], [ns.Segment(1, 1, 10, 10, 5)])
    k, v = segment_kv(9, 0, w.history[0], 2)
    k[::7] = 0.0
    v[::5] = 0.0
    g = nb.KVCache(2, 300)
    nb.nomas_kv_append_quant(g, k.to(DEV), v.to(DEV), w.history[0], tables)
    o = oracle.Cache(2, 300)
    o.append(ns.bf16_bits(k), ns.bf16_bits(v), oracle.segment_positions(w.history[0]))
    check_attention(w, tables, gpu_hist=g, orc_hist=o)


def test_attention_is_deterministic(tables):
    w = ns.config5(8_000, 4)
    gh = gpu_history(w, tables)
    a, _ = run_gpu_attention(w, tables, gh)
    b, _ = run_gpu_attention(w, tables, gh)
    assert torch.equal(a, b)


# ------------------------------------------------------------------- failure detection
def test_bounded_wait_reports_timeout_and_context_survives(tables):
    w = ns.config1()
    gh = gpu_history(w, tables)
    q, k, v = (t.to(DEV) for t in current_qkv(w))
    out = torch.full_like(q, 7.0)
    nb.nomas_debug_inject(1)                    # the next launch withholds its Q load
    nb.nomas_seg_attn(q, k, v, [0, w.lq], gh, out)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_stream_check()
    assert e.value.status == nb.NOMAS_ETIMEOUT
    assert torch.all(out == 7.0)                # nothing written
    nb.nomas_stream_check()                     # status word was cleared
    check_attention(w, tables)                  # and the context still works


def test_invalid_calls_raise_before_launch(tables):
    q = torch.zeros((10, 2, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros_like(q)
    h = nb.KVCache(3, 8)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_seg_attn(q, q, q, [0, 10], h, out)           # heads mismatch
    assert e.value.status == nb.NOMAS_EINVAL
    with pytest.raises(nb.NomasError):
        nb.nomas_rope3d(q, q, ns.Segment(600, 1, 1, 10, 0), tables)   # t beyond the tables
    nb.nomas_stream_check()


# ---------------------------------------------------- both variants of the attention kernel
# The library picks the CTA-pair variant for long unsplit calls and the single-CTA one otherwise;
# the test hook forces either, so both run the same cases against the oracle: odd Q-block counts
# (a pair whose second CTA has no live rows), ragged tails, several segments, split key ranges.
@pytest.fixture(params=[1, 2], ids=["single_cta", "cta_pair"])
def variant(request):
    nb.nomas_debug_attn_variant(request.param)
    yield request.param
    nb.nomas_debug_attn_variant(0)


VARIANT_CASES = {
    "config1": lambda: (ns.config1(), None),
    "config1_two_segments": lambda: (ns.config1_two_segments(), None),
    "ragged": lambda: (ns.Workload("edge", 9, 3, [ns.Segment(0, 0, 0, 0, 200)], [ns.Segment(3, 1, 5, 26, 0)]), None),
    "three_segments": lambda: (ns.Workload("edge", 9, 3, [ns.Segment(0, 1, 3, 43, 0)],
                                           [ns.Segment(3, 1, 3, 3, 4), ns.Segment(4, 2, 5, 7, 1),
                                            ns.Segment(6, 1, 11, 13, 100)]), None),
    "odd_q_blocks": lambda: (ns.Workload("edge", 9, 3, [ns.Segment(0, 3, 22, 40, 0)],
                                         [ns.Segment(9, 4, 22, 40, 256)]), None),       # 15 Q blocks
    "config2": lambda: (ns.config2(), 96),
    "split_key_range": lambda: (ns.config5(100_000, 4), 24),                           # 3 splits
    "packed": lambda: (ns.packed(5, 2), 60),
}


@pytest.mark.parametrize("case", sorted(VARIANT_CASES))
def test_attention_variants(tables, variant, case):
    w, n_rows = VARIANT_CASES[case]()
    check_attention(w, tables, n_rows=n_rows)


def test_attention_variants_agree_bitwise_where_the_work_is_split_alike(tables):
    # the two variants issue the same MMAs per row block in the same order: identical outputs
    w = ns.config5(8_000, 4)
    gh = gpu_history(w, tables)
    outs = []
    for v in (1, 2):
        nb.nomas_debug_attn_variant(v)
        try:
            outs.append(run_gpu_attention(w, tables, gh)[0])
        finally:
            nb.nomas_debug_attn_variant(0)
    assert torch.equal(outs[0], outs[1])


def test_pair_variant_bounded_wait_reports_timeout(tables):
    w = ns.config1()
    gh = gpu_history(w, tables)
    q, k, v = (t.to(DEV) for t in current_qkv(w))
    out = torch.full_like(q, 7.0)
    nb.nomas_debug_attn_variant(2)
    try:
        nb.nomas_debug_inject(1)                # the next launch withholds its Q loads
        nb.nomas_seg_attn(q, k, v, [0, w.lq], gh, out)
        with pytest.raises(nb.NomasError) as e:
            nb.nomas_stream_check()
        assert e.value.status == nb.NOMAS_ETIMEOUT
        assert torch.all(out == 7.0)            # nothing written
        nb.nomas_stream_check()
        check_attention(w, tables)              # the context still works, in the pair variant too
    finally:
        nb.nomas_debug_attn_variant(0)
