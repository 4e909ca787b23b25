"""GPU parity of the W8A16 QKV projection with fused 3D RoPE (nomas_qkv_project_rope).

Bar: Q, K, V within the attention tolerance of the float64 oracle (max |gpu - oracle| <= 1e-2 *
max |oracle|, mean relative error <= 2e-3), and element by element within the bound the
arithmetic sets (see projection_rounding_ok): the BF16 roundings plus the fp32 accumulation,
with at least 99 % of the elements exactly the oracle's (its projection rounded once to BF16,
Q and K then rotated by its BF16 RoPE); the fused RoPE bit-exact with nomas_rope3d applied to
the same projection computed without rotation (a text-only segment).
"""
import numpy as np
import pytest
import torch

import nomas_synth as ns
import oracle
import segment_causal_attention_nomas_b300 as nb
from harness import assert_attn_close, bf16_to_f64

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


def weights(heads, hidden, seed):
    """Synthetic INT8 weights: codes uniform in [-127, 127], one fp32 scale per output channel
    sized so that outputs are of order one."""
    g = np.random.default_rng(seed)
    n = 3 * heads * 128
    codes = g.integers(-127, 128, (n, hidden)).astype(np.int8)
    scale = (g.uniform(0.5, 1.5, n) / (127.0 * np.sqrt(hidden) / 3.0)).astype(np.float32)
    return codes, scale


def run(x, codes, scale, seg, tables, heads):
    out = torch.empty((x.shape[0], 3, heads, 128), dtype=torch.bfloat16, device=DEV)
    nb.nomas_qkv_project_rope(x.to(DEV), torch.from_numpy(codes).to(DEV), torch.from_numpy(scale).to(DEV), seg,
                              tables, out)
    nb.nomas_stream_check()
    return out


def reference(x, codes, scale, seg, heads):
    proj = oracle.qkv_project(ns.bf16_bits(x), codes, scale)          # [L, 3*H*128] float64
    L = proj.shape[0]
    pos = oracle.segment_positions(seg)
    q = oracle.rope_f64(proj[:, :heads * 128].reshape(L, heads, 128), pos)
    k = oracle.rope_f64(proj[:, heads * 128:2 * heads * 128].reshape(L, heads, 128), pos)
    v = proj[:, 2 * heads * 128:].reshape(L, heads, 128)
    return q, k, v


def rne_bf16(a):
    """float64 -> the nearest BF16 value (ties to even), as float64: one rounding of the exact
    value to 8 significant bits (the operands here stay far inside BF16's normal range)."""
    m, e = np.frexp(a)
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def bf16_bits_of(a):
    """float64 values exactly representable in BF16 -> uint16 bit patterns."""
    b = a.astype(np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)
    return (b >> 16).astype(np.uint16)


def projection_rounding_ok(out, x, codes, scale, seg, heads, what):
    """Element-wise check of the projection against the oracle's exact float64 values y.

    The kernel forms acc = sum_k x[k] * code[n, k] in fp32 on the tensor cores (the products are
    exact), multiplies by scale[n] in fp32 and rounds to BF16; Q and K are then rotated in fp32
    from the BF16 values (tables rounded once to fp32) and rounded to BF16 again.  Per element:
      V:     |got - y| <= 2^-8 |y| + 1.01 E
      Q, K:  |got - ref| <= 2^-8 |ref| + 1.02 (2^-8 + 2^-20) (|y0| + |y1|) + 1.03 (E0 + E1)
    where ref is the exact rotation of y, (y0, y1) the element's RoPE pair (channels 2i, 2i + 1,
    the same channel for text tokens), 2^-8 the unit roundoff of BF16's 8 significant bits and
    E = 2^-16 * scale[n] * sum_k |x[k] code[n, k]| + 2^-23 |y|: the fp32 multiply's rounding
    and the accumulation's, whose order the tensor core does not document; one fp32 rounding
    per addition, of random sign over hidden <= 2048 terms, stays below sqrt(hidden) * 2^-24 of
    the sum of magnitudes, 4x inside 2^-16 (a sequential fp32 sum measures 2^-23.6).  And at
    least 99 % of the elements equal the oracle's own BF16 path exactly: V = y rounded to BF16,
    Q and K = oracle.rope_bf16 of their BF16-rounded projection (a projection element that the
    fp32 accumulation moves across a rounding boundary differs by one BF16 step)."""
    L = seg.n_tokens
    y = oracle.qkv_project(ns.bf16_bits(x), codes, scale)                 # [L, 3*H*128]
    xa = np.abs(bf16_to_f64(x))
    mag = xa @ np.abs(codes.astype(np.float64)).T * scale.astype(np.float64)[None, :]
    E = (2.0 ** -16 * mag + 2.0 ** -23 * np.abs(y)).reshape(L, 3, heads, 128)
    y = y.reshape(L, 3, heads, 128)
    got_bits = out.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_to_f64(got_bits)
    pos = oracle.segment_positions(seg)
    video = (pos[:, 0] >= 0)[:, None, None]
    # V
    bound = 2.0 ** -8 * np.abs(y[:, 2]) + 1.01 * E[:, 2]
    excess = np.abs(got[:, 2] - y[:, 2]) - bound
    assert np.all(excess <= 0), f"{what} v: worst excess {excess.max():.3e}"
    same = [np.mean(got_bits[:, 2] == bf16_bits_of(rne_bf16(y[:, 2])))]
    # Q, K
    partner = np.arange(128) ^ 1
    for i, name in ((0, "q"), (1, "k")):
        yi, ei = y[:, i], E[:, i]                                          # [L, H, 128]
        ref = oracle.rope_f64(yi, pos)
        pair = np.abs(yi) + np.where(video, np.abs(yi[..., partner]), 0.0)
        e_pair = ei + np.where(video, ei[..., partner], 0.0)
        bound = 2.0 ** -8 * np.abs(ref) + 1.02 * (2.0 ** -8 + 2.0 ** -20) * pair + 1.03 * e_pair
        excess = np.abs(got[:, i] - ref) - bound
        assert np.all(excess <= 0), f"{what} {name}: worst excess {excess.max():.3e}"
        want = oracle.rope_bf16(bf16_bits_of(rne_bf16(y[:, i])), pos)
        same.append(np.mean(got_bits[:, i] == want))
    assert min(same) >= 0.99, f"{what}: fractions equal to the oracle's BF16 path (v, q, k) {same}"
    return same


def test_qkv_projection_matches_oracle(tables):
    heads, hidden = 16, 2048
    seg = ns.Segment(3, 2, 22, 40, 256)                      # 1,760 video + 256 text tokens
    x = ns.bf16_normal((seg.n_tokens, hidden), 41)
    codes, scale = weights(heads, hidden, 42)
    raw = run(x, codes, scale, seg, tables, heads)
    out = bf16_to_f64(raw.cpu())
    q, k, v = reference(x, codes, scale, seg, heads)
    for name, got, ref in (("q", out[:, 0], q), ("k", out[:, 1], k), ("v", out[:, 2], v)):
        assert_attn_close(got, ref, f"qkv projection {name}")
    projection_rounding_ok(raw, x, codes, scale, seg, heads, "qkv projection")


def test_qkv_fused_rope_is_rope3d_of_projection(tables):
    heads, hidden = 4, 512
    seg = ns.Segment(7, 3, 5, 9, 20)                         # 135 video + 20 text tokens
    x = ns.bf16_normal((seg.n_tokens, hidden), 43)
    codes, scale = weights(heads, hidden, 44)
    fused = run(x, codes, scale, seg, tables, heads)
    plain = run(x, codes, scale, ns.Segment(0, 0, 0, 0, seg.n_tokens), tables, heads)  # no rotation
    assert torch.equal(fused[:, 2], plain[:, 2])              # V is never rotated
    for i in (0, 1):
        r = plain[:, i].contiguous()
        nb.nomas_rope3d(r, r, seg, tables)
        nb.nomas_stream_check()
        assert torch.equal(fused[:, i], r)


@pytest.mark.parametrize("heads,hidden,seg", [
    (2, 192, ns.Segment(0, 1, 10, 12, 10)),                  # 130 tokens: a ragged 128-row tile
    (6, 64, ns.Segment(2, 1, 1, 1, 0)),                      # one token, one stage of 64
    (2, 320, ns.Segment(1, 2, 11, 20, 300)),                 # 740 tokens, 5 stages
])
def test_qkv_projection_small_shapes(tables, heads, hidden, seg):
    x = ns.bf16_normal((seg.n_tokens, hidden), 45 + hidden)
    codes, scale = weights(heads, hidden, 46 + heads)
    raw = run(x, codes, scale, seg, tables, heads)
    out = bf16_to_f64(raw.cpu())
    q, k, v = reference(x, codes, scale, seg, heads)
    for name, got, ref in (("q", out[:, 0], q), ("k", out[:, 1], k), ("v", out[:, 2], v)):
        assert_attn_close(got, ref, f"qkv projection {name} heads {heads} hidden {hidden}")
    projection_rounding_ok(raw, x, codes, scale, seg, heads, f"qkv projection heads {heads} hidden {hidden}")


def test_qkv_projection_rejects_bad_shapes(tables):
    seg = ns.Segment(0, 1, 2, 2, 0)
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.full((4, 3, 3, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros((3 * 3 * 128, 128), dtype=torch.int8, device=DEV)
    scale = torch.ones(3 * 3 * 128, dtype=torch.float32, device=DEV)
    with pytest.raises(nb.NomasError) as e:                  # odd head count
        nb.nomas_qkv_project_rope(x, codes, scale, seg, tables, out)
    assert e.value.status == nb.NOMAS_EUNSUPPORTED
    x2 = torch.zeros((4, 100), dtype=torch.bfloat16, device=DEV)
    codes2 = torch.zeros((3 * 2 * 128, 100), dtype=torch.int8, device=DEV)
    out2 = torch.full((4, 3, 2, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nb.NomasError) as e:                  # hidden not a multiple of 64
        nb.nomas_qkv_project_rope(x2, codes2, scale[:768], seg, tables, out2)
    assert e.value.status == nb.NOMAS_EUNSUPPORTED
    nb.nomas_stream_check()
    assert torch.all(out == 5.0) and torch.all(out2 == 5.0)  # nothing written


def test_qkv_fused_append_equals_append_of_the_unrotated_projection(tables):
    # the fused final-step call writes the cache rows nomas_kv_append_quant writes from the
    # projection's K and V before RoPE, bit for bit, behind rows already in the cache
    heads, hidden = 4, 512
    seg = ns.Segment(7, 3, 5, 9, 20)                          # 155 tokens: a ragged second row tile
    x = ns.bf16_normal((seg.n_tokens, hidden), 47)
    codes, scale = weights(heads, hidden, 48)
    pre = ns.Segment(0, 2, 5, 9, 0)                           # 90 earlier tokens already cached
    pk = ns.bf16_normal((pre.n_tokens, heads, 128), 49).to(DEV)
    pv = ns.bf16_normal((pre.n_tokens, heads, 128), 50).to(DEV)
    caches = []
    for _ in range(2):
        c = nb.KVCache(heads, 400)
        nb.nomas_kv_append_quant(c, pk, pv, pre, tables)
        caches.append(c)
    fused = torch.empty((seg.n_tokens, 3, heads, 128), dtype=torch.bfloat16, device=DEV)
    nb.nomas_qkv_project_rope(x.to(DEV), torch.from_numpy(codes).to(DEV), torch.from_numpy(scale).to(DEV), seg,
                              tables, fused, append_to=caches[0])
    nb.nomas_stream_check()
    assert caches[0].length == pre.n_tokens + seg.n_tokens
    assert torch.equal(fused, run(x, codes, scale, seg, tables, heads))           # same Q, K, V as without
    plain = run(x, codes, scale, ns.Segment(0, 0, 0, 0, seg.n_tokens), tables, heads)  # no rotation
    nb.nomas_kv_append_quant(caches[1], plain[:, 1].contiguous(), plain[:, 2].contiguous(), seg, tables)
    nb.nomas_stream_check()
    n = pre.n_tokens + seg.n_tokens
    a, b = caches
    assert torch.equal(a.k[:, :n], b.k[:, :n]) and torch.equal(a.v[:, :n], b.v[:, :n])
    assert torch.equal(a.k_scale[:, :n], b.k_scale[:, :n]) and torch.equal(a.v_scale[:, :n], b.v_scale[:, :n])


def test_qkv_fused_append_against_the_oracle(tables):
    # dequantised cache rows against the oracle's rotated K and V in float64: each within half a
    # quantisation step of the BF16 value the kernel quantised, which is within two BF16
    # roundings of the exact value (the projection's, carried through the rotation of its pair,
    # and the rotation's): at most 3.5 * 2^-9 of the pair norm, below 2^-6 of the row maximum
    heads, hidden = 2, 320
    seg = ns.Segment(1, 2, 11, 20, 300)                       # 740 tokens
    x = ns.bf16_normal((seg.n_tokens, hidden), 51)
    codes, scale = weights(heads, hidden, 52)
    cache = nb.KVCache(heads, 800)
    out = torch.empty((seg.n_tokens, 3, heads, 128), dtype=torch.bfloat16, device=DEV)
    nb.nomas_qkv_project_rope(x.to(DEV), torch.from_numpy(codes).to(DEV), torch.from_numpy(scale).to(DEV), seg,
                              tables, out, append_to=cache)
    nb.nomas_stream_check()
    _, k_ref, v_ref = reference(x, codes, scale, seg, heads)  # [L, H, 128] float64
    L = seg.n_tokens
    for name, c, s, ref in (("k", cache.k, cache.k_scale, k_ref), ("v", cache.v, cache.v_scale, v_ref)):
        cd = c[:, :L].cpu().numpy().astype(np.float64)         # [H, L, 128]
        sc = s[:, :L].cpu().numpy().astype(np.float64)         # [H, L]
        deq = cd * sc[:, :, None]
        r = ref.transpose(1, 0, 2)
        bound = 0.5 * sc[:, :, None] * (1 + 2.0 ** -20) + 2.0 ** -6 * np.abs(r).max(axis=2, keepdims=True) + 1e-6
        assert np.all(np.abs(deq - r) <= bound), f"{name}: worst excess {np.max(np.abs(deq - r) - bound):.3e}"
        assert np.all(np.abs(cd) <= 127)


def test_qkv_fused_append_checks_capacity(tables):
    heads, hidden = 2, 64
    seg = ns.Segment(0, 1, 4, 4, 0)                           # 16 tokens
    cache = nb.KVCache(heads, 12)
    x = torch.zeros((16, hidden), dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros((3 * heads * 128, hidden), dtype=torch.int8, device=DEV)
    scale = torch.ones(3 * heads * 128, dtype=torch.float32, device=DEV)
    out = torch.full((16, 3, heads, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_qkv_project_rope(x, codes, scale, seg, tables, out, append_to=cache)
    assert e.value.status == nb.NOMAS_ECAPACITY
    nb.nomas_stream_check()
    assert cache.length == 0 and torch.all(out == 5.0)


def test_qkv_fused_append_at_config2_size(tables):
    # the full 16,096-token segment at 16 heads x 2,048 hidden, as bench.py times it: cache rows
    # bit-exact with the separate append of the unrotated projection
    heads, hidden = 16, 2048
    seg = ns.config2().current[0]
    x = ns.bf16_normal((seg.n_tokens, hidden), 53)
    codes, scale = weights(heads, hidden, 54)
    a, b = nb.KVCache(heads, seg.n_tokens), nb.KVCache(heads, seg.n_tokens)
    fused = torch.empty((seg.n_tokens, 3, heads, 128), dtype=torch.bfloat16, device=DEV)
    nb.nomas_qkv_project_rope(x.to(DEV), torch.from_numpy(codes).to(DEV), torch.from_numpy(scale).to(DEV), seg,
                              tables, fused, append_to=a)
    plain = run(x, codes, scale, ns.Segment(0, 0, 0, 0, seg.n_tokens), tables, heads)
    nb.nomas_kv_append_quant(b, plain[:, 1], plain[:, 2], seg, tables)
    nb.nomas_stream_check()
    assert a.length == b.length == seg.n_tokens
    assert torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert torch.equal(a.k_scale, b.k_scale) and torch.equal(a.v_scale, b.v_scale)
