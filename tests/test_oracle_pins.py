"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes a part of the oracle against a closed form, an invariant, a
special case or brute force in 50-digit arithmetic, chosen so that a plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, a wrong
axis split, an off-by-one in the mask) fails at least one of them.

Sources: Hy-Nomas pages -- comfyui-wiki news, architecture table (16 heads x 128,
3D RoPE [16, 56, 56], theta 256) and sections "一个世界，分段生成" (segment-causal
attention over the K/V cache of every earlier segment) and "单张 4090 配置"
(INT8 cached K/V, BF16 compute, 18 temporal_context frames).
"""
import math

import mpmath
import numpy as np
import pytest

import oracle
from nomas_synth import bf16_bits, bf16_normal, Segment

SPLIT = (16, 56, 56)
BASES = (0, 16, 72)


def f32(x):
    return float(np.float32(x))


def bf16_of(values):
    """float values (exactly representable in BF16) -> uint16 bits."""
    a = np.asarray(values, dtype=np.float32).view(np.uint32)
    assert np.all((a & 0xFFFF) == 0), "value not exactly representable in BF16"
    return (a >> 16).astype(np.uint16)


# ------------------------------------------------------------------ RoPE
def test_rope_table_closed_form_time_axis():
    # d = 16, theta = 256 = 2^8  =>  omega_i = 256^(-2i/16) = 2^-i exactly.
    cos, sin = oracle.rope_table(5, 16)
    for p in range(5):
        for i in range(8):
            assert cos[p, i] == f32(math.cos(p * 2.0 ** -i))
            assert sin[p, i] == f32(math.sin(p * 2.0 ** -i))


def test_rope_table_closed_form_spatial_axes():
    # d = 56  =>  omega_i = 2^(-8*2i/56) = 2^(-2i/7); i = 0, 7, 14, 21 give 1, 1/4, 1/16, 1/64.
    cos, sin = oracle.rope_table(40, 56)
    for p in (0, 1, 3, 21, 39):
        for i, om in ((0, 1.0), (7, 0.25), (14, 1.0 / 16), (21, 1.0 / 64)):
            assert cos[p, i] == f32(math.cos(p * om))
            assert sin[p, i] == f32(math.sin(p * om))


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_rope_basis_vector_axis_split_and_pairing(axis):
    # A unit vector on channel base+2i at a position that is non-zero on `axis` only
    # must come out as (cos(p*omega_i), sin(p*omega_i)) on channels (base+2i, base+2i+1)
    # and leave every other channel zero.
    d = SPLIT[axis]
    base = BASES[axis]
    p = 3
    pos = np.zeros((1, 3), np.int32)
    pos[0, axis] = p
    for i in range(d // 2):
        x = np.zeros((1, 1, 128), np.float32)
        x[0, 0, base + 2 * i] = 1.0
        y = oracle.bf16_to_f64(oracle.rope_bf16(bf16_of(x), pos))[0, 0]
        ang = p * 256.0 ** (-2.0 * i / d)
        expect = np.zeros(128)
        expect[base + 2 * i] = math.cos(ang)
        expect[base + 2 * i + 1] = math.sin(ang)
        assert np.max(np.abs(y - expect)) <= 2.0 ** -8, (axis, i)
        # second member of the pair rotates the other way round: (-sin, cos)
        x = np.zeros((1, 1, 128), np.float32)
        x[0, 0, base + 2 * i + 1] = 1.0
        y = oracle.bf16_to_f64(oracle.rope_bf16(bf16_of(x), pos))[0, 0]
        expect = np.zeros(128)
        expect[base + 2 * i] = -math.sin(ang)
        expect[base + 2 * i + 1] = math.cos(ang)
        assert np.max(np.abs(y - expect)) <= 2.0 ** -8, (axis, i)


def test_rope_relative_offset_invariance():
    # score(R(p + D) q, R(p' + D) k) == score(R(p) q, R(p') k) for any shift D.
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 2, 128))
    k = rng.standard_normal((1, 2, 128))
    for p, pk, shift in [((3, 5, 7), (1, 2, 30), (10, 4, 2)),
                         ((0, 0, 0), (17, 21, 39), (300, 1, 1)),
                         ((9, 13, 3), (9, 13, 3), (5, 6, 7))]:
        def dots(a, b):
            qa = oracle.rope_f64(q, np.array([a], np.int32))
            kb = oracle.rope_f64(k, np.array([b], np.int32))
            return np.sum(qa * kb, axis=-1)
        base = dots(p, pk)
        shifted = dots(tuple(x + s for x, s in zip(p, shift)), tuple(x + s for x, s in zip(pk, shift)))
        assert np.allclose(base, shifted, rtol=0, atol=1e-11)
    # and depends on the offset: a different relative offset changes the score
    assert not np.allclose(dots((0, 0, 0), (1, 0, 0)), dots((0, 0, 0), (2, 0, 0)), atol=1e-6)


def test_rope_identity_at_origin_and_norms():
    x_bits = bf16_bits(bf16_normal((6, 3, 128), 11))
    pos0 = np.zeros((6, 3), np.int32)
    assert np.array_equal(oracle.rope_bf16(x_bits, pos0), x_bits)
    x = oracle.bf16_to_f64(x_bits)
    pos = np.array([[1, 2, 3], [4, 5, 6], [7, 8, 9], [10, 0, 39], [0, 21, 0], [359, 21, 39]], np.int32)
    y = oracle.rope_f64(x, pos)
    pair_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    pair_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(pair_x, pair_y, rtol=1e-13, atol=0)


def test_rope_time_offset_touches_only_time_channels():
    x_bits = bf16_bits(bf16_normal((1, 4, 128), 12))
    a = oracle.rope_bf16(x_bits, np.array([[2, 7, 9]], np.int32))
    b = oracle.rope_bf16(x_bits, np.array([[5, 7, 9]], np.int32))
    assert np.array_equal(a[..., 16:], b[..., 16:])
    assert not np.array_equal(a[..., :16], b[..., :16])
    c = oracle.rope_bf16(x_bits, np.array([[2, 8, 9]], np.int32))
    assert np.array_equal(a[..., :16], c[..., :16]) and np.array_equal(a[..., 72:], c[..., 72:])
    assert not np.array_equal(a[..., 16:72], c[..., 16:72])


def test_rope_bf16_path_matches_exact_rotation():
    x_bits = bf16_bits(bf16_normal((50, 2, 128), 13))
    rng = np.random.default_rng(3)
    pos = np.stack([rng.integers(0, 400, 50), rng.integers(0, 22, 50), rng.integers(0, 40, 50)], 1).astype(np.int32)
    y = oracle.bf16_to_f64(oracle.rope_bf16(x_bits, pos))
    ye = oracle.rope_f64(oracle.bf16_to_f64(x_bits), pos)
    x = oracle.bf16_to_f64(x_bits)
    pair_mag = np.repeat(np.abs(x[..., 0::2]) + np.abs(x[..., 1::2]), 2, axis=-1)
    # BF16 output rounding (half an ulp, <= 2^-8 relative) + fp32 table/op rounding
    assert np.all(np.abs(y - ye) <= 2.0 ** -8 * np.abs(ye) + 1e-6 * pair_mag + 1e-30)


def test_rope_text_tokens_unrotated():
    seg = Segment(3, 1, 2, 2, 5)
    pos = oracle.segment_positions(seg)
    assert pos.shape == (9, 3)
    assert np.all(pos[4:] == -1)
    assert pos[:4].tolist() == [[3, 0, 0], [3, 0, 1], [3, 1, 0], [3, 1, 1]]
    x_bits = bf16_bits(bf16_normal((9, 2, 128), 14))
    y = oracle.rope_bf16(x_bits, pos)
    assert np.array_equal(y[4:], x_bits[4:])
    assert not np.array_equal(y[1:4], x_bits[1:4])


# -------------------------------------------------------------- quantisation
def test_quant_absmax_maps_to_127_and_bound():
    x_bits = bf16_bits(bf16_normal((300, 128), 21))
    x = oracle.bf16_to_f64(x_bits)
    x[::7, 5] *= 8                       # outlier channels, still exact in BF16
    x_bits = bf16_of(x.astype(np.float32))
    codes, scales = oracle.quantize_rows(x_bits)
    assert codes.dtype == np.int8 and np.all(np.abs(codes.astype(np.int32)) <= 127)
    amax_idx = np.argmax(np.abs(x), axis=1)
    got = codes[np.arange(300), amax_idx].astype(np.int32)
    assert np.array_equal(got, np.sign(x[np.arange(300), amax_idx]).astype(np.int32) * 127)
    # scale * 127 reproduces absmax to within one fp32 ulp
    amax = np.abs(x).max(1)
    assert np.all(np.abs(scales.astype(np.float64) * 127 - amax) <= np.spacing(amax.astype(np.float32)))
    # dequantisation error <= scale/2, up to the rounding of the fp32 quotient x/scale
    # (half an fp32 ulp of |x/scale|, i.e. |x/scale| * 2^-24) taken before round-half-even
    err = np.abs(codes.astype(np.float64) * scales[:, None] - x)
    s64 = scales[:, None].astype(np.float64)
    assert np.all(err <= s64 / 2 + np.abs(x) * 2.0 ** -24)
    # the code is the nearest integer to the exact quotient, within that allowance
    quot = x / s64
    assert np.all(np.abs(codes - quot) <= 0.5 + np.abs(quot) * 2.0 ** -24)
    # beyond exact scale/2 only where the exact quotient sits within that allowance of a tie
    beyond = err > s64 / 2
    assert np.all(np.abs(np.abs(quot[beyond]) % 1.0 - 0.5) <= np.abs(quot[beyond]) * 2.0 ** -24)


def test_quant_ties_round_half_even():
    # absmax 127 gives scale = 1 exactly, so x/scale = x and ties are exact.
    row = np.zeros(128, np.float32)
    row[:9] = [127, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, 126.5]
    codes, scales = oracle.quantize_rows(bf16_of(row)[None])
    assert scales[0] == 1.0
    assert codes[0, :9].tolist() == [127, 2, 4, -2, -4, 0, 2, 0, 126]
    # absmax 63.5 gives scale = 0.5: x = 0.75 -> 1.5 -> 2; x = 1.25 -> 2.5 -> 2
    row = np.zeros(128, np.float32)
    row[:3] = [63.5, 0.75, 1.25]
    codes, scales = oracle.quantize_rows(bf16_of(row)[None])
    assert scales[0] == np.float32(63.5) / np.float32(127) and scales[0] == 0.5
    assert codes[0, :3].tolist() == [127, 2, 2]


def test_quant_zero_row():
    codes, scales = oracle.quantize_rows(np.zeros((2, 128), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 0)
    neg0 = np.full((1, 128), 0x8000, np.uint16)      # -0.0 everywhere
    codes, scales = oracle.quantize_rows(neg0)
    assert np.all(codes == 0) and scales[0] == 0


def test_append_is_rotate_round_then_quantise_and_placement():
    seg = Segment(1, 2, 3, 4, 5)          # 24 video + 5 text tokens
    heads = 3
    k = bf16_bits(bf16_normal((seg.n_tokens, heads, 128), 31))
    v = bf16_bits(bf16_normal((seg.n_tokens, heads, 128), 32))
    pos = oracle.segment_positions(seg)
    cache = oracle.Cache(heads, 100)
    cache.length = 40                     # append lands at 40..68
    cache.append(k, v, pos)
    assert cache.length == 40 + seg.n_tokens
    kr = oracle.rope_bf16(k, pos)
    kq, ks = oracle.quantize_rows(kr)
    vq, vs = oracle.quantize_rows(v)
    for h in range(heads):
        assert np.array_equal(cache.k[h, 40:69], kq[:, h])
        assert np.array_equal(cache.ks[h, 40:69], ks[:, h])
        assert np.array_equal(cache.v[h, 40:69], vq[:, h])
        assert np.array_equal(cache.vs[h, 40:69], vs[:, h])
        assert np.all(cache.k[h, :40] == 0) and np.all(cache.k[h, 69:] == 0)
    # text K is quantised unrotated
    tq, _ = oracle.quantize_rows(k[24:])
    assert np.array_equal(cache.k[:, 64:69].transpose(1, 0, 2), tq)
    with pytest.raises(ValueError):
        cache.append(k, v, pos)          # 69 + 29 fits; a third would not
        cache.append(k, v, pos)


# ------------------------------------------------------------------- gather
def test_gather_index_map_closed_form_and_rows():
    heads, tpf = 2, 6
    arch = oracle.Cache(heads, 10 * tpf + 3)
    rng = np.random.default_rng(5)
    arch.k[:] = rng.integers(-127, 128, arch.k.shape, dtype=np.int8)
    arch.v[:] = rng.integers(-127, 128, arch.v.shape, dtype=np.int8)
    arch.ks[:] = rng.random(arch.ks.shape, dtype=np.float32)
    arch.vs[:] = rng.random(arch.vs.shape, dtype=np.float32)
    # frames interleaved with 1 text token after frame 4 (offsets skip it)
    fto = [f * tpf + (1 if f > 4 else 0) for f in range(10)]
    frames = [0, 3, 5, 9]
    dst, idx = oracle.gather(arch, fto, tpf, frames)
    expect = [fto[frames[j // tpf]] + j % tpf for j in range(len(frames) * tpf)]
    assert idx.tolist() == expect
    assert dst.length == len(frames) * tpf
    for h in range(heads):
        assert np.array_equal(dst.k[h, :dst.length], arch.k[h, expect])
        assert np.array_equal(dst.v[h, :dst.length], arch.v[h, expect])
        assert np.array_equal(dst.ks[h, :dst.length], arch.ks[h, expect])
        assert np.array_equal(dst.vs[h, :dst.length], arch.vs[h, expect])


# ----------------------------------------------------------------- attention
def _tiny_problem(seed=40, heads=2, lh=56, segs=(56,), history=True):
    lq = sum(segs)
    q = bf16_bits(bf16_normal((lq, heads, 128), seed))
    k = bf16_bits(bf16_normal((lq, heads, 128), seed + 1))
    v = bf16_bits(bf16_normal((lq, heads, 128), seed + 2))
    offs = np.concatenate([[0], np.cumsum(segs)]).astype(np.int32)
    hist = None
    if history and lh:
        hist = oracle.Cache(heads, lh)
        hk = bf16_bits(bf16_normal((lh, heads, 128), seed + 3))
        hv = bf16_bits(bf16_normal((lh, heads, 128), seed + 4))
        hist.append(hk, hv, np.zeros((lh, 3), np.int32) - 1)   # unrotated keys are fine here
    return q, k, v, offs, hist


def _brute_force_row(q, k, v, offs, hist, i, h, scale, dps=50):
    """Attention of query i, head h in exact/50-digit arithmetic, written out from the definition."""
    mpmath.mp.dps = dps
    qf = oracle.bf16_to_f64(q[i, h])
    keys, vals = [], []
    if hist is not None:
        for j in range(hist.length):
            keys.append([mpmath.mpf(int(c)) * mpmath.mpf(float(hist.ks[h, j])) for c in hist.k[h, j]])
            vals.append([mpmath.mpf(int(c)) * mpmath.mpf(float(hist.vs[h, j])) for c in hist.v[h, j]])
    seg = int(np.searchsorted(offs, i, side="right")) - 1
    for j in range(int(offs[seg + 1])):       # current keys of segments 0..seg
        keys.append([mpmath.mpf(float(x)) for x in oracle.bf16_to_f64(k[j, h])])
        vals.append([mpmath.mpf(float(x)) for x in oracle.bf16_to_f64(v[j, h])])
    qm = [mpmath.mpf(float(x)) for x in qf]
    s = [mpmath.fsum(a * b for a, b in zip(qm, kk)) * mpmath.mpf(scale) for kk in keys]
    e = [mpmath.exp(x) for x in s]
    z = mpmath.fsum(e)
    out = [mpmath.fsum(e[j] * vals[j][d] for j in range(len(e))) / z for d in range(128)]
    return np.array([float(x) for x in out]), float(mpmath.log(z))


def test_attention_brute_force_50_digits():
    q, k, v, offs, hist = _tiny_problem(segs=(28, 28))
    scale = 1.0 / math.sqrt(128)
    rows = [0, 13, 27, 28, 41, 55]
    out, lse = oracle.seg_attn(q, k, v, offs, hist, rows=rows)
    for r, i in enumerate(rows):
        for h in range(2):
            ref, ref_lse = _brute_force_row(q, k, v, offs, hist, i, h, scale)
            assert np.max(np.abs(out[r, h] - ref)) <= 1e-13 * np.max(np.abs(ref))
            assert abs(lse[r, h] - ref_lse) <= 1e-12 * max(1.0, abs(ref_lse))


def test_attention_constant_v_gives_v():
    q, k, v, offs, hist = _tiny_problem(seed=50)
    # history V: code 64 * scale 2^-5 = 2.0 ; current V: 2.0 in BF16
    hist.v[:] = 64
    hist.vs[:] = 2.0 ** -5
    v = np.full_like(v, bf16_of([2.0])[0])
    out, _ = oracle.seg_attn(q, k, v, offs, hist)
    assert np.max(np.abs(out - 2.0)) <= 1e-14


def test_attention_single_key_gives_v():
    q, k, v, offs, _ = _tiny_problem(seed=60, segs=(1,), history=False)
    out, lse = oracle.seg_attn(q, k, v, offs, None)
    assert np.array_equal(out[0], oracle.bf16_to_f64(v[0]))
    qk = np.sum(oracle.bf16_to_f64(q[0]) * oracle.bf16_to_f64(k[0]), axis=-1) / math.sqrt(128)
    assert np.allclose(lse[0], qk, rtol=0, atol=1e-13)


def test_attention_zero_query_gives_mean_of_visible_v():
    q, k, v, offs, hist = _tiny_problem(seed=70, segs=(20, 36))
    q = np.zeros_like(q)
    out, lse = oracle.seg_attn(q, k, v, offs, hist)
    hv = hist.v.astype(np.float64) * hist.vs[..., None]         # [H][Lh][D]
    vc = oracle.bf16_to_f64(v)                                     # [Lq][H][D]
    for i in (0, 19, 20, 55):
        end = 20 if i < 20 else 56
        for h in range(2):
            allv = np.concatenate([hv[h], vc[:end, h]], 0)
            assert np.allclose(out[i, h], allv.mean(0), rtol=0, atol=1e-14)
            assert abs(lse[i, h] - math.log(56 + end)) < 1e-13


def test_attention_key_permutation_invariance():
    q, k, v, offs, hist = _tiny_problem(seed=80)
    out, lse = oracle.seg_attn(q, k, v, offs, hist)
    perm = np.random.default_rng(1).permutation(hist.length)
    hist.k[:] = hist.k[:, perm]
    hist.v[:] = hist.v[:, perm]
    hist.ks[:] = hist.ks[:, perm]
    hist.vs[:] = hist.vs[:, perm]
    out2, lse2 = oracle.seg_attn(q, k, v, offs, hist)
    assert np.allclose(out, out2, rtol=0, atol=1e-13) and np.allclose(lse, lse2, rtol=0, atol=1e-13)


def test_attention_split_and_lse_merge_equals_whole():
    q, k, v, offs, hist = _tiny_problem(seed=90)
    out, lse = oracle.seg_attn(q, k, v, offs, hist)
    o1, l1 = oracle.seg_attn(q, k, v, offs, hist, key_parts=1)     # history keys only
    o2, l2 = oracle.seg_attn(q, k, v, offs, hist, key_parts=2)     # current keys only
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    merged = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    assert np.allclose(out, merged, rtol=0, atol=1e-13)
    assert np.allclose(lse, m + np.log(w1 + w2), rtol=0, atol=1e-13)


def test_segment_causality_future_segment_leaves_outputs_unchanged():
    q, k, v, offs, hist = _tiny_problem(seed=100, segs=(30, 26))
    out, lse = oracle.seg_attn(q, k, v, offs, hist)
    out0, lse0 = oracle.seg_attn(q[:30], k[:30], v[:30], np.array([0, 30], np.int32), hist)
    assert np.array_equal(out[:30], out0) and np.array_equal(lse[:30], lse0)
    # and the later segment does see the earlier one (so the mask is not "own segment only")
    out1, _ = oracle.seg_attn(q[30:], k[30:], v[30:], np.array([0, 26], np.int32), hist)
    assert not np.allclose(out[30:], out1, atol=1e-6)


def test_attention_row_sampling_matches_full():
    q, k, v, offs, hist = _tiny_problem(seed=110, segs=(10, 46))
    out, lse = oracle.seg_attn(q, k, v, offs, hist)
    rows = [55, 0, 9, 10, 31]
    o, l = oracle.seg_attn(q, k, v, offs, hist, rows=rows)
    assert np.array_equal(o, out[rows]) and np.array_equal(l, lse[rows])


def test_attention_softmax_scale_default():
    q, k, v, offs, hist = _tiny_problem(seed=120)
    out, _ = oracle.seg_attn(q, k, v, offs, hist)
    q2 = bf16_of((oracle.bf16_to_f64(q) * 2).astype(np.float32))    # exact doubling
    out2, _ = oracle.seg_attn(q2, k, v, offs, hist, sm_scale=0.5 / math.sqrt(128))
    assert np.allclose(out, out2, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------- W8A16 QKV projection
def test_qkv_projection_against_exact_loops():
    # explicit sums in exact rationals, with every operand distinct, so a transposed weight, a
    # scale applied per input channel instead of per output channel, or a dropped term fails
    from fractions import Fraction
    rng = np.random.default_rng(11)
    L, K, N = 3, 5, 7
    x = rng.standard_normal((L, K)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)           # truncate to BF16 bit patterns
    codes = rng.integers(-127, 128, (N, K)).astype(np.int8)
    scale = (rng.random(N) + 0.1).astype(np.float32)
    y = oracle.qkv_project(xb, codes, scale)
    xv = oracle.bf16_to_f64(xb)
    for l in range(L):
        for n in range(N):
            ref = sum(Fraction(float(xv[l, k])) * int(codes[n, k]) for k in range(K)) * Fraction(float(scale[n]))
            assert abs(Fraction(float(y[l, n])) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 1000)


def test_qkv_projection_unit_basis_closed_form():
    # x = e_k picks column k of the dequantised weights: y[n] = codes[n, k] * scale[n]
    K, N = 8, 6
    codes = np.arange(N * K, dtype=np.int64).reshape(N, K).astype(np.int8) - 20
    scale = np.linspace(0.5, 3.0, N).astype(np.float32)
    for k in range(K):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        y = oracle.qkv_project(xb, codes, scale)[0]
        assert np.array_equal(y, codes[:, k].astype(np.float64) * scale.astype(np.float64))



# ------------------------------------------------------------------------ camera tokens
def _rz(deg):
    c, s = math.cos(math.radians(deg)), math.sin(math.radians(deg))
    return np.array([[c, -s, 0.0], [s, c, 0.0], [0.0, 0.0, 1.0]])


def _pose(r, t):
    m = np.eye(4)
    m[:3, :3] = r
    m[:3, 3] = t
    return m


def test_camera_tokens_identity_trajectory():
    toks = oracle.camera_tokens(np.tile(np.eye(4), (8, 1, 1)))
    assert toks.shape == (2, 64)
    frame = np.diag([2.5, 2.5, 2.5, 1.0]).reshape(16)
    assert np.array_equal(toks, np.tile(frame, (2, 4)))


def test_camera_tokens_worked_example():
    # first camera turned 90 degrees about z and placed at (1, 2, 3); by hand, inverse(c2w0) =
    # [R0^T | -R0^T t0] with R0^T = [[0, 1, 0], [-1, 0, 0], [0, 0, 1]], so
    #   frame 1 (identity pose):           R = R0^T, t = R0^T (0 - t0) = (-2, 1, -3)
    #   frame 2 (first pose, +1 along z):  R = I,    t = (0, 0, 1)
    #   frame 3 (first pose, +1 along x):  R = I,    t = (0, -1, 0)   (world x is camera -y)
    r0 = np.array([[0.0, -1.0, 0.0], [1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    c2w = np.stack([_pose(r0, (1, 2, 3)), np.eye(4), _pose(r0, (1, 2, 4)), _pose(r0, (2, 2, 3))])
    want = np.array([
        2.5, 0, 0, 0, 0, 2.5, 0, 0, 0, 0, 2.5, 0, 0, 0, 0, 1,
        0, 2.5, 0, -2, -2.5, 0, 0, 1, 0, 0, 2.5, -3, 0, 0, 0, 1,
        2.5, 0, 0, 0, 0, 2.5, 0, 0, 0, 0, 2.5, 1, 0, 0, 0, 1,
        2.5, 0, 0, 0, 0, 2.5, 0, -1, 0, 0, 2.5, 0, 0, 0, 0, 1,
    ], np.float64)
    assert np.array_equal(oracle.camera_tokens(c2w)[0], want)
    # the translation scale multiplies the translation column only, the rotation scale the block
    toks = oracle.camera_tokens(c2w, translation_scale=2.0, rotation_scale=1.0)[0].reshape(4, 4, 4)
    assert np.array_equal(toks[1, :3, 3], [-4.0, 2.0, -6.0])
    assert np.array_equal(toks[1, :3, :3], r0.T)


def test_camera_tokens_invariant_to_a_common_world_transform():
    # E_i = inverse(c2w0) . c2w_i does not change when every pose is moved by one rigid G
    rng = np.random.default_rng(5)
    c2w = []
    for i in range(12):
        q, _ = np.linalg.qr(rng.standard_normal((3, 3)))
        c2w.append(_pose(q * np.sign(np.linalg.det(q)), rng.standard_normal(3) * 4))
    c2w = np.stack(c2w)
    qg, _ = np.linalg.qr(rng.standard_normal((3, 3)))
    g = _pose(qg * np.sign(np.linalg.det(qg)), (10.0, -3.0, 7.0))
    a = oracle.camera_tokens(c2w, 1.5, 2.5)
    b = oracle.camera_tokens(g[None] @ c2w, 1.5, 2.5)
    assert np.max(np.abs(a - b)) < 1e-12
    # the first frame of every trajectory normalises to diag(r, r, r, 1)
    assert np.allclose(a[0, :16], np.diag([2.5, 2.5, 2.5, 1.0]).reshape(16), atol=1e-14)


def test_camera_tokens_layout_and_bad_shapes():
    # pure translations: frame 4g + j sits at columns 16 j .. 16 j + 15 of token g, row-major
    c2w = np.stack([_pose(np.eye(3), (i, 2 * i, -i)) for i in range(12)])
    toks = oracle.camera_tokens(c2w, 1.0, 1.0)
    for i in range(12):
        m = toks[i // 4, 16 * (i % 4):16 * (i % 4) + 16].reshape(4, 4)
        assert np.array_equal(m, _pose(np.eye(3), (i, 2 * i, -i)))
    with pytest.raises(ValueError):
        oracle.camera_tokens(np.tile(np.eye(4), (6, 1, 1)))


# ---------------------------------------------------------------- camera cross-attention
def _cam_problem(L, Tc, H, seed):
    return (bf16_bits(bf16_normal((L, H, 128), seed)), bf16_bits(bf16_normal((Tc, H, 128), seed + 1)),
            bf16_bits(bf16_normal((Tc, H, 128), seed + 2)))


def test_camera_xattn_single_camera_token_returns_its_value():
    q, k, v = _cam_problem(5, 1, 2, 130)
    out = oracle.camera_cross_attn(q, k, v)
    assert np.array_equal(out, np.broadcast_to(oracle.bf16_to_f64(v), out.shape))


def test_camera_xattn_constant_values_and_zero_query():
    q, k, v = _cam_problem(6, 9, 2, 131)
    vc = np.broadcast_to(v[:1], v.shape).copy()
    out = oracle.camera_cross_attn(q, k, vc)
    assert np.max(np.abs(out - oracle.bf16_to_f64(vc[:1]))) < 1e-14
    out0 = oracle.camera_cross_attn(np.zeros_like(q), k, v)          # q = 0: the mean of V
    assert np.max(np.abs(out0 - oracle.bf16_to_f64(v).mean(axis=0)[None])) < 1e-14


def test_camera_xattn_two_tokens_logistic_closed_form():
    # softmax over two keys: O = v0 + sigma(d) (v1 - v0), d = scale q.(k1 - k0)
    q, k, v = _cam_problem(4, 2, 3, 132)
    qf, kf, vf = (oracle.bf16_to_f64(x) for x in (q, k, v))
    for scale in (None, 0.3):
        out = oracle.camera_cross_attn(q, k, v, sm_scale=scale)
        sc = 1.0 / math.sqrt(128) if scale is None else scale
        for l in range(4):
            for h in range(3):
                d = sc * float(np.dot(qf[l, h], kf[1, h] - kf[0, h]))
                sig = 1.0 / (1.0 + math.exp(-d))
                want = vf[0, h] + sig * (vf[1, h] - vf[0, h])
                assert np.max(np.abs(out[l, h] - want)) < 1e-13


def test_camera_xattn_permutation_heads_and_rows():
    q, k, v = _cam_problem(7, 11, 3, 133)
    out = oracle.camera_cross_attn(q, k, v)
    perm = np.random.default_rng(0).permutation(11)
    assert np.max(np.abs(oracle.camera_cross_attn(q, k[perm], v[perm]) - out)) < 1e-14
    k2 = k.copy()
    k2[:, 1] = k[::-1, 1]                                            # touch head 1 only
    out2 = oracle.camera_cross_attn(q, k2, v)
    assert np.array_equal(out2[:, 0], out[:, 0]) and np.array_equal(out2[:, 2], out[:, 2])
    assert np.array_equal(oracle.camera_cross_attn(q, k, v, rows=[6, 0, 3]), out[[6, 0, 3]])


def test_camera_tokens_relative_poses_compose():
    # with unit scales E_i = inverse(c2w0) c2w_i, so inverse(E_j) E_i = inverse(c2w_j) c2w_i for
    # every pair: the tokens keep every relative pose of the trajectory
    rng = np.random.default_rng(9)
    c2w = []
    for i in range(8):
        q, _ = np.linalg.qr(rng.standard_normal((3, 3)))
        c2w.append(_pose(q * np.sign(np.linalg.det(q)), rng.standard_normal(3) * 3))
    c2w = np.stack(c2w)
    e = oracle.camera_tokens(c2w, 1.0, 1.0).reshape(8, 4, 4)
    for i in range(8):
        for j in range(8):
            assert np.max(np.abs(np.linalg.inv(e[j]) @ e[i] - np.linalg.inv(c2w[j]) @ c2w[i])) < 1e-12


def test_camera_xattn_agrees_with_the_segment_attention_oracle():
    # with the queries' own tokens as the camera tokens, the cross-attention is the single-segment
    # attention without history, computed independently by the C oracle (pinned above by 50-digit
    # brute force)
    q, k, v = _cam_problem(9, 9, 2, 134)
    want, _ = oracle.seg_attn(q, k, v, [0, 9])
    assert np.max(np.abs(oracle.camera_cross_attn(q, k, v) - want)) < 1e-14
