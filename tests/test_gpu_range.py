"""GPU parity over the whole BF16 input range, and the history staged once per segment.

The tensor-core operands are FP16, whose normal range (2^-14 .. 65,504) is far narrower than
BF16's.  The library multiplies every operand block by an exact power of two chosen from the
block's maximum and undoes it in fp32, so inputs of any finite magnitude must still meet the
attention tolerance against the float64 oracle (max |gpu - oracle| <= 1e-2 max |oracle|,
sum |gpu - oracle| / sum |oracle| <= 2e-3).  The inputs here are the seeded N(0,1) BF16 tensors
of the other tests, multiplied by powers of two (exact in BF16) or by other factors (rounded to
BF16 once; both sides receive the same BF16 values): uniformly scaled by 2^17 and by 2^-20, a
history with row maxima near 1e5, query rows spread over fifty binary orders, heads of different
magnitudes, and current values far from the history's in both directions.  The operands' FP16
rounding (2^-12 relative for the dequantised history) bounds the score error by about 2^-12 of the
score's magnitude, so inputs whose softmax is an arg-max over near-ties at that level are not a
meaningful comparison; the cases here keep either well-separated or moderate scores.  Magnitudes
beyond what the fp32 softmax represents must be reported as NOMAS_ERANGE rather than returned as a
result.
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
CFG = 21   # seed family of this file


@pytest.fixture(scope="module")
def tables():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from segment_causal_attention_nomas_b300 import build
    build.build()
    t = nb.nomas_rope_tables_create(256.0, (16, 56, 56), 512, 64, 64)
    yield t
    t.close()


def scaled(t: torch.Tensor, f) -> torch.Tensor:
    """t * f in fp32, rounded once to BF16 (f a number or a tensor broadcasting against t)."""
    return (t.float() * f).to(torch.bfloat16)


def pow2_rows(n: int, lo: int, hi: int, step: int) -> torch.Tensor:
    """Per-row factors 2^e with e cycling through [lo, hi] by `step` (shape [n, 1, 1])."""
    e = lo + (np.arange(n) * step) % (hi - lo + 1)
    return torch.from_numpy(np.ldexp(1.0, e).astype(np.float32)).view(n, 1, 1)


def inputs(heads, hist_seg, cur_seg, step=0):
    h = ns.bf16_normal((hist_seg.n_tokens, heads, 128), ns.seed_of(CFG, ns.T_HK)) if hist_seg else None
    hv = ns.bf16_normal((hist_seg.n_tokens, heads, 128), ns.seed_of(CFG, ns.T_HV)) if hist_seg else None
    q, k, v = (ns.bf16_normal((cur_seg.n_tokens, heads, 128), ns.seed_of(CFG, t, 0, step))
               for t in (ns.T_Q, ns.T_K, ns.T_V))
    return q, k, v, h, hv


def gpu_run(tables, heads, hist_seg, cur_seg, q, k, v, hk, hv, staged=False, lse=False):
    hist = None
    if hist_seg is not None:
        hist = nb.KVCache(heads, hist_seg.n_tokens)
        nb.nomas_kv_append_quant(hist, hk.to(DEV), hv.to(DEV), hist_seg, tables)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    nb.nomas_rope3d(qd, qd, cur_seg, tables)
    nb.nomas_rope3d(kd, kd, cur_seg, tables)
    out = torch.full_like(qd, float("nan"))         # an unwritten element fails the finiteness check
    lse_t = torch.full((heads, cur_seg.n_tokens), float("nan"), dtype=torch.float32, device=DEV) if lse else None
    lq = cur_seg.n_tokens
    if staged:
        sh = nb.StagedHistory(heads, hist.length + 64) if hist is not None else None
        if sh is not None:
            nb.nomas_seg_attn_stage_history(hist, sh)
        nb.nomas_seg_attn_staged(qd, kd, vd, [0, lq], sh, out, lse_t)
    else:
        nb.nomas_seg_attn(qd, kd, vd, [0, lq], hist, out, lse_t)
    return out, lse_t, hist


def oracle_run(heads, hist_seg, cur_seg, q, k, v, hk, hv, rows=None):
    hist = None
    if hist_seg is not None:
        hist = oracle.Cache(heads, hist_seg.n_tokens)
        hist.append(ns.bf16_bits(hk), ns.bf16_bits(hv), oracle.segment_positions(hist_seg))
    pos = oracle.segment_positions(cur_seg)
    qr = oracle.rope_bf16(ns.bf16_bits(q), pos)
    kr = oracle.rope_bf16(ns.bf16_bits(k), pos)
    return oracle.seg_attn(qr, kr, ns.bf16_bits(v), [0, cur_seg.n_tokens], hist, rows=rows)


def check(tables, heads, hist_seg, cur_seg, q, k, v, hk, hv, what, rows=None):
    out, lse, _ = gpu_run(tables, heads, hist_seg, cur_seg, q, k, v, hk, hv, lse=True)
    nb.nomas_stream_check()
    ref, ref_lse = oracle_run(heads, hist_seg, cur_seg, q, k, v, hk, hv, rows)
    got = bf16_to_f64(out)
    gl = lse.cpu().numpy().astype(np.float64).T
    if rows is not None:
        got, gl = got[rows], gl[rows]
    res = assert_attn_close(got, ref, what)
    # the log-sum-exp in natural-log units, relative to its own magnitude (scores may be huge)
    assert np.max(np.abs(gl - ref_lse)) <= 1e-3 * max(1.0, np.max(np.abs(ref_lse))), f"{what}: lse"
    return res


HEADS = 3
HIST = ns.Segment(0, 2, 11, 23, 7)    # 506 video + 7 text = 513 history tokens (ragged tile)
CUR = ns.Segment(2, 1, 13, 29, 11)    # 377 video + 11 text = 388 query tokens (ragged tile)


@pytest.mark.parametrize("e", [17, -20])
def test_attention_uniformly_scaled_inputs(tables, e):
    # every input times 2^e: beyond FP16's largest value (2^17 * |N(0,1)| up to ~6e5) and below
    # its normal range (2^-20 * |N(0,1)|); the softmax at 2^17 is an arg-max, at 2^-20 uniform
    q, k, v, hk, hv = inputs(HEADS, HIST, CUR)
    f = 2.0 ** e
    check(tables, HEADS, HIST, CUR, scaled(q, f), scaled(k, f), scaled(v, f), scaled(hk, f), scaled(hv, f),
          f"all inputs x 2^{e}")


@pytest.mark.parametrize("which", ["k_and_v", "v_only"])
def test_attention_history_rows_of_absmax_1e5(tables, which):
    # A quarter of the history (token, head) rows scaled to a maximum near 1e5, so the dequantised
    # code * scale reaches 1e5 (above FP16's 65,504); the current segment N(0,1).  With the large
    # K rows the queries are scaled by 2^-14, which keeps the scores of those rows in the usual
    # range (|score| of a few units): scores of 1e5 would make the softmax an arg-max whose
    # near-ties (gaps below 2^-12 of the score) no FP16- or BF16-operand kernel resolves as the
    # float64 oracle does, a question of the softmax's conditioning rather than of the range.
    q, k, v, hk, hv = inputs(HEADS, HIST, CUR)
    g = torch.Generator().manual_seed(ns.seed_of(CFG, ns.T_MISC))
    big = (torch.rand((HIST.n_tokens, HEADS, 1), generator=g) < 0.25).float()
    fv = 1.0 + big * (1e5 / hv.float().abs().amax(-1, keepdim=True) - 1.0)
    hv2 = scaled(hv, fv)
    assert float(hv2.float().abs().max()) > 65504
    hk2 = hk
    if which == "k_and_v":
        fk = 1.0 + big * (1e5 / hk.float().abs().amax(-1, keepdim=True) - 1.0)
        hk2 = scaled(hk, fk)
        assert float(hk2.float().abs().max()) > 65504
        q = scaled(q, 2.0 ** -14)
    check(tables, HEADS, HIST, CUR, q, k, v, hk2, hv2, f"history row absmax 1e5 ({which})")


@pytest.mark.parametrize("v_cur_e,v_hist_e", [(-10, 30), (25, -25)])
def test_attention_mixed_magnitudes(tables, v_cur_e, v_hist_e):
    # query rows spread over 2^-34 .. 2^0 (each row its own exponent), heads of K at 2^-10, 2^0,
    # 2^2 (each head its own, shared by history and current K), and current values 2^40 or 2^-50
    # away from the history's (the accumulator is rescaled between the two); the largest scores
    # stay moderate, so the comparison is about the exponents, not the softmax's conditioning
    q, k, v, hk, hv = inputs(HEADS, HIST, CUR)
    head_f = torch.tensor([2.0 ** -10, 1.0, 2.0 ** 2]).view(1, HEADS, 1)
    q2 = scaled(q, pow2_rows(CUR.n_tokens, -34, 0, 7))
    k2 = scaled(k, head_f)
    hk2 = scaled(hk, head_f)
    v2 = scaled(v, 2.0 ** v_cur_e)
    hv2 = scaled(hv, 2.0 ** v_hist_e)
    check(tables, HEADS, HIST, CUR, q2, k2, v2, hk2, hv2, f"mixed, V 2^{v_cur_e} / history V 2^{v_hist_e}")


@pytest.mark.parametrize("v_cur_e,v_hist_e", [(3, -3), (-20, 12)])
def test_attention_scaled_split_kv(tables, v_cur_e, v_hist_e):
    # a short segment over a long history takes the split-KV path (partials merged by a second
    # kernel); some splits hold only history tiles, one holds the last history and the current
    # tiles, so the per-split output exponents and the in-split rescale are both exercised.  Q at
    # 2^-3 and K at 2^3 keep the scores in the usual range; V and history V differ by 2^6 or 2^32.
    heads = 2
    hist_seg = ns.Segment(0, 12, 22, 40, 0)      # 10,560 history tokens
    cur_seg = ns.Segment(12, 1, 11, 17, 13)      # 200 query tokens
    lq, lh = cur_seg.n_tokens, hist_seg.n_tokens
    no_split = (3 * lq * heads * 256 + (-(-8 * heads // 1024) * 1024 + 2 * lh * heads * 256)
                + -(-lq * heads // 256) * 256 + -(-8 * heads // 256) * 256)
    assert nb.nomas_seg_attn_workspace_size(lq, lh, heads) > no_split      # partials in the workspace
    q, k, v, hk, hv = inputs(heads, hist_seg, cur_seg)
    check(tables, heads, hist_seg, cur_seg, scaled(q, 2.0 ** -3), scaled(k, 2.0 ** 3), scaled(v, 2.0 ** v_cur_e),
          scaled(hk, 2.0 ** 3), scaled(hv, 2.0 ** v_hist_e), f"split-KV, V 2^{v_cur_e} / history V 2^{v_hist_e}")


@pytest.mark.parametrize("case", ["scores", "values"])
def test_attention_out_of_range_is_reported(tables, case):
    # scores beyond ~1e34 (Q and K at 2^60), or current and history V maxima 2^90 apart: the
    # call completes, nomas_stream_check reports NOMAS_ERANGE, and the next call is unaffected
    q, k, v, hk, hv = inputs(HEADS, HIST, CUR)
    if case == "scores":
        q, k = scaled(q, 2.0 ** 60), scaled(k, 2.0 ** 60)
    else:
        v, hv = scaled(v, 2.0 ** -30), scaled(hv, 2.0 ** 60)
    gpu_run(tables, HEADS, HIST, CUR, q, k, v, hk, hv)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_stream_check()
    assert e.value.status == nb.NOMAS_ERANGE
    nb.nomas_stream_check()   # the status word was cleared
    q, k, v, hk, hv = inputs(HEADS, HIST, CUR)
    check(tables, HEADS, HIST, CUR, q, k, v, hk, hv, "after a range report")


# ------------------------------------------------------------- history staged once
def test_staged_history_bit_identical_over_two_steps(tables):
    # One staging of the history serves two Euler steps with fresh Q/K/V: each step's output
    # (and LSE) equals nomas_seg_attn's on the INT8 history bit for bit, and the oracle's within
    # the tolerance.  The staged buffer has spare capacity (rows past the length are not read).
    heads = HEADS
    hist = nb.KVCache(heads, HIST.n_tokens)
    _, _, _, hk, hv = inputs(heads, HIST, CUR)
    hk, hv = scaled(hk, 2.0 ** -2), scaled(hv, 2.0 ** 9)
    nb.nomas_kv_append_quant(hist, hk.to(DEV), hv.to(DEV), HIST, tables)
    sh = nb.StagedHistory(heads, HIST.n_tokens + 300)
    nb.nomas_seg_attn_stage_history(hist, sh)
    assert sh.length == HIST.n_tokens
    lq = CUR.n_tokens
    for step in (0, 1):
        q, k, v, _, _ = inputs(heads, HIST, CUR, step)
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        nb.nomas_rope3d(qd, qd, CUR, tables)
        nb.nomas_rope3d(kd, kd, CUR, tables)
        out_a, out_b = torch.empty_like(qd), torch.empty_like(qd)
        lse_a = torch.empty((heads, lq), dtype=torch.float32, device=DEV)
        lse_b = torch.empty_like(lse_a)
        nb.nomas_seg_attn(qd, kd, vd, [0, lq], hist, out_a, lse_a)
        nb.nomas_seg_attn_staged(qd, kd, vd, [0, lq], sh, out_b, lse_b)
        nb.nomas_stream_check()
        assert torch.equal(out_a, out_b), f"step {step}"
        assert torch.equal(lse_a, lse_b), f"step {step}"
        ref, _ = oracle_run(heads, HIST, CUR, q, k, v, hk, hv)
        assert_attn_close(bf16_to_f64(out_b), ref, f"staged step {step}")


def test_staged_empty_history_equals_no_history(tables):
    heads = 2
    seg = ns.Segment(0, 1, 9, 15, 5)
    q, k, v = (ns.bf16_normal((seg.n_tokens, heads, 128), ns.seed_of(CFG, t, 3)).to(DEV)
               for t in (ns.T_Q, ns.T_K, ns.T_V))
    empty = nb.KVCache(heads, 8)
    sh = nb.StagedHistory(heads, 8)
    nb.nomas_seg_attn_stage_history(empty, sh)
    assert sh.length == 0
    a, b = torch.empty_like(q), torch.empty_like(q)
    nb.nomas_seg_attn(q, k, v, [0, seg.n_tokens], None, a)
    nb.nomas_seg_attn_staged(q, k, v, [0, seg.n_tokens], sh, b)
    nb.nomas_stream_check()
    assert torch.equal(a, b)
