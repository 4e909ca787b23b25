"""nomas_seg_attn_noalloc against nomas_seg_attn, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory where they
run attention; its scratch (the staged FP16 operands, the split-KV partials and the operand
exponents) comes from a fixed array inside the library.  This file checks, on shapes whose scratch fits that array and
whose split-KV path is taken, that two calls in a row give the output of the ordinary entry
point (which takes a caller workspace) within the attention tolerance of the parity tests, and
that shapes needing more scratch than the array holds are refused before anything is written.
It builds its own inputs so it passes in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import nomas_synth as ns
import segment_causal_attention_nomas_b300 as nb
from harness import assert_attn_close, bf16_to_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
HEADS = 4
HIST = ns.Segment(0, 5, 20, 40, 0)         # 4,000 history tokens
CUR = ns.Segment(5, 1, 22, 40, 120)        # 880 video + 120 text = 1,000 query tokens


@pytest.fixture(scope="module")
def setup():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from segment_causal_attention_nomas_b300 import build
    build.build()
    tables = nb.nomas_rope_tables_create(256.0, (16, 56, 56), 512, 64, 64)
    hist = nb.KVCache(HEADS, HIST.n_tokens)
    k = ns.bf16_normal((HIST.n_tokens, HEADS, 128), ns.seed_of(11, ns.T_HK)).to(DEV)
    v = ns.bf16_normal((HIST.n_tokens, HEADS, 128), ns.seed_of(11, ns.T_HV)).to(DEV)
    nb.nomas_kv_append_quant(hist, k, v, HIST, tables)
    nb.nomas_stream_check()
    yield tables, hist
    tables.close()


def current_inputs(tables, step):
    q, k, v = (ns.bf16_normal((CUR.n_tokens, HEADS, 128), ns.seed_of(11, t, 0, step)).to(DEV)
               for t in (ns.T_Q, ns.T_K, ns.T_V))
    nb.nomas_rope3d(q, q, CUR, tables)
    nb.nomas_rope3d(k, k, CUR, tables)
    return q, k, v


def test_noalloc_matches_workspace_entry_point_on_two_calls(setup):
    tables, hist = setup
    lq = CUR.n_tokens
    lh = hist.length
    need = nb.nomas_seg_attn_workspace_size(lq, lh, HEADS)
    assert 0 < need <= nb.NOMAS_NOALLOC_SCRATCH_BYTES, need
    # everything but the split-KV partials: staged Q, K, V and history (with its scale maxima),
    # the query-row exponents and the current K/V maxima; the rest of `need` is at least two
    # splits' partials, so this shape's split path keeps its partials in the fixed scratch
    ru = lambda x, a: -(-x // a) * a
    no_split = (3 * lq * HEADS * 256 + ru(8 * HEADS, 1024) + 2 * lh * HEADS * 256 + ru(lq * HEADS, 256)
                + ru(8 * HEADS, 256))
    assert need - no_split >= 2 * lq * HEADS * 129 * 4, (need, no_split)
    for step in (0, 1):
        q, k, v = current_inputs(tables, step)
        ref = torch.empty_like(q)
        ref_lse = torch.empty((HEADS, lq), dtype=torch.float32, device=DEV)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        nb.nomas_seg_attn(q, k, v, [0, lq], hist, ref, ref_lse, workspace=ws)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((HEADS, lq), float("nan"), dtype=torch.float32, device=DEV)
        nb.nomas_seg_attn_noalloc(q, k, v, [0, lq], hist, out, lse)
        nb.nomas_stream_check()
        assert_attn_close(bf16_to_f64(out), bf16_to_f64(ref), f"noalloc call {step + 1}")
        assert torch.allclose(lse, ref_lse, rtol=1e-5, atol=1e-5)


def test_noalloc_refuses_shapes_beyond_its_scratch(setup):
    heads, lq, lh = 16, 3776, 300_000
    need = nb.nomas_seg_attn_workspace_size(lq, lh, heads)
    assert need > nb.NOMAS_NOALLOC_SCRATCH_BYTES, need
    hist = nb.KVCache(heads, lh)
    hist.length = lh
    q = torch.zeros((lq, heads, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.full_like(q, 3.0)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_seg_attn_noalloc(q, q, q, [0, lq], hist, out)
    assert e.value.status == nb.NOMAS_ECAPACITY
    assert "scratch" in nb.nomas_last_error()
    nb.nomas_stream_check()
    assert torch.all(out == 3.0)                 # nothing launched, nothing written
    del hist
    torch.cuda.empty_cache()
