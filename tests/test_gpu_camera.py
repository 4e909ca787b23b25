"""GPU parity of the camera conditioning path: nomas_camera_tokens and nomas_camera_cross_attn.

Bars:
* camera tokens: every entry within a forward error bound of the fp32 evaluation (each entry is
  a three-term dot product times a scale: |err| <= 8u * scale * sum of |terms|, u = 2^-24), the
  constant bottom rows exact, exact results where every product is exact;
* cross-attention: the attention tolerance against the float64 oracle (max |gpu - oracle| <=
  1e-2 * max |oracle|, mean relative error <= 2e-3), exact where the method is (one camera
  token).
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
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from segment_causal_attention_nomas_b300 import build
    build.build()


def gpu_tokens(c2w: np.ndarray, ts=1.0, rs=2.5) -> np.ndarray:
    c = torch.from_numpy(np.ascontiguousarray(c2w, np.float32)).to(DEV)
    out = torch.full((c.shape[0] // 4, 64), float("nan"), dtype=torch.float32, device=DEV)
    nb.nomas_camera_tokens(c, out, ts, rs)
    nb.nomas_stream_check()
    return out.cpu().numpy().astype(np.float64)


def token_bound(c2w: np.ndarray, ts: float, rs: float) -> np.ndarray:
    """8u * |scale| * (sum of |terms|) per entry, float64, laid out like the tokens."""
    c = np.asarray(c2w, np.float64)
    r0, t0 = np.abs(c[0, :3, :3]), np.abs(c[0, :3, 3])
    b = np.zeros((c.shape[0], 4, 4))
    for i in range(c.shape[0]):
        b[i, :3, :3] = 8 * U * abs(rs) * (r0.T @ np.abs(c[i, :3, :3]))
        b[i, :3, 3] = 8 * U * abs(ts) * (r0.T @ (np.abs(c[i, :3, 3]) + t0))
    return b.reshape(-1, 64)


@pytest.mark.parametrize("n_frames,ts,rs", [(72, 1.0, 2.5), (288, 1.0, 2.5), (4, 1.0, 2.5), (96, 0.7, 1.3)])
def test_camera_tokens_match_oracle(n_frames, ts, rs):
    c2w = ns.camera_trajectory(n_frames, ns.seed_of(2, ns.T_CAMERA, step=n_frames))
    got = gpu_tokens(c2w, ts, rs)
    want = oracle.camera_tokens(c2w, ts, rs)
    assert got.shape == want.shape == (n_frames // 4, 64)
    err = np.abs(got - want)
    bound = token_bound(c2w, ts, rs)
    assert np.all(err <= bound), f"worst excess {np.max(err - bound):.3e}"
    bottom = got.reshape(-1, 4, 4, 4)[:, :, 3, :]
    assert np.array_equal(bottom, np.broadcast_to([0.0, 0.0, 0.0, 1.0], bottom.shape))


def test_camera_tokens_worked_example_is_exact():
    # poses whose products are all exact in fp32: the GPU must reproduce the hand-derived tokens
    r0 = np.array([[0.0, -1.0, 0.0], [1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    poses = []
    for r, t in ((r0, (1, 2, 3)), (np.eye(3), (0, 0, 0)), (r0, (1, 2, 4)), (r0, (2, 2, 3))):
        m = np.eye(4)
        m[:3, :3], m[:3, 3] = r, t
        poses.append(m)
    c2w = np.stack(poses)
    assert np.array_equal(gpu_tokens(c2w), oracle.camera_tokens(c2w))
    assert np.array_equal(gpu_tokens(c2w, 2.0, 1.0), oracle.camera_tokens(c2w, 2.0, 1.0))


def test_camera_tokens_rejects_bad_arguments():
    c = torch.eye(4, device=DEV).repeat(8, 1, 1)
    out = torch.full((2, 64), 7.0, device=DEV)
    with pytest.raises(nb.NomasError) as e:                   # not a multiple of 4 frames
        nb._check(nb.lib().nomas_camera_tokens(c.data_ptr(), 6, 1.0, 2.5, out.data_ptr(), None), "t")
    assert e.value.status == nb.NOMAS_EINVAL
    with pytest.raises(nb.NomasError) as e:                   # non-finite scale
        nb.nomas_camera_tokens(c, out, float("inf"), 2.5)
    assert e.value.status == nb.NOMAS_EINVAL
    with pytest.raises(nb.NomasError) as e:                   # tokens overlapping c2w
        nb._check(nb.lib().nomas_camera_tokens(c.data_ptr(), 8, 1.0, 2.5, c.data_ptr() + 64, None), "t")
    assert e.value.status == nb.NOMAS_EINVAL
    nb.nomas_stream_check()
    assert torch.all(out == 7.0)                              # nothing written


# ------------------------------------------------------------------- cross-attention
def problem(lq, heads, n_cam, seed):
    q = ns.bf16_normal((lq, heads, 128), seed)
    k = ns.bf16_normal((n_cam, heads, 128), seed + 1)
    v = ns.bf16_normal((n_cam, heads, 128), seed + 2)
    return q, k, v


def run_xattn(q, k, v, scale=0.0):
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    nb.nomas_camera_cross_attn(q.to(DEV), k.to(DEV), v.to(DEV), out, scale)
    nb.nomas_stream_check()
    return out.cpu()


@pytest.mark.parametrize("cfg", [2, 4])
def test_camera_xattn_config_shapes_full(cfg):
    w = ns.config2() if cfg == 2 else ns.config4()
    _, n_cam, lq = ns.camera_workload(w)                       # 18 or 24 camera tokens
    q, k, v = problem(lq, w.heads, n_cam, ns.seed_of(cfg, ns.T_CAMERA))
    got = bf16_to_f64(run_xattn(q, k, v))
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(got, want, f"camera cross-attention, config {cfg}")


def test_camera_xattn_config3_sampled_rows():
    w = ns.config3()
    _, n_cam, lq = ns.camera_workload(w)                       # 72 camera tokens, 63,360 queries
    q, k, v = problem(lq, w.heads, n_cam, ns.seed_of(3, ns.T_CAMERA))
    got = run_xattn(q, k, v)
    rows = np.unique(np.concatenate([np.arange(0, lq, 31), np.arange(lq - 130, lq)]))
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v), rows=rows)
    assert_attn_close(bf16_to_f64(got[rows]), want, "camera cross-attention, config 3 rows")


@pytest.mark.parametrize("lq,heads,n_cam", [
    (1, 1, 1),          # one query, one camera token
    (130, 2, 5),        # a ragged second tile
    (300, 3, 32),       # exactly one 32-column S block
    (257, 2, 33),       # 64 padded columns, one real past the first block
    (129, 1, 97),       # 128 padded columns
    (200, 2, 128),      # the maximum
    (130, 150, 40),     # more heads than SMs: persistent CTAs run across head boundaries
    (260, 300, 72),     #   (K and V reloaded, V converted once per head)
    (130, 300, 18),     #   the same with 32 columns
])
def test_camera_xattn_small_shapes(lq, heads, n_cam):
    q, k, v = problem(lq, heads, n_cam, 7000 + lq + n_cam)
    got = bf16_to_f64(run_xattn(q, k, v))
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(got, want, f"camera cross-attention lq {lq} heads {heads} n_cam {n_cam}")


def test_camera_xattn_special_cases():
    # one camera token: softmax weight exactly 1, so out = v bit for bit
    q, k, v = problem(260, 2, 1, 7100)
    assert torch.equal(run_xattn(q, k, v), v.expand(260, 2, 128).contiguous())
    # zero queries and a zero scale both give the mean of V
    q, k, v = problem(140, 2, 9, 7101)
    want = oracle.camera_cross_attn(ns.bf16_bits(torch.zeros_like(q)), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(bf16_to_f64(run_xattn(torch.zeros_like(q), k, v)), want, "zero queries")
    got = bf16_to_f64(run_xattn(q, k, v, scale=1e-30))
    assert_attn_close(got, want, "vanishing scale")
    # an explicit scale
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v), sm_scale=0.25)
    assert_attn_close(bf16_to_f64(run_xattn(q, k, v, scale=0.25)), want, "scale 0.25")


def test_camera_xattn_in_place_on_a_fused_buffer():
    # queries as one slice of a fused [L][3][H][128] tensor, the output written over them
    lq, heads, n_cam = 777, 4, 20
    fused = ns.bf16_normal((lq, 3, heads, 128), 7200).to(DEV)
    k = ns.bf16_normal((n_cam, heads, 128), 7201)
    v = ns.bf16_normal((n_cam, heads, 128), 7202)
    q_host = fused[:, 1].cpu()
    rest = fused[:, [0, 2]].clone()
    nb.nomas_camera_cross_attn(fused[:, 1], k.to(DEV), v.to(DEV), fused[:, 1])
    nb.nomas_stream_check()
    want = oracle.camera_cross_attn(ns.bf16_bits(q_host), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(bf16_to_f64(fused[:, 1].cpu()), want, "in place, strided")
    assert torch.equal(fused[:, [0, 2]], rest)                 # the neighbouring slices untouched


def test_camera_xattn_rejects_bad_arguments():
    q = torch.zeros((4, 2, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.full((4, 2, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    big = torch.zeros((129, 2, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_camera_cross_attn(q, big, big, out)           # 129 camera tokens
    assert e.value.status == nb.NOMAS_EUNSUPPORTED
    none = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_camera_cross_attn(q, none, none, out)         # no camera token
    assert e.value.status == nb.NOMAS_EINVAL
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_camera_cross_attn(q, big[:3], big[:3], out, softmax_scale=-1.0)
    assert e.value.status == nb.NOMAS_EINVAL
    nb.nomas_stream_check()
    assert torch.all(out == 5.0)                               # nothing written


def _scaled(t, f):
    return (t.float() * f).to(torch.bfloat16)


@pytest.mark.parametrize("lq,heads,n_cam", [(300, 3, 18), (260, 20, 72)])      # 32 and 96 columns
@pytest.mark.parametrize("eq,ek,ev", [(17, 17, 17), (-20, -20, -20), (0, 0, 20), (5, -5, -30)])
def test_camera_xattn_over_the_bf16_range(lq, heads, n_cam, eq, ek, ev):
    # Q, K, V times 2^eq, 2^ek, 2^ev (exact in BF16): V beyond FP16's largest value or below its
    # normal range is scaled into range by a power of two per head and scaled back exactly; heads
    # get different magnitudes of V (x 2^(4h mod 24)) so each head's own exponent matters
    q, k, v = problem(lq, heads, n_cam, 7300 + lq + n_cam)
    head_f = torch.from_numpy(np.ldexp(1.0, (4 * np.arange(heads)) % 24).astype(np.float32)).view(1, heads, 1)
    q, k, v = _scaled(q, 2.0 ** eq), _scaled(k, 2.0 ** ek), _scaled(v, head_f * 2.0 ** ev)
    got = bf16_to_f64(run_xattn(q, k, v))
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(got, want, f"camera cross-attention at 2^({eq}, {ek}, {ev})")


def test_camera_xattn_score_overflow_is_reported():
    # q . k beyond the fp32 range (both near 2^100): NOMAS_ERANGE instead of a result, then the
    # next call is unaffected
    q, k, v = problem(140, 2, 9, 7400)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=DEV)
    nb.nomas_camera_cross_attn(_scaled(q, 2.0 ** 100).to(DEV), _scaled(k, 2.0 ** 100).to(DEV), v.to(DEV), out)
    with pytest.raises(nb.NomasError) as e:
        nb.nomas_stream_check()
    assert e.value.status == nb.NOMAS_ERANGE
    got = bf16_to_f64(run_xattn(q, k, v))
    want = oracle.camera_cross_attn(ns.bf16_bits(q), ns.bf16_bits(k), ns.bf16_bits(v))
    assert_attn_close(got, want, "after a range report")
