"""Shared workload construction for the GPU parity tests (and smoke()).

Both sides start from the same seeded BF16 host tensors (nomas_synth).  The CUDA side runs
them through the C ABI (segment_causal_attention_nomas_b300); the oracle side through the
CPU oracle.  Nothing produced by the CUDA path ever feeds the oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import nomas_synth as ns

ATTN_MAX_ABS_REL = 1e-2     # max |gpu - oracle| <= 1e-2 * max |oracle|
ATTN_MEAN_REL = 2e-3        # sum |gpu - oracle| / sum |oracle| <= 2e-3


def seg_offsets(segs):
    offs = [0]
    for s in segs:
        offs.append(offs[-1] + s.n_tokens)
    return np.array(offs, np.int32)


def segment_kv(cfg: int, seg_index: int, seg: ns.Segment, heads: int, outliers=None, tensor_k=ns.T_HK,
               tensor_v=ns.T_HV, step: int = 0):
    """Seeded BF16 K and V [n][heads][128] for one segment (outlier columns x8 on K)."""
    k = ns.bf16_normal((seg.n_tokens, heads, 128), ns.seed_of(cfg, tensor_k, seg_index, step))
    v = ns.bf16_normal((seg.n_tokens, heads, 128), ns.seed_of(cfg, tensor_v, seg_index, step))
    if outliers:
        k = ns.apply_outliers(k, outliers)
    return k, v


def current_qkv(w: ns.Workload, step: int = 0, outliers=None):
    """Seeded BF16 Q, K, V [Lq][heads][128] of the current segment(s), before RoPE."""
    q = ns.bf16_normal((w.lq, w.heads, 128), ns.seed_of(w.config, ns.T_Q, 0, step))
    k = ns.bf16_normal((w.lq, w.heads, 128), ns.seed_of(w.config, ns.T_K, 0, step))
    v = ns.bf16_normal((w.lq, w.heads, 128), ns.seed_of(w.config, ns.T_V, 0, step))
    if outliers:
        k = ns.apply_outliers(k, outliers)
    return q, k, v


def workload_outliers(w: ns.Workload):
    return ns.outlier_pairs(w.heads, ns.seed_of(w.config, ns.T_OUTLIER)) if w.outliers else None


ARCHIVE_CHUNK_FRAMES = 24


def archive_chunks(w: ns.Workload):
    """The gather workload's archive: frames [0, archive_frames) as 24-frame segments."""
    segs = []
    for c in range(0, w.archive_frames, ARCHIVE_CHUNK_FRAMES):
        segs.append(ns.Segment(c, min(ARCHIVE_CHUNK_FRAMES, w.archive_frames - c), ns.GRID_H, ns.GRID_W, 0))
    return segs


def sample_rows(lq: int, n: int, segs=None):
    """n query rows strided uniformly over [0, lq), including the first and last, plus the
    first and last rows of every segment (segment boundaries, text tokens)."""
    rows = set(np.linspace(0, lq - 1, num=min(n, lq)).round().astype(int).tolist())
    if segs is not None:
        offs = seg_offsets(segs)
        for a, b in zip(offs[:-1], offs[1:]):
            if b > a:
                rows.update([int(a), int(b) - 1])
    return np.array(sorted(rows), np.int64)


def attn_errors(gpu: np.ndarray, ref: np.ndarray):
    err = np.abs(gpu.astype(np.float64) - ref)
    max_abs_rel = float(err.max() / max(np.abs(ref).max(), 1e-300))
    mean_rel = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    return max_abs_rel, mean_rel


def assert_attn_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    mx, mean = attn_errors(gpu, ref)
    assert mx <= ATTN_MAX_ABS_REL and mean <= ATTN_MEAN_REL, f"{what}: max_abs_rel {mx:.3e} mean_rel {mean:.3e}"
    return mx, mean


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def default_scale() -> float:
    return 1.0 / math.sqrt(128)
