"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds *no* arithmetic of the method (no RoPE, no quantisation, no
attention).  It only defines the workload shapes of the five configurations and
draws the random numbers both sides consume:

* BF16 ~ N(0, 1) tensors: ``torch.randn`` in fp32 from a seeded CPU generator,
  rounded once to BF16 (round-to-nearest-even by ``Tensor.to``).
* the temporal_context frame selection of the gather workload (6 most recent
  frames + 12 stratified older frames, offsets from splitmix64),
* the 1 % outlier (head, channel) pairs of the lifelong-cache workload.

Shapes follow the Hy-Nomas pages: 16 heads x 128 (architecture table,
comfyui-wiki "模型内部"), 880 tokens per 704x1280 latent frame (22 x 40 after
32x spatial compression of DCAE-V f32t4c32, same table), an 18-frame
temporal_context budget (same page, "单张 4090 配置"), context up to 360K
tokens (huaweicloud blog, spec table).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np
import torch

HEAD_DIM = 128
ROPE_SPLIT = (16, 56, 56)   # (t, h, w) channel split of the head dim
ROPE_THETA = 256.0
GRID_H, GRID_W = 22, 40     # 704/32 x 1280/32
TOKENS_PER_FRAME = GRID_H * GRID_W  # 880
TEXT_TOKENS = 256


# --------------------------------------------------------------------------
# random sources
# --------------------------------------------------------------------------
MASK64 = (1 << 64) - 1


def splitmix64(state: int) -> Tuple[int, int]:
    """One step of splitmix64 (Steele, Lea & Flood 2014; Vigna's constants).

    Returns (new_state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return state, z ^ (z >> 31)


def seed_of(config: int, tensor: int, seg: int = 0, step: int = 0) -> int:
    """Deterministic seed for one tensor of one workload."""
    return 1_000_000 * config + 10_000 * tensor + 100 * seg + step


T_Q, T_K, T_V, T_HK, T_HV, T_OUTLIER, T_FRAMES, T_MISC = 1, 2, 3, 4, 5, 6, 7, 8


def bf16_normal(shape, seed: int) -> torch.Tensor:
    """BF16 N(0,1) CPU tensor: fp32 randn from a seeded generator, rounded to BF16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 view of a contiguous BF16 CPU tensor (what the oracle consumes)."""
    t = t.contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def outlier_pairs(heads: int, seed: int, frac: float = 0.01) -> List[Tuple[int, int]]:
    """1 % of the (head, channel) pairs, drawn without replacement (seeded)."""
    n = int(heads * HEAD_DIM * frac)
    rng = np.random.default_rng(seed)
    flat = rng.choice(heads * HEAD_DIM, size=n, replace=False)
    return sorted((int(f) // HEAD_DIM, int(f) % HEAD_DIM) for f in flat)


def apply_outliers(k: torch.Tensor, pairs, factor: float = 8.0) -> torch.Tensor:
    """Scale the chosen (head, channel) columns of a [L][H][128] BF16 tensor.

    A power-of-two factor keeps every value exactly representable in BF16."""
    k = k.clone()
    for h, c in pairs:
        k[:, h, c] = k[:, h, c] * factor
    return k


def select_frames(n_archive_frames: int, seed: int, n_recent: int = 6,
                  n_strided: int = 12) -> List[int]:
    """temporal_context selection used by the gather workload.

    The n_recent most recent frames plus one frame from each of n_strided equal
    strata of the older frames, [floor(j*N/n), floor((j+1)*N/n)), the offset in a
    stratum drawn from splitmix64.  Returned sorted ascending."""
    older = n_archive_frames - n_recent
    picks = []
    state = seed & MASK64
    for j in range(n_strided):
        lo = (j * older) // n_strided
        hi = ((j + 1) * older) // n_strided
        state, r = splitmix64(state)
        picks.append(lo + (r % (hi - lo)))
    picks += list(range(older, n_archive_frames))
    return sorted(picks)


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Segment:
    """Video tokens (t, h, w) in row-major order, then n_text unrotated text tokens."""
    t0: int
    T: int
    grid_h: int
    grid_w: int
    n_text: int

    @property
    def n_video(self) -> int:
        return self.T * self.grid_h * self.grid_w

    @property
    def n_tokens(self) -> int:
        return self.n_video + self.n_text


@dataclass
class Workload:
    name: str
    config: int
    heads: int
    history: List[Segment]          # appended to the INT8 cache, in order
    current: List[Segment]          # the segment(s) being denoised (one attention call)
    steps: int = 1                  # Euler steps (fresh Q/K/V each step)
    outliers: bool = False          # x8 on 1 % of K (head, channel) pairs before RoPE
    archive_frames: int = 0         # gather workload: archive size in frames
    gather: List[int] = field(default_factory=list)

    @property
    def lq(self) -> int:
        return sum(s.n_tokens for s in self.current)

    @property
    def lh(self) -> int:
        if self.archive_frames:
            return len(self.gather) * TOKENS_PER_FRAME
        return sum(s.n_tokens for s in self.history)

    def attn_flops(self) -> float:
        """4*D*H*sum over visible (query, key) pairs (QK^T and PV)."""
        offs = [0]
        for s in self.current:
            offs.append(offs[-1] + s.n_tokens)
        vis = 0
        for i in range(len(self.current)):
            vis += (offs[i + 1] - offs[i]) * (self.lh + offs[i + 1])
        return 4.0 * HEAD_DIM * self.heads * vis


def _frames_then_partial(t0: int, n_tokens: int) -> List[Segment]:
    """History token i at t = t0 + i // 880, (h, w) from i mod 880 (whole rows)."""
    full, rem = divmod(n_tokens, TOKENS_PER_FRAME)
    segs = []
    if full:
        segs.append(Segment(t0, full, GRID_H, GRID_W, 0))
    if rem:
        assert rem % GRID_W == 0, "partial frame must be whole latent rows"
        segs.append(Segment(t0 + full, 1, rem // GRID_W, GRID_W, 0))
    return segs


def config1() -> Workload:
    seg0 = Segment(0, 2, 4, 6, 8)
    seg1 = Segment(2, 2, 4, 6, 8)
    return Workload("tiny: 2 segments of 2x4x6 video + 8 text, 2 heads", 1, 2, [seg0], [seg1])


def config1_two_segments() -> Workload:
    """Same tiny shapes, both segments current: exercises the segment-causal mask."""
    seg0 = Segment(0, 2, 4, 6, 8)
    seg1 = Segment(2, 2, 4, 6, 8)
    return Workload("tiny causal: segments 0 and 1 current, empty history", 1, 2, [], [seg0, seg1])


def config2() -> Workload:
    hist = [Segment(0, 18, GRID_H, GRID_W, 0)]
    cur = [Segment(18, 18, GRID_H, GRID_W, TEXT_TOKENS)]
    return Workload("704x1280 segment, 18-frame history, 8 Euler steps", 2, 16, hist, cur, steps=8)


def config3() -> Workload:
    hist = [Segment(72 * s, 72, GRID_H, GRID_W, TEXT_TOKENS) for s in range(4)]
    cur = [Segment(288, 72, GRID_H, GRID_W, TEXT_TOKENS)]
    return Workload("lifelong cache, turn 5 of five 12-s turns", 3, 16, hist, cur, outliers=True)


def config4(seed: int = None) -> Workload:
    seed = seed_of(4, T_FRAMES) if seed is None else seed
    frames = select_frames(240, seed)
    cur = [Segment(240, 24, GRID_H, GRID_W, TEXT_TOKENS)]
    return Workload("temporal_context gather (18 of 240 frames) + 4-s segment", 4, 16, [], cur,
                    archive_frames=240, gather=frames)


SWEEP_LH = (0, 8_000, 32_000, 100_000, 200_000, 300_000)
SWEEP_T = (4, 24, 72)   # 3,520 / 21,120 / 63,360 video tokens


def config5(lh: int, T: int) -> Workload:
    hist = _frames_then_partial(0, lh)
    t0 = -(-lh // TOKENS_PER_FRAME)
    cur = [Segment(t0, T, GRID_H, GRID_W, TEXT_TOKENS)]
    return Workload(f"sweep Lh={lh} T={T}", 5, 16, hist, cur)


def packed(n_seg: int, T: int) -> Workload:
    """Packed multi-segment forward: n_seg consecutive segments of T frames (+ text), all in one
    attention call with the segment-causal mask, no cached history."""
    cur = [Segment(s * T, T, GRID_H, GRID_W, TEXT_TOKENS) for s in range(n_seg)]
    return Workload(f"packed forward: {n_seg} segments of {T} frames in one call", 6, 16, [], cur)


VIDEO_FRAMES_PER_LATENT = 4   # DCAE-V f32t4c32: 4x temporal compression
T_CAMERA = 9


def camera_trajectory(n_frames: int, seed: int) -> np.ndarray:
    """A seeded, smooth synthetic camera path: float32 camera-to-world matrices [n_frames][4][4].

    The camera yaws by a drifting angle per frame, pitches a little, and moves forward along its
    heading with seeded jitter (a walk through a generated world, as with WASD and the mouse).
    Only the input is drawn here; the normalisation and grouping of the method live in the
    library and the oracle."""
    g = np.random.default_rng(seed)
    yaw_rate = g.uniform(-0.02, 0.02)
    yaw, pitch = g.uniform(-np.pi, np.pi), 0.0
    pos = g.normal(0.0, 2.0, 3)
    out = np.zeros((n_frames, 4, 4), np.float32)
    for i in range(n_frames):
        yaw += yaw_rate + g.normal(0.0, 0.004)
        pitch = float(np.clip(pitch + g.normal(0.0, 0.003), -0.3, 0.3))
        cy, sy, cp, sp = np.cos(yaw), np.sin(yaw), np.cos(pitch), np.sin(pitch)
        r = np.array([[cy, 0.0, sy], [0.0, 1.0, 0.0], [-sy, 0.0, cy]]) @ \
            np.array([[1.0, 0.0, 0.0], [0.0, cp, -sp], [0.0, sp, cp]])
        pos = pos + r[:, 2] * 0.05 + g.normal(0.0, 0.005, 3)
        out[i, :3, :3] = r
        out[i, :3, 3] = pos
        out[i, 3, 3] = 1.0
    return out


def camera_workload(w: Workload):
    """The camera cross-attention of a workload's (last) current segment: (video frames of the
    trajectory, camera tokens, video-token queries).  One camera token per four video frames,
    i.e. one per latent frame."""
    seg = w.current[-1]
    return seg.T * VIDEO_FRAMES_PER_LATENT, seg.T, seg.n_video


def max_t(w: Workload) -> int:
    ts = [s.t0 + s.T for s in w.history + w.current]
    if w.archive_frames:
        ts.append(w.archive_frames)
    return max(ts)
