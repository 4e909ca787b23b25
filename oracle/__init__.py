"""CPU oracle for the segment-causal attention hot path (TEST INFRASTRUCTURE ONLY).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline / reference
arm may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or executes anything here, and this package never
imports the product.  The arithmetic lives in ``nomas_oracle.c`` (plain C,
float64 for attention, fp32-exact RoPE/quantisation as the method fixes it),
built with gcc on first use.

Every function is pinned by tests/test_oracle_pins.py against closed forms,
invariants, brute force in 50-digit arithmetic and the pages' constants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nomas_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libnomas_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile nomas_oracle.c with gcc (if missing or stale); returns the .so path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.orc_rope_table.argtypes = [f64, i32, i32, P, P]
            lib.orc_positions.argtypes = [i32, i32, i32, i32, i32, P]
            lib.orc_rope_bf16.argtypes = [P, P, i64, i32, i64, i32, P, P, f64]
            lib.orc_rope_f64.argtypes = [P, P, i64, i32, i32, P, P, f64]
            lib.orc_quantize_rows.argtypes = [P, i64, i32, P, P]
            lib.orc_append.argtypes = [P, P, i64, i64, i32, i32, P, P, f64, P, P, P, P, i64, i64]
            lib.orc_gather.argtypes = [P, P, P, P, i64, i32, i32, P, i32, P, i32, P, P, P, P, i64, P]
            lib.orc_seg_attn.argtypes = [i32, i32, P, P, P, i64, i64, P, i32, P, P, P, P, i64, i64,
                                         i32, f64, P, i64, P, P, i32]
            lib.orc_seg_attn.restype = ctypes.c_int
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = f64
            lib.orc_float_to_bf16.argtypes = [ctypes.c_float]
            lib.orc_float_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


HEAD_DIM = 128
SPLIT = np.array([16, 56, 56], dtype=np.int32)
THETA = 256.0


def num_threads() -> int:
    return int(_load().orc_num_threads())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    b = _c(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def rope_table(n_pos: int, d_axis: int, theta: float = THETA):
    cos = np.empty((n_pos, d_axis // 2), np.float32)
    sin = np.empty((n_pos, d_axis // 2), np.float32)
    _load().orc_rope_table(theta, d_axis, n_pos, _p(cos), _p(sin))
    return cos, sin


def positions(t0: int, T: int, gh: int, gw: int, n_text: int) -> np.ndarray:
    """[n_tok][3] int32 (t, h, w); text tokens are (-1, -1, -1)."""
    n = T * gh * gw + n_text
    pos = np.empty((max(n, 1), 3), np.int32)
    _load().orc_positions(t0, T, gh, gw, n_text, _p(pos))
    return pos[:n]


def segment_positions(seg) -> np.ndarray:
    return positions(seg.t0, seg.T, seg.grid_h, seg.grid_w, seg.n_text)


def rope_bf16(x_bits: np.ndarray, pos: np.ndarray, split=SPLIT, theta: float = THETA) -> np.ndarray:
    """x_bits: uint16 [n][heads][D] -> rotated uint16 [n][heads][D] (fp32 ops, no FMA, RNE to BF16)."""
    x = _c(x_bits, np.uint16)
    n, heads, d = x.shape
    y = np.empty_like(x)
    _load().orc_rope_bf16(_p(x), _p(y), n, heads, heads * d, d, _p(_c(pos, np.int32)),
                          _p(_c(split, np.int32)), theta)
    return y


def rope_f64(x: np.ndarray, pos: np.ndarray, split=SPLIT, theta: float = THETA) -> np.ndarray:
    x = _c(x, np.float64)
    n, heads, d = x.shape
    y = np.empty_like(x)
    _load().orc_rope_f64(_p(x), _p(y), n, heads, d, _p(_c(pos, np.int32)), _p(_c(split, np.int32)), theta)
    return y


def qkv_project(x_bits: np.ndarray, w_codes: np.ndarray, w_scale: np.ndarray) -> np.ndarray:
    """The QKV linear of a dual-stream block with INT8 weights and BF16 activations (comfyui-wiki
    news, 模型内部: hidden 2,048 = 16 heads x 128; 单张 4090 配置: DiT weights stored INT8, linear
    layers computed in BF16).  Output channel n has INT8 codes w_codes[n, :] and one fp32 scale
    w_scale[n]; y[l, n] = sum_k x[l, k] * w_codes[n, k] * w_scale[n], in float64 (a library
    matmul of the exact operands).  Channels [0, H*128), [H*128, 2H*128) and [2H*128, 3H*128) are
    Q, K and V, head-major inside each."""
    x = bf16_to_f64(x_bits)                                   # [L, hidden]
    w = _c(w_codes, np.int8).astype(np.float64) * _c(w_scale, np.float32).astype(np.float64)[:, None]
    return x @ w.T                                            # [L, 3*H*128]


def camera_tokens(c2w, translation_scale: float = 1.0, rotation_scale: float = 2.5) -> np.ndarray:
    """Camera tokens of a trajectory (comfyui-wiki news, 相机控制作为一等输入: camera-to-world
    matrices c2ws [N, 4, 4]; the extrinsics are normalised, grouped by four video frames and each
    group flattened to a 64-value input; trajectory_translation_scale 1.0 and
    trajectory_rotation_scale 2.5 by default).

    Readings (the page fixes none of these): normalising expresses every pose in the first
    frame's camera, E_i = inverse(c2w[0]) . c2w[i], with the rigid inverse [R0^T | -R0^T t0];
    the 3 x 3 rotation block of E_i is multiplied by rotation_scale and its translation column
    by translation_scale; the bottom row stays (0, 0, 0, 1); token g holds frames 4g .. 4g+3,
    each matrix row-major, in frame order.  The intrinsics are not part of the token.

    c2w: [N, 4, 4] (N a multiple of 4; the bottom rows are not read).  Returns float64
    [N / 4, 64]."""
    c = np.asarray(c2w, dtype=np.float64)
    if c.ndim != 3 or c.shape[1:] != (4, 4) or c.shape[0] % 4 != 0:
        raise ValueError("c2w must be [N, 4, 4] with N a multiple of 4")
    n = c.shape[0]
    r0, t0 = c[0, :3, :3], c[0, :3, 3]
    e = np.zeros((n, 4, 4), np.float64)
    for i in range(n):
        e[i, :3, :3] = rotation_scale * (r0.T @ c[i, :3, :3])
        e[i, :3, 3] = translation_scale * (r0.T @ (c[i, :3, 3] - t0))
        e[i, 3, 3] = 1.0
    return e.reshape(n // 4, 64)


def camera_cross_attn(q_bits, k_bits, v_bits, sm_scale: float = None, rows=None) -> np.ndarray:
    """Cross-attention from video tokens to the camera tokens of their segment, float64
    (comfyui-wiki news, 相机控制作为一等输入 and the 相机条件 row of the 模型内部 table: video
    tokens query the camera input through cross-attention in every dual-stream block;
    huaweicloud blog, 2.1: the camera path is a cross-attention apart from the text stream).

    Reading: every query attends to every camera token (no mask, no positions), per head,
    scale 1/sqrt(D) unless given: O = softmax(q k^T * scale) v.
    q_bits: uint16 BF16 [L][H][D]; k_bits, v_bits: uint16 BF16 [Tc][H][D].  Returns float64
    [L][H][D], or [len(rows)][H][D] for the selected query rows."""
    q = bf16_to_f64(q_bits)
    k = bf16_to_f64(k_bits)
    v = bf16_to_f64(v_bits)
    if q.ndim != 3 or k.shape != v.shape or k.shape[1:] != q.shape[1:] or k.shape[0] < 1:
        raise ValueError("q [L][H][D], k and v [Tc][H][D] with Tc >= 1")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(q.shape[2])
    if rows is not None:
        q = q[np.asarray(rows, np.int64)]
    out = np.empty(q.shape, np.float64)
    for a in range(0, q.shape[0], 2048):
        s = np.einsum("lhd,thd->lht", q[a:a + 2048], k) * sm_scale
        p = np.exp(s - s.max(axis=2, keepdims=True))
        p /= p.sum(axis=2, keepdims=True)
        out[a:a + 2048] = np.einsum("lht,thd->lhd", p, v)
    return out


def quantize_rows(x_bits: np.ndarray):
    """x_bits: uint16 [..., d] -> (int8 codes [..., d], float32 scales [...])."""
    x = _c(x_bits, np.uint16)
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    codes = np.empty(rows.shape, np.int8)
    scales = np.empty(rows.shape[0], np.float32)
    _load().orc_quantize_rows(_p(rows), rows.shape[0], d, _p(codes), _p(scales))
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])


class Cache:
    """Host INT8 KV cache, head-major: codes [heads][cap][D], scales [heads][cap]."""

    def __init__(self, heads: int, cap: int, head_dim: int = HEAD_DIM):
        self.heads, self.cap, self.head_dim = heads, cap, head_dim
        self.k = np.zeros((heads, cap, head_dim), np.int8)
        self.v = np.zeros((heads, cap, head_dim), np.int8)
        self.ks = np.zeros((heads, cap), np.float32)
        self.vs = np.zeros((heads, cap), np.float32)
        self.length = 0

    def append(self, k_bits: np.ndarray, v_bits: np.ndarray, pos: np.ndarray,
               split=SPLIT, theta: float = THETA) -> None:
        k = _c(k_bits, np.uint16)
        v = _c(v_bits, np.uint16)
        n, heads, d = k.shape
        assert heads == self.heads and d == self.head_dim and v.shape == k.shape
        if self.length + n > self.cap:
            raise ValueError("cache capacity exceeded")
        _load().orc_append(_p(k), _p(v), heads * d, n, heads, d, _p(_c(pos, np.int32)),
                           _p(_c(split, np.int32)), theta, _p(self.k), _p(self.v), _p(self.ks),
                           _p(self.vs), self.cap, self.length)
        self.length += n


def gather(archive: Cache, frame_token_offset, tokens_per_frame: int, frames):
    """Pack the selected frames into a new Cache; returns (cache, index_map int32)."""
    frames = _c(frames, np.int32)
    fto = _c(frame_token_offset, np.int32)
    n = len(frames) * tokens_per_frame
    dst = Cache(archive.heads, max(n, 1), archive.head_dim)
    idx = np.empty(max(n, 1), np.int32)
    _load().orc_gather(_p(archive.k), _p(archive.v), _p(archive.ks), _p(archive.vs), archive.cap,
                       archive.heads, archive.head_dim, _p(fto), tokens_per_frame, _p(frames),
                       len(frames), _p(dst.k), _p(dst.v), _p(dst.ks), _p(dst.vs), dst.cap, _p(idx))
    dst.length = n
    return dst, idx[:n]


def seg_attn(q_bits, k_bits, v_bits, seg_offsets, history: Cache = None, sm_scale: float = None,
             rows=None, key_parts: int = 3, threads: int = 0):
    """Float64 segment-causal attention.

    q_bits, k_bits, v_bits: uint16 [Lq][heads][D] (q, k already rotated).
    seg_offsets: [n_seg + 1] current-segment boundaries (0 ... Lq).
    Returns (out float64 [n_rows][heads][D], lse float64 [n_rows][heads])."""
    q = _c(q_bits, np.uint16)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    lq, heads, d = q.shape
    offs = _c(seg_offsets, np.int32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    if rows is None:
        rows_a = None
        n_rows = lq
    else:
        rows_a = _c(rows, np.int64)
        n_rows = len(rows_a)
    out = np.empty((max(n_rows, 1), heads, d), np.float64)
    lse = np.empty((max(n_rows, 1), heads), np.float64)
    if history is None:
        hk = hv = np.zeros((1,), np.int8)
        hks = hvs = np.zeros((1,), np.float32)
        hcap, lh = 0, 0
    else:
        hk, hv, hks, hvs, hcap, lh = history.k, history.v, history.ks, history.vs, history.cap, history.length
    rc = _load().orc_seg_attn(heads, d, _p(q), _p(k), _p(v), heads * d, lq, _p(offs), len(offs) - 1,
                              _p(hk), _p(hv), _p(hks), _p(hvs), hcap, lh, key_parts, float(sm_scale),
                              None if rows_a is None else _p(rows_a), n_rows, _p(out), _p(lse), threads)
    if rc != 0:
        raise ValueError("oracle seg_attn: invalid arguments")
    return out[:n_rows], lse[:n_rows]
