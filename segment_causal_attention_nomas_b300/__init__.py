"""Python binding of libnomas: the B300 (sm_103a) segment-causal attention hot path.

Argument marshalling only.  Every step of the path runs in the CUDA kernels of
``libnomas.so`` behind the C ABI declared in ``include/nomas.h``; the functions here carry
the same names as the C entry points.  PyTorch supplies device memory and streams.  There
is no CPU fallback: if the library is missing or a call fails, a ``NomasError`` is raised.

Build the library with ``python -m segment_causal_attention_nomas_b300.build``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnomas.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "nomas.h")
HEAD_DIM = 128

NOMAS_OK, NOMAS_EINVAL, NOMAS_ECAPACITY, NOMAS_EUNSUPPORTED, NOMAS_ECUDA, NOMAS_ETIMEOUT, NOMAS_ERANGE = range(7)


class NomasError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status


class nomas_segment(ctypes.Structure):
    _fields_ = [("t0", ctypes.c_int32), ("T", ctypes.c_int32), ("grid_h", ctypes.c_int32),
                ("grid_w", ctypes.c_int32), ("n_text", ctypes.c_int32)]


class nomas_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("capacity", ctypes.c_int64), ("length", ctypes.c_int64),
                ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class nomas_staged_history(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("bytes", ctypes.c_size_t), ("capacity", ctypes.c_int64),
                ("length", ctypes.c_int64), ("heads", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libnomas (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libnomas.so is not built ({LIB_PATH}); run "
                                  "`python -m segment_causal_attention_nomas_b300.build`")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            st = ctypes.c_int
            SEG = ctypes.POINTER(nomas_segment)
            KV = ctypes.POINTER(nomas_kv_cache)
            SH = ctypes.POINTER(nomas_staged_history)
            sz = ctypes.c_size_t
            sig = {
                "nomas_rope_tables_create": (st, [f32, P, i32, i32, i32, ctypes.POINTER(P)]),
                "nomas_rope_tables_destroy": (None, [P]),
                "nomas_rope_tables_read": (st, [P, i32, P, P]),
                "nomas_rope3d": (st, [P, P, i64, SEG, i32, P, P]),
                "nomas_kv_append_quant": (st, [KV, P, P, i64, SEG, P, P]),
                "nomas_kv_gather_context": (st, [KV, P, i32, i32, P, i32, KV, P, P]),
                "nomas_kv_gather_context_host": (st, [KV, P, i32, i32, P, i32, KV, P, P]),
                "nomas_seg_attn": (st, [P, P, P, i64, i32, P, i32, KV, f32, P, P, P, ctypes.c_size_t, P]),
                "nomas_seg_attn_workspace_size": (ctypes.c_size_t, [i64, i64, i32]),
                "nomas_staged_history_size": (sz, [i64, i32]),
                "nomas_seg_attn_stage_history": (st, [KV, SH, P]),
                "nomas_seg_attn_staged": (st, [P, P, P, i64, i32, P, i32, SH, f32, P, P, P, sz, P]),
                "nomas_seg_attn_staged_workspace_size": (sz, [i64, i64, i32]),
                "nomas_qkv_project_rope": (st, [P, i64, i32, P, P, i32, SEG, P, P, i64, P, ctypes.c_size_t, P]),
                "nomas_qkv_project_workspace_size": (ctypes.c_size_t, [i32, i32]),
                "nomas_qkv_project_rope_append": (st, [P, i64, i32, P, P, i32, SEG, P, P, i64, P, ctypes.c_size_t, KV,
                                                       P]),
                "nomas_camera_tokens": (st, [P, i32, f32, f32, P, P]),
                "nomas_camera_cross_attn": (st, [P, i64, i32, i32, P, P, i64, i32, f32, P, i64, P]),
                "nomas_seg_attn_noalloc": (st, [P, P, P, i64, i32, P, i32, KV, f32, P, P, P]),
                "nomas_stream_check": (st, [P]),
                "nomas_status_string": (ctypes.c_char_p, [st]),
                "nomas_last_error": (ctypes.c_char_p, []),
                "nomas_version": (ctypes.c_char_p, []),
                "nomas_debug_inject": (None, [i32]),
                "nomas_debug_attn_variant": (None, [i32]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def declared_entry_points() -> list:
    """Function names declared in include/nomas.h (for the export check)."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nomas_\w+)\s*\(", text)))


def _check(status: int, where: str) -> None:
    if status != NOMAS_OK:
        msg = lib().nomas_last_error().decode(errors="replace")
        raise NomasError(status, where, msg)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _seg(seg) -> nomas_segment:
    if isinstance(seg, nomas_segment):
        return seg
    return nomas_segment(seg.t0, seg.T, seg.grid_h, seg.grid_w, seg.n_text)


def _tok_tensor(x: torch.Tensor, heads: Optional[int], what: str) -> int:
    """Checks a [L][H][128] BF16 device tensor with unit inner strides; returns its token stride."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 3 or x.shape[2] != HEAD_DIM:
        raise ValueError(f"{what}: expected a CUDA bf16 tensor [L][H][128], got {tuple(x.shape)} {x.dtype}")
    if heads is not None and x.shape[1] != heads:
        raise ValueError(f"{what}: {x.shape[1]} heads, expected {heads}")
    if x.stride(2) != 1 or x.stride(1) != HEAD_DIM:
        raise ValueError(f"{what}: channels and heads must be contiguous")
    return x.stride(0)


def nomas_version() -> str:
    return lib().nomas_version().decode()


def nomas_status_string(status: int) -> str:
    return lib().nomas_status_string(status).decode()


def nomas_last_error() -> str:
    return lib().nomas_last_error().decode()


def nomas_debug_inject(what: int) -> None:
    lib().nomas_debug_inject(int(what))


def nomas_debug_attn_variant(variant: int) -> None:
    """Test hook: 1 the single-CTA attention kernel, 2 the CTA-pair one, 0 chosen by shape."""
    lib().nomas_debug_attn_variant(int(variant))


class RopeTables:
    """Owns a nomas_rope_tables handle (device cos/sin tables)."""

    def __init__(self, handle: int, split, max_pos):
        self.handle = ctypes.c_void_p(handle)
        self.split = tuple(split)
        self.max_pos = tuple(max_pos)

    def close(self) -> None:
        if self.handle and self.handle.value:
            lib().nomas_rope_tables_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def nomas_rope_tables_create(theta: float = 256.0, split=(16, 56, 56), max_t: int = 512, max_h: int = 64,
                             max_w: int = 64) -> RopeTables:
    sp = (ctypes.c_int32 * 3)(*split)
    out = ctypes.c_void_p()
    _check(lib().nomas_rope_tables_create(float(theta), sp, max_t, max_h, max_w, ctypes.byref(out)),
           "nomas_rope_tables_create")
    return RopeTables(out.value, split, (max_t, max_h, max_w))


def nomas_rope_tables_read(tables: RopeTables, axis: int):
    n = tables.max_pos[axis] * (tables.split[axis] // 2)
    cos = np.empty(n, np.float32)
    sin = np.empty(n, np.float32)
    _check(lib().nomas_rope_tables_read(tables.handle, axis, cos.ctypes.data, sin.ctypes.data),
           "nomas_rope_tables_read")
    return cos.reshape(tables.max_pos[axis], -1), sin.reshape(tables.max_pos[axis], -1)


def nomas_rope3d(x: torch.Tensor, y: torch.Tensor, seg, tables: RopeTables, stream=None) -> None:
    """y = RoPE(x) for one segment's tokens (y may be x)."""
    rs = _tok_tensor(x, None, "x")
    if _tok_tensor(y, x.shape[1], "y") != rs or y.shape[0] != x.shape[0]:
        raise ValueError("y must have the shape and token stride of x")
    s = _seg(seg)
    if x.shape[0] != s.T * s.grid_h * s.grid_w + s.n_text:
        raise ValueError("x rows != segment tokens")
    _check(lib().nomas_rope3d(x.data_ptr(), y.data_ptr(), rs, ctypes.byref(s), x.shape[1], tables.handle,
                              _stream(stream)), "nomas_rope3d")


class KVCache:
    """An INT8 KV cache in device memory (torch-allocated), head-major."""

    def __init__(self, heads: int, capacity: int, device="cuda"):
        capacity = (int(capacity) + 3) // 4 * 4
        self.k = torch.zeros((heads, capacity, HEAD_DIM), dtype=torch.int8, device=device)
        self.v = torch.zeros((heads, capacity, HEAD_DIM), dtype=torch.int8, device=device)
        self.k_scale = torch.zeros((heads, capacity), dtype=torch.float32, device=device)
        self.v_scale = torch.zeros((heads, capacity), dtype=torch.float32, device=device)
        self.c = nomas_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.k_scale.data_ptr(),
                                self.v_scale.data_ptr(), capacity, 0, heads, HEAD_DIM)

    @property
    def heads(self) -> int:
        return self.c.heads

    @property
    def capacity(self) -> int:
        return self.c.capacity

    @property
    def length(self) -> int:
        return self.c.length

    @length.setter
    def length(self, n: int) -> None:
        self.c.length = int(n)


class HostKVCache(KVCache):
    """An INT8 KV cache in pinned host memory (the archive of nomas_kv_gather_context_host)."""

    def __init__(self, heads: int, capacity: int):
        capacity = (int(capacity) + 3) // 4 * 4
        self.k = torch.zeros((heads, capacity, HEAD_DIM), dtype=torch.int8).pin_memory()
        self.v = torch.zeros((heads, capacity, HEAD_DIM), dtype=torch.int8).pin_memory()
        self.k_scale = torch.zeros((heads, capacity), dtype=torch.float32).pin_memory()
        self.v_scale = torch.zeros((heads, capacity), dtype=torch.float32).pin_memory()
        self.c = nomas_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.k_scale.data_ptr(),
                                self.v_scale.data_ptr(), capacity, 0, heads, HEAD_DIM)

    @classmethod
    def from_device(cls, cache: KVCache) -> "HostKVCache":
        """A pinned host copy of a device cache (codes, scales and length)."""
        h = cls(cache.heads, cache.capacity)
        h.k.copy_(cache.k)
        h.v.copy_(cache.v)
        h.k_scale.copy_(cache.k_scale)
        h.v_scale.copy_(cache.v_scale)
        h.length = cache.length
        return h


def nomas_kv_append_quant(cache: KVCache, k: torch.Tensor, v: torch.Tensor, seg, tables: RopeTables,
                          stream=None) -> None:
    rs = _tok_tensor(k, cache.heads, "k")
    if _tok_tensor(v, cache.heads, "v") != rs or v.shape[0] != k.shape[0]:
        raise ValueError("v must have the shape and token stride of k")
    s = _seg(seg)
    if k.shape[0] != s.T * s.grid_h * s.grid_w + s.n_text:
        raise ValueError("k rows != segment tokens")
    _check(lib().nomas_kv_append_quant(ctypes.byref(cache.c), k.data_ptr(), v.data_ptr(), rs, ctypes.byref(s),
                                       tables.handle, _stream(stream)), "nomas_kv_append_quant")


def nomas_kv_gather_context(archive: KVCache, frame_token_offset: Sequence[int], tokens_per_frame: int,
                            frames: Sequence[int], dst: KVCache, index_map: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    fto = np.ascontiguousarray(frame_token_offset, dtype=np.int32)
    fr = np.ascontiguousarray(frames, dtype=np.int32)
    if index_map is not None and (index_map.dtype != torch.int32 or not index_map.is_cuda
                                  or index_map.numel() < len(fr) * tokens_per_frame):
        raise ValueError("index_map: CUDA int32 tensor with n_frames * tokens_per_frame elements")
    _check(lib().nomas_kv_gather_context(ctypes.byref(archive.c), fto.ctypes.data, len(fto), tokens_per_frame,
                                         fr.ctypes.data, len(fr), ctypes.byref(dst.c),
                                         None if index_map is None else index_map.data_ptr(), _stream(stream)),
           "nomas_kv_gather_context")


def nomas_kv_gather_context_host(archive: HostKVCache, frame_token_offset: Sequence[int], tokens_per_frame: int,
                                 frames: Sequence[int], dst: KVCache, index_map: Optional[torch.Tensor] = None,
                                 stream=None) -> None:
    fto = np.ascontiguousarray(frame_token_offset, dtype=np.int32)
    fr = np.ascontiguousarray(frames, dtype=np.int32)
    if index_map is not None and (index_map.dtype != torch.int32 or not index_map.is_cuda
                                  or index_map.numel() < len(fr) * tokens_per_frame):
        raise ValueError("index_map: CUDA int32 tensor with n_frames * tokens_per_frame elements")
    _check(lib().nomas_kv_gather_context_host(ctypes.byref(archive.c), fto.ctypes.data, len(fto), tokens_per_frame,
                                              fr.ctypes.data, len(fr), ctypes.byref(dst.c),
                                              None if index_map is None else index_map.data_ptr(),
                                              _stream(stream)), "nomas_kv_gather_context_host")


def nomas_qkv_project_workspace_size(heads: int, hidden: int) -> int:
    return int(lib().nomas_qkv_project_workspace_size(heads, hidden))


def nomas_qkv_project_rope(x: torch.Tensor, w_codes: torch.Tensor, w_scale: torch.Tensor, seg,
                           tables: RopeTables, out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                           stream=None, append_to: Optional["KVCache"] = None) -> None:
    """out[l] = (Q, K, V) of token l: the INT8-weight projection of x, Q and K rotated by RoPE.
    With append_to, the same call also appends K and V to that INT8 cache (the segment's final
    step; nomas_qkv_project_rope_append)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a bf16 [L][hidden] tensor with unit channel stride")
    hidden = x.shape[1]
    n_out = w_codes.shape[0]
    if w_codes.dtype != torch.int8 or w_codes.dim() != 2 or w_codes.shape[1] != hidden or not w_codes.is_contiguous():
        raise ValueError("w_codes must be a contiguous int8 [3*H*128][hidden] tensor")
    if n_out % (3 * HEAD_DIM):
        raise ValueError("w_codes rows must be 3 * heads * 128")
    heads = n_out // (3 * HEAD_DIM)
    if w_scale.dtype != torch.float32 or w_scale.numel() != n_out or not w_scale.is_contiguous():
        raise ValueError("w_scale must be a contiguous float32 [3*H*128] tensor")
    rs = _tok_tensor(out.view(out.shape[0], 3 * heads, HEAD_DIM), 3 * heads, "out")
    s = _seg(seg)
    need = nomas_qkv_project_workspace_size(heads, hidden)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if append_to is None:
        _check(lib().nomas_qkv_project_rope(x.data_ptr(), x.stride(0), hidden, w_codes.data_ptr(),
                                            w_scale.data_ptr(), heads, ctypes.byref(s), tables.handle, out.data_ptr(),
                                            rs, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                            _stream(stream)), "nomas_qkv_project_rope")
    else:
        _check(lib().nomas_qkv_project_rope_append(x.data_ptr(), x.stride(0), hidden, w_codes.data_ptr(),
                                                   w_scale.data_ptr(), heads, ctypes.byref(s), tables.handle,
                                                   out.data_ptr(), rs, workspace.data_ptr(),
                                                   workspace.numel() * workspace.element_size(),
                                                   ctypes.byref(append_to.c), _stream(stream)),
               "nomas_qkv_project_rope_append")


def nomas_camera_tokens(c2w: torch.Tensor, tokens: torch.Tensor, translation_scale: float = 1.0,
                        rotation_scale: float = 2.5, stream=None) -> None:
    """tokens[g] = the first-frame-relative, scaled extrinsics of video frames 4g .. 4g+3,
    row-major (c2w: CUDA float32 [N][4][4], tokens: CUDA float32 [N/4][64])."""
    if c2w.dtype != torch.float32 or not c2w.is_cuda or c2w.dim() != 3 or tuple(c2w.shape[1:]) != (4, 4) \
            or not c2w.is_contiguous():
        raise ValueError("c2w must be a contiguous CUDA float32 [N][4][4] tensor")
    n = c2w.shape[0]
    if tokens.dtype != torch.float32 or not tokens.is_cuda or tuple(tokens.shape) != (n // 4, 64) \
            or not tokens.is_contiguous():
        raise ValueError("tokens must be a contiguous CUDA float32 [N/4][64] tensor")
    _check(lib().nomas_camera_tokens(c2w.data_ptr(), n, float(translation_scale), float(rotation_scale),
                                     tokens.data_ptr(), _stream(stream)), "nomas_camera_tokens")


def nomas_camera_cross_attn(q: torch.Tensor, k_cam: torch.Tensor, v_cam: torch.Tensor, out: torch.Tensor,
                            softmax_scale: float = 0.0, stream=None) -> None:
    """out = softmax(q k_cam^T * scale) v_cam per head, every query over every camera token
    (q, out: [L][H][128]; k_cam, v_cam: [Tc][H][128]; BF16; out may be q)."""
    rq = _tok_tensor(q, None, "q")
    heads = q.shape[1]
    rk = _tok_tensor(k_cam, heads, "k_cam")
    if _tok_tensor(v_cam, heads, "v_cam") != rk or v_cam.shape[0] != k_cam.shape[0]:
        raise ValueError("v_cam must have the shape and token stride of k_cam")
    ro = _tok_tensor(out, heads, "out")
    if out.shape[0] != q.shape[0]:
        raise ValueError("out rows != q rows")
    _check(lib().nomas_camera_cross_attn(q.data_ptr(), rq, q.shape[0], heads, k_cam.data_ptr(), v_cam.data_ptr(),
                                         rk, k_cam.shape[0], float(softmax_scale), out.data_ptr(), ro,
                                         _stream(stream)), "nomas_camera_cross_attn")


def nomas_seg_attn_workspace_size(lq: int, lh: int, heads: int) -> int:
    return int(lib().nomas_seg_attn_workspace_size(lq, lh, heads))


def nomas_seg_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seg_offsets: Sequence[int],
                   history: Optional[KVCache], out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                   softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out = segment-causal attention of q over [history ; current k/v]."""
    heads, rs, offs, lq = _attn_args(q, k, v, seg_offsets, out, lse)
    lh = history.length if history is not None else 0
    need = nomas_seg_attn_workspace_size(lq, lh, heads)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().nomas_seg_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), rs, heads, offs.ctypes.data,
                                len(offs) - 1, None if history is None else ctypes.byref(history.c),
                                float(softmax_scale), out.data_ptr(), None if lse is None else lse.data_ptr(),
                                ws_ptr, ws_bytes, _stream(stream)), "nomas_seg_attn")


def nomas_staged_history_size(capacity: int, heads: int) -> int:
    return int(lib().nomas_staged_history_size(capacity, heads))


def nomas_seg_attn_staged_workspace_size(lq: int, lh: int, heads: int) -> int:
    return int(lib().nomas_seg_attn_staged_workspace_size(lq, lh, heads))


class StagedHistory:
    """A history's FP16 attention operands, staged once (device memory allocated here by torch);
    see nomas_seg_attn_stage_history."""

    def __init__(self, heads: int, capacity: int, device="cuda"):
        n = max(nomas_staged_history_size(capacity, heads), 16)
        self.buf = torch.empty(n, dtype=torch.uint8, device=device)
        self.c = nomas_staged_history(self.buf.data_ptr(), n, int(capacity), 0, int(heads))

    @property
    def length(self) -> int:
        return self.c.length

    @property
    def heads(self) -> int:
        return self.c.heads


def nomas_seg_attn_stage_history(history: KVCache, staged: StagedHistory, stream=None) -> None:
    """Stages rows [0, history.length) of the INT8 history into `staged` (FP16 operands)."""
    _check(lib().nomas_seg_attn_stage_history(ctypes.byref(history.c), ctypes.byref(staged.c), _stream(stream)),
           "nomas_seg_attn_stage_history")


def _attn_args(q, k, v, seg_offsets, out, lse):
    heads = q.shape[1]
    rs = _tok_tensor(q, heads, "q")
    if _tok_tensor(k, heads, "k") != rs or _tok_tensor(v, heads, "v") != rs:
        raise ValueError("q, k, v must share one token stride")
    offs = np.ascontiguousarray(seg_offsets, dtype=np.int32)
    lq = int(offs[-1])
    if q.shape[0] < lq or k.shape[0] < lq or v.shape[0] < lq:
        raise ValueError("q/k/v shorter than the segment offsets")
    if _tok_tensor(out, heads, "out") != heads * HEAD_DIM or out.shape[0] < lq:
        raise ValueError("out must be a contiguous [Lq][H][128] bf16 tensor")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or lse.numel() < heads * lq):
        raise ValueError("lse must be a contiguous float32 [H][Lq] tensor")
    return heads, rs, offs, lq


def nomas_seg_attn_staged(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seg_offsets: Sequence[int],
                          history: Optional[StagedHistory], out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          softmax_scale: float = 0.0, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """nomas_seg_attn over a history staged by nomas_seg_attn_stage_history."""
    heads, rs, offs, lq = _attn_args(q, k, v, seg_offsets, out, lse)
    lh = history.length if history is not None else 0
    need = nomas_seg_attn_staged_workspace_size(lq, lh, heads)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().nomas_seg_attn_staged(q.data_ptr(), k.data_ptr(), v.data_ptr(), rs, heads, offs.ctypes.data,
                                       len(offs) - 1, None if history is None else ctypes.byref(history.c),
                                       float(softmax_scale), out.data_ptr(), None if lse is None else lse.data_ptr(),
                                       ws_ptr, ws_bytes, _stream(stream)), "nomas_seg_attn_staged")


NOMAS_NOALLOC_SCRATCH_BYTES = 32 << 20


def nomas_seg_attn_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seg_offsets: Sequence[int],
                           history: Optional[KVCache], out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                           softmax_scale: float = 0.0, stream=None) -> None:
    """nomas_seg_attn with the split-KV scratch taken from the library's fixed device array
    (for callers that cannot allocate); raises NomasError(NOMAS_ECAPACITY) when the shapes need
    more than NOMAS_NOALLOC_SCRATCH_BYTES."""
    heads, rs, offs, lq = _attn_args(q, k, v, seg_offsets, out, lse)
    _check(lib().nomas_seg_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), rs, heads, offs.ctypes.data,
                                        len(offs) - 1, None if history is None else ctypes.byref(history.c),
                                        float(softmax_scale), out.data_ptr(),
                                        None if lse is None else lse.data_ptr(), _stream(stream)),
           "nomas_seg_attn_noalloc")


def nomas_stream_check(stream=None) -> None:
    _check(lib().nomas_stream_check(_stream(stream)), "nomas_stream_check")
