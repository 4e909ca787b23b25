"""The C-ABI library without a GPU: it loads, exports every entry point include/nomas.h
declares, and its host-side argument checks reject bad calls before touching the device."""
import ctypes

import numpy as np
import pytest

import segment_causal_attention_nomas_b300 as nb


@pytest.fixture(scope="module")
def L():
    from segment_causal_attention_nomas_b300 import build
    build.build()
    return nb.lib()


def test_exports_every_declared_entry_point(L):
    declared = nb.declared_entry_points()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(L, name), f"{name} declared in include/nomas.h but not exported"


def test_status_strings_and_version(L):
    assert nb.nomas_version().startswith("nomas-b300")
    for s in range(7):
        assert nb.nomas_status_string(s).startswith("NOMAS_")
    assert "RANGE" in nb.nomas_status_string(nb.NOMAS_ERANGE)
    assert "unknown" in nb.nomas_status_string(99)


def test_seg_attn_rejects_bad_arguments_on_host(L):
    offs = (ctypes.c_int32 * 3)(0, 5, 3)       # decreasing offsets
    st = L.nomas_seg_attn(16, 16, 16, 128, 1, offs, 2, None, 0.0, 16, None, None, 0, None)
    assert st == nb.NOMAS_EINVAL and "decrease" in nb.nomas_last_error()
    offs = (ctypes.c_int32 * 2)(1, 5)          # offsets[0] != 0
    assert L.nomas_seg_attn(16, 16, 16, 128, 1, offs, 1, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_EINVAL
    offs = (ctypes.c_int32 * 2)(0, 5)
    assert L.nomas_seg_attn(16, 16, 16, 128, 0, offs, 1, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_EINVAL
    assert L.nomas_seg_attn(16, 16, 16, 100, 1, offs, 1, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_EINVAL
    assert L.nomas_seg_attn(18, 16, 16, 128, 1, offs, 1, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_EINVAL
    assert L.nomas_seg_attn(16, 16, 16, 128, 1, offs, 1, None, -1.0, 16, None, None, 0, None) == nb.NOMAS_EINVAL
    many = (ctypes.c_int32 * 66)(*range(66))
    assert L.nomas_seg_attn(16, 16, 16, 128, 1, many, 65, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_EUNSUPPORTED
    # empty query set is a no-op
    zero = (ctypes.c_int32 * 2)(0, 0)
    assert L.nomas_seg_attn(16, 16, 16, 128, 1, zero, 1, None, 0.0, 16, None, None, 0, None) == nb.NOMAS_OK


def test_noalloc_reports_the_errors_of_seg_attn(L):
    # The no-allocation variant checks its arguments as nomas_seg_attn does, before its scratch
    # size check, so malformed calls get the same status (not ECAPACITY for the scratch).
    offs = (ctypes.c_int32 * 4)(0, 2_000_000, 1_000_000, 3_000_000)   # decreasing, ends large
    st = L.nomas_seg_attn_noalloc(16, 16, 16, 128, 1, offs, 3, None, 0.0, 16, None, None)
    assert st == nb.NOMAS_EINVAL and "decrease" in nb.nomas_last_error()
    offs = (ctypes.c_int32 * 2)(0, 5)
    st = L.nomas_seg_attn_noalloc(16, 16, 16, 5000 * 128, 5000, offs, 1, None, 0.0, 16, None, None)
    assert st == nb.NOMAS_EUNSUPPORTED and "heads" in nb.nomas_last_error()
    hist = nb.nomas_kv_cache(16, 16, 16, 16, 1 << 20, 1 << 20, 3, 128)   # 3 heads, caller says 2
    st = L.nomas_seg_attn_noalloc(16, 16, 16, 256, 2, offs, 1, ctypes.byref(hist), 0.0, 16, None, None)
    assert st == nb.NOMAS_EINVAL and "heads" in nb.nomas_last_error()
    assert L.nomas_seg_attn(16, 16, 16, 256, 2, offs, 1, ctypes.byref(hist), 0.0, 16, None, None, 0,
                            None) == nb.NOMAS_EINVAL


def test_staged_history_entry_points_reject_bad_arguments_on_host(L):
    cache = nb.nomas_kv_cache(16, 16, 16, 16, 64, 40, 2, 128)
    need = nb.nomas_staged_history_size(64, 2)
    ok_buf = nb.nomas_staged_history(4096, need, 64, 7, 2)
    # heads differ, capacity too small, buffer too small or misaligned: nothing is written
    for sh, want in [(nb.nomas_staged_history(4096, need, 64, 7, 3), nb.NOMAS_EINVAL),
                     (nb.nomas_staged_history(4096, need, 32, 7, 2), nb.NOMAS_ECAPACITY),
                     (nb.nomas_staged_history(4096, need - 1, 64, 7, 2), nb.NOMAS_EINVAL),
                     (nb.nomas_staged_history(4100, need, 64, 7, 2), nb.NOMAS_EINVAL)]:
        assert L.nomas_seg_attn_stage_history(ctypes.byref(cache), ctypes.byref(sh), None) == want
        assert sh.length == 7
    assert L.nomas_seg_attn_stage_history(None, ctypes.byref(ok_buf), None) == nb.NOMAS_EINVAL
    # attention over a staged history: heads mismatch, length beyond capacity, small buffer
    offs = (ctypes.c_int32 * 2)(0, 5)
    for sh in (nb.nomas_staged_history(4096, need, 64, 40, 3), nb.nomas_staged_history(4096, need, 64, 65, 2),
               nb.nomas_staged_history(4096, 1024, 64, 40, 2)):
        assert L.nomas_seg_attn_staged(16, 16, 16, 256, 2, offs, 1, ctypes.byref(sh), 0.0, 16, None, 16, 1 << 30,
                                       None) == nb.NOMAS_EINVAL
    # a workspace smaller than nomas_seg_attn_staged_workspace_size
    sh = nb.nomas_staged_history(4096, need, 64, 40, 2)
    small = nb.nomas_seg_attn_staged_workspace_size(5, 40, 2) - 1
    assert L.nomas_seg_attn_staged(16, 16, 16, 256, 2, offs, 1, ctypes.byref(sh), 0.0, 16, None, 16, small,
                                   None) == nb.NOMAS_EINVAL
    assert "workspace" in nb.nomas_last_error()


def test_camera_entry_points_reject_bad_arguments_on_host(L):
    # camera tokens: frame count, scales, pointers, overlap
    assert L.nomas_camera_tokens(16, 6, 1.0, 2.5, 4096, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_tokens(16, 0, 1.0, 2.5, 4096, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_tokens(16, 8, float("nan"), 2.5, 4096, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_tokens(None, 8, 1.0, 2.5, 4096, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_tokens(16, 8, 1.0, 2.5, 24, None) == nb.NOMAS_EINVAL          # misaligned
    assert L.nomas_camera_tokens(4096, 8, 1.0, 2.5, 4096 + 256, None) == nb.NOMAS_EINVAL  # overlap
    assert "overlaps" in nb.nomas_last_error()
    # cross-attention: counts, limits, strides, scale; lq = 0 is a no-op
    x = 4096
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, x, 256, 0, 0.0, x, 256, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, x, 256, 129, 0.0, x, 256, None) == nb.NOMAS_EUNSUPPORTED
    assert L.nomas_camera_cross_attn(x, 256, 10, 4097, x, x, 256, 4, 0.0, x, 256, None) == nb.NOMAS_EUNSUPPORTED
    assert L.nomas_camera_cross_attn(x, 255, 10, 2, x, x, 256, 4, 0.0, x, 256, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, x, 264, 4, 0.0, x, 252, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, x, 256, 4, -1.0, x, 256, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, None, 256, 4, 0.0, x, 256, None) == nb.NOMAS_EINVAL
    assert L.nomas_camera_cross_attn(x, 256, 10, 2, x, x, 256, 4, 0.0, x, 264, None) == nb.NOMAS_EINVAL  # q alias
    assert L.nomas_camera_cross_attn(x, 256, 0, 2, x, x, 256, 4, 0.0, x, 256, None) == nb.NOMAS_OK


def test_projection_append_rejects_a_missing_cache_on_host(L):
    seg = nb.nomas_segment(0, 1, 2, 2, 0)
    st = L.nomas_qkv_project_rope_append(16, 64, 64, 16, 16, 2, ctypes.byref(seg), None, 16, 768, 16, 1 << 20,
                                         None, None)
    assert st == nb.NOMAS_EINVAL and "cache is NULL" in nb.nomas_last_error()


def test_cache_checks_on_host(L):
    bad = nb.nomas_kv_cache(16, 16, 16, 16, 8, 9, 1, 128)        # length > capacity
    seg = nb.nomas_segment(0, 1, 1, 1, 0)
    assert L.nomas_kv_append_quant(ctypes.byref(bad), 16, 16, 128, ctypes.byref(seg), 16, None) == nb.NOMAS_EINVAL
    hd = nb.nomas_kv_cache(16, 16, 16, 16, 8, 0, 1, 64)          # head_dim 64
    assert L.nomas_kv_append_quant(ctypes.byref(hd), 16, 16, 128, ctypes.byref(seg), 16, None) == nb.NOMAS_EUNSUPPORTED
    cap = nb.nomas_kv_cache(16, 16, 16, 16, 6, 0, 1, 128)        # capacity not a multiple of 4
    assert L.nomas_kv_append_quant(ctypes.byref(cap), 16, 16, 128, ctypes.byref(seg), 16, None) == nb.NOMAS_EINVAL
    full = nb.nomas_kv_cache(16, 16, 16, 16, 8, 8, 1, 128)       # full: one more token overflows
    assert L.nomas_kv_append_quant(ctypes.byref(full), 16, 16, 128, ctypes.byref(seg), 16, None) == nb.NOMAS_ECAPACITY
    assert full.length == 8
    mis = nb.nomas_kv_cache(17, 16, 16, 16, 8, 0, 1, 128)        # misaligned codes
    assert L.nomas_kv_append_quant(ctypes.byref(mis), 16, 16, 128, ctypes.byref(seg), 16, None) == nb.NOMAS_EINVAL


def test_gather_checks_on_host(L):
    arch = nb.nomas_kv_cache(16, 16, 16, 16, 40, 40, 2, 128)
    dst = nb.nomas_kv_cache(32, 32, 32, 32, 12, 0, 2, 128)
    fto = (ctypes.c_int32 * 4)(0, 10, 20, 30)
    for frames, want in [((2, 1), nb.NOMAS_EINVAL),        # not increasing
                         ((1, 1), nb.NOMAS_EINVAL),        # duplicate
                         ((0, 4), nb.NOMAS_EINVAL),        # out of range
                         ((0, 1, 2), nb.NOMAS_ECAPACITY)]:  # 3 x 5 tokens > 12
        fr = (ctypes.c_int32 * len(frames))(*frames)
        assert L.nomas_kv_gather_context(ctypes.byref(arch), fto, 4, 5, fr, len(frames), ctypes.byref(dst),
                                         None, None) == want
    # a frame reaching past the archive length
    short = nb.nomas_kv_cache(16, 16, 16, 16, 40, 22, 2, 128)
    fr = (ctypes.c_int32 * 1)(2)
    assert L.nomas_kv_gather_context(ctypes.byref(short), fto, 4, 5, fr, 1, ctypes.byref(dst), None,
                                     None) == nb.NOMAS_EINVAL
    assert dst.length == 0
    # on an error the destination's length is left as it was (both gathers)
    dst.length = 7
    for fn in (L.nomas_kv_gather_context, L.nomas_kv_gather_context_host):
        for frames in ((2, 1), (0, 1, 2)):
            fr = (ctypes.c_int32 * len(frames))(*frames)
            assert fn(ctypes.byref(arch), fto, 4, 5, fr, len(frames), ctypes.byref(dst), None, None) != nb.NOMAS_OK
            assert dst.length == 7


def test_rope_tables_arguments(L):
    out = ctypes.c_void_p()
    bad_split = (ctypes.c_int32 * 3)(16, 56, 48)
    assert L.nomas_rope_tables_create(256.0, bad_split, 8, 8, 8, ctypes.byref(out)) == nb.NOMAS_EUNSUPPORTED
    split = (ctypes.c_int32 * 3)(16, 56, 56)
    assert L.nomas_rope_tables_create(0.5, split, 8, 8, 8, ctypes.byref(out)) == nb.NOMAS_EINVAL
    assert L.nomas_rope_tables_create(256.0, split, 0, 8, 8, ctypes.byref(out)) == nb.NOMAS_EINVAL
    seg = nb.nomas_segment(0, 1, 1, 1, 0)
    assert L.nomas_rope3d(16, 16, 128, ctypes.byref(seg), 1, None, None) == nb.NOMAS_EINVAL


def _ru(x, a):
    return (x + a - 1) // a * a


def _layout(lq, lh, h, splits, with_history=True):
    """Bytes of the attention workspace as include/nomas.h lays it out: staged FP16 Q, K, V; the
    staged history (per-head scale maxima, FP16 K, V) when the call stages it; n_splits fp32
    partial rows (O and LSE) when the key range is split; int8 query-row exponents; the per-head
    current K/V maxima."""
    n = 3 * lq * h * 256
    if with_history and lh > 0:
        n += _ru(8 * h, 1024) + 2 * lh * h * 256
    if splits > 1:
        n += _ru(splits * lq * h * 129 * 4, 256)
    return n + _ru(lq * h, 256) + _ru(8 * h, 256)


def test_workspace_size_is_host_only(L):
    assert nb.nomas_seg_attn_workspace_size(0, 0, 16) == 0
    assert nb.nomas_seg_attn_staged_workspace_size(0, 10, 16) == 0
    # sizes nomas_seg_attn refuses get 0, not a wrapped product
    for lq, lh, h in ((1 << 30, 0, 16), (2 ** 62, 0, 16), (100, 1 << 30, 1), (100, 2 ** 62, 16),
                      (100, 0, 4097), (100, 70_000_000, 16), (100, -1, 16)):
        assert nb.nomas_seg_attn_workspace_size(lq, lh, h) == 0, (lq, lh, h)
        assert nb.nomas_seg_attn_staged_workspace_size(lq, lh, h) == 0, (lq, lh, h)
    assert nb.nomas_seg_attn_workspace_size((1 << 30) - 1, 0, 1) > 0
    lq, lh, h = 3776, 300000, 16
    assert nb.nomas_seg_attn_workspace_size(lq, 0, h) == _layout(lq, 0, h, 1)
    # large Lh / short Lq adds split-KV partials: whole fp32 partial rows (O and LSE)
    n = nb.nomas_seg_attn_workspace_size(lq, lh, h)
    assert n > _layout(lq, lh, h, 1)
    # the staged variant needs the same minus the history block
    assert nb.nomas_seg_attn_staged_workspace_size(lq, lh, h) == n - (_ru(8 * h, 1024) + 2 * lh * h * 256)
    assert nb.nomas_staged_history_size(lh, h) == _ru(8 * h, 1024) + 2 * lh * h * 256
    assert nb.nomas_staged_history_size(0, h) == 0


def _splits(lq, lh, heads=16):
    # the split count that reproduces the workspace size
    n = nb.nomas_seg_attn_workspace_size(lq, lh, heads)
    found = [s for s in range(1, 17) if _layout(lq, lh, heads, s) == n]
    assert len(found) == 1, (lq, lh, n)
    return found[0]


def test_split_kv_choice(L):
    # Host-side split choice (148 SMs without a GPU): long query sets keep one split (config 2 is
    # seven full waves, config 3 twenty-seven); short ones over long histories split the key
    # range; short ones without history do not (the merge would cost more than the idle SMs).
    assert _splits(16096, 15840) == 1
    assert _splits(63616, 254464) == 1
    assert _splits(10816, 0) == 1
    assert _splits(3776, 100000) == 3
    assert _splits(21376, 300000) == 3
    for lq, lh in ((1, 0), (3776, 300000), (128, 1000000)):
        s = _splits(lq, lh)
        tiles = -(-lh // 128) + -(-lq // 128)
        assert 1 <= s <= 16 and (s == 1 or tiles // s >= 8)


def test_declared_names_parse():
    names = nb.declared_entry_points()
    for n in ["nomas_kv_append_quant", "nomas_rope3d", "nomas_seg_attn", "nomas_kv_gather_context",
              "nomas_stream_check", "nomas_seg_attn_workspace_size"]:
        assert n in names
    assert np.all([n.startswith("nomas_") for n in names])
