"""The Python binding's own argument checks, which run before any call into the library: wrong
devices, dtypes, shapes and strides are refused with ValueError (no GPU needed)."""
import pytest
import torch

import nomas_synth as ns
import segment_causal_attention_nomas_b300 as nb


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_token_tensors_must_be_cuda_bf16_with_contiguous_heads():
    with pytest.raises(ValueError, match="CUDA bf16"):
        nb._tok_tensor(bf16(4, 2, 128), None, "x")                       # host memory
    with pytest.raises(ValueError, match="CUDA bf16"):
        nb._tok_tensor(torch.zeros(4, 2, 128), None, "x")                 # fp32
    with pytest.raises(ValueError, match="CUDA bf16"):
        nb._tok_tensor(bf16(4, 2, 64), None, "x")                         # head dim 64


def test_camera_tokens_binding_checks():
    with pytest.raises(ValueError, match="c2w"):
        nb.nomas_camera_tokens(torch.zeros(8, 4, 4), torch.zeros(2, 64))  # host tensors
    with pytest.raises(ValueError, match="c2w"):
        nb.nomas_camera_tokens(torch.zeros(8, 3, 4), torch.zeros(2, 64))  # not 4 x 4


def test_camera_cross_attn_binding_checks():
    with pytest.raises(ValueError, match="q"):
        nb.nomas_camera_cross_attn(bf16(4, 2, 128), bf16(3, 2, 128), bf16(3, 2, 128), bf16(4, 2, 128))


def test_rope_and_append_binding_checks():
    seg = ns.Segment(0, 1, 2, 2, 0)
    with pytest.raises(ValueError):
        nb.nomas_rope3d(bf16(4, 2, 128), bf16(4, 2, 128), seg, None)


def test_projection_binding_checks():
    seg = ns.Segment(0, 1, 2, 2, 0)
    with pytest.raises(ValueError, match="x must be"):
        nb.nomas_qkv_project_rope(torch.zeros(4, 64), torch.zeros(768, 64, dtype=torch.int8), torch.ones(768), seg,
                                  None, bf16(4, 3, 2, 128))
    with pytest.raises(ValueError, match="w_codes"):
        nb.nomas_qkv_project_rope(bf16(4, 64), torch.zeros(768, 32, dtype=torch.int8), torch.ones(768), seg,
                                  None, bf16(4, 3, 2, 128))
    with pytest.raises(ValueError, match="3 \\* heads"):
        nb.nomas_qkv_project_rope(bf16(4, 64), torch.zeros(700, 64, dtype=torch.int8), torch.ones(700), seg,
                                  None, bf16(4, 3, 2, 128))
    with pytest.raises(ValueError, match="w_scale"):
        nb.nomas_qkv_project_rope(bf16(4, 64), torch.zeros(768, 64, dtype=torch.int8), torch.ones(768).double(), seg,
                                  None, bf16(4, 3, 2, 128))
