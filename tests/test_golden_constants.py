"""The workload shapes and the oracle's RoPE constants against the values the pages print
(tests/golden/page_constants.json, each entry citing its page and section)."""
import json
import math
import os

import numpy as np

import nomas_synth as ns
import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def v(key):
    return GOLDEN[key]["value"]


def test_head_geometry_matches_pages():
    assert v("heads") * v("head_dim") == v("hidden")
    assert ns.HEAD_DIM == oracle.HEAD_DIM == v("head_dim")
    assert tuple(ns.ROPE_SPLIT) == tuple(oracle.SPLIT.tolist()) == tuple(v("rope_split"))
    assert sum(v("rope_split")) == GOLDEN["derived"]["head_dim_from_split"]["value"] == v("head_dim")
    assert ns.ROPE_THETA == oracle.THETA == v("rope_theta")
    assert ns.config2().heads == v("heads")


def test_tokens_per_latent_frame_derivation():
    w, h = v("width_height")
    s = v("spatial_compression")
    assert v("latent_patch") == [1, 1, 1]
    grid = [h // s, w // s]
    assert h % s == 0 and w % s == 0
    assert grid == GOLDEN["derived"]["latent_grid"]["value"] == [ns.GRID_H, ns.GRID_W]
    assert grid[0] * grid[1] == GOLDEN["derived"]["tokens_per_latent_frame"]["value"] == ns.TOKENS_PER_FRAME


def test_history_budget_and_context_ceiling():
    w2 = ns.config2()
    assert w2.lh == v("history_frames") * ns.TOKENS_PER_FRAME
    assert w2.steps == v("euler_steps")
    w4 = ns.config4()
    assert len(w4.gather) == v("history_frames")
    # the lifelong-cache workload stays within the stated context
    w3 = ns.config3()
    assert w3.lh + w3.lq <= v("context_tokens")
    # 12 s at 24 fps with 4x temporal compression = 72 latent frames per turn
    assert 12 * v("fps") // v("temporal_compression") == w3.current[0].T


def test_rope_time_axis_frequencies_are_powers_of_two():
    # theta 256 = 2^8 and d_t = 16: omega_i = 256^(-2i/16) = 2^-i, a closed form the
    # printed constants fix exactly
    cos, sin = oracle.rope_table(3, v("rope_split")[0], float(v("rope_theta")))
    for i in range(8):
        assert cos[1, i] == np.float32(math.cos(2.0 ** -i))
        assert sin[2, i] == np.float32(math.sin(2.0 * 2.0 ** -i))
