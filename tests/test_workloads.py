"""The seeded input recipes and workload table (CPU): the same seed gives the
same inputs on every call, the shapes and dtypes follow the workload, and the
derived sizes (tokens, algorithmic bytes and flops) follow their definitions."""
import torch

from gated_linear_attention_attn_b300.workloads import (WORKLOADS, Workload, make_attnres_inputs,
                                                        make_inputs, sample_rows)


def test_make_inputs_is_seeded_and_shaped():
    wl = Workload("t", B=1, H=2, grid=(2, 3, 4), rope=True)
    a = make_inputs(wl, seed=7)
    b = make_inputs(wl, seed=7)
    c = make_inputs(wl, seed=8)
    for x, y, z in zip(a, b, c):
        assert x.shape == (1, 2, 24, 128) and x.dtype == torch.bfloat16
        assert torch.equal(x, y) and not torch.equal(x, z)


def test_make_inputs_scales_keys():
    wl = Workload("t", B=1, H=1, grid=(1, 1, 64), dtype=torch.float32)
    q, k, _, _ = make_inputs(wl, seed=3)
    q2, k2, _, _ = make_inputs(wl.with_(k_scale=0.5), seed=3)
    assert torch.equal(q, q2) and torch.allclose(k2, 0.5 * k)


def test_make_attnres_inputs_recipe():
    wl = Workload("a", B=1, H=3, grid=(1, 1, 50), d=256, layer="attnres")
    s, w = make_attnres_inputs(wl, seed=5)
    s2, w2 = make_attnres_inputs(wl, seed=5)
    assert s.shape == (3, 50, 256) and s.dtype == torch.bfloat16
    assert w.shape == (256,) and w.dtype == torch.float32
    assert torch.equal(s, s2) and torch.equal(w, w2)
    # source n is drawn at scale 1 + n
    rms = s.float().pow(2).mean(dim=(1, 2)).sqrt()
    assert rms[0] < rms[1] < rms[2]


def test_derived_sizes():
    wl = WORKLOADS["5b_720p"]
    assert wl.N == 22000 and wl.token_heads == 2 * 20 * 22000
    assert wl.algorithmic_bytes == 5 * 2 * 20 * 22000 * 128 * 2
    an = WORKLOADS["anchor_5b_720p"]
    assert an.algorithmic_flops == 4 * 2 * 10 * 22000 * 22000 * 256
    ar = WORKLOADS["attnres_5b_720p"]
    assert ar.tokens == 44000 and ar.algorithmic_bytes == 5 * 44000 * 2560 * 2
    b736 = WORKLOADS["5b_720p_736"]
    assert b736.N == 25 * 23 * 40 == 23000 and b736.rope
    bc = WORKLOADS["5b_720p_block5"]
    assert bc.block_tokens == 5 * 22 * 40 and bc.N % bc.block_tokens == 0


def test_sample_rows_cover_both_ends():
    rows = sample_rows(4290, 24)
    assert rows[0] == 0 and rows[-1] == 4289 and rows == sorted(set(rows))
    assert sample_rows(4290, 24) == rows
