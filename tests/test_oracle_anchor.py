"""Pins for the gated-softmax anchor oracle (oracle/softmax_anchor.py),
checked against mathematics other than itself.

- Library routine: with the gate saturated (sigmoid(60) == 1.0 in float64)
  and no RoPE, the layer is scaled dot-product attention, which torch computes
  in float64 by its own code (torch.nn.functional.scaled_dot_product_attention).
- Closed forms: a zero query attends uniformly (the output is the mean of the
  values); one key gives that key's value; g = 0 halves the ungated output;
  near-one-hot scores pick one value.
- Invariants: adding one vector to every key leaves each softmax row
  unchanged; permuting keys and values together changes nothing, permuting
  queries and gates permutes the rows; RoPE depends only on relative
  positions, so shifting the grid by whole frames changes nothing; zero angles
  are the identity.
- The split rule gives the (44, 42, 42) printed for D = 128.
- The row-sampled form matches the full one.

``test_anchor_pins_catch_planted_mistakes`` plants plausible mistakes in the
oracle and checks that each one fails a pin.
"""
import numpy as np
import pytest
import torch

import oracle.linattn as ol
import oracle.softmax_anchor as oa
from oracle.block_causal import block_angles


def _rng(extra=0):
    return np.random.default_rng(2026 + extra)


def _rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _head(seed, N=9, D=16, scale=1.0):
    rng = _rng(seed)
    q, k, v, g = (rng.standard_normal((N, D)) for _ in range(4))
    return scale * q, scale * k, v, g


def pin_sdpa_without_rope_saturated_gate():
    rng = _rng(1)
    B, H, N, D = 2, 3, 11, 16
    q, k, v = (rng.standard_normal((B, H, N, D)) * 2.0 for _ in range(3))
    g = np.full((B, H, N, D), 60.0)
    got = oa.anchor_forward(q, k, v, g)
    want = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x) for x in (q, k, v))).numpy()
    assert _rel_err(got, want) < 1e-12


def pin_gate_zero_halves():
    q, k, v, _ = _head(2)
    half = oa.anchor_head(q, k, v, np.zeros_like(q))
    full = oa.anchor_head(q, k, v, np.full_like(q, 60.0))
    assert _rel_err(half, 0.5 * full) < 1e-14


def pin_zero_query_gives_mean_of_values():
    _, k, v, g = _head(3)
    got = oa.anchor_head(np.zeros_like(k), k, v, g)
    want = ol.sigmoid(g) * v.mean(axis=0)[None, :]
    assert _rel_err(got, want) < 1e-13


def pin_single_key():
    q, k, v, g = _head(4, N=1)
    got = oa.anchor_head(q, k, v, g)
    assert _rel_err(got, ol.sigmoid(g) * v) < 1e-15


def pin_one_hot_scores():
    # k_j = a e_j and q_i = a e_c(i): s_ic(i) = a^2 / sqrt(D) = 100, all others 0
    N = D = 16
    a = np.sqrt(100.0 * np.sqrt(D))
    c = _rng(5).permutation(N)
    k = a * np.eye(N, D)
    q = a * np.eye(D)[c]
    v = _rng(6).standard_normal((N, D))
    g = _rng(7).standard_normal((N, D))
    got = oa.anchor_head(q, k, v, g)
    assert _rel_err(got, ol.sigmoid(g) * v[c]) < 1e-13


def pin_key_shift_invariance():
    q, k, v, g = _head(8)
    shift = _rng(9).standard_normal((1, k.shape[1])) * 3.0
    a = oa.anchor_head(q, k, v, g)
    b = oa.anchor_head(q, k + shift, v, g)
    assert _rel_err(a, b) < 1e-12


def pin_permutation_equivariance():
    q, k, v, g = _head(10, N=13, D=8)
    pk = _rng(11).permutation(13)
    pq = _rng(12).permutation(13)
    a = oa.anchor_head(q, k, v, g)
    assert _rel_err(oa.anchor_head(q, k[pk], v[pk], g), a) < 1e-13
    assert _rel_err(oa.anchor_head(q[pq], k, v, g[pq]), a[pq]) < 1e-13


def pin_rope_relative_positions():
    # a grid of 3 frames read at frames [0, 3) and at [2, 5) of a 5-frame grid
    T, Hs, Ws, D = 3, 2, 3, 24
    split = oa.anchor_split(D)
    N = T * Hs * Ws
    q, k, v, g = _head(13, N=N, D=D, scale=2.0)
    a = oa.anchor_forward(*(x[None, None] for x in (q, k, v, g)),
                          rope=ol.RopeSpec(T, Hs, Ws, *split))
    wide = ol.RopeSpec(T + 2, Hs, Ws, *split)
    ang = block_angles(wide, N, D, rope_offset=2 * Hs * Ws)
    b = oa.anchor_forward(*(x[None, None] for x in (q, k, v, g)), rope=ang)
    none = oa.anchor_forward(*(x[None, None] for x in (q, k, v, g)))
    assert _rel_err(a, b) < 1e-12
    assert _rel_err(a, none) > 1e-3            # the rotation does act


def pin_zero_angles_are_identity():
    q, k, v, g = _head(14, N=6, D=12)
    a = oa.anchor_head(q, k, v, g, np.zeros((6, 6)))
    assert _rel_err(a, oa.anchor_head(q, k, v, g)) < 1e-15


def pin_split_rule():
    assert oa.anchor_split(128) == (44, 42, 42)
    assert oa.anchor_split(256) == (88, 84, 84)


def pin_rows_match_full():
    rng = _rng(15)
    B, H, T, Hs, Ws, D = 1, 2, 2, 3, 2, 12
    N = T * Hs * Ws
    q, k, v, g = (rng.standard_normal((B, H, N, D)) for _ in range(4))
    spec = ol.RopeSpec(T, Hs, Ws, *oa.anchor_split(D))
    full = oa.anchor_forward(q, k, v, g, spec)
    rows = np.array([0, 4, 11])
    part = oa.anchor_forward_rows(q, k, v, g, rows, spec)
    for (b, h), o in part.items():
        assert _rel_err(o, full[b, h][rows]) < 1e-14


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_anchor_oracle_pin(pin):
    pin()


# ------------------------------------------------------- planted mistakes ---

_ORIG_ROTATE = oa._rotate


def _mutant_no_scale(qr, kr):
    return qr @ kr.T


def _mutant_softmax_over_queries(s):
    e = np.exp(s - s.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def _mutant_no_max_for_sum(s):
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / np.exp(s).sum(axis=1, keepdims=True)


def _mutant_ungated(g, y):
    return y


def _mutant_transposed_angles(x, angles):
    return x if angles is None else _ORIG_ROTATE(x, angles[::-1])


def _mutant_relu_features(qr, kr):
    return np.maximum(qr, 0.0) @ np.maximum(kr, 0.0).T / np.sqrt(qr.shape[1])


def _mutant_query_only_rope(q, k, v, g, angles=None, q_angles=None):
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    qa = angles if q_angles is None else q_angles
    return oa._gate(g, oa._softmax(oa._scores(_ORIG_ROTATE(q, qa), k)) @ v)


MUTANTS = {
    "no_scale": ("_scores", _mutant_no_scale),
    "softmax_over_queries": ("_softmax", _mutant_softmax_over_queries),
    "unnormalised_rows": ("_softmax", _mutant_no_max_for_sum),
    "ungated": ("_gate", _mutant_ungated),
    "angles_of_other_tokens": ("_rotate", _mutant_transposed_angles),
    "relu_feature_map": ("_scores", _mutant_relu_features),
    "rope_on_queries_only": ("anchor_head", _mutant_query_only_rope),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_anchor_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(oa, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant!r}"
