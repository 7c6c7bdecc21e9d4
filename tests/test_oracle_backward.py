"""Pins for the backward oracle (oracle/backward.py), checked against
mathematics other than itself.

- Central finite differences of the forward oracle (itself pinned in
  test_oracle.py) check every gradient element of small heads, with and
  without rotary embeddings.
- Invariants: a zero upstream gradient gives zero gradients; a saturated gate
  has no gate gradient; permuting the tokens permutes the gradients
  (no RoPE).
- The row-sampled form matches the full one.

``test_backward_pins_catch_planted_mistakes`` plants plausible mistakes in
the oracle and checks that each one fails a pin.
"""
import numpy as np
import pytest

import oracle.backward as ob
import oracle.linattn as ol


def _rng(extra=0):
    return np.random.default_rng(777 + extra)


def _away_from_zero(x, margin=0.05):
    """Inputs whose ReLU kinks are far from the finite-difference step."""
    return np.where(np.abs(x) < margin, np.sign(x + 1e-12) * margin, x)


def _rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _finite_difference(q, k, v, g, do, eps, angles, step=1e-6):
    """dL/dx for L = sum(do * o), by central differences of the forward oracle."""
    grads = []
    base = [q, k, v, g]
    for which in range(4):
        x = base[which]
        grad = np.empty_like(x)
        for idx in np.ndindex(*x.shape):
            plus = [y.copy() for y in base]
            minus = [y.copy() for y in base]
            plus[which][idx] += step
            minus[which][idx] -= step
            lp = float(np.sum(do * ol.linattn_head(*plus, eps, angles)))
            lm = float(np.sum(do * ol.linattn_head(*minus, eps, angles)))
            grad[idx] = (lp - lm) / (2.0 * step)
        grads.append(grad)
    return grads


def _small_head(seed, N=5, d=6):
    rng = _rng(seed)
    q, k = (_away_from_zero(rng.standard_normal((N, d))) for _ in range(2))
    v, g, do = (rng.standard_normal((N, d)) for _ in range(3))
    return q, k, v, g, do


def pin_finite_differences_no_rope():
    q, k, v, g, do = _small_head(1)
    got = ob.linattn_head_backward(q, k, v, g, do, 1e-3)
    want = _finite_difference(q, k, v, g, do, 1e-3, None)
    for name, a, b in zip("dq dk dv dg".split(), got, want):
        assert _rel_err(a, b) < 1e-6, name


def pin_finite_differences_rope():
    q, k, v, g, do = _small_head(2, N=6, d=8)
    angles = _rng(3).uniform(-np.pi, np.pi, (6, 4))
    got = ob.linattn_head_backward(q, k, v, g, do, 1e-3, angles)
    want = _finite_difference(q, k, v, g, do, 1e-3, angles)
    for name, a, b in zip("dq dk dv dg".split(), got, want):
        assert _rel_err(a, b) < 1e-6, name


def pin_finite_differences_3d_grid():
    spec = ol.RopeSpec(2, 2, 2, 2, 2, 2)           # 8 tokens, d = 6
    q, k, v, g, do = _small_head(4, N=8, d=6)
    ang = ol.rope3d_angles(spec)
    got = ob.linattn_head_backward(q, k, v, g, do, 1e-2, ang)
    want = _finite_difference(q, k, v, g, do, 1e-2, ang)
    for name, a, b in zip("dq dk dv dg".split(), got, want):
        assert _rel_err(a, b) < 1e-6, name


def pin_zero_upstream_gradient():
    q, k, v, g, _ = _small_head(5)
    for grad in ob.linattn_head_backward(q, k, v, g, np.zeros_like(q), 1e-6):
        assert np.all(grad == 0.0)


def pin_saturated_gate_has_no_gate_gradient():
    q, k, v, _, do = _small_head(6)
    g = np.full_like(q, 60.0)
    _, _, _, dg = ob.linattn_head_backward(q, k, v, g, do, 1e-6)
    assert np.max(np.abs(dg)) < 1e-20


def pin_permutation_equivariance():
    q, k, v, g, do = _small_head(7, N=7, d=5)
    perm = _rng(8).permutation(7)
    a = ob.linattn_head_backward(q, k, v, g, do, 1e-6)
    b = ob.linattn_head_backward(q[perm], k[perm], v[perm], g[perm], do[perm], 1e-6)
    for x, y in zip(a, b):
        assert _rel_err(x[perm], y) < 1e-12


def pin_rows_match_full():
    rng = _rng(9)
    B, H, N, d = 1, 2, 12, 8
    q, k, v, g, do = (rng.standard_normal((B, H, N, d)) for _ in range(5))
    spec = ol.RopeSpec(3, 2, 2, 4, 2, 2)
    full = ob.linattn_backward(q, k, v, g, do, 1e-6, spec)
    rows = np.array([0, 5, 11])
    part = ob.linattn_backward_rows(q, k, v, g, do, rows, 1e-6, spec)
    for (b, h), grads in part.items():
        for x, y in zip(grads, full):
            assert _rel_err(x, y[b, h][rows]) < 1e-13


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_oracle_pin(pin):
    pin()


# ------------------------------------------------------- planted mistakes ---

_ORIG_QUERY = ob._query_terms
_ORIG_ROT = ob._rot


def _mutant_gate_derivative(q, g, do, S, z, eps, angles):
    qp, qr, a, dg, dden = _ORIG_QUERY(q, g, do, S, z, eps, angles)
    return qp, qr, a, dg / (1.0 - ol.sigmoid(g)), dden      # s instead of s (1 - s)


def _mutant_no_den_gradient(q, g, do, S, z, eps, angles):
    qp, qr, a, dg, dden = _ORIG_QUERY(q, g, do, S, z, eps, angles)
    return qp, qr, a, dg, 0.0 * dden


def _mutant_den_sign(q, g, do, S, z, eps, angles):
    qp, qr, a, dg, dden = _ORIG_QUERY(q, g, do, S, z, eps, angles)
    return qp, qr, a, dg, -dden


def _mutant_forward_rotation(x, angles, sign=1.0):
    return _ORIG_ROT(x, angles, 1.0)                       # R instead of R^T


MUTANTS = {
    "gate_derivative": ("_query_terms", _mutant_gate_derivative),
    "no_denominator_gradient": ("_query_terms", _mutant_no_den_gradient),
    "denominator_sign": ("_query_terms", _mutant_den_sign),
    "forward_rotation_in_backward": ("_rot", _mutant_forward_rotation),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_backward_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(ob, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant!r}"
