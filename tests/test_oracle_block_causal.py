"""Pins for the block-causal oracle (oracle/block_causal.py), checked against
mathematics other than itself.

The O(N^2) form with a block mask, written out below pair by pair, pins the
running-state formulation for several block sizes, with and without rotary
embeddings.  A hand-worked two-token case pins the values.  Invariants pin
the rest:

- one block is the bidirectional layer;
- the last block sees every token;
- chained calls with the carried state and the RoPE offset equal one call;
- an incoming state acts as a prefix.

``test_block_pins_catch_planted_mistakes`` plants plausible mistakes in the
oracle and checks that each one fails a pin.
"""
import numpy as np
import pytest

import oracle.block_causal as bc
import oracle.linattn as ol


def _rng(extra=0):
    return np.random.default_rng(4321 + extra)


def _rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _pairwise_block_mask(q, k, v, g, block_tokens, eps, angles=None):
    """Every (query i, key j) pair with block(j) <= block(i) adds the weight
    (R_i phi(q_i)) . (R_j phi(k_j)) to the numerator and phi(q_i) . phi(k_j)
    to the denominator; the gate multiplies the ratio."""
    N, d = q.shape
    qp, kp = np.maximum(q, 0.0), np.maximum(k, 0.0)
    if angles is None:
        qr, kr = qp, kp
    else:
        # RoFormer's complex form: pair p of x is x_2p + i x_2p+1
        def rot(x):
            c = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * angles)
            out = np.empty_like(x)
            out[:, 0::2], out[:, 1::2] = c.real, c.imag
            return out
        qr, kr = rot(qp), rot(kp)
    out = np.empty((N, d))
    for i in range(N):
        num, den = np.zeros(d), eps
        for j in range(N):
            if j // block_tokens <= i // block_tokens:
                num += float(qr[i] @ kr[j]) * v[j]
                den += float(qp[i] @ kp[j])
        out[i] = num / den / (1.0 + np.exp(-g[i]))
    return out


def pin_block_mask_bruteforce():
    rng = _rng(1)
    N, d = 12, 8
    q, k, v, g = (rng.standard_normal((N, d)) for _ in range(4))
    angles = rng.uniform(-np.pi, np.pi, (N, d // 2))
    for bt in (1, 2, 3, 4, 6, 12):
        for ang in (None, angles):
            o, _, _ = bc.linattn_block_causal_head(q, k, v, g, bt, 1e-6, ang)
            ref = _pairwise_block_mask(q, k, v, g, bt, 1e-6, ang)
            assert _rel_err(o, ref) < 1e-11, (bt, ang is None)


def pin_hand_two_tokens():
    # d = 1, q = (1, 1), k = (1, 2), v = (3, 5), eps = 0, g large (gate ~ 1):
    # token blocks: o_0 = 3, o_1 = (1*3 + 2*5) / (1 + 2) = 13/3; one block: both 13/3
    q = np.array([[1.0], [1.0]]); k = np.array([[1.0], [2.0]])
    v = np.array([[3.0], [5.0]]); g = np.full((2, 1), 60.0)
    o1, S, z = bc.linattn_block_causal_head(q, k, v, g, 1, 0.0)
    assert abs(o1[0, 0] - 3.0) < 1e-12 and abs(o1[1, 0] - 13.0 / 3.0) < 1e-12
    assert abs(S[0, 0] - 13.0) < 1e-12 and abs(z[0] - 3.0) < 1e-12
    o2, _, _ = bc.linattn_block_causal_head(q, k, v, g, 2, 0.0)
    assert np.allclose(o2[:, 0], 13.0 / 3.0, rtol=0, atol=1e-12)


def pin_one_block_is_bidirectional():
    rng = _rng(2)
    N, d = 20, 16
    q, k, v, g = (rng.standard_normal((N, d)) for _ in range(4))
    spec = ol.RopeSpec(1, 4, 5, 6, 6, 4)
    ang = ol.rope3d_angles(spec)
    o, S, z = bc.linattn_block_causal_head(q, k, v, g, N, 1e-6, ang)
    assert _rel_err(o, ol.linattn_head(q, k, v, g, 1e-6, ang)) < 1e-13
    S_ref, z_ref = ol.linattn_state(k, v, ang)
    assert _rel_err(S, S_ref) < 1e-13 and _rel_err(z, z_ref) < 1e-13


def pin_last_block_sees_every_token():
    rng = _rng(3)
    N, d, bt = 24, 8, 6
    q, k, v, g = (rng.standard_normal((N, d)) for _ in range(4))
    o, _, _ = bc.linattn_block_causal_head(q, k, v, g, bt, 1e-6)
    full = ol.linattn_head(q, k, v, g, 1e-6)
    assert _rel_err(o[-bt:], full[-bt:]) < 1e-13
    assert _rel_err(o[:bt], ol.linattn_head(q[:bt], k[:bt], v[:bt], g[:bt], 1e-6)) < 1e-13


def pin_chained_calls_equal_one_call():
    rng = _rng(4)
    spec = ol.RopeSpec(6, 2, 3, 6, 6, 4)          # 6 frames of 6 tokens, d = 16
    B, H, N, d, bt = 1, 2, spec.n_tokens, 16, 6
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    whole, (S, z) = bc.linattn_forward_block_causal(q, k, v, g, bt, 1e-6, spec)
    cut = 4 * bt
    a, st = bc.linattn_forward_block_causal(q[:, :, :cut], k[:, :, :cut], v[:, :, :cut],
                                            g[:, :, :cut], bt, 1e-6, spec, 0)
    b, (S2, z2) = bc.linattn_forward_block_causal(q[:, :, cut:], k[:, :, cut:], v[:, :, cut:],
                                                  g[:, :, cut:], bt, 1e-6, spec, cut, st)
    assert _rel_err(np.concatenate([a, b], axis=2), whole) < 1e-13
    assert _rel_err(S2, S) < 1e-13 and _rel_err(z2, z) < 1e-13


def pin_incoming_state_acts_as_prefix():
    rng = _rng(5)
    N, d, bt = 12, 8, 4
    P = 8                                         # prefix tokens, two blocks
    q, k, v, g = (rng.standard_normal((P + N, d)) for _ in range(4))
    o_all, _, _ = bc.linattn_block_causal_head(q, k, v, g, bt, 1e-6)
    S0, z0 = ol.linattn_state(k[:P], v[:P])
    o, _, _ = bc.linattn_block_causal_head(q[P:], k[P:], v[P:], g[P:], bt, 1e-6, None, S0, z0)
    assert _rel_err(o, o_all[P:]) < 1e-13


def pin_rows_match_full():
    rng = _rng(6)
    spec = ol.RopeSpec(4, 2, 5, 6, 6, 4)
    B, H, N, d, bt = 1, 2, spec.n_tokens, 16, 10
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    full, _ = bc.linattn_forward_block_causal(q, k, v, g, bt, 1e-6, spec)
    rows = np.array([0, 9, 10, 25, 39])
    part = bc.linattn_block_causal_rows(q, k, v, g, bt, rows, 1e-6, spec)
    for (b, h), o in part.items():
        assert _rel_err(o, full[b, h][rows]) < 1e-13


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_block_oracle_pin(pin):
    pin()


def test_blocks_must_divide_the_tokens():
    with pytest.raises(ValueError):
        bc.linattn_block_causal_head(np.ones((5, 2)), np.ones((5, 2)), np.ones((5, 2)),
                                     np.ones((5, 2)), 2, 1e-6)


# ------------------------------------------------------- planted mistakes ---

_ORIG_HEAD = bc.linattn_block_causal_head
_ORIG_ANGLES = bc.block_angles


def _mutant_own_block_excluded(q, k, v, g, block_tokens, eps, angles=None, S0=None, z0=None):
    N, d = q.shape
    S = np.zeros((d, d)) if S0 is None else np.array(S0, dtype=np.float64)
    z = np.zeros(d) if z0 is None else np.array(z0, dtype=np.float64)
    out = np.empty((N, d))
    for b in range(N // block_tokens):
        sl = slice(b * block_tokens, (b + 1) * block_tokens)
        ang = None if angles is None else angles[sl]
        out[sl] = ol.linattn_apply(q[sl], g[sl], S, z, eps, ang)
        Sb, zb = ol.linattn_state(k[sl], v[sl], ang)
        S, z = S + Sb, z + zb
    return out, S, z


def _mutant_state_not_carried(q, k, v, g, block_tokens, eps, angles=None, S0=None, z0=None):
    N, d = q.shape
    out = np.empty((N, d))
    S, z = np.zeros((d, d)), np.zeros(d)
    for b in range(N // block_tokens):
        sl = slice(b * block_tokens, (b + 1) * block_tokens)
        ang = None if angles is None else angles[sl]
        S, z = ol.linattn_state(k[sl], v[sl], ang)
        out[sl] = ol.linattn_apply(q[sl], g[sl], S, z, eps, ang)
    return out, S, z


def _mutant_state_in_ignored(q, k, v, g, block_tokens, eps, angles=None, S0=None, z0=None):
    return _ORIG_HEAD(q, k, v, g, block_tokens, eps, angles)


def _mutant_offset_ignored(rope, N, d, rope_offset=0):
    return _ORIG_ANGLES(rope, N, d, 0)


MUTANTS = {
    "own_block_excluded": ("linattn_block_causal_head", _mutant_own_block_excluded),
    "state_not_carried": ("linattn_block_causal_head", _mutant_state_not_carried),
    "state_in_ignored": ("linattn_block_causal_head", _mutant_state_in_ignored),
    "rope_offset_ignored": ("block_angles", _mutant_offset_ignored),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_block_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(bc, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant!r}"
