"""Pins for the fp64 oracle, checked against mathematics other than itself.

Each ``pin_*`` below checks the oracle against something it does not compute
the same way: a hand-worked example, the O(N^2) quadratic form of linear
attention, RoFormer's complex-number form of the rotary embedding, closed
forms (a single token, a one-hot scatter-add) and invariants (constant values,
token permutations, the gate's limits, rotation by a constant angle).

``test_pins_catch_planted_mistakes`` plants plausible mistakes in the oracle
(on the CPU) and checks that each one fails at least one pin.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle.linattn as ol

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG_SEED = 1234


def _rng(extra=0):
    return np.random.default_rng(RNG_SEED + extra)


def _rand_head(N, d, rng, gate_scale=1.0):
    q = rng.standard_normal((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    g = gate_scale * rng.standard_normal((N, d))
    return q, k, v, g


def _rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- golden ----

def _parse_value(tok):
    sign = -1.0 if tok.startswith("-") else 1.0
    body = tok.lstrip("+-")
    if body == "ln3":
        return sign * math.log(3.0)
    return sign * float(Fraction(body))


def _load_golden(name):
    data = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows = [[_parse_value(t) for t in r.split()] for r in rest.split("|")]
            data[key] = np.array(rows, dtype=np.float64)
    return data


def pin_golden_hand_example():
    gd = _load_golden("hand_example_norope.txt")
    eps = float(gd["eps"][0, 0])
    S, z = ol.linattn_state(gd["k"], gd["v"])
    assert np.array_equal(S, gd["S"]), (S, gd["S"])
    assert np.array_equal(z, gd["z"][0]), (z, gd["z"])
    o = ol.linattn_head(gd["q"], gd["k"], gd["v"], gd["g"], eps)
    assert _rel_err(o, gd["o"]) < 1e-15, (o, gd["o"])


# ----------------------------------------------------- quadratic form -------

def _bruteforce(q, k, v, g, eps, angles=None):
    """o_i = sigmoid(g_i) sum_j w_ij v_j / (sum_j (phi(q_i).phi(k_j)) + eps).

    Without RoPE, w_ij = phi(q_i).phi(k_j).  With RoPE, w_ij follows RoFormer's
    complex form: each pair is X_p = x_{2p} + i x_{2p+1}, and the rotated dot
    product is Re sum_p conj(Q_ip) K_jp exp(i (a_jp - a_ip)); the denominator
    keeps the unrotated features.
    """
    qp = np.maximum(q, 0.0)
    kp = np.maximum(k, 0.0)
    dots = qp @ kp.T                         # N x N, unrotated
    if angles is None:
        w = dots
    else:
        Qc = qp[:, 0::2] + 1j * qp[:, 1::2]
        Kc = kp[:, 0::2] + 1j * kp[:, 1::2]
        N = q.shape[0]
        w = np.empty((N, N))
        for i in range(N):
            phase = np.exp(1j * (angles - angles[i][None, :]))   # [N, d/2]
            w[i] = np.real((np.conj(Qc[i])[None, :] * Kc * phase).sum(axis=1))
    num = w @ v
    den = dots.sum(axis=1) + eps
    gate = np.array([[1.0 / (1.0 + math.exp(-x)) for x in row] for row in g])
    return gate * num / den[:, None]


def pin_bruteforce_norope_small():
    for n_idx, (N, d) in enumerate([(1, 4), (2, 8), (7, 16), (129, 128)]):
        q, k, v, g = _rand_head(N, d, _rng(n_idx))
        o = ol.linattn_head(q, k, v, g, 1e-6)
        ref = _bruteforce(q, k, v, g, 1e-6)
        assert _rel_err(o, ref) < 1e-12, (N, d, _rel_err(o, ref))


def pin_bruteforce_norope_eps_large():
    # a large eps makes the eps placement visible in every row
    q, k, v, g = _rand_head(9, 8, _rng(11))
    o = ol.linattn_head(q, k, v, g, 3.0)
    ref = _bruteforce(q, k, v, g, 3.0)
    assert _rel_err(o, ref) < 1e-12


def pin_bruteforce_rope_random_angles():
    N, d = 11, 12
    rng = _rng(21)
    q, k, v, g = _rand_head(N, d, rng)
    angles = rng.uniform(-4.0, 4.0, size=(N, d // 2))
    o = ol.linattn_head(q, k, v, g, 1e-6, angles)
    ref = _bruteforce(q, k, v, g, 1e-6, angles)
    assert _rel_err(o, ref) < 1e-12, _rel_err(o, ref)


def pin_bruteforce_rope_grid():
    spec = ol.RopeSpec(3, 4, 5, dt=8, dh=6, dw=6, base=10000.0)   # N = 60, d = 20
    rng = _rng(22)
    q, k, v, g = _rand_head(spec.n_tokens, spec.d, rng)
    angles = ol.rope3d_angles(spec)
    o = ol.linattn_forward(q[None, None], k[None, None], v[None, None], g[None, None],
                           1e-6, spec)[0, 0]
    ref = _bruteforce(q, k, v, g, 1e-6, angles)
    assert _rel_err(o, ref) < 1e-12


def pin_bruteforce_tiny_workload_shape():
    # the shape of the smallest workload: B=1, H=2, N=256, d=128
    rng = _rng(31)
    for _ in range(2):
        q, k, v, g = _rand_head(256, 128, rng)
        o = ol.linattn_head(q, k, v, g, 1e-6)
        assert _rel_err(o, _bruteforce(q, k, v, g, 1e-6)) < 1e-12


# -------------------------------------------------------- RoPE table --------

def pin_rope_positions_row_major():
    spec = ol.RopeSpec(2, 3, 4, dt=2, dh=2, dw=2)
    t, h, w = ol.rope3d_positions(spec)
    # token 23 is the last one: (1, 2, 3); token 5 = (0*3 + 1)*4 + 1
    assert (t[23], h[23], w[23]) == (1, 2, 3)
    assert (t[5], h[5], w[5]) == (0, 1, 1)
    assert (t[12], h[12], w[12]) == (1, 0, 0)


def pin_rope_bands_move_one_axis_each():
    dt, dh, dw = 44, 42, 42
    for axis, grid in enumerate([(7, 1, 1), (1, 7, 1), (1, 1, 7)]):
        spec = ol.RopeSpec(*grid, dt=dt, dh=dh, dw=dw)
        a = ol.rope3d_angles(spec)
        bounds = [(0, dt // 2), (dt // 2, (dt + dh) // 2), ((dt + dh) // 2, 64)]
        for band, (lo, hi) in enumerate(bounds):
            moving = np.any(a[:, lo:hi] != 0.0)
            assert moving == (band == axis), (axis, band)
        lo, hi = bounds[axis]
        width = (dt, dh, dw)[axis]
        # pair 0 of the band turns by exactly one radian per position
        assert np.array_equal(a[:, lo], np.arange(7, dtype=np.float64))
        # the ladder falls by base^(-2/width) from one pair to the next
        ratio = a[3, lo + 1:hi] / a[3, lo:hi - 1]
        assert np.allclose(ratio, 10000.0 ** (-2.0 / width), rtol=1e-13, atol=0)
        # the last pair of the band turns at base^(-(width-2)/width) per position
        assert math.isclose(a[1, hi - 1], 10000.0 ** (-(width - 2) / width), rel_tol=1e-13)


def pin_rope_origin_and_separability():
    spec = ol.RopeSpec(3, 4, 5, dt=44, dh=42, dw=42)
    a = ol.rope3d_angles(spec)
    assert np.all(a[0] == 0.0)
    t, h, w = ol.rope3d_positions(spec)
    # tokens that share a coordinate share that band's angles, whatever the others are
    same_t = np.where(t == 2)[0]
    assert np.all(a[same_t, :22] == a[same_t[0], :22])
    same_w = np.where(w == 3)[0]
    assert np.all(a[same_w, 43:] == a[same_w[0], 43:])


def pin_rotation_is_orthogonal():
    rng = _rng(41)
    x = rng.standard_normal((50, 128))
    ang = rng.uniform(-100, 100, size=(50, 64))
    y = ol.rope_rotate(x, ang)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # a quarter turn maps (1, 0) to (0, 1): the complex product with exp(i pi/2)
    e = np.zeros((1, 2))
    e[0, 0] = 1.0
    r = ol.rope_rotate(e, np.array([[math.pi / 2]]))
    assert abs(r[0, 0]) < 1e-15 and abs(r[0, 1] - 1.0) < 1e-15


# ------------------------------------------------ closed forms/invariants ----

def pin_single_token_closed_form():
    rng = _rng(51)
    spec = ol.RopeSpec(1, 1, 1, dt=44, dh=42, dw=42)
    for rope in (None, spec):
        q, k, v, g = _rand_head(1, 128, rng)
        q = np.abs(q)
        k = np.abs(k)
        o = ol.linattn_forward(q[None, None], k[None, None], v[None, None], g[None, None],
                               1e-6, rope)[0, 0, 0]
        s = float(np.dot(q[0], k[0]))
        expect = v[0] * s / (s + 1e-6) / (1.0 + np.exp(-g[0]))
        assert _rel_err(o, expect) < 1e-14
    # one token away from the origin: the rotation is the same for q and k and cancels
    spec = ol.RopeSpec(1, 1, 1, dt=44, dh=42, dw=42)
    q, k, v, g = _rand_head(1, 128, rng)
    ang = rng.uniform(-9, 9, size=(1, 64))
    o = ol.linattn_head(q, k, v, g, 1e-6, ang)
    s = float(np.dot(np.maximum(q[0], 0), np.maximum(k[0], 0)))
    expect = v[0] * s / (s + 1e-6) / (1.0 + np.exp(-g[0]))
    assert _rel_err(o[0], expect) < 1e-13


def pin_one_hot_state_is_scatter_add():
    rng = _rng(61)
    N, d = 40, 16
    bucket = rng.integers(0, d, size=N)
    scale = rng.uniform(0.5, 2.0, size=N)
    k = -np.abs(rng.standard_normal((N, d)))        # phi(k) = 0 except the hot entry
    k[np.arange(N), bucket] = scale
    v = rng.standard_normal((N, d))
    S, z = ol.linattn_state(k, v)
    expect_S = np.zeros((d, d))
    np.add.at(expect_S, bucket, scale[:, None] * v)
    expect_z = np.bincount(bucket, weights=scale, minlength=d)
    assert np.allclose(S, expect_S, rtol=1e-14, atol=1e-14)
    assert np.allclose(z, expect_z, rtol=1e-14, atol=1e-14)


def pin_constant_values_pass_through():
    rng = _rng(71)
    N, d = 33, 32
    q, k, _, _ = _rand_head(N, d, rng)
    c = rng.standard_normal(d)
    v = np.tile(c, (N, 1))
    g = np.full((N, d), 40.0)                      # sigmoid(40) == 1 in float64
    o = ol.linattn_head(q, k, v, g, 1e-6)
    # sum_j (phi(q).phi(k_j)) c / (sum_j phi(q).phi(k_j) + eps) = c * a/(a + eps)
    a = np.maximum(q, 0) @ np.maximum(k, 0).sum(axis=0)
    assert _rel_err(o, np.outer(a / (a + 1e-6), c)) < 1e-13
    assert np.max(np.abs(o - c)) < 1e-4 * np.max(np.abs(c))


def pin_permutation_equivariance():
    rng = _rng(81)
    N, d = 30, 16
    q, k, v, g = _rand_head(N, d, rng)
    perm = rng.permutation(N)
    o = ol.linattn_head(q, k, v, g, 1e-6)
    op = ol.linattn_head(q[perm], k[perm], v[perm], g[perm], 1e-6)
    assert _rel_err(op, o[perm]) < 1e-13


def pin_gate_limits():
    rng = _rng(91)
    q, k, v, _ = _rand_head(17, 16, rng)
    sat = ol.linattn_head(q, k, v, np.full_like(q, 40.0), 1e-6)
    half = ol.linattn_head(q, k, v, np.zeros_like(q), 1e-6)
    assert np.array_equal(half * 2.0, sat)
    # saturated gate == ungated linear attention (quadratic form without a gate)
    qp, kp = np.maximum(q, 0), np.maximum(k, 0)
    w = qp @ kp.T
    assert _rel_err(sat, (w @ v) / (w.sum(axis=1) + 1e-6)[:, None]) < 1e-12
    # a very negative gate closes the output
    shut = ol.linattn_head(q, k, v, np.full_like(q, -800.0), 1e-6)
    assert np.all(shut == 0.0)


def pin_zero_angles_equal_no_rope():
    rng = _rng(101)
    q, k, v, g = _rand_head(25, 24, rng)
    a = ol.linattn_head(q, k, v, g, 1e-6, np.zeros((25, 12)))
    b = ol.linattn_head(q, k, v, g, 1e-6)
    assert np.array_equal(a, b)


def pin_rope_shift_invariance():
    # moving every token by the same offset (per pair) leaves the output unchanged:
    # the rotated dot product depends only on angle differences
    spec = ol.RopeSpec(4, 3, 5, dt=8, dh=8, dw=8)
    rng = _rng(111)
    q, k, v, g = _rand_head(spec.n_tokens, spec.d, rng)
    a = ol.rope3d_angles(spec)
    shift_t = 7.0 * ol.rope3d_thetas(8, 10000.0)             # t origin moved by 7
    a2 = a.copy()
    a2[:, :4] += shift_t[None, :]
    o1 = ol.linattn_head(q, k, v, g, 1e-6, a)
    o2 = ol.linattn_head(q, k, v, g, 1e-6, a2)
    assert _rel_err(o2, o1) < 1e-11
    # but a shift of q's angles alone does change it
    o3 = ol.linattn_apply(q, g, *ol.linattn_state(k, v, a), 1e-6, a2)
    assert _rel_err(o3, o1) > 1e-3


def pin_rope_leaves_denominator_unrotated():
    # v = 1 everywhere and a saturated gate leave o_i = num_i / den_i in each column;
    # num_i is the rotated dot product summed over j (RoFormer's complex form), den_i
    # the unrotated one.
    spec = ol.RopeSpec(2, 3, 4, dt=8, dh=4, dw=4)
    rng = _rng(121)
    N, d = spec.n_tokens, spec.d
    q, k, _, _ = _rand_head(N, d, rng)
    ones = np.ones((N, d))
    g = np.full((N, d), 40.0)
    a = ol.rope3d_angles(spec)
    o_rope = ol.linattn_head(q, k, ones, g, 1e-6, a)
    # num_i = (R_i phi q_i) . sum_j R_j phi k_j  ;  den_i = phi q_i . z + eps
    qp, kp = np.maximum(q, 0), np.maximum(k, 0)
    num = np.array([
        sum(np.real(np.vdot((qp[i, 0::2] + 1j * qp[i, 1::2]) * np.exp(1j * a[i]),
                            (kp[j, 0::2] + 1j * kp[j, 1::2]) * np.exp(1j * a[j])))
            for j in range(N))
        for i in range(N)])
    den = qp @ kp.sum(axis=0) + 1e-6
    assert _rel_err(o_rope[:, 0], num / den) < 1e-11


def pin_dead_query_row_is_zero():
    rng = _rng(131)
    q, k, v, g = _rand_head(10, 16, rng)
    q[3] = -np.abs(q[3])                           # phi(q_3) = 0: num = 0, den = eps
    o = ol.linattn_head(q, k, v, g, 1e-6)
    assert np.all(o[3] == 0.0)
    assert np.all(np.isfinite(o))


def pin_forward_rows_matches_full():
    rng = _rng(141)
    B, H, N, d = 1, 2, 40, 16
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    full = ol.linattn_forward(q, k, v, g, 1e-6)
    rows = np.array([0, 7, 39])
    part = ol.linattn_forward_rows(q, k, v, g, rows, 1e-6)
    for (b, h), o in part.items():
        assert _rel_err(o, full[b, h][rows]) < 1e-14


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


# ------------------------------------------------------- planted mistakes ---

def _mutant_no_eps(q, g, S, z, eps, angles=None):
    return _ORIG["linattn_apply"](q, g, S, z, 0.0 * eps, angles)


def _mutant_transposed_state(q, g, S, z, eps, angles=None):
    return _ORIG["linattn_apply"](q, g, S.T, z, eps, angles)


def _mutant_rotation_sign(x, angles):
    return _ORIG["rope_rotate"](x, -angles)


def _mutant_halves_pairing(x, angles):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[1]
    c, s = np.cos(angles), np.sin(angles)
    lo, hi = x[:, : d // 2], x[:, d // 2:]
    return np.concatenate([lo * c - hi * s, lo * s + hi * c], axis=1)


def _mutant_no_relu(x):
    return np.asarray(x, dtype=np.float64)


def _mutant_gate_sign(g):
    return _ORIG["sigmoid"](-np.asarray(g))


def _mutant_rotated_denominator(q, g, S, z, eps, angles=None):
    qp = ol.feature_map(q)
    qr = qp if angles is None else ol.rope_rotate(qp, angles)
    return ol.sigmoid(g) * (qr @ S) / (qr @ z + eps)[:, None]


def _mutant_rope_q_only(k, v, angles=None):
    return _ORIG["linattn_state"](k, v, None)


def _mutant_ladder(width, base):
    j = np.arange(width // 2, dtype=np.float64)
    return base ** (-j / width)


def _mutant_band_order(spec):
    t, h, w = ol.rope3d_positions(spec)
    bands = []
    for pos, width in ((w, spec.dw), (h, spec.dh), (t, spec.dt)):
        bands.append(np.outer(pos.astype(np.float64), ol.rope3d_thetas(width, spec.base)))
    return np.concatenate(bands, axis=1)


def _mutant_column_major_tokens(spec):
    n = np.arange(spec.n_tokens, dtype=np.int64)
    t = n % spec.T
    h = (n // spec.T) % spec.Hs
    w = n // (spec.T * spec.Hs)
    return t, h, w


_ORIG = {name: getattr(ol, name) for name in
         ("linattn_apply", "rope_rotate", "sigmoid", "linattn_state")}

MUTANTS = {
    "dropped_eps": ("linattn_apply", _mutant_no_eps),
    "transposed_state": ("linattn_apply", _mutant_transposed_state),
    "rotation_sign": ("rope_rotate", _mutant_rotation_sign),
    "halves_pairing": ("rope_rotate", _mutant_halves_pairing),
    "no_relu": ("feature_map", _mutant_no_relu),
    "gate_sign": ("sigmoid", _mutant_gate_sign),
    "rotated_denominator": ("linattn_apply", _mutant_rotated_denominator),
    "rope_on_q_only": ("linattn_state", _mutant_rope_q_only),
    "ladder_exponent": ("rope3d_thetas", _mutant_ladder),
    "band_order": ("rope3d_angles", _mutant_band_order),
    "token_order": ("rope3d_positions", _mutant_column_major_tokens),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(ol, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant!r}"
