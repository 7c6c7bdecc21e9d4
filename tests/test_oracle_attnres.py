"""Pins for the AttnRes aggregation oracle (oracle/attnres.py), checked
against mathematics other than itself.

- Library routines: the weights equal torch's rms_norm followed by torch's
  softmax over the sources, in float64.
- Closed forms: w = 0 gives the mean of the sources; one source gives itself
  for any w; a query aligned with one normalised source, scaled up, selects
  that source.
- Invariants: a positive scale of a source leaves every weight unchanged
  (the keys are normalised; the values are not); permuting the sources
  changes nothing; tokens are independent (a token's output depends on its
  own rows only).

``test_attnres_pins_catch_planted_mistakes`` plants plausible mistakes in the
oracle and checks that each one fails a pin.
"""
import numpy as np
import pytest
import torch

import oracle.attnres as oa


def _rng(extra=0):
    return np.random.default_rng(4242 + extra)


def _rel_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _case(seed, M=4, T=6, C=32):
    rng = _rng(seed)
    s = rng.standard_normal((M, T, C)) * (1.0 + np.arange(M))[:, None, None]
    w = rng.standard_normal(C) / np.sqrt(C) * 3.0
    return s, w


def pin_library_rms_norm_and_softmax():
    s, w = _case(1)
    eps = 1e-6
    st = torch.from_numpy(s)
    k = torch.nn.functional.rms_norm(st, (s.shape[2],), eps=eps)
    a = torch.softmax(k @ torch.from_numpy(w), dim=0)
    assert _rel_err(oa.attnres_weights(s, w, eps), a.numpy()) < 1e-13
    want = (a[:, :, None] * st).sum(dim=0).numpy()
    assert _rel_err(oa.attnres_aggregate(s, w, eps), want) < 1e-13


def pin_zero_query_gives_mean():
    s, w = _case(2)
    assert _rel_err(oa.attnres_aggregate(s, np.zeros_like(w)), s.mean(axis=0)) < 1e-14


def pin_one_source_is_identity():
    s, w = _case(3, M=1)
    assert _rel_err(oa.attnres_aggregate(s, w), s[0]) < 1e-15


def pin_aligned_query_selects_source():
    s, _ = _case(4, M=3, T=1, C=64)
    k1 = s[1, 0] / np.sqrt(np.mean(s[1, 0] ** 2) + 1e-6)
    w = 200.0 * k1 / np.linalg.norm(k1) ** 2 * 1.0      # w . k_1 = 200, others far below
    got = oa.attnres_aggregate(s, w)
    assert _rel_err(got, s[1]) < 1e-12


def pin_source_scale_keeps_weights():
    s, w = _case(5)
    scaled = s.copy()
    scaled[2] *= 7.5
    a = oa.attnres_weights(s, w, 0.0)
    b = oa.attnres_weights(scaled, w, 0.0)
    assert _rel_err(a, b) < 1e-13
    x = oa.attnres_aggregate(scaled, w, 0.0)
    want = (a[:, :, None] * scaled).sum(axis=0)
    assert _rel_err(x, want) < 1e-13


def pin_source_permutation():
    s, w = _case(6, M=5)
    perm = _rng(7).permutation(5)
    assert _rel_err(oa.attnres_aggregate(s[perm], w), oa.attnres_aggregate(s, w)) < 1e-14


def pin_tokens_independent():
    s, w = _case(8, T=9)
    full = oa.attnres_aggregate(s, w)
    for t in (0, 4, 8):
        assert _rel_err(oa.attnres_aggregate(s[:, t:t + 1], w), full[t:t + 1]) < 1e-15


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_attnres_oracle_pin(pin):
    pin()


# ------------------------------------------------------- planted mistakes ---

def _mutant_softmax_over_tokens(logits):
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _mutant_l2_norm(s, eps):
    return s / np.sqrt(np.sum(s * s, axis=-1, keepdims=True) + eps)


def _mutant_no_norm(s, eps):
    return s


def _mutant_normalised_values(sources, w, eps=1e-6):
    k = oa.attnres_keys(sources, eps)
    return np.einsum("nt,ntc->tc", oa.attnres_weights(sources, w, eps), k)


MUTANTS = {
    "softmax_over_tokens": ("_softmax_sources", _mutant_softmax_over_tokens),
    "l2_instead_of_rms": ("_rms_normalise", _mutant_l2_norm),
    "keys_not_normalised": ("_rms_normalise", _mutant_no_norm),
    "normalised_values": ("attnres_aggregate", _mutant_normalised_values),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_attnres_pins_catch_planted_mistakes(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(oa, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant!r}"
