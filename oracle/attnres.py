"""Plain fp64 CPU oracle for the Block Attention Residual (AttnRes) aggregation.

TEST INFRASTRUCTURE ONLY, like ``oracle.linattn``: nothing in the library
imports this module and it shares no code with the CUDA path.

Sources.  "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section
"Architecture"): both models use a shared, timestep-independent Attention
Residual aggregation in blocks of eight layers.  The arXiv abstract of
2607.21553 and the article "SANA-Video 2.0: Hybrid Attention for Faster
High-Resolution Video Generation" (its key points, "Attention residuals
across depth") say that completed block summaries are routed into later
linear layers.  No page gives a formula.

Reading.  This is the plainest reading the pages support, and the design notes
list it:

* the layers form blocks of eight; each completed block leaves one summary
  s_n of shape T x C (T tokens, C the hidden size); a layer's input may also
  include the running summary of its own block as one more source;
* a later layer aggregates its M sources token by token, by attention over
  depth.  Each source is a key after an RMS normalisation, and the query is one
  learned vector w of length C.  That w is shared by all tokens and does not
  depend on the diffusion timestep, and it absorbs the normalisation's gain:

      k_n(t)  = s_n(t) / sqrt(mean_c s_n(t, c)^2 + eps)
      a_n(t)  = softmax over n of (w . k_n(t))
      x(t)    = sum_n a_n(t) s_n(t)

  The values are the raw summaries.

Every function works in float64 on numpy arrays, in the order of the formula.
"""
from __future__ import annotations

import numpy as np

__all__ = ["attnres_keys", "attnres_weights", "attnres_aggregate"]


def _rms_normalise(s, eps):
    """k = s / sqrt(mean over the last axis of s^2 + eps)."""
    return s / np.sqrt(np.mean(s * s, axis=-1, keepdims=True) + eps)


def _softmax_sources(logits):
    """Softmax over axis 0 (the sources)."""
    e = np.exp(logits - logits.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def attnres_keys(sources, eps):
    """k_n(t): the RMS-normalised sources, [M, T, C]."""
    return _rms_normalise(np.asarray(sources, dtype=np.float64), eps)


def attnres_weights(sources, w, eps):
    """a_n(t): the attention over the M sources of every token, [M, T]."""
    k = attnres_keys(sources, eps)
    logits = k @ np.asarray(w, dtype=np.float64)
    return _softmax_sources(logits)


def attnres_aggregate(sources, w, eps=1e-6):
    """x(t) = sum_n a_n(t) s_n(t) for sources [M, T, C] and the query w [C]; returns [T, C]."""
    s = np.asarray(sources, dtype=np.float64)
    if s.ndim != 3 or np.asarray(w).shape != (s.shape[2],):
        raise ValueError("sources must be [M, T, C] and w [C]")
    a = attnres_weights(s, w, eps)
    return np.einsum("nt,ntc->tc", a, s)
