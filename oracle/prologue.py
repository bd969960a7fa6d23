"""fp64 CPU oracle for the fused input prologue of the KDA mixer.

TEST INFRASTRUCTURE ONLY.  Like the rest of ``oracle/``, only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
it imports nothing from the CUDA library.

What the layer does to its raw projections before the recurrence
("Linear Attention, From Scratch to Kimi 3", sec. 6, "Exactly how K3
computes the forget values", and sec. 7, "Q/K normalization and query
scaling"):

* q and k are L2-normalised per head (the query scale 1/sqrt(d_k) stays the
  recurrence's ``scale`` argument);
* beta = sigmoid(raw beta) ("applies sigmoid inside the kernel");
* the log retention is -5 * sigmoid(.) of the token's gate projection g,
  shifted by a learned per-channel bias b and scaled by one learned
  sensitivity per head, A_log.

Readings: the gate's formula is stripped from the page text; the page fixes
a sigmoid, a factor of -5 giving a log retention in (-5, 0), and the three
ingredients.  We take log_alpha = -5 * sigmoid(exp(A_log[h]) * (g + b[h, j])):
the sensitivity acts inside the sigmoid (outside it would leave (-5, 0)),
and A_log is a logarithm, so exp(A_log) > 0.  The L2 norm is
x / sqrt(sum x^2 + 1e-6) (the epsilon keeps a zero vector at zero).

Parity partly unpinned: the pins fix the range, the midpoint, monotonicity
and the closed forms; where exp(A_log) enters the gate is this reading's
choice, which no printed value checks.
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp(-x) = inf for x < -709 gives the exact limit 0
        return 1.0 / (1.0 + np.exp(-x))


def l2_normalise(x):
    """Per head (last axis): x / sqrt(sum(x^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def k3_log_alpha(g, gate_bias, A_log):
    """g [T, H, d_k] raw gate projection; gate_bias [H, d_k]; A_log [H]."""
    g = np.asarray(g, dtype=np.float64)
    z = np.exp(np.asarray(A_log, dtype=np.float64))[None, :, None] * (
        g + np.asarray(gate_bias, dtype=np.float64)[None])
    return -5.0 * sigmoid(z)


def apply(q, k, beta, g, *, l2norm=False, beta_logits=False, gate=None):
    """The transformed (q, k, beta, log_alpha), fp64.  gate = (bias, A_log)
    turns g from gate logits into log retentions; otherwise g is returned as
    given (already log_alpha)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if l2norm:
        q, k = l2_normalise(q), l2_normalise(k)
    b = sigmoid(beta) if beta_logits else np.asarray(beta, dtype=np.float64)
    la = k3_log_alpha(g, *gate) if gate is not None else np.asarray(g, dtype=np.float64)
    return q, k, b, la
