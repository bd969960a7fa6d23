"""fp64 CPU oracle for the short causal convolution of the KDA layer.

TEST INFRASTRUCTURE ONLY.  Like the rest of ``oracle/``, only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
it imports nothing from the CUDA library.

What it computes ("Linear Attention, From Scratch to Kimi 3", sec. 7, "The
short convolution is temporal, not channel mixing"): every channel c owns a
W-tap filter over time and nothing mixes channels; q, k and v each have
their own convolution and their own cache of the most recent
pre-convolution inputs, which decode extends by one token at a time; packed
sequences (cu_seqlens, sec. 9) never see each other's tokens.

Readings (the tap formula itself is not in the page text): the output at
token t of a sequence is

    y[t, c] = sum_{i=0}^{W-1} w[c, i] * x[t - W + 1 + i, c]   (+ bias[c])

followed by SiLU(z) = z * sigmoid(z) when asked; inputs before a sequence's
first token come from its cache (slot W-1 the most recent), or are zero
without one; after the call the cache holds the sequence's W most recent
inputs.  A decode step is the same filter over the cache shifted by one with
the new token appended.

Parity partly unpinned: the pins are closed forms of this reading (impulse
and step responses, a hand-worked example, decode equal to prefill); the
tap order itself is the reading's, since the page's formula is stripped.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def _act(z: np.ndarray, silu: bool) -> np.ndarray:
    return z / (1.0 + np.exp(-z)) if silu else z


def short_conv(x, weight, bias=None, cu_seqlens=None, cache=None, silu: bool = False
               ) -> Tuple[np.ndarray, np.ndarray]:
    """Prefill over packed sequences.

    x [T, C]; weight [C, W]; bias [C] or None; cu_seqlens [N + 1] or None (one
    sequence); cache [N, C, W] or None.  Returns (y [T, C], cache_out [N, C, W]),
    float64.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    T, C = x.shape
    W = w.shape[1]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    cin = (np.zeros((N, C, W)) if cache is None else np.asarray(cache, dtype=np.float64))
    y = np.zeros((T, C))
    cout = np.zeros((N, C, W))
    for s in range(N):
        a, b = int(cu[s]), int(cu[s + 1])
        # the sequence's input history: its cache (oldest first), then its tokens
        hist = np.concatenate([cin[s].T, x[a:b]], axis=0)        # [W + L, C]
        for j in range(b - a):
            z = np.zeros(C)
            for i in range(W):
                # tap i sees x[t - W + 1 + i]: history row (W + j) - (W - 1) + i
                z += w[:, i] * hist[j + 1 + i]
            if bias is not None:
                z += np.asarray(bias, dtype=np.float64)
            y[a + j] = _act(z, silu)
        cout[s] = hist[-W:].T
    return y, cout


def short_conv_step(x, weight, bias=None, cache=None, silu: bool = False
                    ) -> Tuple[np.ndarray, np.ndarray]:
    """One decode token per sequence: x [N, C]; cache [N, C, W] (updated copy
    returned).  Shift the cache by one, append x, filter."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    N, C = x.shape
    W = w.shape[1]
    c = np.zeros((N, C, W)) if cache is None else np.array(cache, dtype=np.float64)
    c[:, :, :-1] = c[:, :, 1:]
    c[:, :, -1] = x
    z = np.einsum("ncw,cw->nc", c, w)
    if bias is not None:
        z = z + np.asarray(bias, dtype=np.float64)[None, :]
    return _act(z, silu), c
