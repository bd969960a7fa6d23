"""fp64 CPU oracle for the gradients of the KDA recurrence.

TEST INFRASTRUCTURE ONLY.  Like the rest of ``oracle/``, only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
it imports nothing from the CUDA library.

The pages derive no gradients ("Kimi Unveils Delta Attention and K3
Architecture Updates", sec. 6 and 6.6, say only that the chunkwise form
serves training).  This is reverse-mode differentiation of the token
recurrence of sec. 4.1, written out step by step.  Forward, per token:

    Sb = Diag(a) S_prev            a = exp(log_alpha_t)
    p  = Sb^T k
    e  = b (v - p)
    S  = Sb + k e^T
    o  = S^T (s q)

Backward, per token in reverse, with dS the gradient of the loss in S (the
state after the token; at the end of a sequence, the final-state gradient):

    dS  += (s q) do^T                 o = S^T (s q)
    dq   = s S do
    dk   = dS e,   de = dS^T k        S = Sb + k e^T   (dSb = dS)
    db   = de . (v - p),  dv = b de,  dp = -b de
    dSb  = dS + k dp^T,   dk += Sb dp p = Sb^T k
    da_i = sum_j dSb_ij S_prev_ij,  dlog_alpha = a * da
    dS   = Diag(a) dSb                Sb = Diag(a) S_prev

and the gradient of the initial state is dS after the sequence's first token.
"""
from __future__ import annotations

import numpy as np


def recurrent_backward(q, k, v, log_alpha, beta, scale, initial_state=None, cu_seqlens=None,
                       d_out=None, d_final_state=None):
    """Gradients of (out, final_state) with respect to every input.

    Shapes as the forward oracle: q, k [T, H, d_k]; v [T, H, d_v]; log_alpha
    [T, H, d_k]; beta [T, H]; initial_state [N, H, d_k, d_v] or None;
    cu_seqlens [N + 1] or None; d_out [T, H, d_v] or None (zero); d_final_state
    [N, H, d_k, d_v] or None (zero).  Returns (dq, dk, dv, dlog_alpha, dbeta,
    d_initial_state), float64.
    """
    f = lambda x: np.asarray(x, dtype=np.float64)
    q, k, v, g, b = f(q), f(k), f(v), f(log_alpha), f(beta)
    T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    S0 = np.zeros((N, H, dk_, dv_)) if initial_state is None else f(initial_state)
    dO = np.zeros((T, H, dv_)) if d_out is None else f(d_out)
    dSf = np.zeros((N, H, dk_, dv_)) if d_final_state is None else f(d_final_state)
    gq, gk, gv, gg = (np.zeros_like(x) for x in (q, k, v, g))
    gb = np.zeros_like(b)
    gS0 = np.zeros_like(S0)
    for s in range(N):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            # forward, keeping what the reverse sweep needs
            S = S0[s, h].copy()
            saved = []
            for t in range(t0, t1):
                a = np.exp(g[t, h])
                Sp = S
                Sb = a[:, None] * Sp
                p = Sb.T @ k[t, h]
                e = b[t, h] * (v[t, h] - p)
                S = Sb + np.outer(k[t, h], e)
                saved.append((Sp, Sb, S, a, p, e))
            # reverse
            dS = dSf[s, h].copy()
            for t in range(t1 - 1, t0 - 1, -1):
                Sp, Sb, St, a, p, e = saved[t - t0]
                dS = dS + np.outer(scale * q[t, h], dO[t, h])
                gq[t, h] = scale * (St @ dO[t, h])
                dkt = dS @ e
                de = dS.T @ k[t, h]
                gb[t, h] = de @ (v[t, h] - p)
                gv[t, h] = b[t, h] * de
                dp = -b[t, h] * de
                dSb = dS + np.outer(k[t, h], dp)
                dkt = dkt + Sb @ dp
                gk[t, h] = dkt
                gg[t, h] = a * np.sum(dSb * Sp, axis=1)
                dS = a[:, None] * dSb
            gS0[s, h] = dS
    return gq, gk, gv, gg, gb, gS0
