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


def chunk_backward(q, k, v, log_alpha, beta, scale, initial_state=None, cu_seqlens=None,
                   d_out=None, d_final_state=None, chunk_size=64):
    """The same gradients, through the chunkwise form ("Kimi Unveils Delta
    Attention and K3 Architecture Updates", sec. 6): the blueprint of a
    chunk-parallel backward.  Per chunk (tokens i, j of the chunk; G the
    chunk-local cumulative log decay, G_l its last row; D_ij = exp(G_i - G_j)
    per key channel), the forward of sec. 6 is

        R    = tril_-1( Diag(b) [k_i . (D_ij * k_j)] )      A  = (I + R)^-1
        Aqk  = tril_0( s [q_i . (D_ij * k_j)] )
        W    = A Diag(b) (exp(G) * K),   U = A Diag(b) V,    E = U - W S0
        O    = (s exp(G) * Q) S0 + Aqk E
        S1   = Diag(exp(G_l)) S0 + K_end^T E,  K_end = exp(G_l - G) * K

    and its reverse-mode derivative, with dO and dS1 given (dS1 of a chunk is
    dS0 of the next; at the end of a sequence, the final-state gradient):

        dE   = Aqk^T dO + K_end dS1
        dS0  = (s exp(G) * Q)^T dO + Diag(exp(G_l)) dS1 - W^T dE
        dAqk = tril_0(dO E^T),   dK_end = E dS1^T,   dU = dE,   dW = -dE S0^T
        dA   = dU (Diag(b) V)^T + dW (Diag(b) exp(G) * K)^T
        dR   = tril_-1(-A^T dA A^T)                       (A = (I + R)^-1)

    then through the products above to q, k, v, b and G, and dlog_alpha as
    the reverse cumulative sum of dG within the chunk.  fp64, one head of one
    chunk at a time (no blocking beyond the chunks).  Returns the tuple of
    ``recurrent_backward``.
    """
    f = lambda x: np.asarray(x, dtype=np.float64)
    q, k, v, g, b = f(q), f(k), f(v), f(log_alpha), f(beta)
    T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    S0all = np.zeros((N, H, dk_, dv_)) if initial_state is None else f(initial_state)
    dO = np.zeros((T, H, dv_)) if d_out is None else f(d_out)
    dSf = np.zeros((N, H, dk_, dv_)) if d_final_state is None else f(d_final_state)
    gq, gk, gv, gg = (np.zeros_like(x) for x in (q, k, v, g))
    gb = np.zeros_like(b)
    gS0 = np.zeros_like(S0all)
    for s in range(N):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        starts = list(range(t0, t1, chunk_size))
        for h in range(H):
            # forward over the chunks: the state entering each, and each
            # chunk's intermediates
            S = S0all[s, h].copy()
            fwd = []
            for c0 in starts:
                c1 = min(c0 + chunk_size, t1)
                K, Q, V = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h]
                B = b[c0:c1, h]
                L = c1 - c0
                G = np.cumsum(g[c0:c1, h], axis=0)
                Gl = G[-1]
                Dx = np.exp(G[:, None, :] - G[None, :, :])           # [i, j, channel]
                low = np.tril(np.ones((L, L)), -1)
                low0 = np.tril(np.ones((L, L)))
                KK = np.einsum("ic,jc,ijc->ij", K, K, Dx)
                QK = np.einsum("ic,jc,ijc->ij", Q, K, Dx)
                R = low * (B[:, None] * KK)
                A = np.linalg.inv(np.eye(L) + R)
                Aqk = low0 * (scale * QK)
                KG = np.exp(G) * K
                W = A @ (B[:, None] * KG)
                U = A @ (B[:, None] * V)
                E = U - W @ S
                QG = scale * np.exp(G) * Q
                Kend = np.exp(Gl - G) * K
                fwd.append(dict(c0=c0, c1=c1, K=K, Q=Q, V=V, B=B, G=G, Gl=Gl, Dx=Dx, low=low,
                                low0=low0, KK=KK, QK=QK, A=A, Aqk=Aqk, KG=KG, W=W, E=E, QG=QG,
                                Kend=Kend, S0=S.copy()))
                S = np.exp(Gl)[:, None] * S + Kend.T @ E
            # reverse over the chunks
            dS1 = dSf[s, h].copy()
            for ch in reversed(fwd):
                c0, c1 = ch["c0"], ch["c1"]
                K, Q, V, B, G, Gl, Dx = ch["K"], ch["Q"], ch["V"], ch["B"], ch["G"], ch["Gl"], ch["Dx"]
                A, Aqk, KG, W, E, QG, Kend, S0 = (ch[x] for x in ("A", "Aqk", "KG", "W", "E",
                                                                   "QG", "Kend", "S0"))
                dOc = dO[c0:c1, h]
                dE = Aqk.T @ dOc + Kend @ dS1
                dQG = dOc @ S0.T
                dS0 = QG.T @ dOc + np.exp(Gl)[:, None] * dS1 - W.T @ dE
                dAqk = ch["low0"] * (dOc @ E.T)
                dKend = E @ dS1.T
                dGl = np.exp(Gl) * np.sum(S0 * dS1, axis=1)
                dU, dW = dE, -dE @ S0.T
                BV, BK = B[:, None] * V, B[:, None] * KG
                dA = dU @ BV.T + dW @ BK.T
                dBV, dBK = A.T @ dU, A.T @ dW
                dV = B[:, None] * dBV
                dB = np.sum(V * dBV, axis=1) + np.sum(KG * dBK, axis=1)
                dKG = B[:, None] * dBK
                dR = ch["low"] * (-(A.T @ dA @ A.T))
                # R_ij = b_i sum_c k_ic k_jc D_ijc
                dB += np.sum(dR * ch["KK"], axis=1)
                wR = (B[:, None] * dR)[:, :, None] * Dx                 # [i, j, c]
                dK = np.einsum("ijc,jc->ic", wR, K) + np.einsum("ijc,ic->jc", wR, K)
                tR = wR * K[:, None, :] * K[None, :, :]
                dG = tR.sum(axis=1) - tR.sum(axis=0)
                # Aqk_ij = s sum_c q_ic k_jc D_ijc
                wQ = (scale * dAqk)[:, :, None] * Dx
                dQ = np.einsum("ijc,jc->ic", wQ, K)
                dK += np.einsum("ijc,ic->jc", wQ, Q)
                tQ = wQ * Q[:, None, :] * K[None, :, :]
                dG += tQ.sum(axis=1) - tQ.sum(axis=0)
                # the elementwise exp(G) factors
                dK += np.exp(G) * dKG
                dG += KG * dKG
                dQ += scale * np.exp(G) * dQG
                dG += QG * dQG
                dK += np.exp(Gl - G) * dKend
                dG -= Kend * dKend
                dGl += np.sum(Kend * dKend, axis=0)
                dG[-1] += dGl
                # G = cumsum(log_alpha): dlog_alpha_t = sum_{i >= t} dG_i
                gg[c0:c1, h] = np.cumsum(dG[::-1], axis=0)[::-1]
                gq[c0:c1, h], gk[c0:c1, h], gv[c0:c1, h], gb[c0:c1, h] = dQ, dK, dV, dB
                dS1 = dS0
            gS0[s, h] = dS1
    return gq, gk, gv, gg, gb, gS0


def folded_chunk_backward(q, k, v, log_alpha, beta, scale, initial_state=None,
                          cu_seqlens=None, d_out=None, d_final_state=None, chunk_size=64):
    """The same gradients through the folded chunk form that the forward
    engine stores per chunk: M' = K_end^T W, P' = K_end^T A, Q' = Q_hat - Aqk W,
    Z = Aqk A (A = (I + R)^-1, W = A Diag(b)(exp(G) * K), Q_hat = s exp(G) * Q),
    with

        S1 = Diag(exp(G_l)) S0 + P' (b V) - M' S0,      O = Q' S0 + Z (b V).

    Reverse mode, chunk by chunk from the end (the serial part is the forward
    scan transposed, on the same images):

        dS0   = Q'^T dO + Diag(exp(G_l)) dS1 - M'^T dS1
        d(bV) = Z^T dO + P'^T dS1
        dQ'   = dO S0^T,   dZ = dO (bV)^T,   dP' = dS1 (bV)^T,   dM' = -dS1 S0^T
        dK_end = W dM'^T + A dP'^T,          dW = K_end dM' - Aqk^T dQ'
        dA    = K_end dP' + Aqk^T dZ + dW (b exp(G) K)^T
        dAqk  = tril_0(-dQ' W^T + dZ A^T),   dR = tril_-1(-A^T dA A^T)

    then the decayed products and exp(G) factors as in ``chunk_backward``.
    fp64.  Returns the tuple of ``recurrent_backward``.
    """
    f = lambda x: np.asarray(x, dtype=np.float64)
    q, k, v, g, b = f(q), f(k), f(v), f(log_alpha), f(beta)
    T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    S0all = np.zeros((N, H, dk_, dv_)) if initial_state is None else f(initial_state)
    dO = np.zeros((T, H, dv_)) if d_out is None else f(d_out)
    dSf = np.zeros((N, H, dk_, dv_)) if d_final_state is None else f(d_final_state)
    gq, gk, gv, gg = (np.zeros_like(x) for x in (q, k, v, g))
    gb = np.zeros_like(b)
    gS0 = np.zeros_like(S0all)
    for s in range(N):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            S = S0all[s, h].copy()
            fwd = []
            for c0 in range(t0, t1, chunk_size):
                c1 = min(c0 + chunk_size, t1)
                K, Q, V, B = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h], b[c0:c1, h]
                L = c1 - c0
                G = np.cumsum(g[c0:c1, h], axis=0)
                Gl = G[-1]
                Dx = np.exp(G[:, None, :] - G[None, :, :])
                low, low0 = np.tril(np.ones((L, L)), -1), np.tril(np.ones((L, L)))
                KK = np.einsum("ic,jc,ijc->ij", K, K, Dx)
                QK = np.einsum("ic,jc,ijc->ij", Q, K, Dx)
                A = np.linalg.inv(np.eye(L) + low * (B[:, None] * KK))
                Aqk = low0 * (scale * QK)
                KG = np.exp(G) * K
                W = A @ (B[:, None] * KG)
                Kend = np.exp(Gl - G) * K
                QG = scale * np.exp(G) * Q
                Mp, Pp, Qp, Zm = Kend.T @ W, Kend.T @ A, QG - Aqk @ W, Aqk @ A
                BV = B[:, None] * V
                fwd.append(dict(c0=c0, c1=c1, K=K, Q=Q, V=V, B=B, G=G, Gl=Gl, Dx=Dx, low=low,
                                low0=low0, KK=KK, A=A, Aqk=Aqk, KG=KG, W=W, Kend=Kend, QG=QG,
                                Mp=Mp, Pp=Pp, Qp=Qp, Zm=Zm, BV=BV, S0=S.copy()))
                S = np.exp(Gl)[:, None] * S + Pp @ BV - Mp @ S
            dS1 = dSf[s, h].copy()
            for ch in reversed(fwd):
                c0, c1 = ch["c0"], ch["c1"]
                K, Q, V, B, G, Gl, Dx = (ch[x] for x in ("K", "Q", "V", "B", "G", "Gl", "Dx"))
                A, Aqk, KG, W, Kend, QG = (ch[x] for x in ("A", "Aqk", "KG", "W", "Kend", "QG"))
                Mp, Pp, Qp, Zm, BV, S0 = (ch[x] for x in ("Mp", "Pp", "Qp", "Zm", "BV", "S0"))
                dOc = dO[c0:c1, h]
                # the serial part: the forward scan, transposed
                dS0 = Qp.T @ dOc + np.exp(Gl)[:, None] * dS1 - Mp.T @ dS1
                dBV = Zm.T @ dOc + Pp.T @ dS1
                dQp, dZ, dPp, dMp = dOc @ S0.T, dOc @ BV.T, dS1 @ BV.T, -dS1 @ S0.T
                dGl = np.exp(Gl) * np.sum(S0 * dS1, axis=1)
                # the folded factors
                dKend = W @ dMp.T + A @ dPp.T
                dW = Kend @ dMp - Aqk.T @ dQp
                dA = Kend @ dPp + Aqk.T @ dZ
                dAqk = ch["low0"] * (-dQp @ W.T + dZ @ A.T)
                dQG = dQp
                # W = A Diag(b) KG
                BK = B[:, None] * KG
                dA += dW @ BK.T
                dBK = A.T @ dW
                dKG = B[:, None] * dBK
                dB = np.sum(KG * dBK, axis=1) + np.sum(V * dBV, axis=1)
                dV = B[:, None] * dBV
                dR = ch["low"] * (-(A.T @ dA @ A.T))
                dB += np.sum(dR * ch["KK"], axis=1)
                wR = (B[:, None] * dR)[:, :, None] * Dx
                dK = np.einsum("ijc,jc->ic", wR, K) + np.einsum("ijc,ic->jc", wR, K)
                tR = wR * K[:, None, :] * K[None, :, :]
                dG = tR.sum(axis=1) - tR.sum(axis=0)
                wQ = (scale * dAqk)[:, :, None] * Dx
                dQ = np.einsum("ijc,jc->ic", wQ, K)
                dK += np.einsum("ijc,ic->jc", wQ, Q)
                tQ = wQ * Q[:, None, :] * K[None, :, :]
                dG += tQ.sum(axis=1) - tQ.sum(axis=0)
                dK += np.exp(G) * dKG
                dG += KG * dKG
                dQ += scale * np.exp(G) * dQG
                dG += QG * dQG
                dK += np.exp(Gl - G) * dKend
                dG -= Kend * dKend
                dGl += np.sum(Kend * dKend, axis=0)
                dG[-1] += dGl
                gg[c0:c1, h] = np.cumsum(dG[::-1], axis=0)[::-1]
                gq[c0:c1, h], gk[c0:c1, h], gv[c0:c1, h], gb[c0:c1, h] = dQ, dK, dV, dB
                dS1 = dS0
            gS0[s, h] = dS1
    return gq, gk, gv, gg, gb, gS0
