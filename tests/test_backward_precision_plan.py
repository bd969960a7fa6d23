"""Operand precision for a tensor-core chunkwise backward, on the CPU.

The chunkwise backward (the folded form of ``oracle.backward``) is a chain of
dense products per chunk.  On tensor cores each product rounds its operands
(tf32, f16 or bf16) and accumulates in fp32.  This test emulates that rounding
in every product of the folded chunk backward and compares the gradients
with the fp64 token-recurrence gradients, to fix the operand type that a GPU
kernel of this form has to use:

- tf32 operands keep every gradient well inside the bf16 parity bound at any
  gradient scale (tf32 has the fp32 exponent range);
- f16 operands match tf32 at unit scale but fail once the incoming gradients
  are small (1e-6: training-sized values fall into f16's subnormal range);
- bf16 operands cost about ten times the error of tf32.

The second half emulates the whole planned decomposition at tile level: the
forward recompute as the forward prep forms it (mid-chunk decay
factorisation with its range fallback, f16 factors, zero-padded partial
chunks), the forward scan (f16 state operand), X_c = Q'^T dO_c, the reverse
scan dS_c = Diag(Gamma_last) dS_{c+1} - M'^T dS_{c+1} + X_c, and the
per-chunk gradient pass, whose decayed-product gradients reuse the forward's
tf32 operands (K_tilde, Q_tilde, K_hat) in two products.  A dP'^T is taken as
U dS_{c+1}^T (U = A (beta V)), which halves the dlog_alpha error.
"""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, nerr


def _tf32(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)).astype(np.float64)


def _f16(x):
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


def _bf16(x):
    return inputs.bf16_round(np.asarray(x, np.float32)).astype(np.float64)


def _fp32(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def _emulated_chunk_backward(w, dO, rnd, C=64):
    """Folded chunk backward of one-sequence inputs, every product taken as
    rnd(a) @ rnd(b) with the result rounded to fp32.  The forward factors are
    exact (fp64): only the backward's products are under test."""
    mm = lambda a, b: _fp32(rnd(a) @ rnd(b))
    q, k, v, g, b = (np.asarray(x, np.float64) for x in (w.q, w.k, w.v, w.log_alpha, w.beta))
    T, H, d = q.shape
    s = w.scale
    gq, gk, gv, gg = (np.zeros_like(x) for x in (q, k, v, g))
    gb = np.zeros_like(b)
    for h in range(H):
        S, fwd = np.zeros((d, d)), []
        for c0 in range(0, T, C):
            c1 = min(c0 + C, T)
            L = c1 - c0
            K, Q, V, B = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h], b[c0:c1, h]
            G = np.cumsum(g[c0:c1, h], axis=0)
            Gl = G[-1]
            Dx = np.exp(G[:, None, :] - G[None, :, :])
            low, low0 = np.tril(np.ones((L, L)), -1), np.tril(np.ones((L, L)))
            KK = np.einsum("ic,jc,ijc->ij", K, K, Dx)
            A = np.linalg.inv(np.eye(L) + low * (B[:, None] * KK))
            Aqk = low0 * (s * np.einsum("ic,jc,ijc->ij", Q, K, Dx))
            KG = np.exp(G) * K
            W = A @ (B[:, None] * KG)
            Kend = np.exp(Gl - G) * K
            Mp, Pp, Zm = Kend.T @ W, Kend.T @ A, Aqk @ A
            Qp = s * np.exp(G) * Q - Aqk @ W
            BV = B[:, None] * V
            fwd.append((c0, c1, K, Q, V, B, G, Gl, Dx, low, low0, KK, A, Aqk, KG, W, Kend,
                        Mp, Pp, Qp, Zm, BV, S.copy()))
            S = np.exp(Gl)[:, None] * S + Pp @ BV - Mp @ S
        dS1 = np.zeros((d, d))
        for (c0, c1, K, Q, V, B, G, Gl, Dx, low, low0, KK, A, Aqk, KG, W, Kend,
             Mp, Pp, Qp, Zm, BV, S0) in reversed(fwd):
            dOc = dO[c0:c1, h]
            dS0 = _fp32(mm(Qp.T, dOc) + np.exp(Gl)[:, None] * dS1 - mm(Mp.T, dS1))
            dBV = mm(Zm.T, dOc) + mm(Pp.T, dS1)
            dQp, dZ = mm(dOc, S0.T), mm(dOc, BV.T)
            dPp, dMp = mm(dS1, BV.T), -mm(dS1, S0.T)
            dGl = np.exp(Gl) * np.sum(S0 * dS1, axis=1)
            dKend = mm(W, dMp.T) + mm(A, dPp.T)
            dW = mm(Kend, dMp) - mm(Aqk.T, dQp)
            BK = B[:, None] * KG
            dA = mm(Kend, dPp) + mm(Aqk.T, dZ) + mm(dW, BK.T)
            dAqk = low0 * (-mm(dQp, W.T) + mm(dZ, A.T))
            dBK = mm(A.T, dW)
            dKG = B[:, None] * dBK
            dB = np.sum(KG * dBK, axis=1) + np.sum(V * dBV, axis=1)
            dR = low * (-mm(mm(A.T, dA), A.T))
            dB += np.sum(dR * KK, axis=1)
            wR = (B[:, None] * dR)[:, :, None] * Dx
            dK = np.einsum("ijc,jc->ic", wR, K) + np.einsum("ijc,ic->jc", wR, K)
            tR = wR * K[:, None, :] * K[None, :, :]
            dG = tR.sum(axis=1) - tR.sum(axis=0)
            wQ = (s * dAqk)[:, :, None] * Dx
            dQ = np.einsum("ijc,jc->ic", wQ, K)
            dK += np.einsum("ijc,ic->jc", wQ, Q)
            tQ = wQ * Q[:, None, :] * K[None, :, :]
            dG += tQ.sum(axis=1) - tQ.sum(axis=0)
            dK += np.exp(G) * dKG
            dG += KG * dKG
            dQ += s * np.exp(G) * dQp
            dG += s * np.exp(G) * Q * dQp
            dK += np.exp(Gl - G) * dKend
            dG -= Kend * dKend
            dGl += np.sum(Kend * dKend, axis=0)
            dG[-1] += dGl
            gg[c0:c1, h] = np.cumsum(dG[::-1], axis=0)[::-1]
            gq[c0:c1, h], gk[c0:c1, h], gv[c0:c1, h], gb[c0:c1, h] = dQ, dK, B[:, None] * dBV, dB
            dS1 = dS0
    return gq, gk, gv, gg, gb


@pytest.fixture(scope="module")
def case():
    from oracle.backward import recurrent_backward
    w = inputs.prefill(7, [256], H=1, d=128, dtype="bf16")
    rng = np.random.default_rng(9)
    base = rng.standard_normal(w.q.shape).astype(np.float32)
    out = {}
    for scale in (1.0, 1e-6):
        dO = inputs.bf16_round(base * np.float32(scale)).astype(np.float64)
        ref = recurrent_backward(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, None, None, dO,
                                 None)[:5]
        out[scale] = (w, dO, ref)
    return out


def _errors(case, scale, rnd):
    w, dO, ref = case[scale]
    got = _emulated_chunk_backward(w, dO, rnd)
    return [nerr(a, r) for a, r in zip(got, ref)]


def test_exact_products_reproduce_the_recurrent_gradients(case):
    assert max(_errors(case, 1.0, lambda x: np.asarray(x, np.float64))) < 1e-5


@pytest.mark.parametrize("scale", [1.0, 1e-6])
def test_tf32_operands_keep_the_bound_at_any_gradient_scale(case, scale):
    assert max(_errors(case, scale, _tf32)) < 0.25 * TOL_BF16


def test_f16_operands_fail_for_small_gradients(case):
    assert max(_errors(case, 1.0, _f16)) < 0.25 * TOL_BF16
    assert max(_errors(case, 1e-6, _f16)) > TOL_BF16


def test_bf16_operands_cost_several_times_tf32(case):
    assert max(_errors(case, 1.0, _bf16)) > 4 * max(_errors(case, 1.0, _tf32))


# ---------------------------------------------------------------------------
# the planned kernels, tile by tile
# ---------------------------------------------------------------------------

C, MID, SPAN = 64, 32, 80.0


def _mm(a, b, kind):
    r = _tf32 if kind == "tf32" else _f16
    return _fp32(r(a) @ r(b))


def _chunk_forward(K, Q, V, B, g, L, s):
    """One zero-padded chunk's forward factors, as the forward prep forms them."""
    G = np.cumsum(g, axis=0)
    Gm, Gl = G[MID], G[-1]
    fast = np.max(np.abs(G - Gm)) <= SPAN
    low, low0 = np.tril(np.ones((C, C)), -1), np.tril(np.ones((C, C)))
    valid = (np.arange(C) < L).astype(np.float64)[:, None]
    Ep, Em = np.exp(G - Gm), np.exp(Gm - G)
    Kt, Qt, Kh = Ep * K, Ep * Q, Em * K
    if fast:
        P = _mm(np.vstack([Kt, Qt]), Kh.T, "tf32")
        KK, QK = P[:C], P[C:]
    else:
        Dx = np.exp(G[:, None, :] - G[None, :, :])
        KK = np.einsum("ic,jc,ijc->ij", K, K, Dx)
        QK = np.einsum("ic,jc,ijc->ij", Q, K, Dx)
    R = low * valid * (B[:, None] * KK)
    Aqk = low0 * valid * (s * QK)
    A = _fp32(np.linalg.inv(np.eye(C) + R))
    KG = np.exp(G) * K
    W = _mm(A, B[:, None] * KG, "f16")
    Kend = np.exp(Gl - G) * K
    QG = s * np.exp(G) * Q
    return dict(G=G, Gl=Gl, Ep=Ep, Em=Em, Kt=Kt, Qt=Qt, Kh=Kh, fast=fast, KK=KK, A=A,
                Aqk=Aqk, KG=KG, W=W, Kend=Kend, QG=QG, low=low * valid, low0=low0 * valid,
                Mp=_mm(Kend.T, W, "f16"), Pp=_mm(Kend.T, A, "f16"),
                Qp=_fp32(QG - _mm(Aqk, W, "f16")), Zm=_mm(Aqk, A, "f16"))


def _grad_pass(f, K, Q, V, B, dO, S0, dS1, L, s):
    """One chunk's gradients from S_c (S0) and dS_{c+1} (dS1), tf32 products."""
    t = "tf32"
    BV = B[:, None] * V
    dBV = _mm(f["Zm"].T, dO, t) + _mm(f["Pp"].T, dS1, t)
    dQp, dZ = _mm(dO, S0.T, t), _mm(dO, BV.T, t)
    dPp, dMp = _mm(dS1, BV.T, t), -_mm(dS1, S0.T, t)
    dGl = np.exp(f["Gl"]) * np.sum(S0 * dS1, axis=1)
    U = _mm(f["A"], BV, t)
    dKend = _mm(f["W"], dMp.T, t) + _mm(U, dS1.T, t)
    dW = _mm(f["Kend"], dMp, t) - _mm(f["Aqk"].T, dQp, t)
    BK = B[:, None] * f["KG"]
    dA = _mm(f["Kend"], dPp, t) + _mm(f["Aqk"].T, dZ, t) + _mm(dW, BK.T, t)
    dAqk = f["low0"] * (-_mm(dQp, f["W"].T, t) + _mm(dZ, f["A"].T, t))
    dBK = _mm(f["A"].T, dW, t)
    dR = f["low"] * (-_mm(_mm(f["A"].T, dA, t), f["A"].T, t))
    dKG = B[:, None] * dBK
    dB = np.sum(f["KG"] * dBK, axis=1) + np.sum(V * dBV, axis=1)
    G, Ep, Em = f["G"], f["Ep"], f["Em"]
    if f["fast"]:
        rows = _mm(np.vstack([dR, s * dAqk]), f["Kh"], t)
        Rrow0, Arow = rows[:C], rows[C:]
        Ccol = _mm(np.hstack([(B[:, None] * dR).T, (s * dAqk).T]),
                   np.vstack([f["Kt"], f["Qt"]]), t)
        Rrow = B[:, None] * Rrow0
        dK = Ep * Rrow + Em * Ccol
        dQ = Ep * Arow
        dG = K * Ep * Rrow + Q * Ep * Arow - K * Em * Ccol
        dB += np.sum(K * Ep * Rrow0, axis=1)
    else:
        Dx = np.exp(G[:, None, :] - G[None, :, :])
        wR = (B[:, None] * dR)[:, :, None] * Dx
        wQ = (s * dAqk)[:, :, None] * Dx
        dK = (np.einsum("ijc,jc->ic", wR, K) + np.einsum("ijc,ic->jc", wR, K)
              + np.einsum("ijc,ic->jc", wQ, Q))
        dQ = np.einsum("ijc,jc->ic", wQ, K)
        tR, tQ = wR * K[:, None, :] * K[None, :, :], wQ * Q[:, None, :] * K[None, :, :]
        dG = tR.sum(axis=1) - tR.sum(axis=0) + tQ.sum(axis=1) - tQ.sum(axis=0)
        dB += np.sum(dR * f["KK"], axis=1)
    dK += np.exp(G) * dKG + np.exp(f["Gl"] - G) * dKend
    dQ += s * np.exp(G) * dQp
    dG += f["KG"] * dKG + f["QG"] * dQp - f["Kend"] * dKend
    dG[L - 1] += dGl + np.sum(f["Kend"] * dKend, axis=0)
    dG[L:] = 0.0
    dla = np.cumsum(dG[::-1], axis=0)[::-1]
    return dQ[:L], dK[:L], (B[:, None] * dBV)[:L], dla[:L], dB[:L]


def _planned_backward(w, dO, dSf):
    q, k, v, g, b = (np.asarray(x, np.float64) for x in (w.q, w.k, w.v, w.log_alpha, w.beta))
    T, H, d = q.shape
    cu = np.asarray(w.cu_seqlens, dtype=np.int64)
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(g),
           np.zeros_like(b)]
    dS_init = np.zeros((len(cu) - 1, H, d, d))
    for n in range(len(cu) - 1):
        for h in range(H):
            S = (np.zeros((d, d)) if w.initial_state is None
                 else np.asarray(w.initial_state[n, h], np.float64))
            chunks = []
            for c0 in range(int(cu[n]), int(cu[n + 1]), C):
                L = min(C, int(cu[n + 1]) - c0)
                pad = lambda a: np.concatenate([a[c0:c0 + L, h],
                                                np.zeros((C - L,) + a.shape[2:])])
                K, Q, V, B = pad(k), pad(q), pad(v), pad(b)
                f = _chunk_forward(K, Q, V, B, pad(g), L, w.scale)
                chunks.append((c0, L, K, Q, V, B, f, S.copy()))
                S = _fp32(np.exp(f["Gl"])[:, None] * S + _mm(f["Pp"], B[:, None] * V, "f16")
                          - _mm(f["Mp"], S, "f16"))
            dS = np.asarray(dSf[n, h], np.float64).copy()
            for c0, L, K, Q, V, B, f, S0 in reversed(chunks):
                dOc = np.concatenate([dO[c0:c0 + L, h], np.zeros((C - L, d))])
                res = _grad_pass(f, K, Q, V, B, dOc, _f16(S0), dS, L, w.scale)
                for o, r in zip(out, res):
                    o[c0:c0 + L, h] = r
                X = _mm(f["Qp"].T, dOc, "tf32")
                dS = _fp32(np.exp(f["Gl"])[:, None] * dS - _mm(f["Mp"].T, dS, "tf32") + X)
            dS_init[n, h] = dS
    return out + [dS_init]


def _strong_decay(w, seed):
    """Log-decays down to -6 per token over the first 100 tokens: chunks whose
    cumulative decay spans more than 80 take the direct-exponent path."""
    rng = np.random.default_rng(seed)
    la = w.log_alpha.copy()
    la[:100] = -rng.uniform(0, 6, size=la[:100].shape).astype(np.float32)
    w.log_alpha = la
    return w


@pytest.mark.parametrize("name,make,gscale", [
    ("one sequence", lambda: inputs.prefill(11, [384], H=1, d=128, dtype="bf16"), 1.0),
    ("packed ragged, initial states",
     lambda: inputs.prefill(12, [1, 63, 64, 65, 130], H=1, d=128, dtype="bf16", init_std=0.02),
     1.0),
    ("direct-exponent chunks",
     lambda: _strong_decay(inputs.prefill(15, [200], H=1, d=128, dtype="bf16"), 5), 1.0),
    ("small gradients", lambda: inputs.prefill(14, [200], H=1, d=128, dtype="bf16"), 1e-6),
])
def test_planned_decomposition_keeps_the_bound(name, make, gscale):
    from oracle.backward import recurrent_backward
    w = make()
    rng = np.random.default_rng(3)
    dO = inputs.bf16_round(rng.standard_normal(w.q.shape).astype(np.float32)
                           * np.float32(gscale)).astype(np.float64)
    dSf = rng.standard_normal((len(w.cu_seqlens) - 1, w.H, 128, 128)) * 0.1 * gscale
    ref = recurrent_backward(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, w.initial_state,
                             w.cu_seqlens, dO, dSf)
    got = _planned_backward(w, dO, dSf)
    errs = [nerr(a, r) for a, r in zip(got, ref)]
    assert max(errs) < 0.6 * TOL_BF16, (name, errs)
