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
