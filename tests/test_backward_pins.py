"""Pins for the gradient oracle: central finite differences of the
independent forward oracle (the C token recurrence), entry by entry, on
small packed problems; and the gradient of a linear read, which has a closed
form."""
import numpy as np
import pytest

import oracle
from oracle.backward import recurrent_backward


def _problem(seed, lengths, H, dk, dv):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.05, 0.8, (T, H, dk))
    b = rng.uniform(0.1, 0.9, (T, H))
    S0 = rng.standard_normal((len(lengths), H, dk, dv)) * 0.3
    R = rng.standard_normal((T, H, dv))            # loss weights on the outputs
    Q = rng.standard_normal((len(lengths), H, dk, dv))  # ... and on the final states
    return dict(q=q, k=k, v=v, g=g, b=b, S0=S0, cu=cu, R=R, Q=Q, s=dk ** -0.5)


def _loss(P, **over):
    x = dict(P, **over)
    o, f = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["b"], x["s"], x["S0"], x["cu"])
    return float(np.sum(o * x["R"]) + np.sum(f * x["Q"]))


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "b", "S0"])
def test_finite_differences(name):
    P = _problem(10, [4, 1, 3], H=2, dk=3, dv=2)
    grads = dict(zip(["q", "k", "v", "g", "b", "S0"],
                     recurrent_backward(P["q"], P["k"], P["v"], P["g"], P["b"], P["s"], P["S0"],
                                        P["cu"], P["R"], P["Q"])))
    x = P[name]
    eps = 1e-6
    fd = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        fd[idx] = (_loss(P, **{name: xp}) - _loss(P, **{name: xm})) / (2 * eps)
    np.testing.assert_allclose(grads[name], fd, rtol=1e-6, atol=1e-8)


def test_read_gradient_closed_form():
    """With beta = 0 nothing is written and alpha = 1 forgets nothing: o_t =
    S0^T (s q_t), so dq_t = s S0 do_t and dS0 = s sum_t q_t do_t^T."""
    rng = np.random.default_rng(3)
    T, dk, dv = 5, 4, 3
    q, k, v = rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dk, dv))
    dO = rng.standard_normal((T, 1, dv))
    s = 0.7
    dq, dk_, dvv, dg, db, dS0 = recurrent_backward(q, k, v, np.zeros((T, 1, dk)), np.zeros((T, 1)),
                                                   s, S0, None, dO, None)
    np.testing.assert_allclose(dq[:, 0], s * dO[:, 0] @ S0[0, 0].T, rtol=1e-13)
    np.testing.assert_allclose(dS0[0, 0], s * q[:, 0].T @ dO[:, 0], rtol=1e-13)
    assert not dvv.any()


@pytest.mark.parametrize("folded", [False, True])
@pytest.mark.parametrize("chunk_size", [1, 3, 16, 64])
def test_chunkwise_backward_equals_recurrent(chunk_size, folded):
    """The chunkwise backward (sec. 6's chunk form differentiated, the
    blueprint of a chunk-parallel backward), directly or through the folded
    per-chunk factors M', P', Q', Z the forward engine stores, gives the
    recurrent backward's gradients to rounding, for any chunk size, across
    packed sequences with empty and one-token ones, partial last chunks and
    strong decays."""
    from oracle.backward import chunk_backward, folded_chunk_backward
    P = _problem(20, [37, 0, 1, 70, 16], H=2, dk=8, dv=8)
    P["g"][40:50] -= 6.0   # near-total forgetting inside a chunk
    args = (P["q"], P["k"], P["v"], P["g"], P["b"], P["s"], P["S0"], P["cu"], P["R"], P["Q"])
    ref = recurrent_backward(*args)
    got = (folded_chunk_backward if folded else chunk_backward)(*args, chunk_size=chunk_size)
    for name, x, r in zip(("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial"), got, ref):
        np.testing.assert_allclose(x, r, rtol=0, atol=1e-11 * max(np.abs(r).max(), 1.0),
                                   err_msg=name)


def test_chunkwise_backward_finite_differences():
    """An independent check of the chunk form on its own: central finite
    differences of the C forward oracle for log_alpha and beta (the inputs
    that reach the most factors of the chunk form)."""
    from oracle.backward import chunk_backward
    P = _problem(21, [6, 5], H=1, dk=3, dv=2)
    grads = chunk_backward(P["q"], P["k"], P["v"], P["g"], P["b"], P["s"], P["S0"], P["cu"],
                           P["R"], P["Q"], chunk_size=4)
    for name, gi in (("g", 3), ("b", 4)):
        x = P[name]
        eps = 1e-6
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fd[idx] = (_loss(P, **{name: xp}) - _loss(P, **{name: xm})) / (2 * eps)
        np.testing.assert_allclose(grads[gi], fd, rtol=1e-6, atol=1e-8, err_msg=name)
