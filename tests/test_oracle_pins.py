"""Pins for the fp64 oracle: facts the pages and the mathematics fix.

None of these compares the oracle with itself.  Each check is one of: a
worked example printed on a page (fixtures under tests/golden/, each citing
its page and section), a closed form, an identity a page derives, a reduction
to DeltaNet / Gated DeltaNet written independently here in matrix form, or
brute-force agreement of the chunkwise derivation with the token recurrence.

The last test plants plausible mistakes in a copy of the oracle source
(dropped decay, dropped beta, wrong sign, transposed read, read before write,
missing scale, column instead of row decay, chunk-algebra slips) and checks
that every one of them breaks at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _one(x):
    """[d] -> [1, 1, d] (one token, one head)."""
    return np.asarray(x, dtype=np.float64).reshape(1, 1, -1)


def _rng_inputs(rng, T, H, dk, dv, gate_lo=0.0, gate_hi=0.7):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(gate_lo, gate_hi, size=(T, H, dk))
    b = rng.uniform(0.05, 1.0, size=(T, H))
    return q, k, v, g, b


# ---------------------------------------------------------------------------
# Pins.  Each takes an object with .recurrent / .chunkwise (the oracle or a
# deliberately broken copy of it) and raises AssertionError on disagreement.
# ---------------------------------------------------------------------------

def pin_channel_decay(O):
    """Kimi Delta Attention: Channel-Wise Memory Control, 'What a channel-wise
    decay actually scales': S = I with retention (1, 0.25) -> diag(1, 0.25)."""
    gd = _golden("channel_decay.json")
    s0 = np.asarray(gd["initial_state"]).reshape(1, 1, 2, 2)
    la = _one(np.log(gd["retention"]))
    k, v, b = _one([0.6, 0.8]), _one([5.0, -7.0]), np.zeros((1, 1))
    for qv, want in (([1.0, 0.0], gd["read_e1"]), ([0.0, 1.0], gd["read_e2"])):
        out, fin = O.recurrent(_one(qv), k, v, la, b, 1.0, s0)
        np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)
        np.testing.assert_allclose(fin[0, 0], gd["decayed_state"], rtol=0, atol=1e-15)


def pin_noncommuting(O):
    """Same page, 'The two transformations usually do not commute': one step
    from S = I with k = (1,1)/sqrt2, beta = 1, D = diag(1, 0.5), v = 0 gives the
    transition (I - k k^T) D, not D (I - k k^T)."""
    gd = _golden("noncommuting.json")
    s0 = np.eye(2).reshape(1, 1, 2, 2)
    _, fin = O.recurrent(_one([0.3, -0.2]), _one(gd["k"]), _one([0.0, 0.0]),
                         _one(np.log(gd["retention"])), np.full((1, 1), gd["beta"]),
                         1.0, s0)
    np.testing.assert_allclose(fin[0, 0], gd["I_minus_kkT_times_D"], rtol=0, atol=1e-15)
    assert np.abs(fin[0, 0] - np.asarray(gd["D_times_I_minus_kkT"])).max() > 0.2


def pin_deltanet_overwrite(O):
    """Linear Attention, From Scratch to Kimi 3, sec. 4: the memory maps
    [1,0] -> [3,4]; writing [9,2] with beta = 1 makes the read return [9,2]."""
    gd = _golden("deltanet_overwrite.json")
    key = np.asarray(gd["key"])
    s0 = np.outer(key, gd["old_value"]).reshape(1, 1, 2, 2)
    zero_gate = _one([0.0, 0.0])
    # before the write (beta = 0) the memory returns the old value
    out0, _ = O.recurrent(_one(key), _one(key), _one(gd["new_value"]), zero_gate,
                          np.zeros((1, 1)), 1.0, s0)
    np.testing.assert_allclose(out0[0, 0], gd["old_value"], rtol=0, atol=1e-15)
    out, _ = O.recurrent(_one(key), _one(key), _one(gd["new_value"]), zero_gate,
                         np.full((1, 1), gd["beta"]), 1.0, s0)
    np.testing.assert_allclose(out[0, 0], gd["read_after_write"], rtol=0, atol=1e-15)


def pin_readback_interpolation(O):
    """Kimi Unveils Delta Attention and K3 Architecture Updates, sec. 2.1 (and
    the KDA form of sec. 4): for a unit key, S_t^T k = (1 - beta) S_bar^T k + beta v."""
    rng = np.random.default_rng(11)
    dk, dv = 5, 3
    for _ in range(4):
        s0 = rng.standard_normal((1, 1, dk, dv))
        k = rng.standard_normal(dk)
        k /= np.linalg.norm(k)
        v = rng.standard_normal(dv)
        g = -rng.uniform(0, 1.5, size=dk)
        beta = rng.uniform(0.1, 0.9)
        args = (_one(k), _one(k), _one(v), _one(g))
        read_bar, _ = O.recurrent(*args, np.zeros((1, 1)), 1.0, s0)
        read_t, _ = O.recurrent(*args, np.full((1, 1), beta), 1.0, s0)
        np.testing.assert_allclose(read_t[0, 0], (1 - beta) * read_bar[0, 0] + beta * v,
                                   rtol=0, atol=1e-12)


def pin_orthogonal_locality(O):
    """Same page, sec. 2.1: a query orthogonal to the written key sees no change
    from the write, (S_t - S_bar_t)^T x = 0."""
    rng = np.random.default_rng(12)
    dk, dv = 6, 4
    for _ in range(4):
        s0 = rng.standard_normal((1, 1, dk, dv))
        k = rng.standard_normal(dk)
        x = rng.standard_normal(dk)
        x -= (x @ k) / (k @ k) * k
        v = rng.standard_normal(dv)
        g = -rng.uniform(0, 1.0, size=dk)
        a, _ = O.recurrent(_one(x), _one(k), _one(v), _one(g), np.zeros((1, 1)), 0.7, s0)
        b, _ = O.recurrent(_one(x), _one(k), _one(v), _one(g), np.full((1, 1), 0.8), 0.7, s0)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def _matrix_form(q, k, v, g, b, scale, s0):
    """Kimi Delta Attention: Channel-Wise Memory Control, 'Where
    diagonal-plus-low-rank structure appears': S_t = A_t S_{t-1} + B_t with
    A_t = D_t - beta_t k_t (k_t^T D_t), B_t = beta_t k_t v_t^T, o_t = S_t^T (s q_t).
    Written with explicit d_k x d_k matrices, one head."""
    S = s0.copy()
    outs = []
    for t in range(q.shape[0]):
        D = np.diag(np.exp(g[t]))
        A = D - b[t] * np.outer(k[t], k[t] @ D)
        B = b[t] * np.outer(k[t], v[t])
        S = A @ S + B
        outs.append(S.T @ (scale * q[t]))
    return np.array(outs), S


def pin_expanded_form(O):
    """Same page: the expanded form A_t S_{t-1} + B_t equals the update form,
    one step and over a sequence (the lab check the page describes)."""
    rng = np.random.default_rng(13)
    for T in (1, 9):
        dk, dv = 4, 3
        q, k, v, g, b = _rng_inputs(rng, T, 1, dk, dv, 0.0, 1.2)
        s0 = rng.standard_normal((1, 1, dk, dv))
        out, fin = O.recurrent(q, k, v, g, b, 0.37, s0)
        ref_o, ref_s = _matrix_form(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], 0.37, s0[0, 0])
        np.testing.assert_allclose(out[:, 0], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(fin[0, 0], ref_s, rtol=0, atol=1e-12)


def pin_gated_deltanet(O):
    """Kimi Unveils Delta Attention ..., sec. 3, and Channel-Wise Memory Control
    ('For equal retention factors, this reduces to the scalar-gated update'):
    with alpha equal across channels, S_t = alpha_t (I - beta_t k k^T) S + beta_t k v^T."""
    rng = np.random.default_rng(14)
    T, dk, dv = 11, 5, 4
    q, k, v, _, b = _rng_inputs(rng, T, 1, dk, dv)
    a = rng.uniform(0.3, 1.0, size=T)
    g = np.repeat(np.log(a)[:, None, None], dk, axis=2)
    s0 = rng.standard_normal((1, 1, dk, dv))
    out, fin = O.recurrent(q, k, v, g, b, 0.5, s0)
    S = s0[0, 0].copy()
    for t in range(T):
        kt = k[t, 0]
        S = a[t] * (np.eye(dk) - b[t, 0] * np.outer(kt, kt)) @ S + b[t, 0] * np.outer(kt, v[t, 0])
        np.testing.assert_allclose(out[t, 0], S.T @ (0.5 * q[t, 0]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], S, rtol=0, atol=1e-12)


def pin_deltanet(O):
    """Kimi Unveils Delta Attention ..., sec. 2.3, and Channel-Wise Memory Control
    ('With all factors one, it reduces to DeltaNet'): S_t = S + beta k (v - S^T k)^T."""
    rng = np.random.default_rng(15)
    T, dk, dv = 10, 4, 6
    q, k, v, _, b = _rng_inputs(rng, T, 1, dk, dv)
    g = np.zeros((T, 1, dk))
    s0 = rng.standard_normal((1, 1, dk, dv))
    out, fin = O.recurrent(q, k, v, g, b, 1.0, s0)
    S = s0[0, 0].copy()
    for t in range(T):
        kt = k[t, 0]
        S = S + b[t, 0] * np.outer(kt, v[t, 0] - S.T @ kt)
        np.testing.assert_allclose(out[t, 0], S.T @ q[t, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], S, rtol=0, atol=1e-12)


def pin_half_life(O):
    """thethings.ai Kimi Delta Attention page: a retention of 0.99 halves the
    memory every 69 tokens (ln 2 / -ln 0.99 = 68.97)."""
    gd = _golden("half_life.json")
    n = gd["half_life_tokens"]
    la = math.log(gd["alpha"])
    s0 = np.eye(2).reshape(1, 1, 2, 2)
    T = n
    z = np.zeros((T, 1, 2))
    _, fin = O.recurrent(z, z, z, np.full((T, 1, 2), la), np.zeros((T, 1)), 1.0, s0)
    ratio = fin[0, 0, 0, 0]
    assert abs(ratio - gd["alpha"] ** n) < 1e-13
    assert abs(ratio - 0.5) < 1e-3
    _, fin_before = O.recurrent(z[:-1], z[:-1], z[:-1], np.full((T - 1, 1, 2), la),
                                np.zeros((T - 1, 1)), 1.0, s0)
    assert fin_before[0, 0, 0, 0] > 0.5 > ratio


def pin_chunkwise_equals_recurrent(O):
    """Kimi Unveils Delta Attention ..., sec. 6: the chunkwise schedule must give
    exactly the states and outputs of the token recurrence.  Brute force on
    packed ragged sequences (a length-1 sequence, partial chunks), nonzero
    initial states, and gates from mild down to -80 per token."""
    rng = np.random.default_rng(16)
    cu = np.array([0, 1, 6, 23, 40], dtype=np.int32)
    T, H, dk, dv = 40, 2, 6, 5
    for lo, hi in ((0.0, 0.6), (0.0, 80.0)):
        q, k, v, g, b = _rng_inputs(rng, T, H, dk, dv, lo, hi)
        s0 = rng.standard_normal((4, H, dk, dv))
        ref_o, ref_s = O.recurrent(q, k, v, g, b, 0.45, s0, cu)
        for C in (1, 2, 4, 16):
            out, fin = O.chunkwise(q, k, v, g, b, 0.45, C, s0, cu)
            np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-10)
            np.testing.assert_allclose(fin, ref_s, rtol=0, atol=1e-10)


def pin_four_token_chunk(O):
    """Kimi Unveils Delta Attention ..., sec. 6.1-6.5 written out for one
    four-token chunk with explicit diagonal decay products D_{j+1:i}: provisional
    errors, e_0..e_3 by the causal substitutions, the fast-forwarded state and
    the four outputs (d_k x d_v layout, i.e. the page's expressions transposed)."""
    rng = np.random.default_rng(17)
    dk, dv, s = 5, 4, 0.6
    q, k, v, g, b = _rng_inputs(rng, 4, 1, dk, dv, 0.0, 1.0)
    q, k, v, g, b = q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0]
    Sc = rng.standard_normal((dk, dv))
    Dm = [np.diag(np.exp(g[i])) for i in range(4)]

    def prod(j0, i):  # D_{j0} D_{j0+1} ... D_i (identity when j0 > i)
        P = np.eye(dk)
        for r in range(j0, i + 1):
            P = P @ Dm[r]
        return P

    ebar = [b[i] * (v[i] - Sc.T @ (prod(0, i) @ k[i])) for i in range(4)]
    rho = lambda i, j: b[i] * (k[j] @ prod(j + 1, i) @ k[i])
    e0 = ebar[0]
    e1 = ebar[1] - rho(1, 0) * e0
    e2 = ebar[2] - rho(2, 0) * e0 - rho(2, 1) * e1
    e3 = ebar[3] - rho(3, 0) * e0 - rho(3, 1) * e1 - rho(3, 2) * e2
    E = [e0, e1, e2, e3]
    S_next = prod(0, 3) @ Sc + sum(np.outer(prod(i + 1, 3) @ k[i], E[i]) for i in range(4))
    chi = lambda i, j: s * (k[j] @ prod(j + 1, i) @ q[i])
    outs = [s * Sc.T @ (prod(0, i) @ q[i]) + sum(chi(i, j) * E[j] for j in range(i + 1))
            for i in range(4)]
    args = (q[:, None], k[:, None], v[:, None], g[:, None], b[:, None], s, Sc[None, None])
    for o, fin in (O.chunkwise(*args[:6], 4, args[6]), O.recurrent(*args)):
        np.testing.assert_allclose(o[:, 0], np.array(outs), rtol=0, atol=1e-12)
        np.testing.assert_allclose(fin[0, 0], S_next, rtol=0, atol=1e-12)


def pin_packed_equals_separate(O):
    """Linear Attention, From Scratch to Kimi 3, sec. 9: cu_seqlens [0, 3, 8, 10]
    packs three requests whose states never cross a boundary."""
    cu = np.asarray(_golden("cu_seqlens.json")["cu_seqlens"], dtype=np.int32)
    rng = np.random.default_rng(18)
    T, H, dk, dv = int(cu[-1]), 2, 4, 3
    q, k, v, g, b = _rng_inputs(rng, T, H, dk, dv)
    s0 = rng.standard_normal((3, H, dk, dv))
    out, fin = O.recurrent(q, k, v, g, b, 0.5, s0, cu)
    for n in range(3):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = O.recurrent(q[sl], k[sl], v[sl], g[sl], b[sl], 0.5, s0[n:n + 1])
        np.testing.assert_allclose(out[sl], o1, rtol=0, atol=0)
        np.testing.assert_allclose(fin[n], f1[0], rtol=0, atol=0)


PINS = [pin_channel_decay, pin_noncommuting, pin_deltanet_overwrite,
        pin_readback_interpolation, pin_orthogonal_locality, pin_expanded_form,
        pin_gated_deltanet, pin_deltanet, pin_half_life,
        pin_chunkwise_equals_recurrent, pin_four_token_chunk,
        pin_packed_equals_separate]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod)


def test_empty_sequences_keep_state(oracle_mod):
    """Zero-length packed sequences return their initial state untouched."""
    rng = np.random.default_rng(19)
    cu = np.array([0, 0, 3, 3], dtype=np.int32)
    q, k, v, g, b = _rng_inputs(rng, 3, 1, 3, 2)
    s0 = rng.standard_normal((3, 1, 3, 2))
    for fn in (lambda: oracle_mod.recurrent(q, k, v, g, b, 1.0, s0, cu),
               lambda: oracle_mod.chunkwise(q, k, v, g, b, 1.0, 2, s0, cu)):
        _, fin = fn()
        np.testing.assert_array_equal(fin[0], s0[0])
        np.testing.assert_array_equal(fin[2], s0[2])


def test_oracle_rejects_bad_cu_seqlens(oracle_mod):
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle_mod.recurrent(q, q, q, q, np.zeros((4, 1)), 1.0, None, [0, 3, 2, 4])
    with pytest.raises(ValueError):
        oracle_mod.recurrent(q, q, q, q, np.zeros((4, 1)), 1.0, None, [0, 3])


# ---------------------------------------------------------------------------
# Planted mistakes: each edit of the oracle source must break some pin.
# ---------------------------------------------------------------------------

_WRITE = """        /* write: S_t = S_bar + k e^T */
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] += k[i] * p[j];
"""
_READ = """        /* read after the write: o_t = S_t^T (scale q_t) */
        for (int32_t j = 0; j < dv; ++j) o[j] = 0.0;
        for (int32_t i = 0; i < dk; ++i) {
            const double sq = J->scale * q[i];
            for (int32_t j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * sq;
        }
"""

MUTANTS = {
    "decay_dropped": [("const double a = exp(g[i]);", "const double a = 1.0;")],
    "decay_columns": [(
        "            const double a = exp(g[i]);\n"
        "            for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;",
        "            for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= exp(g[j < dk ? j : 0]);")],
    "beta_dropped": [("p[j] = beta * (v[j] - p[j]);", "p[j] = (v[j] - p[j]);")],
    "error_sign": [("p[j] = beta * (v[j] - p[j]);", "p[j] = beta * (p[j] - v[j]);")],
    "predict_transposed": [("p[j] += S[(size_t)i * dv + j] * k[i];",
                            "p[j] += S[(size_t)(j < dk ? j : 0) * dv + (i < dv ? i : 0)] * k[i];")],
    "scale_dropped": [("const double sq = J->scale * q[i];", "const double sq = q[i];")],
    "read_before_write": [(_WRITE + _READ, _READ + _WRITE)],
    "chunk_rho_sign": [("E[(size_t)i * dv + m] -= rho * E[(size_t)j * dv + m];",
                        "E[(size_t)i * dv + m] += rho * E[(size_t)j * dv + m];")],
    "chunk_diagonal_read_dropped": [("for (int32_t j = 0; j <= i; ++j) {",
                                     "for (int32_t j = 0; j < i; ++j) {")],
    "chunk_provisional_decay_dropped": [(
        "x[d] = exp(G[(size_t)i * dk + d]) * K_(c0 + i)[d];", "x[d] = K_(c0 + i)[d];")],
    "chunk_end_decay_dropped": [(
        "const double kend = exp(Gl[d] - G[(size_t)i * dk + d]) * K_(c0 + i)[d];",
        "const double kend = K_(c0 + i)[d];")],
    "chunk_cumsum_off_by_one": [(
        "(i ? G[(size_t)(i - 1) * dk + d] : 0.0) + G_(c0 + i)[d];",
        "(i ? G[(size_t)(i - 1) * dk + d] + G_(c0 + i - 1)[d] : 0.0);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, name):
    src = oracle_mod.source_text()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation {name} no longer matches the oracle source"
        src = src.replace(old, new)
    broken = oracle_mod.build_variant(src, name)
    caught = []
    for pin in PINS:
        try:
            pin(broken)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
