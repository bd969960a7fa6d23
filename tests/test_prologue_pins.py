"""Pins for the prologue oracle: what the pages fix about it (a sigmoid
beta; a log retention of -5 sigmoid(.) in (-5, 0); unit-norm q and k) and
closed forms of the readings."""
import numpy as np

from oracle import prologue as P


def test_sigmoid_closed_forms():
    assert P.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(P.sigmoid(np.log(3.0)), 0.75, rtol=1e-15)
    assert P.sigmoid(-800.0) == 0.0 and P.sigmoid(800.0) == 1.0


def test_gate_range_and_midpoint():
    rng = np.random.default_rng(0)
    g = rng.standard_normal((50, 3, 8)) * 10
    la = P.k3_log_alpha(g, np.zeros((3, 8)), np.zeros(3))
    assert (la < 0).all() and (la > -5).all()
    # g + b = 0 gives sigmoid(0) = 1/2: log retention -2.5 whatever A_log is
    la0 = P.k3_log_alpha(np.zeros((1, 2, 4)), np.zeros((2, 4)), np.array([-3.0, 4.0]))
    np.testing.assert_array_equal(la0, -2.5)
    # the bias shifts g channel by channel; A_log scales inside the sigmoid
    la1 = P.k3_log_alpha(np.ones((1, 1, 2)), np.array([[-1.0, 0.0]]), np.array([np.log(2.0)]))
    np.testing.assert_allclose(la1[0, 0], [-2.5, -5.0 * P.sigmoid(2.0)], rtol=1e-15)


def test_retention_is_monotone_in_the_gate():
    g = np.linspace(-6, 6, 101).reshape(-1, 1, 1)
    la = P.k3_log_alpha(g, np.zeros((1, 1)), np.zeros(1))[:, 0, 0]
    assert (np.diff(la) < 0).all()        # a larger gate logit forgets more


def test_l2_normalisation():
    x = np.array([[[3.0, 4.0]], [[0.0, 0.0]]])
    y = P.l2_normalise(x)
    np.testing.assert_allclose(y[0, 0], [0.6, 0.8], rtol=1e-6)
    np.testing.assert_array_equal(y[1, 0], [0.0, 0.0])
    rng = np.random.default_rng(1)
    z = P.l2_normalise(rng.standard_normal((7, 3, 128)) * 5)
    np.testing.assert_allclose(np.linalg.norm(z, axis=-1), 1.0, rtol=1e-7)


def test_apply_passes_through_when_off():
    rng = np.random.default_rng(2)
    q, k, b, g = (rng.standard_normal(s) for s in ((4, 2, 8), (4, 2, 8), (4, 2), (4, 2, 8)))
    out = P.apply(q, k, b, g)
    for a, o in zip((q, k, b, g), out):
        np.testing.assert_array_equal(a, o)
