"""Pins for the short-convolution oracle: closed forms and identities the
definition fixes (impulse response, step response, a hand-worked example
with a cache, sequence boundaries, the decode step against prefill, SiLU)."""
import numpy as np

from oracle.short_conv import short_conv, short_conv_step


def test_impulse_response_is_the_reversed_filter():
    W, C = 4, 3
    w = np.arange(1.0, 1.0 + C * W).reshape(C, W)
    x = np.zeros((9, C))
    x[2] = 1.0
    y, _ = short_conv(x, w)
    for m in range(W):
        np.testing.assert_array_equal(y[2 + m], w[:, W - 1 - m])
    assert not y[:2].any() and not y[2 + W:].any()


def test_step_response_sums_the_taps():
    W = 4
    w = np.array([[0.5, -1.0, 2.0, 3.0]])
    y, _ = short_conv(np.ones((7, 1)), w)
    # token t sees min(t + 1, W) ones at the newest taps
    expect = [w[0, W - 1 - t:].sum() if t < W else w[0].sum() for t in range(7)]
    np.testing.assert_allclose(y[:, 0], expect)


def test_hand_worked_example_with_cache():
    # W = 4, w = [1, 2, 3, 4], cache (oldest first) [5, 6, 7, 8], x = [1, 0, 2]:
    #   y0 = 1*6 + 2*7 + 3*8 + 4*1 = 48
    #   y1 = 1*7 + 2*8 + 3*1 + 4*0 = 26
    #   y2 = 1*8 + 2*1 + 3*0 + 4*2 = 18,  cache after: [8, 1, 0, 2]
    y, c = short_conv(np.array([[1.0], [0.0], [2.0]]), np.array([[1.0, 2.0, 3.0, 4.0]]),
                      cache=np.array([[[5.0, 6.0, 7.0, 8.0]]]))
    np.testing.assert_array_equal(y[:, 0], [48.0, 26.0, 18.0])
    np.testing.assert_array_equal(c[0, 0], [8.0, 1.0, 0.0, 2.0])


def test_sequences_do_not_see_each_other():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((11, 5))
    w = rng.standard_normal((5, 4))
    cache = rng.standard_normal((2, 5, 4))
    y, c = short_conv(x, w, cu_seqlens=[0, 6, 11], cache=cache)
    y0, c0 = short_conv(x[:6], w, cache=cache[:1])
    y1, c1 = short_conv(x[6:], w, cache=cache[1:])
    np.testing.assert_array_equal(y, np.concatenate([y0, y1]))
    np.testing.assert_array_equal(c, np.concatenate([c0, c1]))


def test_short_sequence_keeps_part_of_its_cache():
    w = np.ones((1, 4))
    _, c = short_conv(np.array([[9.0]]), w, cache=np.array([[[1.0, 2.0, 3.0, 4.0]]]))
    np.testing.assert_array_equal(c[0, 0], [2.0, 3.0, 4.0, 9.0])


def test_decode_steps_equal_prefill():
    rng = np.random.default_rng(1)
    N, C, W, L = 3, 6, 4, 5
    x = rng.standard_normal((N, L, C))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    cache = rng.standard_normal((N, C, W))
    cu = np.arange(N + 1) * L
    y, cout = short_conv(x.reshape(N * L, C), w, b, cu, cache, silu=True)
    c = cache
    for t in range(L):
        ys, c = short_conv_step(x[:, t], w, b, c, silu=True)
        np.testing.assert_allclose(ys, y.reshape(N, L, C)[:, t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(c, cout, rtol=0, atol=0)


def test_silu_values():
    w = np.array([[0.0, 0.0, 0.0, 1.0]])
    y, _ = short_conv(np.array([[0.0], [20.0], [-20.0], [1.0]]), w, silu=True)
    assert y[0, 0] == 0.0
    assert abs(y[1, 0] - 20.0) < 1e-7
    assert abs(y[2, 0]) < 1e-7
    assert abs(y[3, 0] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
