"""Parity of libkda's short causal convolution (prefill and decode step)
with the fp64 oracle: packed sequences with empty and one-token members,
every supported width, caches in and out (also in place), bias, SiLU, fp32
and bf16, and a K3-sized channel count."""
import numpy as np
import pytest

from kda_testutil import check_bf16_output, nerr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _bf16(a):
    """Round to bfloat16 values (kept as float32), nearest-even."""
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _case(seed, lengths, C, W, dtype, with_cache=True, with_bias=True):
    rng = np.random.default_rng(seed)
    T, N = int(sum(lengths)), len(lengths)
    cu = np.zeros(N + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    x = rng.standard_normal((T, C)).astype(np.float32)
    cache = rng.standard_normal((N, C, W)).astype(np.float32) if with_cache else None
    if dtype == "bf16":
        x = _bf16(x)
        cache = _bf16(cache) if cache is not None else None
    w = (rng.standard_normal((C, W)) * 0.5).astype(np.float32)
    b = rng.standard_normal(C).astype(np.float32) if with_bias else None
    return x, w, b, cu, cache


def _run(x, w, b, cu, cache, dtype, silu, in_place=False):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    to = lambda a, d=None: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", d)
    xc, cin = to(x, dt), to(cache, dt)
    N, C, W = len(cu) - 1, x.shape[1], w.shape[1]
    cout = cin if (in_place and cin is not None) else torch.empty((N, C, W), dtype=dt, device="cuda")
    y = kda.kda_short_conv_fwd(xc, to(w), to(b), to(cu), cin, cout, silu=silu)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), cout.float().cpu().numpy()


@pytest.mark.parametrize("W", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("silu", [False, True])
def test_prefill(W, dtype, silu):
    from oracle.short_conv import short_conv
    x, w, b, cu, cache = _case(800 + W, [37, 1, 0, 70, 5, 2], 64, W, dtype)
    y, cout = _run(x, w, b, cu, cache, dtype, silu)
    ry, rc = short_conv(x, w, b, cu, cache, silu)
    if dtype == "f32":
        assert nerr(y, ry) <= 1e-5
    else:
        check_bf16_output(y, ry, tol=1e-5)
    np.testing.assert_array_equal(cout, rc.astype(np.float32))   # a cache is a copy of inputs


def test_prefill_without_cache_or_bias_and_in_place():
    from oracle.short_conv import short_conv
    x, w, b, cu, cache = _case(820, [9, 30, 4], 128, 4, "f32", with_cache=False, with_bias=False)
    y, cout = _run(x, w, b, cu, None, "f32", False)
    ry, rc = short_conv(x, w, None, cu, None)
    assert nerr(y, ry) <= 1e-5
    np.testing.assert_array_equal(cout, rc.astype(np.float32))
    x, w, b, cu, cache = _case(821, [3, 17, 1], 64, 4, "bf16")
    y, cout = _run(x, w, b, cu, cache, "bf16", True, in_place=True)
    ry, rc = short_conv(x, w, b, cu, cache, True)
    check_bf16_output(y, ry, tol=1e-5)
    np.testing.assert_array_equal(cout, rc.astype(np.float32))


def test_decode_steps_continue_prefill():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from oracle.short_conv import short_conv_step
    x, w, b, cu, cache = _case(830, [5, 9, 2, 11], 256, 4, "bf16")
    _, cout = _run(x, w, b, cu, cache, "bf16", True)
    rng = np.random.default_rng(831)
    cache_dev = torch.from_numpy(cout).to("cuda", torch.bfloat16)
    ref_cache = cout.astype(np.float64)
    for step in range(6):
        xs = _bf16(rng.standard_normal((4, 256)))
        y = kda.kda_short_conv_step(torch.from_numpy(xs).to("cuda", torch.bfloat16),
                                    torch.from_numpy(w).cuda(), cache_dev,
                                    torch.from_numpy(b).cuda(), silu=True)
        ry, ref_cache = short_conv_step(xs, w, b, ref_cache, silu=True)
        torch.cuda.synchronize()
        check_bf16_output(y.float().cpu().numpy(), ry, tol=1e-5)
        np.testing.assert_array_equal(cache_dev.float().cpu().numpy(),
                                      ref_cache.astype(np.float32))


def test_k3_channel_count():
    """q/k/v width of one K3 layer: 96 heads x 128 = 12,288 channels, 4 taps."""
    from oracle.short_conv import short_conv
    x, w, b, cu, cache = _case(840, [1000, 17, 2048, 1031], 12288, 4, "bf16")
    y, cout = _run(x, w, b, cu, cache, "bf16", True)
    ry, rc = short_conv(x, w, b, cu, cache, True)
    check_bf16_output(y, ry, tol=1e-5)
    np.testing.assert_array_equal(cout, rc.astype(np.float32))
