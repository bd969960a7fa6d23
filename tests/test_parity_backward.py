"""Gradients from libkda's recurrent backward against the fp64 gradient
oracle (itself pinned by finite differences): packed sequences across the
8-token checkpoint boundaries (empty and one-token ones included), every
head width, fp32 and bf16 inputs, with and without initial state and
final-state gradient, and one longer sequence."""
import numpy as np
import pytest

from kda_testutil import nerr

pytestmark = pytest.mark.gpu
TOL = 1e-4   # fp32 arithmetic against fp64, normalised by each gradient's RMS


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _bf16(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _case(seed, lengths, H, d, dtype, with_state=True):
    rng = np.random.default_rng(seed)
    T, N = int(sum(lengths)), len(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = rng.standard_normal((T, H, d)).astype(np.float32)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, d)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    do = rng.standard_normal((T, H, d)).astype(np.float32)
    if dtype == "bf16":
        q, k, v, do = _bf16(q), _bf16(k), _bf16(v), _bf16(do)
    g = (-rng.uniform(0.01, 0.6, (T, H, d))).astype(np.float32)
    b = rng.uniform(0.1, 0.9, (T, H)).astype(np.float32)
    S0 = (rng.standard_normal((N, H, d, d)) * 0.1).astype(np.float32) if with_state else None
    dSf = rng.standard_normal((N, H, d, d)).astype(np.float32) if with_state else None
    return dict(q=q, k=k, v=v, g=g, b=b, S0=S0, dSf=dSf, do=do, cu=cu, s=d ** -0.5)


def _check(c, dtype):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from oracle.backward import recurrent_backward
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    to = lambda x, d=None: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda", d)
    got = kda.kda_recurrent_bwd(to(c["q"], dt), to(c["k"], dt), to(c["v"], dt), to(c["g"]),
                                to(c["b"]), c["s"], to(c["S0"]), to(c["cu"]), to(c["do"], dt),
                                to(c["dSf"]))
    torch.cuda.synchronize()
    ref = recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["b"], c["s"], c["S0"], c["cu"],
                             c["do"], c["dSf"])
    for name, x, r in zip(("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial"), got, ref):
        assert nerr(x.cpu().numpy(), r) <= TOL, name


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed(d, dtype):
    _check(_case(1000 + d, [5, 1, 0, 19, 8, 16], 2, d, dtype), dtype)


def test_without_states():
    _check(_case(1100, [9, 3], 3, 64, "f32", with_state=False), "f32")


def test_long_sequence():
    _check(_case(1200, [300], 2, 128, "bf16"), "bf16")


def test_many_heads_whole_state_tiles():
    """Enough (sequence, head) pairs that each CTA keeps the whole state width
    (small problems split the columns into 16-wide tiles and sum partials)."""
    _check(_case(1300, [3, 0, 9] * 14, 8, 128, "f32"), "f32")


@pytest.mark.parametrize("lengths,H", [([130, 64, 1, 200], 2), ([1000], 4), ([0, 70, 3], 3)])
def test_chunk_form_matches_the_oracle(lengths, H):
    """kda_chunk_bwd (forward engine's factors, reverse scan in tf32, the walk
    per 64-token chunk from its boundary values) against the fp64 gradients:
    ragged packs (empty and one-token sequences), initial states and a
    final-state gradient; bf16 bound, since the forward engine's factors and
    states are f16."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from oracle.backward import recurrent_backward
    from kda_testutil import TOL_BF16
    c = _case(1300 + len(lengths), lengths, H, 128, "bf16")
    to = lambda x, d=None: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", d)
    bf = torch.bfloat16
    got = kda.kda_chunk_bwd(to(c["q"], bf), to(c["k"], bf), to(c["v"], bf), to(c["g"]),
                            to(c["b"]), c["s"], to(c["S0"]), to(c["cu"]), to(c["do"], bf),
                            to(c["dSf"]))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    ref = recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["b"], c["s"], c["S0"], c["cu"],
                             c["do"], c["dSf"])
    for name, x, r in zip(("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial"), got, ref):
        assert nerr(x.cpu().numpy(), r) <= TOL_BF16, name
