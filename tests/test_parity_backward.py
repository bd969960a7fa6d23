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


def _case(seed, lengths, H, d, dtype, with_state=True, dsf_scale=1.0):
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
    dSf = ((rng.standard_normal((N, H, d, d)) * dsf_scale).astype(np.float32)
           if with_state else None)
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


# The chunk form multiplies operands with 11-bit significands (tf32, and the
# forward engine's f16 factors and states), so each gradient element carries
# an error of order 2^-11 of the magnitudes it sums.  Against the max-abs /
# RMS metric that is within the bf16 bound when the gradients have the
# spread that output gradients give; a final-state gradient of N(0, 1) per
# element (about 70x the state gradient the output gradients build up) makes
# the last tokens' gradients 60x the RMS, and then the RMS of the error is
# what the operand precision bounds: HEAVY_RMS of the gradient's RMS.
DSF_SCALE = 0.02
HEAVY_RMS = 2e-3


def _chunk_check(c, heavy=False):
    """kda_chunk_bwd against the fp64 gradients: max-abs / RMS within the
    bf16 bound, or, for heavy-tailed gradients, RMS error within HEAVY_RMS."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from oracle.backward import recurrent_backward
    from kda_testutil import TOL_BF16
    to = lambda x, d=None: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda", d)
    bf = torch.bfloat16
    got = kda.kda_chunk_bwd(to(c["q"], bf), to(c["k"], bf), to(c["v"], bf), to(c["g"]),
                            to(c["b"]), c["s"], to(c["S0"]), to(c["cu"]), to(c["do"], bf),
                            to(c["dSf"]))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    ref = recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["b"], c["s"], c["S0"], c["cu"],
                             c["do"], c["dSf"])
    names = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial")
    for name, x, r in zip(names, got, ref):
        if x is None:
            continue
        x = x.cpu().numpy().astype(np.float64)
        if heavy:
            e = float(np.sqrt(np.mean((x - r) ** 2)) / np.sqrt(np.mean(r * r)))
            assert e <= HEAVY_RMS, f"{name}: rms error {e:.3g}"
        else:
            e = nerr(x, r)
            assert e <= TOL_BF16, f"{name}: {e:.3g}"


@pytest.mark.parametrize("lengths,H", [([130, 64, 1, 200], 2), ([1000], 4), ([0, 70, 3], 3)])
def test_chunk_form_matches_the_oracle(lengths, H):
    """kda_chunk_bwd (forward engine's factors, reverse scan in tf32, the
    per-chunk gradient products on the tensor cores) against the fp64
    gradients: ragged packs (empty and one-token sequences, partial last
    chunks), initial states and a final-state gradient."""
    _chunk_check(_case(1300 + len(lengths), lengths, H, 128, "bf16", dsf_scale=DSF_SCALE))


def test_chunk_form_many_heads_one_after_the_other():
    """More reverse-scan CTAs (1 sequence x 4 value tiles x 20 heads = 80)
    than half of the SMs: the X_c kernel runs to completion before the
    reverse scan starts (no flags), instead of beside it."""
    _chunk_check(_case(1310, [200], 20, 128, "bf16", dsf_scale=DSF_SCALE))


def test_chunk_form_heavy_tailed_final_state_gradient():
    """A final-state gradient of N(0, 1) per element over a 1000-token
    sequence: RMS error bound (see HEAVY_RMS)."""
    _chunk_check(_case(1302, [1000], 4, 128, "bf16"), heavy=True)


def test_chunk_form_without_states_or_output_gradient():
    """No initial state, no final-state gradient; then no output gradient
    either (only the final-state gradient drives the gradients)."""
    c = _case(1320, [64, 129], 2, 128, "bf16", with_state=False)
    _chunk_check(c)
    rng = np.random.default_rng(1321)
    c = _case(1322, [100, 28], 2, 128, "bf16")
    c["do"] = None
    c["dSf"] = (rng.standard_normal(c["dSf"].shape) * DSF_SCALE).astype(np.float32)
    _chunk_check(c)


def test_chunk_form_tiny_gradients():
    """Gradients of training size (1e-6): the gradient operands keep fp32
    range (tf32), so the relative error does not grow."""
    c = _case(1330, [200, 77], 2, 128, "bf16", dsf_scale=DSF_SCALE)
    c["do"] = _bf16(c["do"] * 1e-6)
    c["dSf"] = (c["dSf"] * 1e-6).astype(np.float32)
    _chunk_check(c)


def test_chunk_form_strong_decays():
    """Log decays down to -8 per token: the decayed products' gradients
    leave the mid-chunk split (|G_i - G_32| > 80) for direct exponents, and
    the forward prep takes its half-chunk and direct paths."""
    c = _case(1340, [150, 64], 2, 128, "bf16", dsf_scale=DSF_SCALE)
    rng = np.random.default_rng(1341)
    c["g"] = (-rng.uniform(0.5, 8.0, c["g"].shape)).astype(np.float32)
    _chunk_check(c)


def test_chunk_form_k3_gates():
    """K3-range log decays (-5 sigmoid(N(0, 1)) per token) across whole
    chunks."""
    c = _case(1350, [256], 2, 128, "bf16", dsf_scale=DSF_SCALE)
    rng = np.random.default_rng(1351)
    x = rng.standard_normal(c["g"].shape)
    c["g"] = (-5.0 / (1.0 + np.exp(-x))).astype(np.float32)
    _chunk_check(c)


def test_chunk_form_agrees_with_the_token_recurrence_at_bench_size():
    """The single-head-group workload of the benchmark (1 x 16 heads x 4096
    tokens): too large for the fp64 gradient oracle's saved states, so the
    chunk form is checked against the recurrent-form backward (itself pinned
    to the oracle above), within the bf16 bound of the chunk form."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kda_testutil import TOL_BF16
    c = _case(1360, [4096], 16, 128, "bf16", dsf_scale=DSF_SCALE)
    to = lambda x, d=None: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", d)
    bf = torch.bfloat16
    args = (to(c["q"], bf), to(c["k"], bf), to(c["v"], bf), to(c["g"]), to(c["b"]), c["s"],
            to(c["S0"]), to(c["cu"]), to(c["do"], bf), to(c["dSf"]))
    got = kda.kda_chunk_bwd(*args)
    ref = kda.kda_recurrent_bwd(*args)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    for name, x, r in zip(("dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial"), got, ref):
        e = nerr(x.cpu().numpy(), r.cpu().numpy().astype(np.float64))
        assert e <= TOL_BF16, f"{name}: {e:.3g}"
