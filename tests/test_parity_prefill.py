"""Parity of libkda's chunkwise prefill with the fp64 oracle, element by
element, on seeded inputs, through the C ABI (ctypes binding)."""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import (TOL_BF16, TOL_F32, check_bf16_output, nerr, run_oracle,
                          run_prefill, to_device)

pytestmark = pytest.mark.gpu

ENGINES = ["tensor", "simt"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _check(w, engine, tol=TOL_BF16):
    ref_o, ref_s = run_oracle(w)
    o, s = run_prefill(w, engine=engine, out_f32=True)
    e_o, e_s = nerr(o, ref_o), nerr(s, ref_s)
    assert e_o <= tol, f"out error {e_o:.3g}"
    assert e_s <= tol, f"final_state error {e_s:.3g}"
    if w.dtype == "bf16":
        ob, sb = run_prefill(w, engine=engine, out_f32=False)
        check_bf16_output(ob, ref_o, tol)
        assert nerr(sb, ref_s) <= tol
    return e_o, e_s


def test_tiny_fp32_config():
    """B=1, H=1, T=64, d=16, chunk 16, fp32 inputs, seed 0."""
    w = inputs.tiny_f32()
    e_o, e_s = _check(w, "simt", TOL_F32)
    assert e_o < TOL_F32 and e_s < TOL_F32


@pytest.mark.parametrize("engine", ENGINES)
def test_head_group_prefill_config(engine):
    """B=1, H=16, T=4096, d=128, chunk 64, bf16 inputs, fp32 state."""
    _check(inputs.head_group_prefill(), engine)


@pytest.mark.parametrize("engine", ENGINES)
def test_varlen_ragged(engine):
    """Packed ragged sequences: lengths 1, 63, 64, 65, 128, 200 and random
    short ones (partial chunks, single-token sequences), nonzero initial
    states, H = 3."""
    rng = np.random.default_rng(100)
    lengths = [1, 63, 64, 65, 128, 200] + [int(x) for x in rng.integers(1, 300, size=6)]
    w = inputs.prefill(100, lengths, H=3, d=128, dtype="bf16", init_std=0.02)
    _check(w, engine)


def test_long_context_prefix():
    """The 1M-token recipe's checkpoint prefix: T = 8192, H = 32,
    log_alpha = -softplus(N(-6, 1)) (long horizons)."""
    _check(inputs.long_context_prefix(8192), "tensor")


def test_k3_range_gates_stay_on_tensor_cores():
    """log alpha = -5 sigmoid(g), g ~ N(0, 1): the K3 gate's range (-5, 0)
    with its midpoint -2.5 ("Linear Attention, From Scratch to Kimi 3",
    sec. 6).  Over 32 tokens the decay passes e^-80, so the mid-chunk
    reference cannot serve these chunks, but over 16 it cannot: every item
    takes the half-chunk references (tensor cores), none the direct path."""
    import kimi_delta_attention_chunkwise_gb300 as kda
    rng = np.random.default_rng(111)
    w = inputs.prefill(111, [2048, 700, 64, 1], H=4, d=128, dtype="bf16", init_std=0.02)
    g = rng.standard_normal(w.log_alpha.shape)
    w.log_alpha = (-5.0 / (1.0 + np.exp(-g))).astype(np.float32)
    kda.kda_chunk_path_counts()  # clear
    _check(w, "tensor")
    mid, half, direct = kda.kda_chunk_path_counts()
    assert direct == 0, (mid, half, direct)
    assert half > 0 and half >= 4 * mid, (mid, half, direct)


@pytest.mark.parametrize("engine", ENGINES)
def test_gate_extremes(engine):
    """Gates from no decay at all (log alpha = 0) down to -80 per token (the
    state is wiped), beta in {0, 1}, on one packed batch; the tensor engine
    takes its direct-exponent path for the chunks of the strongest decays."""
    import kimi_delta_attention_chunkwise_gb300 as kda
    rng = np.random.default_rng(101)
    w = inputs.prefill(101, [130, 70, 64], H=2, d=128, dtype="bf16", init_std=0.5)
    T = w.T
    la = w.log_alpha.copy()
    la[:40] = 0.0
    la[40:80] = -rng.uniform(0, 80, size=la[40:80].shape).astype(np.float32)
    la[80:90] = -80.0
    w.log_alpha = la
    b = w.beta.copy()
    b[::3] = 0.0
    b[1::3] = 1.0
    w.beta = b
    assert T == 264
    kda.kda_chunk_path_counts()  # clear
    _check(w, engine)
    mid, half, direct = kda.kda_chunk_path_counts()
    if engine == "tensor":
        assert direct > 0 and mid > 0, (mid, half, direct)
    else:
        assert (mid, half, direct) == (0, 0, 0)


@pytest.mark.parametrize("d,C", [(16, 16), (32, 32), (64, 64), (128, 32), (64, 16)])
def test_simt_shapes_fp32(d, C):
    """The fp32 engine across head widths and chunk sizes, with ragged
    sequences and initial states."""
    w = inputs.prefill(102 + d + C, [5, 40, 97], H=2, d=d, dtype="f32", gate="uniform",
                       init_std=0.3, chunk_size=C)
    _check(w, "simt", TOL_F32)


def test_chunk_size_invariance_fp32():
    """Results do not depend on the chunk size (the chunkwise schedule is the
    same recurrence): C = 16, 32, 64 agree with each other to fp32 rounding."""
    w = inputs.prefill(103, [150, 77], H=2, d=64, dtype="f32", gate="uniform", init_std=0.3)
    outs = [run_prefill(w, engine="simt", chunk_size=C) for C in (16, 32, 64)]
    for o, s in outs[1:]:
        assert nerr(o, outs[0][0]) < TOL_F32
        assert nerr(s, outs[0][1]) < TOL_F32


def test_empty_and_zero_length():
    """T = 0 (final = initial), and zero-length sequences inside a pack."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(104, [0, 70, 0, 3], H=2, d=128, dtype="bf16", init_std=0.1)
    ref_o, ref_s = run_oracle(w)
    for engine in ENGINES:
        o, s = run_prefill(w, engine=engine, out_f32=True)
        assert nerr(o, ref_o) < TOL_BF16 and nerr(s, ref_s) < TOL_BF16
        np.testing.assert_array_equal(s[0], w.initial_state[0])
        np.testing.assert_array_equal(s[2], w.initial_state[2])
    # no tokens at all
    z = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    s0 = torch.randn((1, 2, 128, 128), device="cuda")
    fin = torch.full_like(s0, float("nan"))
    for engine in ENGINES:
        kda.kda_chunk_fwd(z, z, z, z.float(), torch.zeros((0, 2), device="cuda"), 0.1, s0,
                          None, None, fin, engine=engine)
        torch.cuda.synchronize()
        assert torch.equal(fin, s0)


@pytest.mark.parametrize("engine", ENGINES)
def test_state_options(engine):
    """NULL initial state (zeros), NULL final state (not written), and
    final_state aliasing initial_state (in-place resume)."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(105, [100, 37], H=2, d=128, dtype="bf16", init_std=0.05)
    ref_o, ref_s = run_oracle(w)
    d = to_device(w)
    st = d["initial_state"].clone()
    out, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                               st, d["cu_seqlens"], None, st, engine=engine, out_f32=True)
    torch.cuda.synchronize()
    assert nerr(out.cpu().numpy(), ref_o) < TOL_BF16
    assert nerr(st.cpu().numpy(), ref_s) < TOL_BF16
    out2, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                                d["initial_state"], d["cu_seqlens"], None, None,
                                engine=engine, out_f32=True)
    torch.cuda.synchronize()
    assert nerr(out2.cpu().numpy(), ref_o) < TOL_BF16
    w.initial_state = None
    ref_o0, ref_s0 = run_oracle(w)
    o0, s0 = run_prefill(w, engine=engine, out_f32=True)
    assert nerr(o0, ref_o0) < TOL_BF16 and nerr(s0, ref_s0) < TOL_BF16


@pytest.mark.parametrize("engine", ENGINES)
def test_split_and_chain(engine):
    """A prefix call followed by a call on the remainder, resumed from the
    prefix's final state, matches the oracle on the whole sequence (the
    fixed-size state is the only thing carried)."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(106, [1000], H=4, d=128, dtype="bf16")
    ref_o, ref_s = run_oracle(w)
    d = to_device(w)
    cut = 389
    st = torch.zeros((1, 4, 128, 128), device="cuda")
    outs = []
    for sl in (slice(0, cut), slice(cut, w.T)):
        o, _ = kda.kda_chunk_fwd(d["q"][sl].contiguous(), d["k"][sl].contiguous(),
                                 d["v"][sl].contiguous(), d["log_alpha"][sl].contiguous(),
                                 d["beta"][sl].contiguous(), w.scale, st, None, None, st,
                                 engine=engine, out_f32=True)
        outs.append(o)
    torch.cuda.synchronize()
    o = torch.cat(outs).cpu().numpy()
    assert nerr(o, ref_o) < TOL_BF16
    assert nerr(st.cpu().numpy(), ref_s) < TOL_BF16


def test_library_scratch_matches_caller_scratch():
    """kda_chunk_fwd (scratch from cudaMallocAsync) and kda_chunk_fwd_ws
    (caller-owned scratch) give bit-identical results."""
    w = inputs.prefill(107, [300, 129], H=2, d=128, dtype="bf16", init_std=0.02)
    a = run_prefill(w, engine="tensor", out_f32=True)
    b = run_prefill(w, engine="tensor", out_f32=True, use_library_scratch=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_engines_agree():
    """The two engines are independent GPU witnesses of the same result."""
    w = inputs.prefill(108, [700, 300], H=4, d=128, dtype="bf16", init_std=0.02)
    a = run_prefill(w, engine="tensor", out_f32=True)
    b = run_prefill(w, engine="simt", out_f32=True)
    assert nerr(a[0], b[0]) < TOL_BF16 and nerr(a[1], b[1]) < TOL_BF16


@pytest.mark.parametrize("lengths,H", [([4096], 16), ([1000, 37, 2000], 8), ([130] * 40, 2),
                                       ([135000], 32)])
def test_launch_orders_agree(lengths, H):
    """When the scan's CTAs fit in half the SMs, the tensor engine runs the
    scan beside the persistent prep on the SMs the prep leaves (image flags)
    for calls of at most 65,536 (chunk, head) items (the first two cases),
    and the prep on every SM, then the scan with the output pass beside it
    (state flags), for larger ones (67,520 items for 135,000 tokens x 32
    heads).  With more scan CTAs (160 for 40 sequences x 2 heads x 2 value
    tiles) or with per-kernel events it runs them in sequence.  All orders
    run the same arithmetic, so the results are bit-identical, and they match
    the oracle."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(109, lengths, H=H, d=128, dtype="bf16", init_std=0.02)
    d = to_device(w)
    fin = [torch.empty((w.N, w.H, 128, 128), dtype=torch.float32, device="cuda")
           for _ in range(2)]
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale, d["initial_state"],
            d["cu_seqlens"])
    o1, _ = kda.kda_chunk_fwd(*args, None, fin[0], engine="tensor", out_f32=True)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev:
        e.record()  # the library records them again; they must exist first
    o2 = torch.empty_like(o1)
    kda.kda_chunk_fwd_ws_timed(*args, o2, fin[1], ev, engine="tensor", out_f32=True)
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    torch.testing.assert_close(o1, o2, rtol=0, atol=0)
    torch.testing.assert_close(fin[0], fin[1], rtol=0, atol=0)
    if w.T <= 4096 and w.H <= 8:
        ref_o, ref_s = run_oracle(w)
        assert nerr(o1.cpu().numpy(), ref_o) < TOL_BF16
        assert nerr(fin[0].cpu().numpy(), ref_s) < TOL_BF16


@pytest.mark.parametrize("lengths,H,out_f32", [([4096], 16, False), ([300, 129, 1], 2, True)])
def test_host_buffers_match_device_entry(lengths, H, out_f32):
    """kda_chunk_fwd_host (host tensors in and out, copies on the stream) gives
    bit-identical results to kda_chunk_fwd on device copies of the same
    inputs; two calls on two streams with two scratch buffers overlap and
    still agree."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(110, lengths, H=H, d=128, dtype="bf16", init_std=0.02)
    d = to_device(w)
    fin = torch.empty((w.N, w.H, 128, 128), dtype=torch.float32, device="cuda")
    ref, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                               d["initial_state"], d["cu_seqlens"], None, fin, engine="tensor",
                               out_f32=out_f32)
    torch.cuda.synchronize()
    pin = lambda x: x.cpu().pin_memory()
    h = {key: (pin(val) if val is not None else None) for key, val in d.items()}
    streams = [torch.cuda.Stream() for _ in range(2)]
    results = []
    for s in streams:
        hfin = torch.empty((w.N, w.H, 128, 128), dtype=torch.float32).pin_memory()
        scratch = torch.empty(320 << 20, dtype=torch.uint8, device="cuda")
        o, f = kda.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["log_alpha"], h["beta"],
                                      w.scale, h["initial_state"], h["cu_seqlens"], None, hfin,
                                      scratch=scratch, engine="tensor", stream=s,
                                      out_f32=out_f32)
        results.append((o, f, scratch))
    torch.cuda.synchronize()
    for o, f, _ in results:
        assert o.device.type == "cpu" and f.device.type == "cpu"
        torch.testing.assert_close(o, ref.cpu(), rtol=0, atol=0)
        torch.testing.assert_close(f, fin.cpu(), rtol=0, atol=0)
