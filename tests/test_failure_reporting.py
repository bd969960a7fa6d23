"""Failure reporting of the tensor-core prefill, provoked without a GPU fault.

Every wait inside libkda's kernels is bounded.  Here a wait is made to run
out on purpose, in the allowed form: the diagnostic entry point launches the
chunk table and the state scan but withholds the chunk-parallel stage whose
flags the scan waits for, with a wait limit of about two milliseconds.  The
scan must give up on its own, leave KDA_ERR_TIMEOUT in the device status
word (the host call itself returns before any kernel runs), write nothing,
and leave the context usable for the next call.
"""
import time

import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, nerr, run_oracle, run_prefill, to_device

pytestmark = pytest.mark.gpu

SHORT_WAIT = 4_000_000  # SM clocks, ~2 ms at 2 GHz


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def test_withheld_producer_times_out_and_is_reported():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(120, [300, 129], H=2, d=128, dtype="bf16", init_std=0.02)
    d = to_device(w)
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    out = torch.full((w.T, w.H, 128), float("nan"), device="cuda")
    fin = torch.full((w.N, w.H, 128, 128), float("nan"), device="cuda")
    t0 = time.perf_counter()
    kda.kda_chunk_fwd_ws_diag(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                              d["initial_state"], d["cu_seqlens"], out, fin,
                              withhold_prep=True, wait_cycles=SHORT_WAIT)
    st = kda.kda_device_status()  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st == kda.KDA_ERR_TIMEOUT, kda.kda_status_string(st)
    assert elapsed < 10.0, f"the kernels took {elapsed:.1f} s to give up"
    # the scan returned before writing any final state, and no output pass ran
    assert torch.isnan(fin).all() and torch.isnan(out).all()
    # the status word was read and cleared, and the next call is right
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    ref_o, ref_s = run_oracle(w)
    o, s = run_prefill(w, engine="tensor", out_f32=True)
    assert nerr(o, ref_o) < TOL_BF16 and nerr(s, ref_s) < TOL_BF16


@pytest.mark.parametrize("lengths,H", [([300, 129], 2), ([130] * 40, 2)])
def test_diag_entry_with_producer_matches(lengths, H):
    """The same entry without withholding anything, with the short wait limit
    and the overlapped order forced (also for 160 scan CTAs, which the plain
    call runs in sequence), is bit-identical to the plain call: no wait comes
    near its limit."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(121, lengths, H=H, d=128, dtype="bf16", init_std=0.02)
    d = to_device(w)
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale, d["initial_state"],
            d["cu_seqlens"])
    fin = [torch.empty((w.N, w.H, 128, 128), device="cuda") for _ in range(2)]
    o1, _ = kda.kda_chunk_fwd(*args, None, fin[0], engine="tensor", out_f32=True)
    o2 = torch.empty_like(o1)
    kda.kda_chunk_fwd_ws_diag(*args, o2, fin[1], withhold_prep=False,
                              wait_cycles=200 * SHORT_WAIT, out_f32=True)
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    torch.testing.assert_close(o1, o2, rtol=0, atol=0)
    torch.testing.assert_close(fin[0], fin[1], rtol=0, atol=0)


def test_diag_entry_rejects_the_simt_engine():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(122, [40], H=1, d=64, dtype="f32")
    d = to_device(w)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_ws_diag(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                                  None, d["cu_seqlens"], None, None, withhold_prep=True)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED
