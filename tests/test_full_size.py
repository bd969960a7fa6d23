"""Parity at the full workload sizes, in the launch configuration the
benchmark times (tensor-core engine, bf16 inputs, fp32 state).

* The packed variable-length workload (32 sequences, ~140k tokens, H = 32)
  is checked element by element against the oracle, one sequence at a time.
* The 1,048,576-token single-sequence workload is drawn on the device.  The
  oracle runs one whole head over all 1M tokens (sampled outputs it can
  compute one by one) and the checkpoint prefix of 8192 tokens for every
  head; and the call must equal, bit for bit, a prefix call followed by a
  call on the remainder resumed from the prefix's final state.
"""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, nerr

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def test_varlen_workload_full():
    import torch
    import oracle
    import kimi_delta_attention_chunkwise_gb300 as kda
    from kda_testutil import to_device
    w = inputs.varlen_prefill()
    assert w.N == 32 and 100_000 < w.T < 200_000
    d = to_device(w)
    fin = torch.empty((w.N, w.H, 128, 128), device="cuda")
    out, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                               d["initial_state"], d["cu_seqlens"], None, fin, engine="tensor",
                               out_f32=True)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    fin = fin.cpu().numpy()
    assert np.isfinite(out).all() and np.isfinite(fin).all()
    worst_o = worst_s = 0.0
    ref_sq_o, ref_sq_s, n_o, n_s = 0.0, 0.0, 0, 0
    max_o = max_s = 0.0
    for n in range(w.N):
        a, b = int(w.cu_seqlens[n]), int(w.cu_seqlens[n + 1])
        ro, rs = oracle.recurrent(w.q[a:b], w.k[a:b], w.v[a:b], w.log_alpha[a:b], w.beta[a:b],
                                  w.scale, w.initial_state[n:n + 1])
        max_o = max(max_o, float(np.abs(out[a:b] - ro).max()))
        max_s = max(max_s, float(np.abs(fin[n] - rs[0]).max()))
        ref_sq_o += float((ro * ro).sum()); n_o += ro.size
        ref_sq_s += float((rs * rs).sum()); n_s += rs.size
    e_o = max_o / np.sqrt(ref_sq_o / n_o)
    e_s = max_s / np.sqrt(ref_sq_s / n_s)
    assert e_o <= TOL_BF16, f"out error {e_o:.3g}"
    assert e_s <= TOL_BF16, f"final_state error {e_s:.3g}"


def test_long_context_full():
    import torch
    import oracle
    import kimi_delta_attention_chunkwise_gb300 as kda
    T, H, cut, head = 1 << 20, 32, 8192, 5
    x = inputs.long_context_device(T=T, H=H)
    q, k, v, la, beta, scale = x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["scale"]
    fin = torch.empty((1, H, 128, 128), device="cuda")
    out, _ = kda.kda_chunk_fwd(q, k, v, la, beta, scale, None, None, None, fin,
                               engine="tensor", out_f32=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()

    # split at the checkpoint and chain through the state: bit-identical
    st = torch.zeros_like(fin)
    o1, _ = kda.kda_chunk_fwd(q[:cut], k[:cut], v[:cut], la[:cut], beta[:cut], scale, None,
                              None, None, st, engine="tensor", out_f32=True)
    torch.cuda.synchronize()
    prefix_state = st.clone()
    o2, _ = kda.kda_chunk_fwd(q[cut:], k[cut:], v[cut:], la[cut:], beta[cut:], scale, st,
                              None, None, st, engine="tensor", out_f32=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, out[:cut]) and torch.equal(o2, out[cut:])
    assert torch.equal(st, fin)

    # the checkpoint prefix, every head, against the oracle
    host = lambda t, sl: t[sl].float().cpu().numpy()
    sl = slice(0, cut)
    ro, rs = oracle.recurrent(host(q, sl), host(k, sl), host(v, sl), host(la, sl),
                              host(beta, sl), scale)
    assert nerr(o1.cpu().numpy(), ro) <= TOL_BF16
    assert nerr(prefix_state.cpu().numpy(), rs) <= TOL_BF16
    del ro, rs

    # one head over all 1M tokens
    hs = slice(head, head + 1)
    sel = lambda t: t[:, hs].float().cpu().numpy()
    ro, rs = oracle.recurrent(sel(q), sel(k), sel(v), sel(la), beta[:, hs].cpu().numpy(), scale)
    oh = out[:, hs].cpu().numpy()
    e_o, e_s = nerr(oh, ro), nerr(fin[:, hs].cpu().numpy(), rs)
    assert e_o <= TOL_BF16, f"head {head} out error {e_o:.3g}"
    assert e_s <= TOL_BF16, f"head {head} final_state error {e_s:.3g}"
