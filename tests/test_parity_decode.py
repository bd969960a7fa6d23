"""Parity of libkda's decode step with the fp64 oracle.  N sequences advance
one token per step; the oracle runs each sequence's steps as one packed
sequence (cu_seqlens) from the same initial state."""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, TOL_F32, check_bf16_output, nerr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _oracle_steps(w):
    """Oracle over `steps` tokens per sequence: returns out [steps,N,H,d], final."""
    import oracle
    steps, N, H, d = w.q.shape
    tr = lambda x: np.ascontiguousarray(np.swapaxes(x, 0, 1)).reshape(N * steps, *x.shape[2:])
    cu = (np.arange(N + 1) * steps).astype(np.int32)
    o, f = oracle.recurrent(tr(w.q), tr(w.k), tr(w.v), tr(w.log_alpha), tr(w.beta), w.scale,
                            w.initial_state, cu)
    return np.swapaxes(o.reshape(N, steps, H, -1), 0, 1), f


def _gpu_steps(w, out_f32):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    qdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = lambda x, dt=None: torch.from_numpy(x).to("cuda", dtype=dt)
    q, k, v = dev(w.q, qdt), dev(w.k, qdt), dev(w.v, qdt)
    la, b = dev(w.log_alpha), dev(w.beta)
    state = dev(w.initial_state).contiguous()
    outs = []
    for t in range(w.q.shape[0]):
        outs.append(kda.kda_recurrent_step(q[t], k[t], v[t], la[t], b[t], w.scale, state,
                                           out_f32=out_f32))
    torch.cuda.synchronize()
    return (torch.stack(outs).float().cpu().numpy().astype(np.float64),
            state.cpu().numpy().astype(np.float64))


def _decode_workload(seed, N, H, d, steps, dtype):
    w = inputs.batched_decode(n_seqs=N, H=H, d=d, steps=steps, seed=seed)
    if dtype == "f32":
        rng = np.random.default_rng(seed + 1)
        w.q = rng.standard_normal(w.q.shape).astype(np.float32) * 0.1
        w.k = (w.k * 1.0).astype(np.float32)
        w.v = rng.standard_normal(w.v.shape).astype(np.float32)
        w.dtype = "f32"
    return w


def test_batched_decode_config():
    """256 sequences x 32 heads, d = 128, fp32 state (512 MiB), 64 steps."""
    w = inputs.batched_decode()
    ref_o, ref_s = _oracle_steps(w)
    o, s = _gpu_steps(w, out_f32=True)
    assert nerr(o, ref_o) <= TOL_BF16
    assert nerr(s, ref_s) <= TOL_BF16
    # the bf16-output variant, steps 0..7 only (same states feed each step)
    w8 = inputs.batched_decode(steps=8)
    ref8, _ = _oracle_steps(w8)
    ob, _ = _gpu_steps(w8, out_f32=False)
    check_bf16_output(ob, ref8)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_shapes(d, dtype):
    w = _decode_workload(200 + d, N=5, H=3, d=d, steps=7, dtype=dtype)
    ref_o, ref_s = _oracle_steps(w)
    o, s = _gpu_steps(w, out_f32=True)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert nerr(o, ref_o) <= tol
    assert nerr(s, ref_s) <= tol


def test_decode_continues_prefill():
    """Decode from states that a prefill produced (the serving hand-off):
    prefill 300 tokens, then 5 decode steps, against one oracle run over all
    305 tokens."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    import oracle
    from kda_testutil import to_device
    w = inputs.prefill(210, [305, 305], H=4, d=128, dtype="bf16")
    ref_o, ref_s = oracle.recurrent(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, None,
                                    w.cu_seqlens)
    d = to_device(w)
    pre = lambda x: torch.cat([x[0:300], x[305:605]]).contiguous()
    st = torch.zeros((2, 4, 128, 128), device="cuda")
    cu = torch.tensor([0, 300, 600], dtype=torch.int32, device="cuda")
    kda.kda_chunk_fwd(pre(d["q"]), pre(d["k"]), pre(d["v"]), pre(d["log_alpha"]),
                      pre(d["beta"]), w.scale, None, cu, None, st)
    outs = []
    for t in range(5):
        idx = torch.tensor([300 + t, 605 + t], device="cuda")
        outs.append(kda.kda_recurrent_step(d["q"][idx].contiguous(), d["k"][idx].contiguous(),
                                           d["v"][idx].contiguous(),
                                           d["log_alpha"][idx].contiguous(),
                                           d["beta"][idx].contiguous(), w.scale, st,
                                           out_f32=True))
    torch.cuda.synchronize()
    o = torch.stack(outs).cpu().numpy()            # [5, 2, H, d]
    ref = np.stack([ref_o[300:305], ref_o[605:610]], axis=1)
    assert nerr(o, ref) <= TOL_BF16
    assert nerr(st.cpu().numpy(), ref_s) <= TOL_BF16
