"""Value-head groups (HV = G * H value heads sharing H q/k heads): every
engine against the fp64 oracle run on q and k repeated across each group,
which is what grouping means -- value head j reads q/k head j // G."""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, TOL_F32, nerr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _grouped(seed, lengths, H, G, d, dtype, init_std=0.02):
    """A workload with H * G value heads; q, k keep H heads (the first H)."""
    w = inputs.prefill(seed, lengths, H=H * G, d=d, dtype=dtype, init_std=init_std)
    q_small, k_small = w.q[:, :H].copy(), w.k[:, :H].copy()
    return w, q_small, k_small


def _oracle(w, q_small, k_small, G):
    import oracle
    rep = lambda x: np.ascontiguousarray(np.repeat(x, G, axis=1))
    return oracle.recurrent(rep(q_small), rep(k_small), w.v, w.log_alpha, w.beta, w.scale,
                            w.initial_state, w.cu_seqlens)


def _to(x, dt=None):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype=dt)


@pytest.mark.parametrize("engine,dtype,d,G", [("tensor", "bf16", 128, 2), ("tensor", "bf16", 128, 4),
                                              ("simt", "f32", 64, 2), ("simt", "bf16", 32, 3)])
def test_prefill_engines(engine, dtype, d, G):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    H = 2
    w, qs, ks = _grouped(700 + G + d, [150, 64, 1, 90], H, G, d, dtype)
    qdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out, fin = kda.kda_chunk_fwd(_to(qs, qdt), _to(ks, qdt), _to(w.v, qdt), _to(w.log_alpha),
                                 _to(w.beta), w.scale, _to(w.initial_state), _to(w.cu_seqlens),
                                 None, torch.empty(w.initial_state.shape, device="cuda"),
                                 engine=engine, out_f32=True)
    torch.cuda.synchronize()
    ref_o, ref_s = _oracle(w, qs, ks, G)
    tol = TOL_F32 if (dtype == "f32" or engine == "simt") else TOL_BF16
    assert nerr(out.cpu().numpy(), ref_o) <= tol
    assert nerr(fin.cpu().numpy(), ref_s) <= tol


def test_recurrent_fwd_and_decode_step():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    H, G, d = 3, 2, 128
    w, qs, ks = _grouped(720, [7, 12, 1], H, G, d, "bf16")
    ref_o, ref_s = _oracle(w, qs, ks, G)
    pool = _to(w.initial_state)
    out = kda.kda_recurrent_fwd(_to(qs, torch.bfloat16), _to(ks, torch.bfloat16),
                                _to(w.v, torch.bfloat16), _to(w.log_alpha), _to(w.beta), w.scale,
                                pool, _to(w.cu_seqlens), out_f32=True)
    torch.cuda.synchronize()
    assert nerr(out.cpu().numpy(), ref_o) <= TOL_F32
    assert nerr(pool.cpu().numpy(), ref_s) <= TOL_F32
    # one decode step per sequence: the first token of each sequence
    first = w.cu_seqlens[:-1]
    wd = inputs.prefill(721, [1, 1, 1], H=H * G, d=d, dtype="bf16", init_std=0.02)
    qd, kd = qs[first], ks[first]
    st = _to(wd.initial_state)
    o = kda.kda_recurrent_step(_to(qd, torch.bfloat16), _to(kd, torch.bfloat16),
                               _to(w.v[first], torch.bfloat16), _to(w.log_alpha[first]),
                               _to(w.beta[first]), w.scale, st, out_f32=True)
    torch.cuda.synchronize()
    import oracle
    rep = lambda x: np.ascontiguousarray(np.repeat(x, G, axis=1))
    ro, rs = oracle.recurrent(rep(qd), rep(kd), w.v[first], w.log_alpha[first], w.beta[first],
                              w.scale, wd.initial_state, np.arange(4, dtype=np.int32))
    assert nerr(o.cpu().numpy(), ro) <= TOL_F32
    assert nerr(st.cpu().numpy(), rs) <= TOL_F32
