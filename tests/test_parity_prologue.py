"""The fused input prologue in every kernel: raw q/k (not normalised), beta
logits and K3 gate projections go in with the prologue flags, and the result
must match the fp64 oracle run on the oracle's own prologue of the same raw
inputs.  The gate's strong decays (log retention down to -5 per token) also
send many tensor-core chunks through their direct-exponent path."""
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


def _bf16(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _raw(seed, lengths, H, d, dtype, G=1):
    """Raw projections: q, k ~ N(0, 2) unnormalised, beta and gate logits."""
    rng = np.random.default_rng(seed)
    T, HV = int(sum(lengths)), H * G
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    q = (rng.standard_normal((T, H, d)) * 2).astype(np.float32)
    k = (rng.standard_normal((T, H, d)) * 2).astype(np.float32)
    v = rng.standard_normal((T, HV, d)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = _bf16(q), _bf16(k), _bf16(v)
    beta = rng.standard_normal((T, HV)).astype(np.float32)
    g = rng.standard_normal((T, HV, d)).astype(np.float32)
    bias = (rng.standard_normal((HV, d)) * 0.5 - 1.5).astype(np.float32)
    a_log = rng.uniform(-1.0, 1.0, HV).astype(np.float32)
    s0 = (rng.standard_normal((len(lengths), HV, d, d)) * 0.02).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, g=g, bias=bias, a_log=a_log, cu=cu, s0=s0,
                scale=d ** -0.5, G=G)


def _oracle(r, l2=True, bl=True, gate=True):
    import oracle
    from oracle import prologue as P
    q, k, b, la = P.apply(r["q"], r["k"], r["beta"], r["g"], l2norm=l2, beta_logits=bl,
                          gate=(r["bias"], r["a_log"]) if gate else None)
    rep = lambda x: np.ascontiguousarray(np.repeat(x, r["G"], axis=1))
    return oracle.recurrent(rep(q), rep(k), r["v"], la, b, r["scale"], r["s0"], r["cu"])


def _to(x, dt=None):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype=dt)


@pytest.mark.parametrize("engine,dtype,d", [("tensor", "bf16", 128), ("simt", "f32", 64),
                                            ("simt", "bf16", 32)])
@pytest.mark.parametrize("flags", [(True, True, True), (True, False, False), (False, True, True)])
def test_prefill(engine, dtype, d, flags):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    l2, bl, gt = flags
    r = _raw(900 + d, [150, 64, 1, 90], 2, d, dtype)
    if not gt:   # log_alpha given as a retention, as without the prologue
        r["g"] = -np.abs(r["g"]) * 0.3
    if not l2:   # without the L2 prologue q and k must arrive normalised (unit keys
        # keep the delta rule's transition contractive)
        for name in ("q", "k"):
            x = r[name] / np.linalg.norm(r[name], axis=-1, keepdims=True)
            r[name] = _bf16(x) if dtype == "bf16" else x.astype(np.float32)
    qdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out, fin = kda.kda_chunk_fwd(
        _to(r["q"], qdt), _to(r["k"], qdt), _to(r["v"], qdt), _to(r["g"]), _to(r["beta"]),
        r["scale"], _to(r["s0"]), _to(r["cu"]), None, torch.empty(r["s0"].shape, device="cuda"),
        engine=engine, out_f32=True, l2norm_qk=l2, beta_logits=bl,
        gate=(_to(r["bias"]), _to(r["a_log"])) if gt else None)
    torch.cuda.synchronize()
    ref_o, ref_s = _oracle(r, l2, bl, gt)
    tol = TOL_BF16 if engine == "tensor" else TOL_F32
    assert nerr(out.cpu().numpy(), ref_o) <= tol
    assert nerr(fin.cpu().numpy(), ref_s) <= tol


def test_recurrent_fwd_and_step_with_groups():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    r = _raw(950, [7, 12, 1], 2, 128, "bf16", G=2)
    ref_o, ref_s = _oracle(r)
    gate = (_to(r["bias"]), _to(r["a_log"]))
    pool = _to(r["s0"])
    out = kda.kda_recurrent_fwd(_to(r["q"], torch.bfloat16), _to(r["k"], torch.bfloat16),
                                _to(r["v"], torch.bfloat16), _to(r["g"]), _to(r["beta"]),
                                r["scale"], pool, _to(r["cu"]), out_f32=True, l2norm_qk=True,
                                beta_logits=True, gate=gate)
    torch.cuda.synchronize()
    assert nerr(out.cpu().numpy(), ref_o) <= TOL_F32
    assert nerr(pool.cpu().numpy(), ref_s) <= TOL_F32
    # one decode step: each sequence's first token from its initial state
    first = r["cu"][:-1]
    rs = dict(r, q=r["q"][first], k=r["k"][first], v=r["v"][first], beta=r["beta"][first],
              g=r["g"][first], cu=np.arange(4, dtype=np.int32))
    ro, rst = _oracle(rs)
    st = _to(r["s0"])
    o = kda.kda_recurrent_step(_to(rs["q"], torch.bfloat16), _to(rs["k"], torch.bfloat16),
                               _to(rs["v"], torch.bfloat16), _to(rs["g"]), _to(rs["beta"]),
                               r["scale"], st, out_f32=True, l2norm_qk=True, beta_logits=True,
                               gate=gate)
    torch.cuda.synchronize()
    assert nerr(o.cpu().numpy(), ro) <= TOL_F32
    assert nerr(st.cpu().numpy(), rst) <= TOL_F32


@pytest.mark.parametrize("G", [1, 2])
def test_launch_orders_agree_with_prologue_and_groups(G):
    """With the prologue (all three parts) and value-head groups, the
    tensor engine's concurrent and sequential launch orders (the latter forced
    by recording per-kernel events) give bit-identical results."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    r = _raw(960 + G, [700, 1, 300, 64], 2, 128, "bf16", G=G)
    args = (_to(r["q"], torch.bfloat16), _to(r["k"], torch.bfloat16), _to(r["v"], torch.bfloat16),
            _to(r["g"]), _to(r["beta"]), r["scale"], _to(r["s0"]), _to(r["cu"]))
    kw = dict(engine="tensor", out_f32=True, l2norm_qk=True, beta_logits=True,
              gate=(_to(r["bias"]), _to(r["a_log"])))
    f1 = torch.empty(r["s0"].shape, device="cuda")
    o1, _ = kda.kda_chunk_fwd(*args, None, f1, **kw)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev:
        e.record()
    o2 = torch.empty_like(o1)
    f2 = torch.empty_like(f1)
    kda.kda_chunk_fwd_ws_timed(*args, o2, f2, ev, **kw)
    torch.cuda.synchronize()
    torch.testing.assert_close(o1, o2, rtol=0, atol=0)
    torch.testing.assert_close(f1, f2, rtol=0, atol=0)
    ref_o, ref_s = _oracle(r)
    assert nerr(o1.cpu().numpy(), ref_o) <= TOL_BF16
    assert nerr(f1.cpu().numpy(), ref_s) <= TOL_BF16


def test_host_entry_with_prologue():
    """kda_chunk_fwd_host with host-side gate parameters equals the device entry."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    r = _raw(970, [150, 64, 1, 90], 2, 128, "bf16")
    dev = (_to(r["q"], torch.bfloat16), _to(r["k"], torch.bfloat16), _to(r["v"], torch.bfloat16),
           _to(r["g"]), _to(r["beta"]), r["scale"], _to(r["s0"]), _to(r["cu"]))
    kw = dict(engine="tensor", out_f32=True, l2norm_qk=True, beta_logits=True)
    f1 = torch.empty(r["s0"].shape, device="cuda")
    o1, _ = kda.kda_chunk_fwd(*dev, None, f1, gate=(_to(r["bias"]), _to(r["a_log"])), **kw)
    torch.cuda.synchronize()
    h = lambda x, dt=None: torch.from_numpy(np.ascontiguousarray(x)).to(dt).pin_memory() \
        if dt is not None else torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    hf = torch.empty(r["s0"].shape).pin_memory()
    o2, _ = kda.kda_chunk_fwd_host(h(r["q"], torch.bfloat16), h(r["k"], torch.bfloat16),
                                   h(r["v"], torch.bfloat16), h(r["g"]), h(r["beta"]), r["scale"],
                                   h(r["s0"]), h(r["cu"]), None, hf,
                                   gate=(h(r["bias"]), h(r["a_log"])), **kw)
    torch.cuda.synchronize()
    torch.testing.assert_close(o2, o1.cpu(), rtol=0, atol=0)
    torch.testing.assert_close(hf, f1.cpu(), rtol=0, atol=0)
