"""Parity of libkda's multi-token recurrent pass (kda_recurrent_fwd) with the
fp64 oracle: packed sequences of mixed lengths (empty ones included), every
head width, fp32 and bf16 inputs, and the slot-indexed state pool (permuted
slots, skipped sequences, untouched slots, an out-of-range index)."""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_F32, check_bf16_output, nerr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _dev(w):
    import torch
    qdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    to = lambda x, dt=None: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype=dt)
    return dict(q=to(w.q, qdt), k=to(w.k, qdt), v=to(w.v, qdt), g=to(w.log_alpha),
                b=to(w.beta), cu=to(w.cu_seqlens))


def _oracle(w, init):
    import oracle
    return oracle.recurrent(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale, init, w.cu_seqlens)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_sequences(d, dtype):
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(500 + d, [5, 1, 17, 0, 33], H=3, d=d, dtype=dtype, init_std=0.02)
    t = _dev(w)
    pool = torch.from_numpy(w.initial_state.copy()).cuda()
    out = kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool, t["cu"],
                                out_f32=True)
    torch.cuda.synchronize()
    ref_o, ref_s = _oracle(w, w.initial_state)
    assert nerr(out.cpu().numpy(), ref_o) <= TOL_F32
    assert nerr(pool.cpu().numpy(), ref_s) <= TOL_F32
    if dtype == "bf16":
        pool = torch.from_numpy(w.initial_state.copy()).cuda()
        ob = kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool, t["cu"])
        torch.cuda.synchronize()
        check_bf16_output(ob.float().cpu().numpy(), ref_o)


def test_one_sequence_without_cu_seqlens():
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(610, [70], H=2, d=64, dtype="f32", init_std=0.05)
    t = _dev(w)
    pool = torch.from_numpy(w.initial_state.copy()).cuda()
    out = kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool)
    torch.cuda.synchronize()
    ref_o, ref_s = _oracle(w, w.initial_state)
    assert nerr(out.cpu().numpy(), ref_o) <= TOL_F32
    assert nerr(pool.cpu().numpy(), ref_s) <= TOL_F32


def test_state_pool_slots():
    """Sequences map to permuted slots of a larger pool; a negative index skips
    its sequence; slots no sequence names stay bit-identical."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(620, [9, 4, 12, 7], H=2, d=128, dtype="bf16")
    S, H, d = 7, 2, 128
    rng = np.random.default_rng(621)
    pool0 = (rng.standard_normal((S, H, d, d)) * 0.05).astype(np.float32)
    slots = np.array([5, 0, -1, 3], dtype=np.int32)
    t = _dev(w)
    pool = torch.from_numpy(pool0.copy()).cuda()
    out = torch.full((w.T, H, d), float("nan"), dtype=torch.float32, device="cuda")
    kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool, t["cu"],
                          torch.from_numpy(slots).cuda(), out=out)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_SUCCESS
    init = np.stack([pool0[s] if s >= 0 else np.zeros((H, d, d), np.float32) for s in slots])
    ref_o, ref_s = _oracle(w, init)
    got_pool, got_out = pool.cpu().numpy(), out.cpu().numpy()
    cu = w.cu_seqlens
    for i, s in enumerate(slots):
        rows = slice(cu[i], cu[i + 1])
        if s < 0:
            assert np.isnan(got_out[rows]).all()      # skipped: outputs not written
            continue
        assert nerr(got_out[rows], ref_o[rows]) <= TOL_F32
        assert nerr(got_pool[s], ref_s[i]) <= TOL_F32
    for s in set(range(S)) - set(int(x) for x in slots):
        np.testing.assert_array_equal(got_pool[s], pool0[s])


def test_out_of_range_slot_sets_status():
    """An index >= num_slots is caught in the kernel's bounds check: that
    sequence is skipped and the device status word reports it."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(630, [6, 5], H=1, d=32, dtype="f32")
    t = _dev(w)
    pool0 = np.zeros((2, 1, 32, 32), np.float32)
    pool = torch.from_numpy(pool0.copy()).cuda()
    kda.kda_device_status()  # clear
    kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool, t["cu"],
                          torch.tensor([1, 2], dtype=torch.int32, device="cuda"))
    assert kda.kda_device_status() == kda.KDA_ERR_INVALID_ARG
    ref_o, ref_s = _oracle(w, np.zeros((2, 1, 32, 32), np.float32))
    assert nerr(pool.cpu().numpy()[1], ref_s[0]) <= TOL_F32   # sequence 0 ran into slot 1
    np.testing.assert_array_equal(pool.cpu().numpy()[0], pool0[0])


def test_multi_token_decode_batch():
    """A speculative-verification-sized step: 256 sequences x 32 heads x 8 new
    tokens each (d = 128, bf16), states from the decode workload's recipe."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(640, [8] * 256, H=32, d=128, dtype="bf16", init_std=0.02)
    t = _dev(w)
    pool = torch.from_numpy(w.initial_state.copy()).cuda()
    out = kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool, t["cu"],
                                out_f32=True)
    torch.cuda.synchronize()
    ref_o, ref_s = _oracle(w, w.initial_state)
    assert nerr(out.cpu().numpy(), ref_o) <= TOL_F32
    assert nerr(pool.cpu().numpy(), ref_s) <= TOL_F32


def test_agrees_with_repeated_decode_steps():
    """T tokens of one sequence through kda_recurrent_fwd equal T calls of
    kda_recurrent_step (same arithmetic per token)."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(650, [12], H=4, d=128, dtype="bf16", init_std=0.02)
    t = _dev(w)
    pool = torch.from_numpy(w.initial_state.copy()).cuda()
    out = kda.kda_recurrent_fwd(t["q"], t["k"], t["v"], t["g"], t["b"], w.scale, pool,
                                out_f32=True)
    st = torch.from_numpy(w.initial_state.copy()).cuda()
    steps = [kda.kda_recurrent_step(t["q"][i:i + 1], t["k"][i:i + 1], t["v"][i:i + 1],
                                    t["g"][i:i + 1], t["b"][i:i + 1], w.scale, st, out_f32=True)
             for i in range(w.T)]
    torch.cuda.synchronize()
    ref = torch.cat(steps).cpu().numpy()
    assert nerr(out.cpu().numpy(), ref) <= 1e-5
    assert nerr(pool.cpu().numpy(), st.cpu().numpy()) <= 1e-5
