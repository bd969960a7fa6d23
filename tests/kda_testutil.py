"""Helpers shared by the GPU parity tests: move a seeded workload to the
device, run libkda through its binding, run the oracle on the same host
arrays, and measure the error the way the parity bar states it."""
import numpy as np

TOL_F32 = 1e-4    # max |gpu - oracle| / rms(oracle), fp32 inputs
TOL_BF16 = 2e-2   # same metric, bf16 inputs (fp32 state)


def nerr(x, ref) -> float:
    """max-abs error normalised by the RMS of the reference (whole tensor)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        return float(np.abs(x - ref).max()) if x.size else 0.0
    return float(np.abs(x - ref).max() / rms) if x.size else 0.0


def bf16_half_ulp(ref) -> np.ndarray:
    """Half a bfloat16 ulp at |ref| (the largest error of rounding ref to bf16)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    return np.exp2(e - 8)


def check_bf16_output(gpu, ref, tol=TOL_BF16):
    """A bf16 output carries its own final rounding (up to half an ulp per
    element, which alone can exceed tol * rms on heavy-tailed outputs), so each
    element must lie within tol * rms(ref) + half_ulp(ref) of the oracle."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(gpu - ref) - (tol * rms + bf16_half_ulp(ref))
    worst = float(excess.max()) if excess.size else -1.0
    assert worst <= 0.0, f"bf16 output exceeds tol*rms + half-ulp by {worst:g}"


def to_device(w, device="cuda"):
    import torch
    qdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = {
        "q": torch.from_numpy(w.q).to(device=device, dtype=qdt),
        "k": torch.from_numpy(w.k).to(device=device, dtype=qdt),
        "v": torch.from_numpy(w.v).to(device=device, dtype=qdt),
        "log_alpha": torch.from_numpy(w.log_alpha).to(device),
        "beta": torch.from_numpy(w.beta).to(device),
        "cu_seqlens": torch.from_numpy(w.cu_seqlens).to(device),
        "initial_state": (torch.from_numpy(w.initial_state).to(device)
                          if w.initial_state is not None else None),
    }
    return dev


def run_prefill(w, engine="auto", out_f32=False, chunk_size=None, dev=None,
                with_final=True, use_library_scratch=False):
    """libkda prefill on the workload; returns (out, final) as float64 numpy."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    d = dev if dev is not None else to_device(w)
    final = (torch.empty((w.N, w.H, w.d_k, w.d_v), dtype=torch.float32, device="cuda")
             if with_final else None)
    out, _ = kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], w.scale,
                               d["initial_state"], d["cu_seqlens"], None, final,
                               chunk_size=(w.chunk_size if chunk_size is None else chunk_size),
                               engine=engine, out_f32=out_f32,
                               use_library_scratch=use_library_scratch)
    check_device_status()
    o = out.float().cpu().numpy().astype(np.float64)
    f = final.cpu().numpy().astype(np.float64) if with_final else None
    return o, f


def check_device_status():
    """Synchronise and assert that no kernel's bounded wait gave up (the
    device status word; the host call returns before the kernels run)."""
    import kimi_delta_attention_chunkwise_gb300 as kda
    st = kda.kda_device_status()
    assert st == kda.KDA_SUCCESS, f"device status: {kda.kda_status_string(st)}"


def run_oracle(w):
    import oracle
    return oracle.recurrent(w.q, w.k, w.v, w.log_alpha, w.beta, w.scale,
                            w.initial_state, w.cu_seqlens)
