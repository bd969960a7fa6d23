"""Seeded synthetic workloads for the KDA token mixer.

This module only draws random inputs.  It holds none of the mixer's
arithmetic, so the CUDA library's tests and the fp64 oracle can both be fed
from it without sharing any code with each other.

Every workload follows one recipe (the pages' workloads: head dim 128, long
contexts, packed variable-length prefill, batched decode):

* q, k, v ~ N(0, 1) drawn in float32; q and k are L2-normalised per
  (token, head) -- the library expects normalised q/k, as the K3 layer
  normalises them upstream of the mixer;
* beta = sigmoid(N(0, 1)) per (token, head);
* log_alpha = -softplus(N(mu, 1)) per (token, head, key channel) (mu = -3 for
  prefill and decode, -6 for the long-context run), or -Uniform(0.001, 0.5)
  for the tiny fp32 case;
* initial states ~ N(0, 0.02) in float32 where a workload has them;
* bf16 workloads round q, k, v to bfloat16 (round to nearest even) here, so
  the float32 arrays hold exactly the values the GPU sees and upcast exactly
  to float64 for the oracle.

Host draws use numpy's PCG64 (``numpy.random.default_rng(seed)``) in the order
lengths (packed runs only), q, k, v, beta logits, gate, initial state.  The
1M-token run is drawn on the device with a seeded torch generator instead
(host generation of 17 GB tensors would dominate the run).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np


@dataclass
class Workload:
    name: str
    q: np.ndarray                 # [T, H, d_k] float32 (bf16-exact when dtype == "bf16")
    k: np.ndarray                 # [T, H, d_k]
    v: np.ndarray                 # [T, H, d_v]
    log_alpha: np.ndarray         # [T, H, d_k] float32, <= 0
    beta: np.ndarray              # [T, H] float32
    cu_seqlens: np.ndarray        # [N + 1] int32
    scale: float
    dtype: str                    # "bf16" or "f32" (q/k/v/out)
    chunk_size: int
    initial_state: Optional[np.ndarray] = None   # [N, H, d_k, d_v] float32
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def d_k(self) -> int:
        return int(self.q.shape[2])

    @property
    def d_v(self) -> int:
        return int(self.v.shape[2])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)


@dataclass
class DecodeWorkload:
    name: str
    q: np.ndarray                 # [steps, N, H, d_k] float32 (bf16-exact)
    k: np.ndarray
    v: np.ndarray                 # [steps, N, H, d_v]
    log_alpha: np.ndarray         # [steps, N, H, d_k]
    beta: np.ndarray              # [steps, N, H]
    initial_state: np.ndarray     # [N, H, d_k, d_v] float32
    scale: float
    dtype: str = "bf16"


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    nan = np.isnan(x)
    out = rounded.astype(np.uint32).view(np.float32).copy()
    out[nan] = np.float32(np.nan)
    return out


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-12)).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _neg_softplus(x: np.ndarray) -> np.ndarray:
    return (-np.logaddexp(0.0, x.astype(np.float64))).astype(np.float32)


def prefill(seed: int, lengths: List[int], H: int, d: int, dtype: str = "bf16",
            gate: str = "softplus", gate_mu: float = -3.0,
            init_std: Optional[float] = None, chunk_size: int = 64,
            name: str = "prefill", rng: Optional[np.random.Generator] = None
            ) -> Workload:
    """Packed prefill workload: sequences of the given lengths, H heads, d = d_k = d_v."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    T = int(sum(lengths))
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    f32 = np.float32
    q = _l2_normalise(rng.standard_normal((T, H, d), dtype=f32))
    k = _l2_normalise(rng.standard_normal((T, H, d), dtype=f32))
    v = rng.standard_normal((T, H, d), dtype=f32)
    beta = _sigmoid(rng.standard_normal((T, H), dtype=f32))
    if gate == "softplus":
        log_alpha = _neg_softplus(rng.standard_normal((T, H, d), dtype=f32) + f32(gate_mu))
    elif gate == "uniform":
        log_alpha = (-rng.uniform(0.001, 0.5, size=(T, H, d))).astype(f32)
    else:
        raise ValueError(gate)
    s0 = None
    if init_std is not None:
        s0 = (rng.standard_normal((len(lengths), H, d, d), dtype=f32) * f32(init_std))
    if dtype == "bf16":
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    elif dtype != "f32":
        raise ValueError(dtype)
    return Workload(name=name, q=q, k=k, v=v, log_alpha=log_alpha, beta=beta,
                    cu_seqlens=cu, scale=float(d) ** -0.5, dtype=dtype,
                    chunk_size=chunk_size, initial_state=s0,
                    meta={"seed": seed, "lengths": lengths, "gate": gate,
                          "gate_mu": gate_mu, "init_std": init_std})


# --------------------------------------------------------------------------
# The five named workloads (seed = workload index - 1).
# --------------------------------------------------------------------------

def tiny_f32() -> Workload:
    """B=1, H=1, T=64, d=16, chunk 16, fp32, zero initial state, seed 0."""
    return prefill(0, [64], H=1, d=16, dtype="f32", gate="uniform",
                   chunk_size=16, name="tiny_f32_T64_H1_d16")


def head_group_prefill(T: int = 4096) -> Workload:
    """B=1, H=16, T=4096, d=128, chunk 64, bf16, zero initial state, seed 1."""
    return prefill(1, [T], H=16, d=128, dtype="bf16", gate_mu=-3.0,
                   name=f"prefill_T{T}_H16_d128")


def varlen_prefill(n_seqs: int = 32, H: int = 32) -> Workload:
    """32 packed sequences, lengths ~ U[512, 8192] (~140k tokens), H=32, d=128,
    bf16, initial states ~ N(0, 0.02), seed 2."""
    rng = np.random.default_rng(2)
    lengths = [int(x) for x in rng.integers(512, 8193, size=n_seqs)]
    return prefill(2, lengths, H=H, d=128, dtype="bf16", gate_mu=-3.0,
                   init_std=0.02, name=f"varlen_{n_seqs}seq_H{H}_d128", rng=rng)


def long_context_prefix(T: int = 8192) -> Workload:
    """The long-context recipe (log_alpha = -softplus(N(-6,1)), H=32, d=128,
    bf16, zero initial state, seed 3) at a host-sized length."""
    return prefill(3, [T], H=32, d=128, dtype="bf16", gate_mu=-6.0,
                   name=f"long_context_T{T}_H32_d128")


def long_context_device(T: int = 1 << 20, H: int = 32, d: int = 128,
                        seed: int = 3, device: str = "cuda"):
    """The 1,048,576-token single-sequence run, drawn on the device.

    Returns a dict of torch tensors: q, k, v (bf16, [T,H,d]), log_alpha
    (fp32 [T,H,d]), beta (fp32 [T,H]), cu_seqlens (int32 [2]).
    """
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normed():
        x = torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(torch.bfloat16)

    q = normed()
    k = normed()
    v = torch.randn((T, H, d), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((T, H), generator=gen, device=device))
    la = torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32)
    la = -torch.nn.functional.softplus(la - 6.0)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    return {"q": q, "k": k, "v": v, "log_alpha": la.contiguous(), "beta": beta,
            "cu_seqlens": cu, "scale": float(d) ** -0.5}


def varlen_device(n_seqs: int = 32, H: int = 32, d: int = 128, seed: int = 2,
                  device: str = "cuda"):
    """The packed 32-sequence workload's shapes and recipe, drawn on the device
    for timing runs: the same sequence lengths as ``varlen_prefill`` (numpy
    PCG64, seed 2), then q, k, v, beta, log_alpha and the initial states from
    a seeded torch generator.  Returns a dict like ``long_context_device``
    plus ``initial_state`` ([N, H, d, d] fp32, N(0, 0.02)) and ``lengths``."""
    import torch
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(512, 8193, size=n_seqs)]
    T = int(sum(lengths))
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normed():
        x = torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(torch.bfloat16)

    q = normed()
    k = normed()
    v = torch.randn((T, H, d), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((T, H), generator=gen, device=device))
    la = -torch.nn.functional.softplus(
        torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32) - 3.0)
    s0 = torch.randn((n_seqs, H, d, d), generator=gen, device=device) * 0.02
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32),
                      device=device)
    return {"q": q, "k": k, "v": v, "log_alpha": la.contiguous(), "beta": beta,
            "cu_seqlens": cu, "scale": float(d) ** -0.5, "initial_state": s0,
            "lengths": lengths}


def batched_decode(n_seqs: int = 256, H: int = 32, d: int = 128, steps: int = 64,
                   seed: int = 4) -> DecodeWorkload:
    """n_seqs independent sequences x H heads, one token per sequence per step,
    fp32 states ~ N(0, 0.02), bf16 q/k/v, seed 4."""
    rng = np.random.default_rng(seed)
    f32 = np.float32
    shp = (steps, n_seqs, H, d)
    q = bf16_round(_l2_normalise(rng.standard_normal(shp, dtype=f32)))
    k = bf16_round(_l2_normalise(rng.standard_normal(shp, dtype=f32)))
    v = bf16_round(rng.standard_normal(shp, dtype=f32))
    beta = _sigmoid(rng.standard_normal((steps, n_seqs, H), dtype=f32))
    log_alpha = _neg_softplus(rng.standard_normal(shp, dtype=f32) + f32(-3.0))
    s0 = rng.standard_normal((n_seqs, H, d, d), dtype=f32) * f32(0.02)
    return DecodeWorkload(name=f"decode_{n_seqs}x{H}_d{d}_{steps}steps", q=q, k=k,
                          v=v, log_alpha=log_alpha, beta=beta, initial_state=s0,
                          scale=float(d) ** -0.5)
