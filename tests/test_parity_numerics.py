"""Numerically hard inputs for the tensor-core prefill, against the fp64 oracle.

The tensor-core engine feeds the state S_c, beta V and the chunk's folded
factors to its MMAs as fp16 (11-bit significand, largest finite value 65504)
and the decayed products as tf32.  The recipe's keys (independent N(0, 1)
directions in d = 128, nearly orthogonal) keep the chunk's triangular system
I + R well conditioned and the state O(1).  These cases do not:

* keys drawn from a rank-4 subspace, with beta = 1: R's rows are strongly
  correlated, so the solve's inverse and the WY factors carry large
  cancelling terms;
* runs of one key repeated with beta = 1 (the DeltaNet overwrite, "Linear
  Attention, From Scratch to Kimi 3", sec. 4): each write replaces the last;
* initial states of magnitude 1e2, 1e3 and 1e4 (near fp16's range at the top);
* log alpha = 0 across whole chunks (no forgetting: the state only grows by
  the writes).
Each must stay within the bf16 parity bound of the oracle.
"""
import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, nerr, run_oracle, run_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import build
    build.build()


def _check(w):
    ref_o, ref_s = run_oracle(w)
    o, s = run_prefill(w, engine="tensor", out_f32=True)
    e_o, e_s = nerr(o, ref_o), nerr(s, ref_s)
    assert e_o <= TOL_BF16, f"out error {e_o:.3g}"
    assert e_s <= TOL_BF16, f"final_state error {e_s:.3g}"
    return e_o, e_s


def _unit_rows(x):
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def test_low_rank_keys_beta_one():
    """Keys (and queries) from a rank-4 subspace of each head, beta = 1."""
    rng = np.random.default_rng(130)
    w = inputs.prefill(130, [700, 190], H=2, d=128, dtype="bf16", init_std=0.02)
    T, H, d = w.q.shape
    for h in range(H):
        basis = rng.standard_normal((4, d))
        w.k[:, h] = _unit_rows(rng.standard_normal((T, 4)) @ basis)
        w.q[:, h] = _unit_rows(rng.standard_normal((T, 4)) @ basis)
    w.k, w.q = inputs.bf16_round(w.k), inputs.bf16_round(w.q)
    w.beta = np.ones_like(w.beta)
    _check(w)


def test_repeated_keys_overwrite():
    """Runs of 1 to 40 tokens sharing one key, beta = 1: every write in a run
    overwrites the value the key holds."""
    rng = np.random.default_rng(131)
    w = inputs.prefill(131, [600], H=2, d=128, dtype="bf16")
    k = w.k.copy()
    t = 0
    while t < w.T:
        run = int(rng.integers(1, 41))
        k[t:t + run] = k[t]
        t += run
    w.k = k
    w.beta = np.ones_like(w.beta)
    _check(w)


@pytest.mark.parametrize("magnitude", [1e2, 1e3, 1e4])
def test_large_initial_states(magnitude):
    """Initial states with entries of the given magnitude (N(0, 1) scaled)."""
    w = inputs.prefill(132, [300, 77], H=2, d=128, dtype="bf16", init_std=1.0)
    w.initial_state = (w.initial_state * np.float32(magnitude)).astype(np.float32)
    _check(w)


def test_no_decay_whole_chunks():
    """log alpha = 0 for every token of the first 192 (three whole chunks),
    then the recipe's gates."""
    w = inputs.prefill(133, [400, 130], H=2, d=128, dtype="bf16", init_std=0.02)
    la = w.log_alpha.copy()
    la[:192] = 0.0
    w.log_alpha = la
    _check(w)
