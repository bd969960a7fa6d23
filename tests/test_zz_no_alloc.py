"""kda_chunk_fwd_static: prefill that allocates no device memory.

Some callers cannot allocate device memory when they run prefill (a host
framework that owns every allocation, a latency-critical path, a service
with a fixed footprint).  kda_chunk_fwd_static serves them with scratch from
a fixed device array inside the library.  This file is collected last on
purpose, so a run that stops at the first failure has run every other test
first; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from kimi_delta_attention_chunkwise_gb300 import inputs
from kda_testutil import TOL_BF16, nerr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kimi_delta_attention_chunkwise_gb300 import binding, build
    build.build()
    lib = binding.load()
    vp = ctypes.c_void_p
    lib.kda_chunk_fwd_static.argtypes = [vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp,
                                         ctypes.POINTER(binding.kdaShape_t), vp]
    lib.kda_chunk_fwd_static.restype = ctypes.c_int
    return lib


def test_static_scratch_matches_allocating_entry(lib):
    """Two calls in a row through the C ABI equal kda_chunk_fwd's results."""
    import torch
    import kimi_delta_attention_chunkwise_gb300 as kda
    w = inputs.prefill(300, [700, 333, 64], H=4, d=128, dtype="bf16", init_std=0.02)
    dev = lambda x, dt=None: torch.from_numpy(x).to("cuda", dt)
    q, k, v = (dev(a, torch.bfloat16) for a in (w.q, w.k, w.v))
    la, b, cu, s0 = dev(w.log_alpha), dev(w.beta), dev(w.cu_seqlens), dev(w.initial_state)
    ref_out = torch.empty((w.T, w.H, 128), device="cuda")
    ref_fin = torch.empty((w.N, w.H, 128, 128), device="cuda")
    kda.kda_chunk_fwd(q, k, v, la, b, w.scale, s0, cu, ref_out, ref_fin,
                      use_library_scratch=True)
    torch.cuda.synchronize()
    shape = kda.make_shape(w.N, w.T, w.H, 128, 128, kda.KDA_DTYPE_BF16, 0,
                           kda.KDA_ENGINE_TENSOR, 1)
    stream = torch.cuda.current_stream().cuda_stream
    results = []
    for _ in range(2):
        out = torch.full((w.T, w.H, 128), float("nan"), device="cuda")
        fin = torch.full((w.N, w.H, 128, 128), float("nan"), device="cuda")
        rc = lib.kda_chunk_fwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), la.data_ptr(),
                                      b.data_ptr(), ctypes.c_float(w.scale), s0.data_ptr(),
                                      cu.data_ptr(), out.data_ptr(), fin.data_ptr(),
                                      ctypes.byref(shape), stream)
        assert rc == kda.KDA_SUCCESS, kda.kda_status_string(rc)
        torch.cuda.synchronize()
        results.append((out.cpu().numpy(), fin.cpu().numpy()))
    ro, rf = ref_out.cpu().numpy(), ref_fin.cpu().numpy()
    for o, f in results:
        assert nerr(o, ro) <= TOL_BF16
        assert nerr(f, rf) <= TOL_BF16
    np.testing.assert_array_equal(results[0][0], results[1][0])
    np.testing.assert_array_equal(results[0][1], results[1][1])


def test_static_scratch_rejects_oversize(lib):
    """A problem needing more scratch than the fixed array is refused before
    anything runs (fake 16-byte-aligned pointers are never touched)."""
    import kimi_delta_attention_chunkwise_gb300 as kda
    shape = kda.make_shape(1, 1 << 20, 32, 128, 128, kda.KDA_DTYPE_BF16)
    fake = 0x10000
    rc = lib.kda_chunk_fwd_static(fake, fake, fake, fake, fake, ctypes.c_float(1.0), None, None,
                                  fake, None, ctypes.byref(shape), None)
    assert rc == kda.KDA_ERR_UNSUPPORTED
