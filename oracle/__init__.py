"""fp64 CPU oracle for the Kimi Delta Attention token mixer.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker that the
CUDA library is compared against.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import it; the library never does, and
this package imports nothing from the library.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, libm ``exp``), built
with gcc into ``oracle/_build/libkda_oracle.so``.  This module only marshals
numpy arrays to it:

* :func:`recurrent` -- the defining token-by-token recurrence
  ("Kimi Unveils Delta Attention and K3 Architecture Updates", sec. 4 and the
  d_k x d_v five-line form at the end of sec. 4.1; "Kimi Delta Attention:
  Channel-Wise Memory Control", "Change one piece of Gated DeltaNet").
* :func:`chunkwise` -- the chunkwise schedule of the same recurrence written
  as the derivation gives it (same page, sec. 6.1-6.5).

Every input is upcast to float64 exactly (bf16 and fp32 values are exactly
representable in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: no -march, no intrinsics)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """ctypes binding of one compiled copy of ``kda_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i32 = ctypes.c_int32
        common = [i32, i32, i32, i32, i32, dp, dp, dp, dp, dp, ctypes.c_double,
                  dp, ip, dp, dp]
        lib.kda_oracle_recurrent.argtypes = common + [i32]
        lib.kda_oracle_recurrent.restype = ctypes.c_int
        lib.kda_oracle_chunkwise.argtypes = common + [i32, i32]
        lib.kda_oracle_chunkwise.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def recurrent(self, q, k, v, log_alpha, beta, scale, initial_state=None,
                  cu_seqlens=None, threads=None):
        return _call(self.lib, False, q, k, v, log_alpha, beta, scale, 0,
                     initial_state, cu_seqlens, threads)

    def chunkwise(self, q, k, v, log_alpha, beta, scale, chunk_size,
                  initial_state=None, cu_seqlens=None, threads=None):
        return _call(self.lib, True, q, k, v, log_alpha, beta, scale, chunk_size,
                     initial_state, cu_seqlens, threads)


def build_variant(source_text: str, tag: str) -> OracleLib:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    src = os.path.join(_OUT_DIR, f"variant_{tag}.c")
    lib = os.path.join(_OUT_DIR, f"libvariant_{tag}_{os.getpid()}.so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-ffp-contract=off", src, "-o", lib, "-lm"], check=True)
    return OracleLib(lib)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _load() -> OracleLib:
    global _lib
    if _lib is None:
        _lib = OracleLib(build())
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _prepare(q, k, v, log_alpha, beta, initial_state, cu_seqlens):
    q, k, v, g, b = (_f64(a) for a in (q, k, v, log_alpha, beta))
    if q.ndim != 3:
        raise ValueError("q must be [T, H, d_k]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != (T, H, dk) or g.shape != (T, H, dk) or v.shape != (T, H, dv):
        raise ValueError("k/log_alpha must be [T,H,d_k] and v [T,H,d_v]")
    if b.shape != (T, H):
        raise ValueError("beta must be [T, H]")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int32)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None
    if initial_state is not None:
        s0 = _f64(initial_state)
        if s0.shape != (N, H, dk, dv):
            raise ValueError("initial_state must be [N, H, d_k, d_v]")
    return q, k, v, g, b, s0, cu, (N, T, H, dk, dv)


def _call(lib, chunked, q, k, v, log_alpha, beta, scale, chunk_size,
          initial_state, cu_seqlens, threads):
    q, k, v, g, b, s0, cu, (N, T, H, dk, dv) = _prepare(
        q, k, v, log_alpha, beta, initial_state, cu_seqlens)
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    dp = ctypes.c_double
    args = [N, T, H, dk, dv, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(g, dp),
            _ptr(b, dp), float(scale), _ptr(s0, dp), _ptr(cu, ctypes.c_int32),
            _ptr(out, dp), _ptr(fin, dp)]
    nthr = int(threads or default_threads())
    if chunked:
        rc = lib.kda_oracle_chunkwise(*args, int(chunk_size), nthr)
    else:
        rc = lib.kda_oracle_recurrent(*args, nthr)
    if rc != 0:
        raise ValueError(f"oracle call failed with code {rc}")
    return out, fin


def recurrent(q, k, v, log_alpha, beta, scale: float, initial_state=None,
              cu_seqlens=None, threads: Optional[int] = None
              ) -> Tuple[np.ndarray, np.ndarray]:
    """Token-by-token KDA in fp64.  Returns ``(out [T,H,d_v], final [N,H,d_k,d_v])``."""
    return _load().recurrent(q, k, v, log_alpha, beta, scale, initial_state,
                             cu_seqlens, threads)


def chunkwise(q, k, v, log_alpha, beta, scale: float, chunk_size: int,
              initial_state=None, cu_seqlens=None, threads: Optional[int] = None
              ) -> Tuple[np.ndarray, np.ndarray]:
    """Chunkwise KDA in fp64 (direct decay exponents, forward substitution)."""
    return _load().chunkwise(q, k, v, log_alpha, beta, scale, chunk_size,
                             initial_state, cu_seqlens, threads)
