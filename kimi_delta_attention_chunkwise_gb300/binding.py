"""Thin Python binding of libkda's C ABI (include/kda.h).

Argument marshalling only: every step of the computation runs in libkda's
CUDA kernels.  Torch supplies device memory and streams.  The shared library
is built in-tree (``build.build()``); if it is missing this module raises --
there is no CPU or PyTorch fallback.

The functions carry the C names:

* ``kda_chunk_fwd``      -- chunkwise prefill over packed sequences;
* ``kda_recurrent_step`` -- one decode token per sequence, state in place;
* ``kda_recurrent_fwd``  -- token-by-token over packed sequences, slot-indexed state pool;
* ``kda_short_conv_fwd`` / ``kda_short_conv_step`` -- the layer's short causal convolution;
* ``kda_chunk_fwd_workspace_size`` / ``kda_chunk_fwd_ws`` -- caller-owned scratch;
* ``kda_chunk_fwd_host`` / ``kda_chunk_fwd_host_scratch_size`` -- prefill on host buffers
  (copies in, prefill, copies out, all on one stream);
* ``kda_recurrent_bwd`` -- gradients of the recurrence;
* ``kda_chunk_fwd_ws_diag`` -- the prefill with a chosen wait limit, optionally
  without its chunk-parallel stage (tests of the timeout path);
* ``kda_chunk_path_counts`` -- how the decayed products were evaluated;
* ``kda_status_string``, ``kda_device_status``.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

from . import build as _build

KDA_SUCCESS = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4

KDA_DTYPE_BF16 = 0
KDA_DTYPE_F32 = 1

KDA_PROLOGUE_L2NORM_QK = 1
KDA_PROLOGUE_BETA_LOGITS = 2
KDA_PROLOGUE_GATE = 4

KDA_ENGINE_AUTO = 0
KDA_ENGINE_TENSOR = 1
KDA_ENGINE_SIMT = 2
_ENGINES = {"auto": KDA_ENGINE_AUTO, "tensor": KDA_ENGINE_TENSOR, "simt": KDA_ENGINE_SIMT}


class kdaShape_t(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("engine", ctypes.c_int32),
                ("out_f32", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("prologue", ctypes.c_int32), ("gate_bias", ctypes.c_void_p),
                ("gate_A_log", ctypes.c_void_p)]


class kdaConvShape_t(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("channels", ctypes.c_int32), ("width", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("activation", ctypes.c_int32)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {kda_status_string(status)}")


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libkda.so not found at {p}; build it with "
            "kimi_delta_attention_chunkwise_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    shp = ctypes.POINTER(kdaShape_t)
    lib.kda_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp, shp, vp]
    lib.kda_chunk_fwd.restype = ctypes.c_int
    lib.kda_chunk_fwd_ws.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp, shp,
                                     vp, ctypes.c_size_t, vp]
    lib.kda_chunk_fwd_ws.restype = ctypes.c_int
    lib.kda_chunk_fwd_ws_timed.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp,
                                           shp, vp, ctypes.c_size_t, vp,
                                           ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_int32)]
    lib.kda_chunk_fwd_ws_timed.restype = ctypes.c_int
    lib.kda_chunk_fwd_ws_diag.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp,
                                          shp, vp, ctypes.c_size_t, ctypes.c_int32,
                                          ctypes.c_int64, vp]
    lib.kda_chunk_fwd_ws_diag.restype = ctypes.c_int
    lib.kda_chunk_path_counts.argtypes = [ctypes.POINTER(ctypes.c_uint64), vp]
    lib.kda_chunk_path_counts.restype = ctypes.c_int
    lib.kda_chunk_fwd_static.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp,
                                         shp, vp]
    lib.kda_chunk_fwd_static.restype = ctypes.c_int
    lib.kda_chunk_fwd_host_scratch_size.argtypes = [shp, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_chunk_fwd_host_scratch_size.restype = ctypes.c_int
    lib.kda_chunk_fwd_host.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp, shp,
                                       vp, ctypes.c_size_t, vp]
    lib.kda_chunk_fwd_host.restype = ctypes.c_int
    lib.kda_chunk_fwd_workspace_size.argtypes = [shp, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_int
    lib.kda_recurrent_step.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, shp, vp]
    lib.kda_recurrent_step.restype = ctypes.c_int
    lib.kda_recurrent_fwd.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, ip, fp, ip,
                                      ctypes.c_int32, vp, shp, vp]
    lib.kda_recurrent_fwd.restype = ctypes.c_int
    cshp = ctypes.POINTER(kdaConvShape_t)
    lib.kda_short_conv_fwd.argtypes = [vp, fp, fp, ip, vp, vp, vp, cshp, vp]
    lib.kda_short_conv_fwd.restype = ctypes.c_int
    lib.kda_short_conv_step.argtypes = [vp, fp, fp, vp, vp, cshp, vp]
    lib.kda_short_conv_step.restype = ctypes.c_int
    lib.kda_recurrent_bwd.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, ip, vp, fp,
                                      fp, fp, fp, fp, fp, fp, shp, vp]
    lib.kda_recurrent_bwd.restype = ctypes.c_int
    lib.kda_chunk_bwd.argtypes = list(lib.kda_recurrent_bwd.argtypes)
    lib.kda_chunk_bwd.restype = ctypes.c_int
    lib.kda_chunk_bwd_ws.argtypes = (list(lib.kda_recurrent_bwd.argtypes[:-1]) +
                                     [vp, ctypes.c_size_t, vp])
    lib.kda_chunk_bwd_ws.restype = ctypes.c_int
    lib.kda_chunk_bwd_workspace_size.argtypes = [shp, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_device_status.argtypes = [vp]
    lib.kda_device_status.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def header_functions() -> list:
    """Names of every function include/kda.h declares."""
    hdr = os.path.join(_build.INCLUDE, "kda.h")
    with open(hdr) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != KDA_SUCCESS:
        raise KdaError(status, where)


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _require(t, name, dtype=None, shape=None, on_host=False):
    torch = _torch()
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if on_host and t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not on_host and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def make_shape(N, T, H, dk, dv, dtype_code, chunk_size=0, engine=KDA_ENGINE_AUTO,
               out_f32=0, num_v_heads=0, prologue=0, gate_bias=None,
               gate_A_log=None) -> kdaShape_t:
    """H: q/k heads; num_v_heads: value heads (0 = H), a multiple of H;
    prologue: KDA_PROLOGUE_* bits; gate_bias / gate_A_log: device addresses."""
    return kdaShape_t(int(N), int(T), int(H), int(dk), int(dv), int(dtype_code),
                      int(chunk_size), int(engine), int(out_f32), int(num_v_heads),
                      int(prologue), gate_bias, gate_A_log)


def _prologue(l2norm_qk, beta_logits, gate, HV, dk, on_host=False):
    """(bits, bias pointer, A_log pointer) of the in-kernel input prologue;
    gate = (bias [HV, d_k] fp32, A_log [HV] fp32) tensors on the device (on
    the host for kda_chunk_fwd_host)."""
    torch = _torch()
    bits = (KDA_PROLOGUE_L2NORM_QK if l2norm_qk else 0) | (
        KDA_PROLOGUE_BETA_LOGITS if beta_logits else 0)
    if gate is None:
        return bits, None, None
    bias, a_log = gate
    _require(bias, "gate bias", torch.float32, (HV, dk), on_host)
    _require(a_log, "gate A_log", torch.float32, (HV,), on_host)
    return bits | KDA_PROLOGUE_GATE, bias.data_ptr(), a_log.data_ptr()


def _value_heads(q, v):
    """Value heads from the tensors: v carries HV heads, q carries H (HV % H == 0)."""
    H, HV = q.shape[-2], v.shape[-2]
    if HV % H:
        raise ValueError(f"v has {HV} heads, not a multiple of q's {H}")
    return HV, (0 if HV == H else HV)


def _out_dtype(q, out, out_f32):
    torch = _torch()
    if out is not None:
        return out.dtype
    return torch.float32 if out_f32 else q.dtype


_ws_cache = {}


def kda_chunk_fwd_workspace_size(shape: kdaShape_t) -> int:
    n = ctypes.c_size_t(0)
    _check(load().kda_chunk_fwd_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "kda_chunk_fwd_workspace_size")
    return int(n.value)


def _workspace(nbytes: int, device, stream=None):
    """A cached scratch buffer of at least nbytes (+256 for alignment), one per
    (device, stream): calls on one stream run in order, so they may share it."""
    torch = _torch()
    if nbytes == 0:
        return None
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           _stream_handle(stream))
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state,
                  chunk_size, engine, out_f32=False, prologue=None, on_host=False):
    torch = _torch()
    _req = lambda t, name, dtype=None, shape=None: _require(t, name, dtype, shape, on_host)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d_k]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    if v.dim() != 3:
        raise ValueError("v must be [T, HV, d_v]")
    HV, nvh = _value_heads(q, v)
    _req(k, "k", q.dtype, (T, H, dk))
    _req(v, "v", q.dtype, (T, HV, dv))
    _req(log_alpha, "log_alpha", torch.float32, (T, HV, dk))
    _req(beta, "beta", torch.float32, (T, HV))
    if cu_seqlens is not None:
        _req(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = 1
    _req(initial_state, "initial_state", torch.float32, (N, HV, dk, dv))
    odt = _out_dtype(q, out, out_f32)
    if odt not in (q.dtype, torch.float32):
        raise TypeError("out must have the dtype of q, or float32")
    if out is None:
        out = torch.empty((T, HV, dv), dtype=odt, device=q.device)
        if on_host:
            out = out.pin_memory()
    _req(out, "out", odt, (T, HV, dv))
    _req(final_state, "final_state", torch.float32, (N, HV, dk, dv))
    eng = _ENGINES[engine] if isinstance(engine, str) else int(engine)
    bits, gb, ga = _prologue(*(prologue or (False, False, None)), HV, dk, on_host)
    shape = make_shape(N, T, H, dk, dv, _dtype_code(q), chunk_size, eng,
                       int(odt == torch.float32 and q.dtype != torch.float32), nvh, bits, gb, ga)
    return shape, out


def kda_chunk_fwd(q, k, v, log_alpha, beta, scale: float, initial_state=None,
                  cu_seqlens=None, out=None, final_state=None, *, chunk_size: int = 0,
                  engine="auto", stream=None, use_library_scratch: bool = False,
                  out_f32: bool = False, l2norm_qk: bool = False, beta_logits: bool = False,
                  gate=None) -> Tuple[object, object]:
    """Chunkwise KDA prefill (C: kda_chunk_fwd).  Returns ``(out, final_state)``.

    q, k: [T, H, d_k] bf16/fp32; v: [T, H, d_v]; log_alpha: [T, H, d_k] fp32;
    beta: [T, H] fp32; initial_state / final_state: [N, H, d_k, d_v] fp32;
    cu_seqlens: int32 [N + 1] on the device.  ``final_state`` may be the same
    tensor as ``initial_state``.  Scratch comes from torch (kda_chunk_fwd_ws)
    unless ``use_library_scratch`` asks libkda to take it with cudaMallocAsync.
    ``out_f32`` (or a float32 ``out``) returns fp32 results for bf16 inputs.
    Prologue (applied in-kernel as the inputs load; kdaPrologue_t):
    ``l2norm_qk`` L2-normalises q and k per head, ``beta_logits`` takes beta as
    logits (sigmoid), ``gate = (bias [HV, d_k], A_log [HV])`` takes log_alpha
    as the K3 gate projection.
    """
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, engine, out_f32,
                               (l2norm_qk, beta_logits, gate))
    lib = load()
    s = _stream_handle(stream)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
            _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
            ctypes.byref(shape))
    if use_library_scratch:
        _check(lib.kda_chunk_fwd(*args, s), "kda_chunk_fwd")
    else:
        nbytes = kda_chunk_fwd_workspace_size(shape)
        ws = _workspace(nbytes, q.device, stream)
        wp = None
        if ws is not None:
            wp = (ws.data_ptr() + 255) // 256 * 256
        _check(lib.kda_chunk_fwd_ws(*args, wp, nbytes, s), "kda_chunk_fwd_ws")
    return out, final_state


def kda_chunk_fwd_static(q, k, v, log_alpha, beta, scale: float, initial_state=None,
                         cu_seqlens=None, out=None, final_state=None, *, chunk_size: int = 0,
                         engine="auto", stream=None, out_f32: bool = False,
                         l2norm_qk: bool = False, beta_logits: bool = False,
                         gate=None) -> Tuple[object, object]:
    """kda_chunk_fwd with the library's fixed scratch array (C:
    kda_chunk_fwd_static): allocates no device memory; problems larger than
    the array are refused (KDA_ERR_UNSUPPORTED).  Arguments as kda_chunk_fwd."""
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, engine, out_f32,
                               (l2norm_qk, beta_logits, gate))
    _check(load().kda_chunk_fwd_static(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        ctypes.byref(shape), _stream_handle(stream)), "kda_chunk_fwd_static")
    return out, final_state


def kda_chunk_fwd_ws_timed(q, k, v, log_alpha, beta, scale: float, initial_state, cu_seqlens,
                           out, final_state, events, *, chunk_size: int = 0, engine="auto",
                           stream=None, out_f32: bool = False, l2norm_qk: bool = False,
                           beta_logits: bool = False, gate=None):
    """kda_chunk_fwd with library-owned stage events: ``events`` is a list of
    already-recorded ``torch.cuda.Event(enable_timing=True)``; libkda records
    events[0] before its first kernel and events[i] after kernel i on the
    launch stream.  Returns ``(out, final_state, n_recorded)``."""
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, engine, out_f32,
                               (l2norm_qk, beta_logits, gate))
    nbytes = kda_chunk_fwd_workspace_size(shape)
    ws = _workspace(nbytes, q.device, stream)
    wp = None if ws is None else (ws.data_ptr() + 255) // 256 * 256
    handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    n = ctypes.c_int32(0)
    _check(load().kda_chunk_fwd_ws_timed(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        ctypes.byref(shape), wp, nbytes, _stream_handle(stream), handles, len(events),
        ctypes.byref(n)), "kda_chunk_fwd_ws_timed")
    return out, final_state, int(n.value)


def kda_chunk_fwd_ws_diag(q, k, v, log_alpha, beta, scale: float, initial_state, cu_seqlens,
                          out, final_state, *, withhold_prep: bool, wait_cycles: int = 0,
                          chunk_size: int = 0, stream=None, out_f32: bool = False):
    """The tensor-core prefill in its overlapped order with every bounded
    device wait limited to ``wait_cycles`` SM clocks (C: kda_chunk_fwd_ws_diag);
    ``withhold_prep`` launches no chunk-parallel stage, so the scan's waits run
    out and the device status word reports KDA_ERR_TIMEOUT.  Returns
    ``(out, final_state)``."""
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, KDA_ENGINE_TENSOR, out_f32)
    nbytes = kda_chunk_fwd_workspace_size(shape)
    ws = _workspace(nbytes, q.device, stream)
    wp = None if ws is None else (ws.data_ptr() + 255) // 256 * 256
    _check(load().kda_chunk_fwd_ws_diag(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        ctypes.byref(shape), wp, nbytes, int(bool(withhold_prep)), int(wait_cycles),
        _stream_handle(stream)), "kda_chunk_fwd_ws_diag")
    return out, final_state


def kda_chunk_path_counts(stream=None):
    """(mid, half, direct): (chunk, head) items per evaluation path of the
    decayed products since the last read on this device (C:
    kda_chunk_path_counts; synchronises the stream, reads and clears)."""
    c = (ctypes.c_uint64 * 3)()
    _check(load().kda_chunk_path_counts(c, _stream_handle(stream)), "kda_chunk_path_counts")
    return tuple(int(x) for x in c)


def kda_chunk_fwd_host_scratch_size(shape: kdaShape_t) -> int:
    n = ctypes.c_size_t(0)
    _check(load().kda_chunk_fwd_host_scratch_size(ctypes.byref(shape), ctypes.byref(n)),
           "kda_chunk_fwd_host_scratch_size")
    return int(n.value)


def kda_chunk_fwd_host(q, k, v, log_alpha, beta, scale: float, initial_state=None,
                       cu_seqlens=None, out=None, final_state=None, *, scratch=None,
                       chunk_size: int = 0, engine="auto", stream=None, out_f32: bool = False,
                       l2norm_qk: bool = False, beta_logits: bool = False, gate=None):
    """kda_chunk_fwd on host tensors (C: kda_chunk_fwd_host): every tensor is a
    CPU tensor (page-locked for asynchronous copies), laid out as for
    kda_chunk_fwd; ``gate`` tensors too.  The call enqueues the copies in,
    the prefill and the copies out on ``stream`` and returns
    ``(out, final_state)``, valid once that stream is synchronised.
    ``scratch``: a uint8 CUDA tensor of at least
    kda_chunk_fwd_host_scratch_size() bytes (plus 256 for alignment), owned
    by the call until its work is done; one per stream for overlapping calls.
    Without it, a cached buffer per (device, stream) serves."""
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, engine, out_f32,
                               (l2norm_qk, beta_logits, gate), on_host=True)
    torch = _torch()
    nbytes = kda_chunk_fwd_host_scratch_size(shape)
    if scratch is None:
        scratch = _workspace(nbytes, torch.device("cuda", torch.cuda.current_device()), stream)
    if not scratch.is_cuda or scratch.numel() * scratch.element_size() < nbytes + 255:
        raise ValueError(f"scratch must be a CUDA buffer of at least {nbytes + 256} bytes")
    sp = (scratch.data_ptr() + 255) // 256 * 256
    _check(load().kda_chunk_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        ctypes.byref(shape), sp, nbytes, _stream_handle(stream)), "kda_chunk_fwd_host")
    return out, final_state


def kda_chunk_fwd_ws(q, k, v, log_alpha, beta, scale: float, initial_state, cu_seqlens,
                     out, final_state, workspace, *, chunk_size: int = 0, engine="auto",
                     stream=None):
    """kda_chunk_fwd with an explicit workspace tensor (uint8, >= the size query)."""
    shape, out = _prefill_args(q, k, v, log_alpha, beta, initial_state, cu_seqlens, out,
                               final_state, chunk_size, engine)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().kda_chunk_fwd_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        ctypes.byref(shape), _ptr(workspace), nbytes, _stream_handle(stream)),
        "kda_chunk_fwd_ws")
    return out, final_state


def kda_recurrent_step(q, k, v, log_alpha, beta, scale: float, state, out=None, *,
                       stream=None, out_f32: bool = False, l2norm_qk: bool = False,
                       beta_logits: bool = False, gate=None):
    """One KDA decode step (C: kda_recurrent_step).  ``state`` is updated in place.

    q, k: [N, H, d_k] bf16/fp32; v: [N, H, d_v]; log_alpha: [N, H, d_k] fp32;
    beta: [N, H] fp32; state: [N, H, d_k, d_v] fp32.  Returns ``out`` [N, H, d_v].
    """
    torch = _torch()
    _require(q, "q")
    if q.dim() != 3:
        raise ValueError("q must be [N, H, d_k]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    if v.dim() != 3:
        raise ValueError("v must be [N, HV, d_v]")
    HV, nvh = _value_heads(q, v)
    _require(k, "k", q.dtype, (N, H, dk))
    _require(v, "v", q.dtype, (N, HV, dv))
    _require(log_alpha, "log_alpha", torch.float32, (N, HV, dk))
    _require(beta, "beta", torch.float32, (N, HV))
    _require(state, "state", torch.float32, (N, HV, dk, dv))
    odt = _out_dtype(q, out, out_f32)
    if odt not in (q.dtype, torch.float32):
        raise TypeError("out must have the dtype of q, or float32")
    if out is None:
        out = torch.empty((N, HV, dv), dtype=odt, device=q.device)
    _require(out, "out", odt, (N, HV, dv))
    bits, gb, ga = _prologue(l2norm_qk, beta_logits, gate, HV, dk)
    shape = make_shape(N, N, H, dk, dv, _dtype_code(q),
                       out_f32=int(odt == torch.float32 and q.dtype != torch.float32),
                       num_v_heads=nvh, prologue=bits, gate_bias=gb, gate_A_log=ga)
    _check(load().kda_recurrent_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale), _ptr(state),
        _ptr(out), ctypes.byref(shape), _stream_handle(stream)), "kda_recurrent_step")
    return out


def kda_recurrent_fwd(q, k, v, log_alpha, beta, scale: float, state_pool, cu_seqlens=None,
                      state_indices=None, out=None, *, stream=None, out_f32: bool = False,
                      l2norm_qk: bool = False, beta_logits: bool = False, gate=None):
    """Token-by-token recurrence over packed sequences against a slot-indexed
    state pool (C: kda_recurrent_fwd).  ``state_pool`` is updated in place.

    q, k: [T, H, d_k] bf16/fp32; v: [T, H, d_v]; log_alpha: [T, H, d_k] fp32;
    beta: [T, H] fp32; state_pool: [S, H, d_k, d_v] fp32; cu_seqlens: int32
    [N + 1] on the device (None: one sequence); state_indices: int32 [N] on the
    device (None: sequence s uses slot s; negative: skip the sequence).
    Returns ``out`` [T, H, d_v].
    """
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d_k]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    if v.dim() != 3:
        raise ValueError("v must be [T, HV, d_v]")
    HV, nvh = _value_heads(q, v)
    _require(k, "k", q.dtype, (T, H, dk))
    _require(v, "v", q.dtype, (T, HV, dv))
    _require(log_alpha, "log_alpha", torch.float32, (T, HV, dk))
    _require(beta, "beta", torch.float32, (T, HV))
    if cu_seqlens is not None:
        _require(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = 1
    _require(state_pool, "state_pool", torch.float32)
    if state_pool is None or state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, dk, dv):
        raise ValueError("state_pool must be [S, HV, d_k, d_v]")
    if state_indices is not None:
        _require(state_indices, "state_indices", torch.int32, (N,))
    odt = _out_dtype(q, out, out_f32)
    if odt not in (q.dtype, torch.float32):
        raise TypeError("out must have the dtype of q, or float32")
    if out is None:
        out = torch.empty((T, HV, dv), dtype=odt, device=q.device)
    _require(out, "out", odt, (T, HV, dv))
    bits, gb, ga = _prologue(l2norm_qk, beta_logits, gate, HV, dk)
    shape = make_shape(N, T, H, dk, dv, _dtype_code(q),
                       out_f32=int(odt == torch.float32 and q.dtype != torch.float32),
                       num_v_heads=nvh, prologue=bits, gate_bias=gb, gate_A_log=ga)
    _check(load().kda_recurrent_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale), _ptr(cu_seqlens),
        _ptr(state_pool), _ptr(state_indices), int(state_pool.shape[0]), _ptr(out),
        ctypes.byref(shape), _stream_handle(stream)), "kda_recurrent_fwd")
    return out


def kda_short_conv_fwd(x, weight, bias=None, cu_seqlens=None, cache_in=None, cache_out=None,
                       y=None, *, silu: bool = False, stream=None):
    """Short causal convolution over packed sequences (C: kda_short_conv_fwd).

    x: [T, C] bf16/fp32; weight: [C, W] fp32; bias: [C] fp32 or None;
    cu_seqlens: int32 [N + 1] on the device (None: one sequence); cache_in /
    cache_out: [N, C, W] of x's dtype or None (cache_out may be cache_in).
    Returns ``y`` [T, C].
    """
    torch = _torch()
    _require(x, "x")
    if x.dim() != 2:
        raise ValueError("x must be [T, C]")
    T, C = x.shape
    _require(weight, "weight", torch.float32)
    if weight is None or weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("weight must be [C, W]")
    W = weight.shape[1]
    _require(bias, "bias", torch.float32, (C,))
    if cu_seqlens is not None:
        _require(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = 1
    _require(cache_in, "cache_in", x.dtype, (N, C, W))
    _require(cache_out, "cache_out", x.dtype, (N, C, W))
    if y is None:
        y = torch.empty_like(x)
    _require(y, "y", x.dtype, (T, C))
    shape = kdaConvShape_t(N, T, C, W, _dtype_code(x), int(bool(silu)))
    _check(load().kda_short_conv_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(cu_seqlens),
                                     _ptr(cache_in), _ptr(cache_out), _ptr(y),
                                     ctypes.byref(shape), _stream_handle(stream)),
           "kda_short_conv_fwd")
    return y


def kda_short_conv_step(x, weight, cache, bias=None, y=None, *, silu: bool = False,
                        stream=None):
    """One decode token per sequence (C: kda_short_conv_step): x [N, C];
    cache [N, C, W] updated in place.  Returns ``y`` [N, C]."""
    torch = _torch()
    _require(x, "x")
    if x.dim() != 2:
        raise ValueError("x must be [N, C]")
    N, C = x.shape
    _require(weight, "weight", torch.float32)
    if weight is None or weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("weight must be [C, W]")
    W = weight.shape[1]
    _require(bias, "bias", torch.float32, (C,))
    _require(cache, "cache", x.dtype, (N, C, W))
    if y is None:
        y = torch.empty_like(x)
    _require(y, "y", x.dtype, (N, C))
    shape = kdaConvShape_t(N, N, C, W, _dtype_code(x), int(bool(silu)))
    _check(load().kda_short_conv_step(_ptr(x), _ptr(weight), _ptr(bias), _ptr(cache), _ptr(y),
                                      ctypes.byref(shape), _stream_handle(stream)),
           "kda_short_conv_step")
    return y


def kda_recurrent_bwd(q, k, v, log_alpha, beta, scale: float, initial_state=None,
                      cu_seqlens=None, d_out=None, d_final_state=None, *, stream=None,
                      want_initial: bool = True):
    """Gradients of the recurrence (C: kda_recurrent_bwd).  Returns ``(dq, dk,
    dv, dlog_alpha, dbeta, d_initial_state)``, float32 (d_initial_state None
    unless ``want_initial``)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d_k]")
    T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    _require(k, "k", q.dtype, (T, H, dk_))
    _require(v, "v", q.dtype, (T, H, dv_))
    _require(log_alpha, "log_alpha", torch.float32, (T, H, dk_))
    _require(beta, "beta", torch.float32, (T, H))
    if cu_seqlens is not None:
        _require(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = 1
    _require(initial_state, "initial_state", torch.float32, (N, H, dk_, dv_))
    _require(d_out, "d_out", q.dtype, (T, H, dv_))
    _require(d_final_state, "d_final_state", torch.float32, (N, H, dk_, dv_))
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dlog = (torch.empty((T, H, dk_), **f32) for _ in range(3))
    dv = torch.empty((T, H, dv_), **f32)
    db = torch.empty((T, H), **f32)
    dS0 = torch.empty((N, H, dk_, dv_), **f32) if want_initial else None
    shape = make_shape(N, T, H, dk_, dv_, _dtype_code(q))
    _check(load().kda_recurrent_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(dlog), _ptr(db), _ptr(dS0), ctypes.byref(shape),
        _stream_handle(stream)), "kda_recurrent_bwd")
    return dq, dk, dv, dlog, db, dS0


def kda_chunk_bwd(q, k, v, log_alpha, beta, scale: float, initial_state=None,
                  cu_seqlens=None, d_out=None, d_final_state=None, *, stream=None,
                  want_initial: bool = True):
    """The same gradients through the chunkwise form (C: kda_chunk_bwd; bf16,
    d = 128).  Returns ``(dq, dk, dv, dlog_alpha, dbeta, d_initial_state)``,
    float32 (d_initial_state None unless ``want_initial``)."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d_k]")
    T, H, dk_ = q.shape
    dv_ = v.shape[-1]
    _require(k, "k", q.dtype, (T, H, dk_))
    _require(v, "v", q.dtype, (T, H, dv_))
    _require(log_alpha, "log_alpha", torch.float32, (T, H, dk_))
    _require(beta, "beta", torch.float32, (T, H))
    if cu_seqlens is not None:
        _require(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    else:
        N = 1
    _require(initial_state, "initial_state", torch.float32, (N, H, dk_, dv_))
    _require(d_out, "d_out", q.dtype, (T, H, dv_))
    _require(d_final_state, "d_final_state", torch.float32, (N, H, dk_, dv_))
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dlog = (torch.empty((T, H, dk_), **f32) for _ in range(3))
    dv = torch.empty((T, H, dv_), **f32)
    db = torch.empty((T, H), **f32)
    dS0 = torch.empty((N, H, dk_, dv_), **f32) if want_initial else None
    shape = make_shape(N, T, H, dk_, dv_, _dtype_code(q))
    # scratch from the binding's per-device cache (no allocation per call)
    n = ctypes.c_size_t(0)
    _check(load().kda_chunk_bwd_workspace_size(ctypes.byref(shape), ctypes.byref(n)),
           "kda_chunk_bwd_workspace_size")
    ws = _workspace(int(n.value), q.device, stream)
    wp = None if ws is None else (ws.data_ptr() + 255) // 256 * 256
    _check(load().kda_chunk_bwd_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq),
        _ptr(dk), _ptr(dv), _ptr(dlog), _ptr(db), _ptr(dS0), ctypes.byref(shape), wp,
        int(n.value), _stream_handle(stream)), "kda_chunk_bwd_ws")
    return dq, dk, dv, dlog, db, dS0


def kda_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device-side status word."""
    return int(load().kda_device_status(_stream_handle(stream)))
