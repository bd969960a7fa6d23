"""libkda: Kimi Delta Attention (KDA) token mixer for GB300 (sm_103a).

The computation lives in the CUDA library ``libkda.so`` (C ABI in
``include/kda.h``); this package holds its sources (``csrc/``), the in-tree
build (``build.py``), a thin ctypes binding (``binding.py``) and seeded
synthetic workloads (``inputs.py``).
"""
from .binding import (  # noqa: F401
    KDA_DTYPE_BF16, KDA_DTYPE_F32, KDA_ENGINE_AUTO, KDA_ENGINE_SIMT, KDA_ENGINE_TENSOR,
    KDA_ERR_CUDA, KDA_ERR_INVALID_ARG, KDA_ERR_TIMEOUT, KDA_ERR_UNSUPPORTED, KDA_SUCCESS,
    KDA_PROLOGUE_BETA_LOGITS, KDA_PROLOGUE_GATE, KDA_PROLOGUE_L2NORM_QK,
    KdaError, kda_chunk_fwd, kda_chunk_fwd_workspace_size, kda_chunk_fwd_ws,
    kda_chunk_fwd_ws_timed, kda_chunk_fwd_host, kda_chunk_fwd_host_scratch_size,
    kda_chunk_fwd_static, kda_chunk_fwd_ws_diag, kda_chunk_path_counts, kda_chunk_bwd,
    kda_device_status, kda_recurrent_bwd, kda_recurrent_fwd, kda_recurrent_step, kda_short_conv_fwd,
    kda_short_conv_step, kda_status_string, kdaConvShape_t, kdaShape_t, lib_path, load,
    make_shape,
)
