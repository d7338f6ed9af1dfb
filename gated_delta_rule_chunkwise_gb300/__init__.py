"""GB300 (sm_103a) chunkwise delta-rule linear attention: DeltaNet, Gated
DeltaNet, KDA and Gated DeltaNet-2 forward, the backward, Residual Linear
Attention / Residual DeltaNet, plus the single-token recurrent decode step.

The computation lives in CUDA kernels behind the C ABI of include/ldn.h
(lib/libldn.so, built by ``build.build()``); this package holds the ctypes
binding (``_native``) and the seeded synthetic workloads (``workloads``).
"""
from ._native import (  # noqa: F401
    EXPORTS, LDN_BF16, LDN_DELTANET, LDN_ERR_CUDA, LDN_ERR_INVALID_ARG, LDN_ERR_TIMEOUT,
    LDN_ERR_UNSUPPORTED, LDN_F32, LDN_GDN, LDN_GDN2, LDN_KDA, LDN_OK, LDN_VARIANT_AUTO, LDN_VARIANT_SIMT,
    LDN_VARIANT_TENSOR, LDN_VARIANT_SPLIT, LDN_VARIANT_PAIR, LDN_VARIANT_PRESOLVED, LIB_PATH, MODES, LdnError, backward, chunk_fwd, chunk_fwd_gdn2, decode_step, decode_steps,
    decode_step_gdn2, device_status, ldn_backward, ldn_backward_workspace_size, ldn_chunk_fwd_gdn2,
    ldn_decode_step_gdn2, ldn_decode_steps, ldn_rla_fwd, ldn_rla_fwd_ws, ldn_rla_fwd_workspace_size, rla_fwd,
    ldn_chunk_fwd, ldn_chunk_fwd_noalloc, ldn_chunk_fwd_select, ldn_chunk_fwd_ws, ldn_chunk_fwd_workspace_size, ldn_chunk_fwd_select_ws, ldn_chunk_fwd_split_segments, ldn_chunk_fwd_variant, ldn_decode_step, ldn_get_device_status, ldn_prologue, ldn_rmsnorm_gated,
    ldn_status_string, ldn_version, load,
)
