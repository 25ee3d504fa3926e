"""Kimi Delta Attention (KDA) chunked forward for one GB300 (sm_103a).

The compute runs in the CUDA library libkda.so (C ABI: include/kda.h); this
package builds it in-tree and binds it with ctypes.
"""
from ._lib import (  # noqa: F401
    EXPORTS,
    KdaError,
    KdaShape,
    kda_backward,
    kda_backward_workspace_size,
    kda_chunk_fwd,
    kda_chunk_fwd_gated,
    kda_chunk_output,
    kda_chunk_states,
    kda_chunk_fwd_static_scratch,
    kda_chunk_fwd_workspace_size,
    kda_chunk_size,
    kda_chunk_fwd_kernel_name,
    kda_chunk_fwd_kernel_launches,
    kda_decode,
    kda_read_device_status,
    kda_recurrent_fwd,
    kda_status_string,
    library_path,
    load_library,
    make_shape,
)
from .builder import build  # noqa: F401
