"""GB300 (sm_103a) token-level multi-head linear attention (MHLA) forward library.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/mhla.h``); :mod:`token_level_head_gb300.binding` is its ctypes
binding.  Build it with :func:`token_level_head_gb300.build.build_library`.
"""

from .binding import (  # noqa: F401
    EXPORTED,
    MhlaError,
    linattn_decode_step,
    linattn_decode_steps,
    load,
    locality_mixing,
    mhla_causal_stream,
    mhla_forward,
    mhla_forward_causal,
    mhla_forward_ex,
    mhla_forward_ex_path,
    mhla_forward_grid,
    mhla_forward_grid_path,
    mhla_forward_noalloc,
    mhla_forward_path,
    mhla_launch_count,
    mhla_query_status,
    mhla_workspace_bytes,
    mhla_backward,
    mhla_backward_path,
    mhla_backward_workspace_bytes,
    new_workspace,
    rala_forward,
    rala_workspace_bytes,
    status_string,
)
