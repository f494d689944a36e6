"""GB300 (sm_103a) MoE layer forward: route -> permute -> grouped SwiGLU -> combine.

The compute lives in the CUDA library `_build/libmoe_gb300.so` (C ABI in
include/moe.h); this package is its thin Python binding.  Build the library
with `mixture_experts_layer_fp32_gb300.build.build()`.
"""

from ._binding import (  # noqa: F401
    EXPORTS,
    LIB_PATH,
    SCORE,
    DTYPE,
    DROP_POLICY,
    MoeConfig,
    MoeError,
    Buffers,
    act_dtype,
    alloc_workspace,
    alloc_workspace_host,
    alloc_workspace_shared,
    capacity,
    check,
    combine,
    combine_shared,
    config,
    forward,
    forward_host,
    forward_shared,
    grouped_fc1,
    grouped_fc2,
    grouped_mlp,
    lib,
    max_rows,
    permute,
    permute_noalloc,
    probe_fp32_fma,
    route,
    selftest_wait_timeout,
    shared_expert,
    workspace_size,
    workspace_size_host,
    workspace_size_shared,
)
