"""Tree/DAG-packed paged attention (forward and backward) for GB300 (sm_103a).

The compute path is libtreeattn (hand-written tcgen05/TMA kernels behind the C ABI declared
in include/treeattn.h); this package is its Python binding.  Importing the package does not
load the library; the first call does, and raises if it has not been built.
"""
from ._native import (  # noqa: F401
    TA_CLAMP_MOUNTS, TA_ERR_CUDA, TA_ERR_DEVICE_BOUNDS, TA_ERR_DEVICE_TIMEOUT, TA_ERR_INVALID, TA_ERR_NOMEM,
    TA_ERR_UNSUPPORTED, TA_NO_MOUNTS, TA_OK, TA_PLAN_HOST_ONLY, TA_PLAN_STREAM_ORDERED, TA_TRANSITIVE_MOUNTS, Plan,
    TreeAttnError, tree_attn_bwd,
    tree_attn_bwd_noalloc,
    tree_attn_bwd_workspace_size, tree_attn_check, tree_attn_fwd, tree_attn_ingest, tree_attn_last_error,
    tree_attn_logprob_bwd, tree_attn_logprob_fwd, tree_attn_logprob_index, tree_attn_owner_mask,
    tree_attn_place, tree_attn_place_units,
    tree_attn_plan, tree_attn_plan_destroy, tree_attn_plan_export, tree_attn_plan_stats, tree_attn_rope,
    tree_attn_selftest_timeout, tree_attn_set_trace_events)
