"""GB300-native sparse-attention token selection over a paged KV cache.

The computation lives in libsel.so (hand-written sm_103a CUDA behind the C ABI in
include/sel.h); this package is its Python binding. Importing it loads the library
and raises if it has not been built.
"""

from .sel import (  # noqa: F401
    Problem,
    SelError,
    new_workspace,
    problem_from_workload,
    sel_error_string,
    sel_host_stage_bytes,
    sel_maxsim_launch_count,
    sel_maxsim_rerank,
    sel_maxsim_workspace_bytes,
    sel_mla_decode,
    sel_mla_launch_count,
    sel_mla_workspace_bytes,
    sel_remap_dcp,
    sel_remap_global,
    sel_remap_workspace,
    sel_score_paged,
    sel_score_workspace_bytes,
    sel_select,
    sel_select_host,
    sel_select_launch_count,
    sel_select_static,
    sel_debug_wait_limit,
    sel_set_trace_events,
    sel_topk_expand,
    sel_version,
    sel_workspace_bytes,
)
