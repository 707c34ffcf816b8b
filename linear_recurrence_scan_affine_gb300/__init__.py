"""GB300 affine-scan kernels for RL credit assignment.

Seven estimators (GAE, TD(lambda) returns, discounted returns, V-trace,
Retrace(lambda), eligibility traces, episodic prefix sum), each one batched
first-order linear recurrence over [N, T] rollouts solved as an associative
scan in hand-written CUDA for sm_103a. The C ABI is include/rlcs.h; this
package is a thin ctypes binding with the same names. Importing it loads
``librlcs.so`` and fails loudly if the library has not been built.
"""
from .binding import (  # noqa: F401
    RLCS_SHAPE_AUTO, RLCS_SHAPE_BLOCK_CHUNK, RLCS_SHAPE_BLOCK_TILE, RLCS_SHAPE_WARP_ROW, RlcsError,
    check_all_workspaces, lib, rlcs_check_status, rlcs_discounted_returns,
    rlcs_eligibility_traces, rlcs_episodic_prefix_sum, rlcs_gae, rlcs_lambda_returns,
    rlcs_retrace, rlcs_set_shape_override, rlcs_vtrace, rlcs_workspace_bytes,
    rlcs_affine_scan, rlcs_gae_and_returns, rlcs_gae_compact, rlcs_diag_stream_copy,
    rlcs_gae_tm, rlcs_lambda_returns_tm, rlcs_discounted_returns_tm, rlcs_vtrace_tm,
    rlcs_retrace_tm, rlcs_eligibility_traces_tm, rlcs_episodic_prefix_sum_tm,
    rlcs_gae_and_returns_tm, rlcs_affine_scan_tm, rlcs_run_group, GROUP_ESTIMATORS, MAX_GROUP,
    workspace_for)
