"""GB300 kernelized linear attention: Python binding of liblinattn.so.

The binding only marshals arguments: torch tensors on the GPU supply device
pointers and the current CUDA stream, and every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if the library has
not been built, every call raises.

Entry points (same names as the C ABI in include/linattn.h):
  la_feature_map, la_forward_bidir, la_forward_causal, la_forward, la_decode_step, la_forward_phase,
  la_forward_causal_noalloc, la_noalloc_error, la_test_force_wait_timeout, la_test_segment_plan, la_backward, la_backward_workspace_bytes, la_workspace_bytes,
  la_check_cu_seqlens, la_workspace_error, la_orthogonal_features,
  la_selected_path, la_status_string, la_version
plus `attention(...)`, which allocates the output and workspace and calls
la_forward_bidir or la_forward_causal.
"""
from ._binding import (  # noqa: F401
    LinAttnError, library_path, load_library, MAP_IDS, DTYPE_IDS, NORM_IDS,
    la_feature_map, la_forward_bidir, la_forward_causal, la_forward, la_decode_step, la_forward_phase,
    la_forward_causal_noalloc, la_noalloc_error, la_test_force_wait_timeout, la_test_segment_plan, la_backward, la_backward_workspace_bytes,
    la_workspace_bytes, la_check_cu_seqlens, la_workspace_error, la_orthogonal_features, la_selected_path,
    la_status_string, la_version, attention, forward_ptrs, forward_general_ptrs,
)
