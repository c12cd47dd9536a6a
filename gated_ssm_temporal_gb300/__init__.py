"""GB300-native gated temporal scan layer (Mamba2-style): C-ABI library + binding.

The forward and backward of the layer (and the bias-gradient column sum of
the same training step) run in hand-written sm_103a kernels in
``libm2scan.so`` (built in-tree by ``gated_ssm_temporal_gb300.build``); this
package only marshals arguments to it.
"""
from .binding import (M2SCAN_OK, NOALLOC_SCRATCH_BYTES, M2ScanError, alloc_bwd_outputs, alloc_workspace, bias_grad,
                      bwd, fwd, header_functions, load_library, m2scan_bwd, m2scan_bwd_noalloc,
                      m2scan_bwd_workspace_bytes, m2scan_fwd, m2scan_last_cuda_error,
                      m2scan_last_launch_count, m2scan_path_for, m2scan_fwd_path_for,
                      m2scan_read_device_flags,
                      m2scan_set_force_generic, m2scan_status_str, m2scan_bias_grad,
                      m2scan_bias_grad_workspace_bytes, m2scan_bwd_ex, m2scan_fwd_ex, fwd_blend,
                      bwd_blend, m2scan_fwd_blend, m2scan_bwd_blend, m2scan_blend_fwd_workspace_bytes,
                      m2scan_blend_bwd_workspace_bytes, fwd_bf16, m2scan_fwd_bf16, bwd_bf16,
                      m2scan_bwd_bf16, m2scan_selftest_wait_timeout)

__all__ = ["M2SCAN_OK", "NOALLOC_SCRATCH_BYTES", "M2ScanError", "alloc_bwd_outputs", "alloc_workspace", "bias_grad",
           "bwd", "fwd", "m2scan_bias_grad", "m2scan_bias_grad_workspace_bytes", "m2scan_bwd_ex",
           "m2scan_fwd_ex", "fwd_blend", "bwd_blend", "m2scan_fwd_blend", "m2scan_bwd_blend",
           "m2scan_blend_fwd_workspace_bytes", "m2scan_blend_bwd_workspace_bytes", "fwd_bf16",
           "m2scan_fwd_bf16", "bwd_bf16", "m2scan_bwd_bf16",
           "header_functions", "load_library", "m2scan_bwd", "m2scan_bwd_noalloc", "m2scan_bwd_workspace_bytes",
           "m2scan_fwd", "m2scan_last_cuda_error", "m2scan_last_launch_count",
           "m2scan_path_for", "m2scan_fwd_path_for", "m2scan_read_device_flags", "m2scan_set_force_generic",
           "m2scan_status_str", "m2scan_selftest_wait_timeout"]
