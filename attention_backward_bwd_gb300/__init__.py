"""GB300-native fused attention backward.

The computation runs in hand-written sm_103a CUDA kernels inside
``libattn_gb300.so`` (C ABI in ``include/attn_bwd.h``); this package only
builds and binds it.  PyTorch provides device memory and streams.
"""
from .binding import (AttnError, alloc_workspace, attn_bwd, attn_bwd_host, attn_bwd_host_varlen,
                      attn_fwd,
                      check_device_status, diag_mma, diag_tanh, diag_wait_timeout,
                      host_buffer_size, lib, set_wait_timeout_ns, version, workspace_layout,
                      workspace_size)

__all__ = ["AttnError", "alloc_workspace", "attn_bwd", "attn_bwd_host", "attn_bwd_host_varlen",
           "attn_fwd",
           "check_device_status", "diag_mma", "diag_tanh", "diag_wait_timeout",
           "host_buffer_size", "lib", "set_wait_timeout_ns", "version", "workspace_layout",
           "workspace_size"]
