"""libssmscan: the Mamba2 selective-state scan as sm_103a CUDA kernels.

    from state_space_model_ssm_gb300 import ssm_scan
    y = ssm_scan(state_slots, x, dt, A, B, C, D, seq_starts, seq_lens, resume_flags)

The C ABI is declared in ``include/ssmscan.h``; ``binding`` wraps it with
ctypes.  ``workloads`` draws the seeded synthetic inputs.
"""
from .binding import (PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_PREFILL_DIRECT,  # noqa: F401
                      SEGMENT_STATE_AUTO, SEGMENT_STATE_FP32, SEGMENT_STATE_TENSOR,
                      Options, SsmScanError, Tuning,
                      load, ssd_workspace_bytes, ssm_conv1d, ssm_scan, ssm_scan_ssd,
                      status_string)

__all__ = ["Options", "ssm_conv1d", "ssm_scan", "ssm_scan_ssd", "ssd_workspace_bytes", "Tuning", "SsmScanError", "PATH_AUTO", "PATH_DECODE",
           "PATH_PREFILL", "PATH_PREFILL_DIRECT", "SEGMENT_STATE_AUTO", "SEGMENT_STATE_FP32",
           "SEGMENT_STATE_TENSOR", "load", "status_string"]
