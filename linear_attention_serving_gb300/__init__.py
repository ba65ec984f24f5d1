"""GB300-native (sm_103a) Kimi Delta Attention forward hot path.

Three calls, each a hand-written CUDA kernel path behind the C ABI in
``include/kda.h``: ``chunk_fwd`` (chunkwise prefill), ``segment_scan``
(intra-device segment-parallel prefill) and ``decode_step`` (in-place decode
with MTP draft replay), plus ``decode_step_fused`` (the decode step with the
short convolution and the gated output norm around the recurrence).
"""
from .kda import (KDAError, chunk_fwd, chunk_fwd_ckpt, chunk_fwd_noalloc, chunk_fwd_plan_segments,
                  chunk_fwd_workspace_size, decode_step, decode_step_fused, launch_count, library_path, load,
                  noalloc_read_device_error, planner_model, profile_collect, profile_enable, read_device_error,
                  segment_scan, segment_scan_auto_segments, segment_scan_workspace_size, set_wait_budget)

__all__ = ["KDAError", "chunk_fwd", "chunk_fwd_ckpt", "chunk_fwd_noalloc", "chunk_fwd_plan_segments",
           "chunk_fwd_workspace_size", "decode_step", "decode_step_fused", "launch_count", "library_path", "load",
           "noalloc_read_device_error", "planner_model", "profile_collect", "profile_enable", "read_device_error",
           "segment_scan", "segment_scan_auto_segments", "segment_scan_workspace_size", "set_wait_budget"]
