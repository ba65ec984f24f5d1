"""GB300-native (sm_103a) Kimi Delta Attention forward hot path.

Three calls, each a hand-written CUDA kernel path behind the C ABI in
``include/kda.h``: ``chunk_fwd`` (chunkwise prefill), ``segment_scan``
(intra-device segment-parallel prefill) and ``decode_step`` (in-place decode
with MTP draft replay).
"""
from .kda import (KDAError, chunk_fwd, chunk_fwd_ckpt, chunk_fwd_plan_segments, chunk_fwd_workspace_size, decode_step, load,
                  library_path, read_device_error, segment_scan, segment_scan_workspace_size)

__all__ = ["KDAError", "chunk_fwd", "chunk_fwd_ckpt", "chunk_fwd_plan_segments", "chunk_fwd_workspace_size", "decode_step", "load",
           "library_path", "read_device_error", "segment_scan", "segment_scan_workspace_size"]
