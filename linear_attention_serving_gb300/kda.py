"""Thin Python binding of the KDA C ABI (include/kda.h).

Argument marshalling only: outputs and the workspace are allocated with torch on
the inputs' device, and every step of the computation runs in the CUDA kernels
of ``libkda.so``.  There is no CPU or PyTorch fallback: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

KDA_OK = 0
KDA_BF16, KDA_F32 = 0, 1
DEVERR_CU_SEQLENS, DEVERR_NUM_ACCEPTED, DEVERR_TIMEOUT = 1, 2, 4
D = 128
G_MIN = -5.0

_lib = None


class KDAError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libkda.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise KDAError(f"libkda.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, L, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kda_status_string.argtypes = [I]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_version.restype = I
    lib.kda_chunk_fwd_workspace_size.argtypes = [L, I, I, I]
    lib.kda_chunk_fwd_workspace_size.restype = S
    lib.kda_segment_scan_workspace_size.argtypes = [L, I, I, I, I]
    lib.kda_segment_scan_workspace_size.restype = S
    lib.kda_chunk_fwd_plan_segments.argtypes = [L, I, I, I, I]
    lib.kda_chunk_fwd_plan_segments.restype = I
    lib.kda_planner_model.argtypes = [P, P]
    lib.kda_planner_model.restype = None
    lib.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, I, L, I, I, I, F, P, P, P, P, S, I, P]
    lib.kda_chunk_fwd.restype = I
    lib.kda_chunk_fwd_ckpt.argtypes = [P, P, P, P, P, P, P, I, L, I, I, I, F, P, P, P, I, P, I, P, I, P, S, I, P]
    lib.kda_chunk_fwd_ckpt.restype = I
    lib.kda_segment_scan.argtypes = [P, P, P, P, P, P, P, I, L, I, I, I, F, P, I, P, P, P, P, P, S, I, P]
    lib.kda_segment_scan.restype = I
    lib.kda_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P, I, P]
    lib.kda_decode_step.restype = I
    lib.kda_decode_step_fused.argtypes = [P, P, P, P, P, P, P, P, P, P, P, F, P, P, P, P, P, P,
                                          I, I, I, I, I, F, P, P, I, P]
    lib.kda_decode_step_fused.restype = I
    lib.kda_read_device_error.argtypes = [P, P, P]
    lib.kda_read_device_error.restype = I
    lib.kda_segment_scan_auto_segments.argtypes = [L, I, I]
    lib.kda_segment_scan_auto_segments.restype = I
    lib.kda_set_wait_budget.argtypes = [ctypes.c_longlong]
    lib.kda_set_wait_budget.restype = ctypes.c_longlong
    lib.kda_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, I, L, I, I, I, F, P, P, P, I, P]
    lib.kda_chunk_fwd_noalloc.restype = I
    lib.kda_noalloc_read_device_error.argtypes = [P, P]
    lib.kda_noalloc_read_device_error.restype = I
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != KDA_OK:
        raise KDAError(f"{what}: {load().kda_status_string(rc).decode()} ({rc})")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise KDAError(f"unsupported dtype {t.dtype}: q, k, v must be bfloat16 or float32")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _contig(*ts):
    """Every tensor the kernels touch: contiguous and on one CUDA device (a host
    tensor would hand the kernels a host pointer)."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_contiguous():
            raise KDAError("all tensors must be contiguous")
        if t.device.type != "cuda":
            raise KDAError("all tensors must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise KDAError("all tensors must be on the same CUDA device")


def chunk_fwd_workspace_size(T_total: int, H: int, n_seqs: int, dtype=torch.bfloat16) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(load().kda_chunk_fwd_workspace_size(T_total, H, n_seqs, code))


def chunk_fwd_plan_segments(T_total: int, H: int, n_seqs: int = 1, dtype=torch.bfloat16,
                            varlen: bool = False) -> int:
    """kda_chunk_fwd_plan_segments: the segment count kda_chunk_fwd uses for this
    shape on the current device (0 = one chain per (document, head))."""
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(load().kda_chunk_fwd_plan_segments(T_total, H, n_seqs, code, int(varlen)))


def planner_model() -> tuple:
    """kda_planner_model: (microseconds per prep unit on one SM, microseconds per
    chain chunk) behind kda_chunk_fwd's segment choice."""
    a, b = ctypes.c_double(0.0), ctypes.c_double(0.0)
    load().kda_planner_model(ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def segment_scan_workspace_size(T_total: int, H: int, n_seqs: int, n_segments: int,
                                dtype=torch.bfloat16) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(load().kda_segment_scan_workspace_size(T_total, H, n_seqs, n_segments, code))


def _n_seqs(cu_seqlens, n_seqs):
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise KDAError("cu_seqlens must be int32")
        return cu_seqlens.numel() - 1
    return n_seqs


KDA_FLAG_QK_L2NORM = 1
KDA_FLAG_BETA_SIGMOID = 2
KDA_FLAG_CONV_SILU = 4
KDA_FLAG_Q_SCALE = 8


def _flags(qk_l2norm: bool, beta_sigmoid: bool, q_scale: bool = False) -> int:
    return ((KDA_FLAG_QK_L2NORM if qk_l2norm else 0) | (KDA_FLAG_BETA_SIGMOID if beta_sigmoid else 0)
            | (KDA_FLAG_Q_SCALE if q_scale else 0))


def chunk_fwd(q, k, v, z, A, beta, cu_seqlens=None, init_state=None, g_min=G_MIN,
              output_final_state=True, n_seqs=1, workspace=None, out=None, qk_l2norm=False,
              beta_sigmoid=False, q_scale=False):
    """kda_chunk_fwd: chunkwise prefill.  q, k, v, z [T, H, 128]; A [H]; beta [T, H];
    cu_seqlens int32 [n+1] (device) or None (n_seqs equal-length sequences).
    Returns (o [T, H, 128] in q's dtype, final_state [n, H, 128, 128] fp32 or None)."""
    lib = load()
    _contig(q, k, v, z, A, beta, cu_seqlens, init_state, workspace, out)
    T, H, Dm = q.shape
    n = _n_seqs(cu_seqlens, n_seqs)
    dt = _dtype_code(q)
    o = out if out is not None else torch.empty_like(q)
    fin = torch.empty((n, H, Dm, Dm), device=q.device, dtype=torch.float32) if output_final_state else None
    if workspace is None:
        # (a caller's own workspace is passed as given: one with room for the
        # single-chain path only keeps that path, a smaller one is refused)
        workspace = torch.empty(lib.kda_chunk_fwd_workspace_size(T, H, n, dt), device=q.device, dtype=torch.uint8)
    rc = lib.kda_chunk_fwd(_p(q), _p(k), _p(v), _p(z), _p(A), _p(beta), _p(cu_seqlens), n, T, H, Dm,
                           dt, float(g_min), _p(init_state), _p(o), _p(fin), _p(workspace),
                           workspace.numel(), _flags(qk_l2norm, beta_sigmoid, q_scale), _stream(q.device))
    _check(rc, "kda_chunk_fwd")
    return o, fin


def chunk_fwd_ckpt(q, k, v, z, A, beta, ckpt_interval, ckpt_slot, ckpt, cu_seqlens=None, init_state=None,
                   g_min=G_MIN, output_final_state=True, n_seqs=1, workspace=None, out=None, qk_l2norm=False,
                   beta_sigmoid=False, q_scale=False):
    """kda_chunk_fwd_ckpt: chunk_fwd that also writes document states at
    ckpt_interval-aligned positions.  ckpt_slot int32 [n, per_seq] (device) maps
    (document, j) -> page of ckpt [n_slots, H, 128, 128] fp32 (device) for the
    state after (j + 1) * ckpt_interval tokens; -1 skips."""
    lib = load()
    _contig(q, k, v, z, A, beta, cu_seqlens, init_state, ckpt_slot, ckpt, workspace, out)
    T, H, Dm = q.shape
    n = _n_seqs(cu_seqlens, n_seqs)
    dt = _dtype_code(q)
    if ckpt_slot.dtype != torch.int32 or ckpt_slot.dim() != 2 or ckpt_slot.shape[0] != n:
        raise KDAError("ckpt_slot must be int32 [n_seqs, per_seq]")
    if ckpt.dtype != torch.float32 or ckpt.dim() != 4 or tuple(ckpt.shape[1:]) != (H, Dm, Dm):
        raise KDAError("ckpt must be fp32 [n_slots, H, 128, 128]")
    o = out if out is not None else torch.empty_like(q)
    fin = torch.empty((n, H, Dm, Dm), device=q.device, dtype=torch.float32) if output_final_state else None
    if workspace is None:
        # (a caller's own workspace is passed as given: one with room for the
        # single-chain path only keeps that path, a smaller one is refused)
        workspace = torch.empty(lib.kda_chunk_fwd_workspace_size(T, H, n, dt), device=q.device, dtype=torch.uint8)
    rc = lib.kda_chunk_fwd_ckpt(_p(q), _p(k), _p(v), _p(z), _p(A), _p(beta), _p(cu_seqlens), n, T, H, Dm,
                                dt, float(g_min), _p(init_state), _p(o), _p(fin), int(ckpt_interval), _p(ckpt_slot),
                                ckpt_slot.shape[1], _p(ckpt), ckpt.shape[0], _p(workspace), workspace.numel(),
                                _flags(qk_l2norm, beta_sigmoid, q_scale), _stream(q.device))
    _check(rc, "kda_chunk_fwd_ckpt")
    return o, fin


def segment_scan(q, k, v, z, A, beta, n_segments, cu_seqlens=None, init_state=None, g_min=G_MIN,
                 output_final_state=True, return_pairs=False, n_seqs=1, workspace=None, qk_l2norm=False,
                 beta_sigmoid=False, q_scale=False):
    """kda_segment_scan: intra-device segment-parallel prefill; n_segments = 0 takes
    the automatic count (segment_scan_auto_segments).
    Returns (o, final_state) or (o, final_state, pairs_M, pairs_S) with pairs [H, n_seg, 128, 128]."""
    lib = load()
    _contig(q, k, v, z, A, beta, cu_seqlens, init_state, workspace)
    T, H, Dm = q.shape
    n = _n_seqs(cu_seqlens, n_seqs)
    if n_segments == 0:
        n_segments = segment_scan_auto_segments(T, H, n)
    dt = _dtype_code(q)
    o = torch.empty_like(q)
    fin = torch.empty((n, H, Dm, Dm), device=q.device, dtype=torch.float32) if output_final_state else None
    pm = ps = None
    if return_pairs:
        pm = torch.empty((H, n_segments, Dm, Dm), device=q.device, dtype=torch.float32)
        ps = torch.empty_like(pm)
    need = lib.kda_segment_scan_workspace_size(T, H, n, n_segments, dt)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    rc = lib.kda_segment_scan(_p(q), _p(k), _p(v), _p(z), _p(A), _p(beta), _p(cu_seqlens), n, T, H, Dm,
                              dt, float(g_min), _p(init_state), int(n_segments), _p(pm), _p(ps),
                              _p(o), _p(fin), _p(workspace), workspace.numel(),
                              _flags(qk_l2norm, beta_sigmoid, q_scale), _stream(q.device))
    _check(rc, "kda_segment_scan")
    if return_pairs:
        return o, fin, pm, ps
    return o, fin


def decode_step(state, q, k, v, z, beta, A, cache, num_accepted=None, g_min=G_MIN,
                error_word=None, out=None, qk_l2norm=False, beta_sigmoid=False, q_scale=False):
    """kda_decode_step: in-place state update with MTP replay.
    state [N, H, 128, 128] fp32 (updated in place); q, k, v, z [N, W, H, 128]; beta [N, W, H];
    cache = (cache_q, cache_k, cache_v, cache_z, cache_beta) with W-1 slots (updated in place);
    num_accepted int32 [N] (device) or None.  Returns o [N, W, H, 128]."""
    lib = load()
    cq, ck, cv, cz, cb = cache if cache is not None else (None,) * 5
    _contig(state, q, k, v, z, beta, A, cq, ck, cv, cz, cb, num_accepted, error_word, out)
    N, W, H, Dm = q.shape
    if num_accepted is not None and num_accepted.dtype != torch.int32:
        raise KDAError("num_accepted must be int32")
    o = out if out is not None else torch.empty_like(q)
    rc = lib.kda_decode_step(_p(state), _p(q), _p(k), _p(v), _p(z), _p(beta), _p(A), _p(cq), _p(ck),
                             _p(cv), _p(cz), _p(cb), _p(num_accepted), N, H, Dm, W, _dtype_code(q),
                             float(g_min), _p(o), _p(error_word), _flags(qk_l2norm, beta_sigmoid, q_scale),
                             _stream(q.device))
    _check(rc, "kda_decode_step")
    return o


def decode_step_fused(state, q, k, v, z, beta, A, conv_w, conv_state, o_gate, o_norm_w, cache,
                      num_accepted=None, o_norm_eps=1e-6, g_min=G_MIN, error_word=None, out=None,
                      qk_l2norm=False, beta_sigmoid=False, conv_silu=False, q_scale=False):
    """kda_decode_step_fused: the decode step with the short convolution of q, k, v in
    front of the recurrence and the gated per-head output norm after it.
    As decode_step, plus conv_w [3, H, 128, 4] fp32 (tap 3 on the current token),
    conv_state [N, H, 3, 3, 128] fp32 (updated in place), o_gate [N, W, H, 128] fp32
    (output-gate logits), o_norm_w [128] fp32.  q, k, v and the cache hold inputs before
    the convolution.  Returns o [N, W, H, 128]."""
    lib = load()
    cq, ck, cv, cz, cb = cache if cache is not None else (None,) * 5
    _contig(state, q, k, v, z, beta, A, conv_w, conv_state, o_gate, o_norm_w, cq, ck, cv, cz, cb,
            num_accepted, error_word, out)
    N, W, H, Dm = q.shape
    if num_accepted is not None and num_accepted.dtype != torch.int32:
        raise KDAError("num_accepted must be int32")
    for t in (conv_w, conv_state, o_gate, o_norm_w):
        if t.dtype != torch.float32:
            raise KDAError("conv_w, conv_state, o_gate and o_norm_w must be float32")
    if tuple(conv_w.shape) != (3, H, Dm, 4) or tuple(conv_state.shape) != (N, H, 3, 3, Dm):
        raise KDAError("conv_w must be [3, H, D, 4] and conv_state [N, H, 3, 3, D]")
    if tuple(o_gate.shape) != (N, W, H, Dm) or tuple(o_norm_w.shape) != (Dm,):
        raise KDAError("o_gate must be [N, W, H, D] and o_norm_w [D]")
    o = out if out is not None else torch.empty_like(q)
    flags = _flags(qk_l2norm, beta_sigmoid, q_scale) | (KDA_FLAG_CONV_SILU if conv_silu else 0)
    rc = lib.kda_decode_step_fused(_p(state), _p(q), _p(k), _p(v), _p(z), _p(beta), _p(A), _p(conv_w),
                                   _p(conv_state), _p(o_gate), _p(o_norm_w), float(o_norm_eps), _p(cq),
                                   _p(ck), _p(cv), _p(cz), _p(cb), _p(num_accepted), N, H, Dm, W,
                                   _dtype_code(q), float(g_min), _p(o), _p(error_word), flags,
                                   _stream(q.device))
    _check(rc, "kda_decode_step_fused")
    return o


def read_device_error(workspace: torch.Tensor) -> int:
    _contig(workspace)
    code = ctypes.c_int32(0)
    rc = load().kda_read_device_error(_p(workspace), ctypes.byref(code), _stream(workspace.device))
    _check(rc, "kda_read_device_error")
    return int(code.value)


def segment_scan_auto_segments(T_total: int, H: int, n_seqs: int = 1) -> int:
    """kda_segment_scan_auto_segments: the count kda_segment_scan takes for n_segments = 0."""
    return int(load().kda_segment_scan_auto_segments(T_total, H, n_seqs))


def set_wait_budget(cycles: int) -> int:
    """kda_set_wait_budget: clock-cycle limit of the waits on other blocks' flags and of
    the decode's copy waits for the calls that follow (<= 0: the default, about one
    second).  Returns the previous limit."""
    return int(load().kda_set_wait_budget(int(cycles)))


def chunk_fwd_noalloc(q, k, v, z, A, beta, cu_seqlens=None, init_state=None, g_min=G_MIN,
                      output_final_state=True, n_seqs=1, out=None, qk_l2norm=False, beta_sigmoid=False,
                      q_scale=False):
    """kda_chunk_fwd_noalloc: chunk_fwd with the library's fixed device array as its
    workspace (the library allocates nothing; this binding still allocates o and the
    final state with torch unless `out` is given and output_final_state is False)."""
    lib = load()
    _contig(q, k, v, z, A, beta, cu_seqlens, init_state, out)
    T, H, Dm = q.shape
    n = _n_seqs(cu_seqlens, n_seqs)
    o = out if out is not None else torch.empty_like(q)
    fin = torch.empty((n, H, Dm, Dm), device=q.device, dtype=torch.float32) if output_final_state else None
    rc = lib.kda_chunk_fwd_noalloc(_p(q), _p(k), _p(v), _p(z), _p(A), _p(beta), _p(cu_seqlens), n, T, H, Dm,
                                   _dtype_code(q), float(g_min), _p(init_state), _p(o), _p(fin),
                                   _flags(qk_l2norm, beta_sigmoid, q_scale), _stream(q.device))
    _check(rc, "kda_chunk_fwd_noalloc")
    return o, fin


def noalloc_read_device_error(device=None) -> int:
    """kda_noalloc_read_device_error: the device error word of the last
    kda_chunk_fwd_noalloc on the current device."""
    code = ctypes.c_int32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    rc = load().kda_noalloc_read_device_error(ctypes.byref(code), _stream(dev))
    _check(rc, "kda_noalloc_read_device_error")
    return int(code.value)


def profile_enable(on: bool = True) -> None:
    _check(load().kda_profile_enable(1 if on else 0), "kda_profile_enable")


def profile_collect(max_marks: int = 256):
    """[(kernel name, ms since the previous mark)] since the last collect."""
    lib = load()
    names = (ctypes.c_char_p * max_marks)()
    ms = (ctypes.c_float * max_marks)()
    lib.kda_profile_collect.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.kda_profile_collect.restype = ctypes.c_int
    n = lib.kda_profile_collect(ctypes.cast(names, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                                max_marks)
    if n < 0:
        raise KDAError("kda_profile_collect failed")
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def launch_count() -> int:
    lib = load()
    lib.kda_launch_count.restype = ctypes.c_longlong
    return int(lib.kda_launch_count())
