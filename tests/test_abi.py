"""Host-side checks of the C ABI: the library loads, exports every symbol that
include/kda.h declares, and rejects bad arguments before launching anything
(no GPU needed: argument validation happens before any CUDA call)."""
import ctypes
import os
import re

import pytest
import torch

import linear_attention_serving_gb300 as kda
from linear_attention_serving_gb300 import kda as kb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("kda_chunk_fwd", "kda_segment_scan", "kda_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol():
    kda.load()
    lib = ctypes.CDLL(kb.library_path())
    for n in declared_functions():
        assert hasattr(lib, n), f"libkda.so does not export {n}"


def test_status_strings_and_version():
    lib = kda.load()
    assert lib.kda_version() >= 100
    for code, name in [(0, b"KDA_OK"), (1, b"KDA_ERR_INVALID_ARG"), (2, b"KDA_ERR_UNSUPPORTED"),
                       (3, b"KDA_ERR_CUDA"), (4, b"KDA_ERR_TIMEOUT"), (5, b"KDA_ERR_WORKSPACE"),
                       (6, b"KDA_ERR_DEVICE_CHECK")]:
        assert lib.kda_status_string(code) == name
    assert lib.kda_status_string(99) == b"KDA_ERR_UNKNOWN"


def test_workspace_sizes_grow_with_work():
    s1 = kda.chunk_fwd_workspace_size(8192, 16, 1)
    s2 = kda.chunk_fwd_workspace_size(16384, 16, 1)
    assert 0 < s1 < s2
    assert kda.segment_scan_workspace_size(8192, 16, 1, 4) > s1
    lib = kda.load()
    assert lib.kda_chunk_fwd_workspace_size(-1, 16, 1, 0) == 0
    assert lib.kda_segment_scan_workspace_size(64, 1, 1, -1, 0) == 0


def test_planner_model_constants():
    """The timing model behind the planner's choice (kda_planner_model): positive,
    the preparation of a (chunk, head) unit slower on one SM than a chain's step
    (what makes long chains over few heads worth splitting), and the rule's
    boundary where the bound says: a single chain just over 1.5x the preparation
    of its batch on the SMs the chain leaves free gets segments."""
    prep_us, chain_us = kda.planner_model()
    assert prep_us > chain_us > 0
    bf16 = torch.bfloat16
    # one document, one head: chains = 2, so the preparation spreads over SMs - 2
    sms = 148 if not torch.cuda.is_available() else torch.cuda.get_device_properties(0).multi_processor_count
    for chunks in (64, 256, 4096):
        units = chunks
        prep = prep_us * units / (sms - 2)
        expect_split = chain_us * chunks > 1.5 * prep
        got = kda.chunk_fwd_plan_segments(chunks * 64, 1, 1, bf16)
        assert (got >= 2) == expect_split, (chunks, got, chain_us * chunks, prep)


def test_segment_planner_host_logic():
    """kda_chunk_fwd's own segment count: none for the bench's H=16, T=8192
    (the chains keep pace with the preparation) or for short documents; a few
    dozen at most for a long document over few heads; for a packed batch, the
    count for the longest document it can hold (the call plans again from its
    actual lengths); never for fp32; and the workspace size has room for it."""
    bf16 = torch.bfloat16
    assert kda.chunk_fwd_plan_segments(8192, 16, 1, bf16) == 0
    assert kda.chunk_fwd_plan_segments(333, 3, 1, bf16) == 0
    n = kda.chunk_fwd_plan_segments(1 << 20, 8, 1, bf16)
    assert 2 <= n <= 64
    assert kda.chunk_fwd_plan_segments(1 << 20, 8, 1, bf16, varlen=True) == n
    # 128 equal documents of 8192 tokens keep one chain each; packed, the same
    # total could be one long document
    assert kda.chunk_fwd_plan_segments(1 << 20, 8, 128, bf16) == 0
    nv = kda.chunk_fwd_plan_segments(1 << 20, 8, 128, bf16, varlen=True)
    assert 2 <= nv <= 64
    assert kda.chunk_fwd_workspace_size(1 << 20, 8, 128) >= kda.segment_scan_workspace_size(1 << 20, 8, 128, nv)
    assert kda.chunk_fwd_plan_segments(1 << 20, 8, 1, torch.float32) == 0
    assert kda.chunk_fwd_plan_segments(-1, 8, 1, bf16) == 0 and kda.chunk_fwd_plan_segments(64, 0, 1, bf16) == 0
    assert kda.chunk_fwd_workspace_size(1 << 20, 8, 1) >= kda.segment_scan_workspace_size(1 << 20, 8, 1, n)
    # more heads leave the chain less exposed: the planner never asks for more segments
    assert kda.chunk_fwd_plan_segments(1 << 20, 64, 1, bf16) <= n
    # whole waves: phase 3 (two blocks per (segment, head)) fits one wave of the SMs
    # and one more segment would not (the device count is 148 without a GPU, 152 on GB300)
    for sms in (148, 152):
        assert 2 * n * 8 <= sms < 2 * (n + 1) * 8
    # short sequences: the composition cap keeps the count small
    assert kda.chunk_fwd_plan_segments(32768, 4, 1, bf16) <= 10


FAKE = ctypes.c_void_p(1 << 20)  # aligned dummy address; never dereferenced on these paths


def _chunk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, A=FAKE, beta=FAKE, cu=None, n=1, T=128, H=2, D=128, dt=0,
             g_min=-5.0, init=None, o=FAKE, fin=None, ws=None, wsb=0, flags=0, s=None)
    a.update(kw)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["z"], a["A"], a["beta"], a["cu"], a["n"], a["T"],
                             a["H"], a["D"], a["dt"], a["g_min"], a["init"], a["o"], a["fin"], a["ws"],
                             a["wsb"], a["flags"], a["s"])


def test_chunk_fwd_rejects_bad_arguments_before_launch():
    lib = kda.load()
    assert _chunk(lib, D=64) == kb.KDA_OK + 2                       # unsupported head dim
    assert _chunk(lib, dt=7) == 1
    assert _chunk(lib, H=0) == 1
    assert _chunk(lib, g_min=-6.0) == 1                             # below the pages' bound
    assert _chunk(lib, g_min=0.0) == 1
    assert _chunk(lib, q=None) == 1
    assert _chunk(lib, A=None) == 1
    assert _chunk(lib, q=ctypes.c_void_p((1 << 20) + 2)) == 1       # misaligned
    assert _chunk(lib, n=3, T=128) == 1                             # T not divisible without cu_seqlens
    assert _chunk(lib, ws=None) == 5                                # no workspace
    assert _chunk(lib, ws=ctypes.c_void_p(1 << 20), wsb=16) == 5    # too small
    assert _chunk(lib, flags=4) == 1                                # unknown input option


def test_segment_scan_and_decode_reject_bad_arguments():
    lib = kda.load()
    r = lib.kda_segment_scan(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 128, 0, -5.0, None, -1,
                             None, None, FAKE, None, None, 0, 0, None)
    assert r == 1  # a negative segment count
    r = lib.kda_segment_scan(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 128, 0, -5.0, None, 0,
                             None, None, FAKE, None, None, 0, 0, None)
    assert r == 5  # zero is the automatic count: accepted, then the missing workspace is reported
    r = lib.kda_segment_scan(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 96, 0, -5.0, None, 4,
                             None, None, FAKE, None, None, 0, 0, None)
    assert r == 2
    dec = lambda **kw: lib.kda_decode_step(
        kw.get("state", FAKE), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("cq", FAKE), FAKE, FAKE, FAKE,
        FAKE, None, kw.get("N", 4), 2, kw.get("D", 128), kw.get("W", 5), 1, -5.0, FAKE, None,
        kw.get("flags", 0), None)
    assert dec(D=64) == 2
    assert dec(W=9) == 1
    assert dec(W=0) == 1
    assert dec(N=0) == 1
    assert dec(state=None) == 1
    assert dec(cq=None) == 1
    assert dec(flags=16) == 1
    assert dec(flags=4) == 1  # the convolution option belongs to the fused step


def test_decode_fused_rejects_bad_arguments():
    lib = kda.load()
    ALIGNED_BAD = 0x1008  # 8-byte aligned only

    def dec(**kw):
        return lib.kda_decode_step_fused(
            FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("conv_w", FAKE), kw.get("conv_state", FAKE),
            kw.get("o_gate", FAKE), kw.get("o_norm_w", FAKE), kw.get("eps", 1e-6), kw.get("cq", FAKE), FAKE,
            FAKE, FAKE, FAKE, None, kw.get("N", 4), 2, kw.get("D", 128), kw.get("W", 5), kw.get("dt", 1),
            kw.get("g_min", -5.0), FAKE, None, kw.get("flags", 0), None)

    assert dec(D=64) == 2
    assert dec(W=9) == 1 and dec(W=0) == 1 and dec(N=0) == 1
    assert dec(dt=7) == 1
    assert dec(g_min=-6.0) == 1
    assert dec(eps=-1.0) == 1 and dec(eps=float("nan")) == 1
    for name in ("conv_w", "conv_state", "o_gate", "o_norm_w", "cq"):
        assert dec(**{name: None}) == 1, name
    assert dec(conv_w=ALIGNED_BAD) == 1 and dec(conv_state=ALIGNED_BAD) == 1
    assert dec(flags=16) == 1


def test_binding_rejects_host_tensors_before_any_launch():
    """Host tensors would hand the kernels host pointers: every call refuses them
    (and tensors spread over devices) before it reaches the library."""
    import torch
    bf = torch.bfloat16
    q = torch.zeros(64, 2, 128, dtype=bf)
    z = torch.zeros(64, 2, 128)
    A, beta = torch.zeros(2), torch.zeros(64, 2)
    with pytest.raises(kda.KDAError, match="CUDA"):
        kda.chunk_fwd(q, q, q, z, A, beta)
    with pytest.raises(kda.KDAError, match="CUDA"):
        kda.segment_scan(q, q, q, z, A, beta, 2)
    qd = torch.zeros(2, 5, 2, 128)
    state = torch.zeros(2, 2, 128, 128)
    cache = tuple(torch.zeros(2, 4, 2, 128) for _ in range(4)) + (torch.zeros(2, 4, 2),)
    with pytest.raises(kda.KDAError, match="CUDA"):
        kda.decode_step(state, qd, qd, qd, qd, torch.zeros(2, 5, 2), A, cache)
    with pytest.raises(kda.KDAError, match="CUDA"):
        kda.decode_step_fused(state, qd, qd, qd, qd, torch.zeros(2, 5, 2), A, torch.zeros(3, 2, 128, 4),
                              torch.zeros(2, 2, 3, 3, 128), qd, torch.ones(128), cache)
    with pytest.raises(kda.KDAError, match="CUDA"):
        kda.read_device_error(torch.zeros(256, dtype=torch.uint8))


def test_binding_rejects_wrong_dtypes_on_cpu_tensors():
    import torch
    q = torch.zeros(4, 1, 128, dtype=torch.float16)
    with pytest.raises(kda.KDAError):
        kb._dtype_code(q)


def test_chunk_fwd_ckpt_rejects_bad_checkpoint_arguments():
    lib = kda.load()
    f = lib.kda_chunk_fwd_ckpt

    def call(interval=256, slot=FAKE, per_seq=4, ck=FAKE, n_slots=2):
        return f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 128, 0, -5.0, None, FAKE, None,
                 interval, slot, per_seq, ck, n_slots, None, 0, 0, None)

    assert call(interval=0) == 1
    assert call(interval=100) == 1        # not a multiple of the 64-token chunk
    assert call(per_seq=0) == 1
    assert call(n_slots=0) == 1
    assert call(slot=None) == 1
    assert call(ck=None) == 1
    assert call(ck=ctypes.c_void_p((1 << 20) + 4)) == 1  # misaligned pages
    assert call() == 5                    # valid checkpoints, but no workspace


def test_wait_budget_setter_returns_previous_and_restores_default():
    lib = kda.load()
    default = kda.set_wait_budget(12345)
    assert default == 2_000_000_000
    assert kda.set_wait_budget(0) == 12345   # <= 0 restores the default
    assert kda.set_wait_budget(-7) == default
    assert kda.set_wait_budget(default) == default


def test_segment_scan_auto_count_host_logic():
    """n_segments = 0: the wave rule's count (two rerun blocks per (segment, head)
    in one wave of the SMs, at most sqrt(chunks / 6), 64 and half the chunks, at
    least 1); the workspace size follows the resolved count."""
    lib = kda.load()
    n = kda.segment_scan_auto_segments(1 << 20, 8, 1)
    assert 2 <= n <= 64
    assert kda.segment_scan_auto_segments(64, 1, 1) == 1
    assert kda.segment_scan_auto_segments(-1, 8, 1) == 0
    assert lib.kda_segment_scan_workspace_size(1 << 20, 8, 1, 0, 0) == \
        lib.kda_segment_scan_workspace_size(1 << 20, 8, 1, n, 0)


def test_q_scale_flag_accepted_unknown_flags_rejected():
    """KDA_FLAG_Q_SCALE is a valid input option of every compute call; an unknown
    bit is rejected before any launch (no GPU touched)."""
    lib = kda.load()
    fake = ctypes.c_void_p(1 << 20)
    args = (fake, fake, fake, fake, fake, fake, None, 1, 64, 1, 128, 0, -5.0, None, fake, None)
    # a workspace of zero bytes: a valid flag gets as far as the workspace check
    assert lib.kda_chunk_fwd(*args, fake, 0, 8, None) == 5
    assert lib.kda_chunk_fwd(*args, fake, 0, 16, None) == 1


def test_noalloc_error_reader_rejects_null():
    lib = kda.load()
    assert lib.kda_noalloc_read_device_error(None, None) == 1
