"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory at call time (an engine that has reserved the whole
device for its own pool, or a latency-critical path where a cudaMalloc and the
device synchronisation it may bring are not acceptable).  It takes its
workspace from a fixed array owned by the library instead of from the caller.

Called through the C ABI with ctypes and checked against kda_chunk_fwd and
against the fp64 oracle on two calls in a row with different inputs, so that
anything the first call leaves in the shared array cannot hide a fault in the
second; and a bad cu_seqlens must show up in the array's error word, which
kda_noalloc_read_device_error reads.  This file is collected last so that a run
stopping at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, err_report, rel_fro, to_dev

P, I, L, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
KDA_ERR_WORKSPACE = 5


def noalloc_fn():
    lib = kda.load()
    fn = lib.kda_chunk_fwd_noalloc
    fn.argtypes = [P, P, P, P, P, P, P, I, L, I, I, I, F, P, P, P, I, P]
    fn.restype = I
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(fn, d, n_seqs):
    q = d["q"]
    T, H, Dm = q.shape
    dt = 0 if q.dtype == torch.bfloat16 else 1
    o = torch.empty_like(q)
    fin = torch.empty((n_seqs, H, Dm, Dm), device=q.device, dtype=torch.float32)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(_p(q), _p(d["k"]), _p(d["v"]), _p(d["z"]), _p(d["A"]), _p(d["beta"]), _p(d["cu_seqlens"]),
            n_seqs, T, H, Dm, dt, -5.0, _p(d["init_state"]), _p(o), _p(fin), 0, stream)
    return rc, o, fin


def test_noalloc_rejects_calls_larger_than_its_array():
    fn = noalloc_fn()
    # 8192 tokens x 16 heads needs ~170 MB of workspace, beyond the fixed array;
    # rejected on the host before anything is launched (no GPU touched)
    fake = ctypes.c_void_p(1 << 20)
    rc = fn(fake, fake, fake, fake, fake, fake, None, 1, 8192, 16, 128, 0, -5.0, None, fake, None, 0, None)
    assert rc == KDA_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_chunk_fwd_on_two_calls(dtype):
    fn = noalloc_fn()
    cases = [
        (kda_synth.cu_from_lengths([300, 1, 0, 700]), 4),   # packed documents
        (None, 1),                                          # one sequence
    ]
    for call, (cu, n) in enumerate(cases):
        inp = kda_synth.prefill_inputs(1001 if cu is not None else 640, 3, dtype, seed=70 + call,
                                       z_std=1.5, A_std=0.5, cu_seqlens=cu, init_std=0.05, n_init=n)
        d = to_dev(inp, "cuda")
        o_ref, f_ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"],
                                     cu_seqlens=d["cu_seqlens"], init_state=d["init_state"])
        rc, o, fin = call_noalloc(fn, d, n)
        torch.cuda.synchronize()
        assert rc == 0, f"call {call}: status {rc}"
        assert kda.noalloc_read_device_error() == 0
        to, tf = TOL[dtype]
        assert rel_fro(o, o_ref) <= to, f"call {call}: o"
        assert rel_fro(fin, f_ref) <= tf, f"call {call}: final state"
        # and against the oracle on the same inputs
        oo, of = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                  cu_seqlens=cu, init_state=inp["init_state"])
        eo, mo = err_report(o, oo, "tokens", cu, n)
        ef, mf = err_report(fin, of, "state")
        assert eo <= to, f"call {call}: o vs oracle {mo}"
        assert ef <= tf, f"call {call}: final state vs oracle {mf}"


@pytest.mark.gpu
def test_noalloc_reports_bad_cu_seqlens():
    """Decreasing document offsets, built on the host: the call returns KDA_OK (the
    check needs device data), writes nothing, and its error word holds
    KDA_DEVERR_CU_SEQLENS; the next good call clears it."""
    fn = noalloc_fn()
    inp = kda_synth.prefill_inputs(256, 1, "bf16", seed=79)
    d = to_dev(inp, "cuda")
    d["cu_seqlens"] = torch.tensor([0, 200, 100, 256], dtype=torch.int32, device="cuda")
    d["init_state"] = None
    rc, o, _ = call_noalloc(fn, d, 3)
    assert rc == 0
    assert kda.noalloc_read_device_error() & 1
    d["cu_seqlens"] = torch.tensor([0, 100, 200, 256], dtype=torch.int32, device="cuda")
    rc, o, fin = call_noalloc(fn, d, 3)
    assert rc == 0
    assert kda.noalloc_read_device_error() == 0
