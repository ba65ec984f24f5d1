"""The bounded waits give up cleanly on the GPU.

A wait that runs out of its clock budget must record KDA_DEVERR_TIMEOUT, let its
block stop (its own copies and tensor-core work finish, its TMEM is freed) and
return, leaving the CUDA context usable.  The tests shorten the budget of the
waits on flags raised by other blocks (the fused prefill's record-ready flags)
and of the decode's copy waits with kda_set_wait_budget, so that those waits
run out on flags that are not yet set and copies that have not yet landed; no
kernel is changed and nothing faults.  The same inputs then run again under the
default budget and must match the oracle."""
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, err_report, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEVERR_TIMEOUT = 4


def test_fused_prefill_flag_wait_times_out_then_recovers():
    """The bench shape (H=16, T=8192, bf16) takes the single fused launch, whose
    chain blocks wait for records other blocks publish; with a one-cycle budget a
    wait on a record not yet published gives up."""
    inp = kda_synth.workload_inputs("prefill_h16_t8k")
    d = to_dev(inp, DEV)
    T, H = inp["q"].shape[0], inp["q"].shape[1]
    assert kda.chunk_fwd_plan_segments(T, H, 1) == 0
    ws = torch.empty(kda.chunk_fwd_workspace_size(T, H, 1), dtype=torch.uint8, device=DEV)
    code = 0
    old = kda.set_wait_budget(1)
    try:
        for _ in range(3):  # the flag waits run out on any record not yet published
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], workspace=ws)
            code = kda.read_device_error(ws)
            if code & DEVERR_TIMEOUT:
                break
    finally:
        kda.set_wait_budget(old)
    assert code & DEVERR_TIMEOUT, f"no wait timed out (error word {code})"
    # the context is still usable and the default budget gives the right answer
    o, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], workspace=ws)
    assert kda.read_device_error(ws) == 0
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"])
    eo, mo = err_report(o, o_ref)
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= TOL["bf16"][0], f"o: {mo}"
    assert ef <= TOL["bf16"][1], f"final state: {mf}"


@pytest.mark.parametrize("fused", [False, True])
def test_decode_copy_wait_times_out_then_recovers(fused):
    """With a one-cycle budget the decode's first wait for an item's state copy
    gives up; the block lets the copy land and stops.  Items processed before the
    timeout may have been updated, so the rerun starts from a saved state."""
    N, H, W, seed = 64, 4, 5, 90
    state0 = kda_synth.decode_state(N, H, seed, device=DEV)
    A = kda_synth.decode_A(H, seed, A_std=0.5, device=DEV)
    z = lambda: torch.zeros((N, W - 1, H, 128), device=DEV)
    if fused:
        prm = kda_synth.decode_fused_params(H, seed, device=DEV)
        cs0 = kda_synth.decode_conv_state(N, H, seed, device=DEV)
        w = kda_synth.decode_fused_window(N, W, H, 0, seed, "f32", device=DEV)
    else:
        w = kda_synth.decode_window(N, W, H, 0, seed, "f32", device=DEV)

    def step(state, cs, err):
        cache = (z(), z(), z(), z(), torch.zeros((N, W - 1, H), device=DEV))
        if fused:
            return kda.decode_step_fused(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, prm["conv_w"], cs,
                                         w["o_gate"], prm["o_norm_w"], cache, error_word=err, qk_l2norm=True,
                                         beta_sigmoid=True, conv_silu=True)
        return kda.decode_step(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, cache, error_word=err)

    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    old = kda.set_wait_budget(1)
    try:
        step(state0.clone(), cs0.clone() if fused else None, err)
        torch.cuda.synchronize()
    finally:
        kda.set_wait_budget(old)
    assert int(err.item()) & DEVERR_TIMEOUT
    err.zero_()
    state = state0.clone()
    cs = cs0.clone() if fused else None
    o = step(state, cs, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    cache0 = tuple(torch.zeros((N, W - 1, H, 128)) for _ in range(4)) + (torch.zeros((N, W - 1, H)),)
    args = [w[n].cpu() for n in ("q", "k", "v", "z", "beta")]
    if fused:
        o_ref, s_ref, _, _ = oracle.decode_step_fused(state0.cpu(), *args, A.cpu(), prm["conv_w"].cpu(), cs0.cpu(),
                                                      w["o_gate"].cpu(), prm["o_norm_w"].cpu(), 1e-6, *cache0,
                                                      qk_l2norm=True, beta_sigmoid=True, conv_silu=True)
    else:
        o_ref, s_ref, _ = oracle.decode_step(state0.cpu(), *args, A.cpu(), *cache0)
    eo, mo = err_report(o, o_ref, "decode")
    es, ms = err_report(state, s_ref, "state")
    assert eo <= 1e-4, f"o: {mo}"
    assert es <= 1e-4, f"state: {ms}"
