"""The segment planner's timing model against the kernels it describes.

kda_chunk_fwd splits a long document's chain into segments when the chain
would take over 1.5 times the preparation; the decision rests on two measured
constants (kda_planner_model).  These tests time the kernels on GB300 and check
that each constant stays within a factor of the measurement, so that a faster
or slower kernel shows up here instead of silently skewing the choice."""
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda

pytestmark = pytest.mark.gpu
DEV = "cuda"
LOW, HIGH = 0.6, 1.6  # model / measurement must lie in [LOW, HIGH]


def kernel_ms(fn, name, reps=3):
    """Fastest of `reps` calls: the summed time of the launches named `name`."""
    best = None
    for _ in range(reps + 1):
        kda.profile_enable(True)
        kda.profile_collect()
        fn()
        torch.cuda.synchronize()
        marks = kda.profile_collect()
        kda.profile_enable(False)
        t = sum(ms for n, ms in marks if n == name)
        assert t > 0, marks
        best = t if best is None else min(best, t)
    return best


def test_prep_time_per_unit_matches_model():
    """Many short documents (H=32, T=16384, 2048-token documents): the standalone
    preparation kernel's time per (chunk, head) unit and SM."""
    T, H, n = 16384, 32, 8
    d = kda_synth.prefill_inputs(T, H, "bf16", seed=5, z_std=1.5, A_std=0.5, device=DEV)
    ms = kernel_ms(lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], n_seqs=n), "prep_tc")
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    measured = ms * 1e3 * n_sm / ((T // 64) * H)
    model = kda.planner_model()[0]
    assert LOW <= model / measured <= HIGH, f"prep: model {model} us/unit, measured {measured:.2f}"


def test_chain_time_per_chunk_matches_model():
    """The prefill's fused launch over one 8192-token document and 16 heads,
    whose time is set by its chains: the time per chunk of one chain."""
    T, H = 8192, 16
    d = kda_synth.prefill_inputs(T, H, "bf16", seed=6, z_std=1.5, A_std=0.5, device=DEV)
    ms = kernel_ms(lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"]), "fused_tc")
    measured = ms * 1e3 / (T // 64)
    model = kda.planner_model()[1]
    assert LOW <= model / measured <= HIGH, f"chain: model {model} us/chunk, measured {measured:.2f}"
