"""Parity of kda_decode_step (CUDA, through the C ABI) with the fp64 oracle."""
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, err_report, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


def empty_cache(N, W, H, dtype):
    t = kda_synth.TORCH_DTYPE[dtype]
    z = lambda: torch.zeros((N, W - 1, H, 128), dtype=t, device=DEV)
    return (z(), z(), z(), torch.zeros((N, W - 1, H, 128), device=DEV),
            torch.zeros((N, W - 1, H), device=DEV))


def run_steps(N, H, W, dtype, steps, seed, sample=None, A_std=0.5, z_mean=0.0, nacc_fill=None):
    """Decode steps on the GPU against the oracle's step over the same windows
    (all sequences unless `sample` names some); o and the state after every step
    at the stated tolerances, the cache exactly.  nacc_fill replaces every
    accepted count after the first step."""
    state = kda_synth.decode_state(N, H, seed, std=0.05, device=DEV)
    A = kda_synth.decode_A(H, seed, A_std=A_std, device=DEV)
    cache = empty_cache(N, W, H, dtype)
    ref_state = state.cpu()
    ref_cache = tuple(c.cpu() for c in cache)
    idx = torch.arange(N) if sample is None else torch.tensor(sample)
    ref_state = ref_state[idx]
    ref_cache = tuple(c[idx] for c in ref_cache)
    tol_o, tol_s = (1e-4, 1e-4) if dtype == "f32" else TOL["bf16"]
    for step in range(steps):
        w = kda_synth.decode_window(N, W, H, step, seed, dtype, z_std=1.5, z_mean=z_mean, device=DEV)
        nacc = None if step == 0 else w["num_accepted"]
        if nacc is not None and nacc_fill is not None:
            nacc = torch.full_like(nacc, nacc_fill)
        o = kda.decode_step(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, cache, num_accepted=nacc)
        torch.cuda.synchronize()
        sel = lambda x: x.cpu()[idx]
        o_ref, ref_state, ref_cache = oracle.decode_step(
            ref_state, sel(w["q"]), sel(w["k"]), sel(w["v"]), sel(w["z"]), sel(w["beta"]), A.cpu(),
            *ref_cache, num_accepted=None if nacc is None else sel(nacc))
        eo, mo = err_report(o.cpu()[idx], o_ref, "decode")
        es, ms = err_report(state.cpu()[idx], ref_state, "state")
        assert eo <= tol_o, f"step {step}: o {mo}"
        assert es <= tol_s, f"step {step}: state {ms}"
        for c, rc in zip(cache, ref_cache):
            assert torch.equal(c.cpu()[idx].double(), torch.from_numpy(rc)), f"step {step}: cache"
    return state


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_small(dtype):
    run_steps(N=7, H=3, W=5, dtype=dtype, steps=4, seed=40)


@pytest.mark.parametrize("W", [1, 2, 8])
def test_decode_window_sizes(W):
    run_steps(N=5, H=2, W=W, dtype="f32", steps=3, seed=41 + W)


def test_decode_mtp_b256_h96_full_size():
    """N=256, H=96, W=5 (1 + 4 drafts), fp32: full-size launch, every sequence
    and head checked against the oracle over three steps."""
    run_steps(N=256, H=96, W=5, dtype="f32", steps=3, seed=5, A_std=0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_gate_at_bound_longest_window(dtype):
    """The numeric extreme of the lazy per-row decay: the gate at its lower
    bound (z ~ N(8, 1), g close to -5 on every channel), the largest window
    (W = 8) and every draft accepted (num_accepted = 7), so one step runs 15
    tokens and the row scale falls to about e^-75 while k / s_t grows to e^75."""
    run_steps(N=6, H=3, W=8, dtype=dtype, steps=3, seed=46, z_mean=8.0, nacc_fill=7)


def test_num_accepted_out_of_range_sets_error_and_skips():
    N, H, W = 4, 2, 5
    state = kda_synth.decode_state(N, H, 50, device=DEV)
    before = state.clone()
    A = torch.zeros(H, device=DEV)
    cache = empty_cache(N, W, H, "f32")
    w = kda_synth.decode_window(N, W, H, 0, 50, "f32", device=DEV)
    nacc = torch.tensor([0, 9, -1, 4], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.decode_step(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, cache, num_accepted=nacc,
                    error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2
    assert torch.equal(state[1], before[1]) and torch.equal(state[2], before[2])
    assert not torch.equal(state[0], before[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("q_scale", [False, True])
def test_decode_input_options(dtype, q_scale):
    """KDA_FLAG_QK_L2NORM | KDA_FLAG_BETA_SIGMOID (and KDA_FLAG_Q_SCALE):
    unnormalised q, k and beta logits in; the oracle runs on the prepared inputs
    (its input_prep), and the cache keeps the drafts' inputs as given."""
    N, H, W, seed = 6, 3, 5, 61
    g = torch.Generator().manual_seed(seed)
    state = kda_synth.decode_state(N, H, seed, std=0.05, device=DEV)
    A = kda_synth.decode_A(H, seed, A_std=0.5, device=DEV)
    cache = empty_cache(N, W, H, dtype)
    ref_state = state.cpu()
    raw_cache = tuple(c.cpu() for c in cache)
    tol_o, tol_s = (1e-4, 1e-4) if dtype == "f32" else TOL["bf16"]
    t = kda_synth.TORCH_DTYPE[dtype]
    for step in range(3):
        w = kda_synth.decode_window(N, W, H, step, seed, dtype, z_std=1.5)
        qr = (w["q"].float() * (0.5 + 2.5 * torch.rand((N, W, H, 1), generator=g))).to(t)
        kr = (w["k"].float() * (0.5 + 2.5 * torch.rand((N, W, H, 1), generator=g))).to(t)
        br = torch.randn((N, W, H), generator=g)
        nacc = None if step == 0 else w["num_accepted"]
        dev = lambda x: x.to(DEV)
        o = kda.decode_step(state, dev(qr), dev(kr), dev(w["v"]), dev(w["z"]), dev(br), A, cache,
                            num_accepted=None if nacc is None else dev(nacc), qk_l2norm=True, beta_sigmoid=True,
                            q_scale=q_scale)
        torch.cuda.synchronize()
        qn, kn, bn = oracle.input_prep(qr, kr, br, qk_l2norm=True, beta_sigmoid=True, q_scale=q_scale)
        cqn, ckn, cbn = oracle.input_prep(raw_cache[0], raw_cache[1], raw_cache[4], qk_l2norm=True, beta_sigmoid=True,
                                          q_scale=q_scale)
        o_ref, ref_state, _ = oracle.decode_step(ref_state, qn, kn, w["v"], w["z"], bn, A.cpu(), cqn, ckn,
                                                 raw_cache[2], raw_cache[3], cbn, num_accepted=nacc)
        eo, mo = err_report(o.cpu(), o_ref, "decode")
        es, ms = err_report(state.cpu(), ref_state, "state")
        assert eo <= tol_o, f"step {step}: o {mo}"
        assert es <= tol_s, f"step {step}: state {ms}"
        # the new drafts' inputs, as given, become the cache
        raw_cache = (qr[:, 1:].contiguous(), kr[:, 1:].contiguous(), w["v"][:, 1:].contiguous(),
                     w["z"][:, 1:].contiguous(), br[:, 1:].contiguous())
        for c, rc in zip(cache, raw_cache):
            assert torch.equal(c.cpu(), rc.to(c.dtype)), f"step {step}: cache"


# ---------------------------------------------------------------- fused step

FUSED_OPTS = dict(qk_l2norm=True, beta_sigmoid=True, conv_silu=True)


def run_fused_steps(N, H, W, dtype, steps, seed, sample=None, opts=FUSED_OPTS, eps=1e-6, scale_qk=1.0):
    """kda_decode_step_fused against oracle.decode_step_fused over several steps with
    replay: outputs and states within the tolerance; the cache and the convolution
    state (pre-convolution inputs) exact."""
    state = kda_synth.decode_state(N, H, seed, std=0.05, device=DEV)
    A = kda_synth.decode_A(H, seed, A_std=0.5, device=DEV)
    prm = kda_synth.decode_fused_params(H, seed, device=DEV)
    cs = kda_synth.decode_conv_state(N, H, seed, device=DEV)
    cache = empty_cache(N, W, H, dtype)
    idx = torch.arange(N) if sample is None else torch.tensor(sample)
    ref_state, ref_cs = state.cpu()[idx], cs.cpu()[idx]
    if scale_qk != 1.0:
        ref_cs[:, :, :2] *= scale_qk
        cs[:, :, :2] *= scale_qk
    ref_cache = tuple(c.cpu()[idx] for c in cache)
    tol_o, tol_s = (1e-4, 1e-4) if dtype == "f32" else TOL["bf16"]
    t = kda_synth.TORCH_DTYPE[dtype]
    for step in range(steps):
        w = kda_synth.decode_fused_window(N, W, H, step, seed, dtype, z_std=1.5, device=DEV)
        if scale_qk != 1.0:
            w["q"] = (w["q"].float() * scale_qk).to(t)
            w["k"] = (w["k"].float() * scale_qk).to(t)
        if not opts.get("beta_sigmoid"):
            w["beta"] = torch.sigmoid(w["beta"])
        nacc = None if step == 0 else w["num_accepted"]
        o = kda.decode_step_fused(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, prm["conv_w"], cs,
                                  w["o_gate"], prm["o_norm_w"], cache, num_accepted=nacc, o_norm_eps=eps,
                                  **opts)
        torch.cuda.synchronize()
        sel = lambda x: x.cpu()[idx]
        o_ref, ref_state, ref_cache, ref_cs = oracle.decode_step_fused(
            ref_state, sel(w["q"]), sel(w["k"]), sel(w["v"]), sel(w["z"]), sel(w["beta"]), A.cpu(),
            prm["conv_w"].cpu(), ref_cs, sel(w["o_gate"]), prm["o_norm_w"].cpu(), eps, *ref_cache,
            num_accepted=None if nacc is None else sel(nacc), **opts)
        eo, mo = err_report(o.cpu()[idx], o_ref, "decode")
        es, ms = err_report(state.cpu()[idx], ref_state, "state")
        assert eo <= tol_o, f"step {step}: o {mo}"
        assert es <= tol_s, f"step {step}: state {ms}"
        assert torch.equal(cs.cpu()[idx].double(), torch.from_numpy(ref_cs)), f"step {step}: conv state"
        for c, rc in zip(cache, ref_cache):
            assert torch.equal(c.cpu()[idx].double(), torch.from_numpy(rc)), f"step {step}: cache"
    return o


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_fused_steps_small(dtype):
    run_fused_steps(N=7, H=3, W=5, dtype=dtype, steps=4, seed=70)


@pytest.mark.parametrize("W", [1, 2, 8])
def test_decode_fused_window_sizes(W):
    run_fused_steps(N=5, H=2, W=W, dtype="f32", steps=3, seed=71 + W)


def test_decode_fused_without_options():
    """No flags: plain convolution, beta as given, q and k not normalised (the inputs are
    scaled down so that the convolved keys keep the delta rule contractive)."""
    run_fused_steps(N=6, H=2, W=5, dtype="f32", steps=3, seed=75, opts={}, scale_qk=0.125)


def test_decode_fused_l2norm_only():
    run_fused_steps(N=6, H=2, W=5, dtype="f32", steps=3, seed=76, opts=dict(qk_l2norm=True, beta_sigmoid=True))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_fused_with_q_scale(dtype):
    run_fused_steps(N=6, H=2, W=5, dtype=dtype, steps=3, seed=78, opts=dict(FUSED_OPTS, q_scale=True))


def test_decode_fused_b256_h96_full_size():
    """N=256, H=96, W=5, fp32, the full-size fused launch; every sequence and head against the oracle."""
    run_fused_steps(N=256, H=96, W=5, dtype="f32", steps=2, seed=5)


def test_decode_fused_out_of_range_keeps_sequence():
    N, H, W = 4, 2, 5
    state = kda_synth.decode_state(N, H, 77, device=DEV)
    prm = kda_synth.decode_fused_params(H, 77, device=DEV)
    cs = kda_synth.decode_conv_state(N, H, 77, device=DEV)
    before, cs_before = state.clone(), cs.clone()
    A = torch.zeros(H, device=DEV)
    cache = empty_cache(N, W, H, "f32")
    w = kda_synth.decode_fused_window(N, W, H, 0, 77, "f32", device=DEV)
    nacc = torch.tensor([0, 9, -1, 4], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.decode_step_fused(state, w["q"], w["k"], w["v"], w["z"], w["beta"], A, prm["conv_w"], cs, w["o_gate"],
                          prm["o_norm_w"], cache, num_accepted=nacc, error_word=err, **FUSED_OPTS)
    torch.cuda.synchronize()
    assert int(err.item()) & 2
    for b in (1, 2):
        assert torch.equal(state[b], before[b]) and torch.equal(cs[b], cs_before[b])
    assert not torch.equal(state[0], before[0]) and not torch.equal(cs[3], cs_before[3])


def test_decode_fused_deterministic():
    outs = []
    for _ in range(2):
        N, H, W = 8, 4, 5
        outs.append(run_fused_steps(N=N, H=H, W=W, dtype="f32", steps=2, seed=79).cpu())
    assert torch.equal(outs[0], outs[1])


def test_decode_fused_unit_conv_matches_plain_step():
    """Cross-path check: with the convolution a unit impulse on the current token and no
    options, the fused step feeds the recurrence the same values as the plain step, so
    the states and caches agree bit for bit, and its outputs are the plain outputs through
    the gated per-head RMS norm."""
    N, H, W, seed = 16, 4, 5, 81
    state_a = kda_synth.decode_state(N, H, seed, device=DEV)
    state_b = state_a.clone()
    A = kda_synth.decode_A(H, seed, A_std=0.5, device=DEV)
    cache_a, cache_b = empty_cache(N, W, H, "f32"), empty_cache(N, W, H, "f32")
    conv_w = torch.zeros((3, H, 128, 4), device=DEV)
    conv_w[..., 3] = 1.0
    cs = torch.zeros((N, H, 3, 3, 128), device=DEV)
    norm_w = kda_synth.decode_fused_params(H, seed, device=DEV)["o_norm_w"]
    for step in range(3):
        w = kda_synth.decode_window(N, W, H, step, seed, "f32", z_std=1.5, device=DEV)
        gate = torch.randn((N, W, H, 128), generator=torch.Generator().manual_seed(step)).to(DEV)
        nacc = None if step == 0 else w["num_accepted"]
        args = [w[n] for n in ("q", "k", "v", "z", "beta")]
        o_a = kda.decode_step(state_a, *args, A, cache_a, num_accepted=nacc)
        o_b = kda.decode_step_fused(state_b, *args, A, conv_w, cs, gate, norm_w, cache_b, num_accepted=nacc,
                                    o_norm_eps=1e-6)
        torch.cuda.synchronize()
        assert torch.equal(state_a, state_b), f"step {step}: state"
        for ca, cb in zip(cache_a, cache_b):
            assert torch.equal(ca, cb), f"step {step}: cache"
        oa = o_a.double().cpu()
        ref = oa / torch.sqrt(oa.pow(2).mean(-1, keepdim=True) + 1e-6) * norm_w.double().cpu() \
            * torch.sigmoid(gate.double().cpu())
        assert rel_fro(o_b.cpu(), ref) <= 1e-5, f"step {step}: o"
