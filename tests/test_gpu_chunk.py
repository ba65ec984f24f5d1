"""Parity of kda_chunk_fwd (CUDA, through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, err_report, rel_fro, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_both(inp, n_seqs=1):
    """kda_chunk_fwd on the GPU and the oracle on the same inputs; returns
    (o, final state, oracle o, oracle final state, cu_seqlens used)."""
    d = to_dev(inp, DEV)
    o, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"],
                           cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], n_seqs=n_seqs)
    torch.cuda.synchronize()
    cu = inp["cu_seqlens"]
    if cu is None and n_seqs > 1:
        T = inp["q"].shape[0]
        cu = torch.arange(0, T + 1, T // n_seqs, dtype=torch.int32)
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    cu_seqlens=cu, init_state=inp["init_state"])
    return o, fin, o_ref, f_ref, cu


def check(o, fin, o_ref, f_ref, dtype, cu=None):
    """Whole-tensor tolerance on o and the final state; the messages also name
    the worst (sequence, head) block."""
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref, "tokens", cu)
    ef, mf = err_report(fin, f_ref, "state")
    assert np.isfinite(eo) and np.isfinite(ef)
    assert eo <= to, f"o: {mo} > {to}"
    assert ef <= tf, f"final_state: {mf} > {tf}"
    return eo, ef, mo, mf


def check_run(res, dtype):
    o, fin, o_ref, f_ref, cu = res
    return check(o, fin, o_ref, f_ref, dtype, cu)


def test_tiny_fp32_workload():
    """B=1, H=2, T=256, fp32, z~N(0,1), A=0, zero init, seed 0."""
    inp = kda_synth.workload_inputs("tiny_fp32")
    check_run(run_both(inp), "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 200, 333])
def test_ragged_lengths(dtype, T):
    inp = kda_synth.prefill_inputs(T, 3, dtype, seed=100 + T, z_std=1.5, A_std=0.5, init_std=0.05)
    check_run(run_both(inp), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slow_decay_carries_state_across_chunks(dtype):
    """z ~ N(-10, 1): g ~ -2e-4 per token, small beta: the state entering a chunk
    dominates its outputs, so the inter-chunk path is exercised (not washed out)."""
    inp = kda_synth.prefill_inputs(700, 2, dtype, seed=7, z_mean=-10.0, beta_mean=-4.0, init_std=0.5)
    check_run(run_both(inp), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_at_lower_bound(dtype):
    """z ~ N(8, 1): g close to g_min = -5 everywhere; the 16-token sub-tile factors
    reach e^{+-80} and must stay finite."""
    inp = kda_synth.prefill_inputs(256, 2, dtype, seed=8, z_mean=8.0, init_std=0.05)
    check_run(run_both(inp), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_documents_with_empty_and_short_docs(dtype):
    lens = [100, 0, 1, 64, 130, 0, 77]
    cu = kda_synth.cu_from_lengths(lens)
    inp = kda_synth.prefill_inputs(sum(lens), 2, dtype, seed=9, cu_seqlens=cu, init_std=0.05)
    check_run(run_both(inp), dtype)


def test_equal_length_batch_without_cu_seqlens():
    inp = kda_synth.prefill_inputs(4 * 96, 2, "bf16", seed=10, init_std=0.05, n_init=4)
    check_run(run_both(inp, n_seqs=4), "bf16")


def test_prefill_h16_t8k_full_size():
    """Full size prefill: B=1, H=16, T=8192, bf16, z~N(0,1.5), A~N(0,0.5)."""
    inp = kda_synth.workload_inputs("prefill_h16_t8k")
    eo, ef, mo, mf = check_run(run_both(inp), "bf16")
    print(f"prefill_h16_t8k: o {mo}; final_state {mf}")


def test_varlen_32k_h32_full_size():
    inp = kda_synth.workload_inputs("varlen_32k_h32")
    eo, ef, mo, mf = check_run(run_both(inp), "bf16")
    print(f"varlen_32k_h32: o {mo}; final_state {mf}")


def test_bitwise_deterministic():
    inp = to_dev(kda_synth.prefill_inputs(1000, 4, "bf16", seed=11, init_std=0.05), DEV)
    a = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], init_state=inp["init_state"])
    b = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], init_state=inp["init_state"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_linearity_in_values_and_initial_state():
    """o and S are linear in (V, S0) for fixed q, k, z, beta."""
    base = kda_synth.prefill_inputs(300, 2, "f32", seed=12, init_std=0.1)
    other = kda_synth.prefill_inputs(300, 2, "f32", seed=13, init_std=0.1)
    d = to_dev(base, DEV)
    v2, s2 = other["v"].to(DEV), other["init_state"].to(DEV)
    f = lambda v, s: kda.chunk_fwd(d["q"], d["k"], v, d["z"], d["A"], d["beta"], init_state=s)
    o1, f1 = f(d["v"], d["init_state"])
    o2, f2 = f(v2, s2)
    o3, f3 = f(d["v"] + v2, d["init_state"] + s2)
    assert rel_fro(o3, o1 + o2) < 1e-5 and rel_fro(f3, f1 + f2) < 1e-5


def test_resume_from_final_state():
    inp = kda_synth.prefill_inputs(640, 2, "f32", seed=14, init_std=0.1)
    d = to_dev(inp, DEV)
    o, f = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], init_state=d["init_state"])
    t = 192
    sl = lambda x, a, b: x[a:b].contiguous()
    oa, fa = kda.chunk_fwd(*(sl(d[n], 0, t) for n in ("q", "k", "v", "z")), d["A"], sl(d["beta"], 0, t),
                           init_state=d["init_state"])
    ob, fb = kda.chunk_fwd(*(sl(d[n], t, 640) for n in ("q", "k", "v", "z")), d["A"], sl(d["beta"], t, 640),
                           init_state=fa)
    assert rel_fro(torch.cat([oa, ob]), o) < 1e-5 and rel_fro(fb, f) < 1e-5


def test_invalid_cu_seqlens_is_reported_on_device():
    inp = to_dev(kda_synth.prefill_inputs(256, 1, "bf16", seed=15), DEV)
    bad = torch.tensor([0, 200, 100, 256], dtype=torch.int32, device=DEV)  # decreasing
    ws = torch.empty(kda.chunk_fwd_workspace_size(256, 1, 3), dtype=torch.uint8, device=DEV)
    o = torch.full_like(inp["q"], 7.0)
    fin_sentinel = None
    kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], cu_seqlens=bad,
                  workspace=ws, out=o, output_final_state=False)
    assert kda.read_device_error(ws) & 1
    assert torch.all(o == 7.0)  # nothing written


@pytest.mark.parametrize("T,H,n_seqs", [(8192, 1, 1), (16384, 1, 2)])
def test_planner_segmented_path(T, H, n_seqs):
    """Long documents over one head: kda_chunk_fwd cuts the chunk list into
    segments by itself (kda_chunk_fwd_plan_segments > 0), and still matches the
    oracle, across the document boundary of the two-document batch too."""
    assert kda.chunk_fwd_plan_segments(T, H, n_seqs) >= 2
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=900 + T, z_std=1.0, init_std=0.05, n_init=n_seqs)
    check_run(run_both(inp, n_seqs=n_seqs), "bf16")


@pytest.mark.parametrize("lens,H", [([128, 12000, 352], 2), ([8192, 64, 1, 4096], 1)])
def test_planner_segments_packed_long_document(lens, H):
    """A packed batch whose longest document would leave one chain setting the
    time: kda_chunk_fwd reads the document lengths, takes the segmented path
    (the composition kernel runs) and matches the oracle, state resets at every
    boundary included; a batch of the same total in short documents keeps one
    chain per (document, head)."""
    T = sum(lens)
    assert kda.chunk_fwd_plan_segments(T, H, len(lens), varlen=True) >= 2
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=950 + T, z_std=1.0, A_std=0.5, init_std=0.05,
                                   cu_seqlens=kda_synth.cu_from_lengths(lens))
    kda.profile_enable(True)
    kda.profile_collect()
    res = run_both(inp, n_seqs=len(lens))
    names = [n for n, _ in kda.profile_collect()]
    kda.profile_enable(False)
    assert "compose" in names, names
    check_run(res, "bf16")
    # the same total in documents of at most 512 tokens: no segments
    short = [512] * (T // 512) + ([T % 512] if T % 512 else [])
    d = to_dev(kda_synth.prefill_inputs(T, H, "bf16", seed=951, cu_seqlens=kda_synth.cu_from_lengths(short)), DEV)
    kda.profile_enable(True)
    kda.profile_collect()
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    names = [n for n, _ in kda.profile_collect()]
    kda.profile_enable(False)
    assert "compose" not in names, names


def raw_inputs(T, H, dtype, seed, n_seqs=1):
    """Prefill inputs with unnormalised q, k (each row scaled by 0.5 .. 3) and beta logits."""
    inp = kda_synth.prefill_inputs(T, H, dtype, seed=seed, z_std=1.0, init_std=0.05, n_init=n_seqs)
    g = torch.Generator().manual_seed(seed)
    t = inp["q"].dtype
    inp["q"] = (inp["q"].float() * (0.5 + 2.5 * torch.rand((T, H, 1), generator=g))).to(t)
    inp["k"] = (inp["k"].float() * (0.5 + 2.5 * torch.rand((T, H, 1), generator=g))).to(t)
    inp["beta"] = torch.randn((T, H), generator=g)
    return inp


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,H,flags", [(333, 3, (True, True, False)), (333, 3, (True, False, False)),
                                       (333, 3, (False, True, False)), (333, 3, (False, False, True)),
                                       (333, 3, (True, True, True)), (2048, 24, (True, True, True)),
                                       (8192, 1, (True, True, True))])
def test_input_options(dtype, T, H, flags):
    """KDA_FLAG_QK_L2NORM / KDA_FLAG_BETA_SIGMOID / KDA_FLAG_Q_SCALE against the
    oracle on the prepared inputs; the shapes take the fused launch (H=3), the
    three-kernel path (H=24: 48 chains) and, in bf16, the automatic segments
    (H=1, T=8192)."""
    l2, sig, qs = flags
    inp = raw_inputs(T, H, dtype, seed=300 + T + H)
    d = to_dev(inp, DEV)
    o, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], init_state=d["init_state"],
                           qk_l2norm=l2, beta_sigmoid=sig, q_scale=qs)
    torch.cuda.synchronize()
    qn, kn, bn = oracle.input_prep(inp["q"], inp["k"], inp["beta"], qk_l2norm=l2, beta_sigmoid=sig, q_scale=qs)
    o_ref, f_ref = oracle.recurrent(qn, kn, inp["v"], inp["z"], inp["A"], bn, init_state=inp["init_state"])
    check(o, fin, o_ref, f_ref, dtype)



def ckpt_reference(inp, cu, positions):
    """State of each document after its first p tokens: the oracle's final state
    on that prefix (the checkpoints' plain definition)."""
    out = {}
    for n, ps in positions.items():
        a = int(cu[n])
        for p in ps:
            sl = lambda x: x[a:a + p]
            init = None if inp["init_state"] is None else inp["init_state"][n:n + 1]
            _, f = oracle.recurrent(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"],
                                    sl(inp["beta"]), init_state=init)
            out[(n, p)] = f[0]
    return out


@pytest.mark.parametrize("dtype,T,H,docs,interval", [
    ("f32", 1000, 3, None, 256), ("bf16", 1000, 3, None, 256),
    ("bf16", 1000, 2, [700, 300], 128), ("f32", 1000, 2, [700, 300], 128),
    ("bf16", 8192, 1, None, 512), ("bf16", 6400, 16, [320] * 20, 128)])
def test_checkpoints(dtype, T, H, docs, interval):
    """kda_chunk_fwd_ckpt: every marked (document, aligned position) page holds
    the oracle's state after that prefix; skipped and out-of-document entries
    leave their pages untouched; o and the final state are unchanged.  The
    bf16 cases with few chains run the fused launch; 8192 x 1 takes the automatic
    segments (the state comes from phase 3); 20 documents x 16 heads take the
    scan blocks that form the outputs themselves."""
    cu = torch.tensor([0] + list(np.cumsum(docs)), dtype=torch.int32) if docs else None
    n = 1 if docs is None else len(docs)
    inp = kda_synth.prefill_inputs(T, H, dtype, seed=500 + T + H, z_std=0.5, init_std=0.05,
                                   cu_seqlens=cu, n_init=n)
    lens = docs or [T]
    per_seq = max(lens) // interval + 1  # includes one position past every document's end
    slot = torch.full((n, per_seq), -1, dtype=torch.int32)
    want, nxt = {}, 0
    for d in range(n):
        for j in range(per_seq):
            if j % 3 == 1:
                continue  # skipped on purpose
            slot[d, j] = nxt
            if (j + 1) * interval <= lens[d]:
                want[(d, (j + 1) * interval)] = nxt
            nxt += 1
    ck = torch.full((nxt, H, 128, 128), float("nan"), device=DEV)
    d_ = to_dev(inp, DEV)
    o, fin = kda.chunk_fwd_ckpt(d_["q"], d_["k"], d_["v"], d_["z"], d_["A"], d_["beta"], interval, slot.to(DEV), ck,
                                cu_seqlens=d_["cu_seqlens"], init_state=d_["init_state"], n_seqs=n)
    torch.cuda.synchronize()
    positions = {}
    for (d, p) in want:
        positions.setdefault(d, []).append(p)
    ref = ckpt_reference(inp, [0] + list(np.cumsum(lens)), positions)
    to, tf = TOL[dtype]
    for key, s_idx in want.items():
        e = rel_fro(ck[s_idx], ref[key])
        assert e <= tf, f"checkpoint {key}: rel err {e:.3e}"
    written = set(want.values())
    for s_idx in range(nxt):
        if s_idx not in written:
            assert torch.isnan(ck[s_idx]).all(), f"page {s_idx} written"
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    cu_seqlens=cu, init_state=inp["init_state"])
    check(o, fin, o_ref, f_ref, dtype, cu)
