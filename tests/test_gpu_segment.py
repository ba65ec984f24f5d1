"""Parity of kda_segment_scan (CUDA, through the C ABI) with the fp64 oracle and
with the unsplit kda_chunk_fwd."""
import numpy as np
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, err_report, rel_fro, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"


def chunk_list(T, cu):
    """(tok, len, doc) of every 64-token chunk, documents cut separately."""
    cu = [0, T] if cu is None else [int(x) for x in cu]
    out = []
    for d in range(len(cu) - 1):
        t = cu[d]
        while t < cu[d + 1]:
            n = min(64, cu[d + 1] - t)
            out.append((t, n, d))
            t += n
    return out


def segment_token_ranges(T, cu, n_seg):
    ch = chunk_list(T, cu)
    out = []
    for a, b in kda_synth.segment_bounds(len(ch), n_seg):
        if a == b:
            out.append((None, None))
        else:
            out.append((ch[a][0], ch[b - 1][0] + ch[b - 1][1]))
    return out


def run(inp, n_seg):
    d = to_dev(inp, DEV)
    return kda.segment_scan(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], n_seg,
                            cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], return_pairs=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_seg", [1, 3, 7, 40])
def test_segment_scan_matches_oracle(dtype, n_seg):
    inp = kda_synth.prefill_inputs(1500, 2, dtype, seed=20 + n_seg, z_std=1.5, A_std=0.5, init_std=0.05)
    o, fin, pm, ps = run(inp, n_seg)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    init_state=inp["init_state"])
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref, "tokens", inp.get("cu_seqlens"))
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= to, f"o: {mo}"
    assert ef <= tf, f"final state: {mf}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pairs_match_oracle_pairs_non_vacuous(dtype):
    """Slow decay (z ~ N(-10,1), small beta): every segment's M carries a large
    share of the exit state, so split == unsplit is a real check."""
    T, H, n_seg = 1280, 2, 5
    inp = kda_synth.prefill_inputs(T, H, dtype, seed=30, z_mean=-10.0, beta_mean=-4.0, init_std=0.5)
    o, fin, pm, ps = run(inp, n_seg)
    torch.cuda.synchronize()
    rng = segment_token_ranges(T, None, n_seg)
    S_in = inp["init_state"][0].double().numpy()
    tol_pair = 1e-4 if dtype == "f32" else 1e-2
    for h in range(H):
        S = None
        for i, (a, b) in enumerate(rng):
            M_ref, St_ref = oracle.pair(inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], a, b, h,
                                        reset_at_begin=(a == 0), init_state=inp["init_state"])
            assert rel_fro(pm[h, i], M_ref) <= tol_pair
            assert rel_fro(ps[h, i], St_ref) <= tol_pair
            if i > 0:
                carried = np.linalg.norm(M_ref @ S) / np.linalg.norm(M_ref @ S + St_ref)
                assert carried > 0.1, f"segment {i}: carried share {carried:.3f}"
            S = St_ref if i == 0 else M_ref @ S + St_ref
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    init_state=inp["init_state"])
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref, "tokens", inp.get("cu_seqlens"))
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= to, f"o: {mo}"
    assert ef <= tf, f"final state: {mf}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_document_boundaries_inside_segments(dtype):
    lens = [300, 0, 450, 1, 190, 700]
    cu = kda_synth.cu_from_lengths(lens)
    inp = kda_synth.prefill_inputs(sum(lens), 2, dtype, seed=31, cu_seqlens=cu, init_std=0.05,
                                   z_mean=-3.0)
    o, fin, pm, ps = run(inp, 6)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    cu_seqlens=cu, init_state=inp["init_state"])
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref, "tokens", inp.get("cu_seqlens"))
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= to, f"o: {mo}"
    assert ef <= tf, f"final state: {mf}"


def oracle_sliced(d, o_gpu, fin_gpu, slice_len=16384):
    """The fp64 oracle over the whole token stream of device inputs d (one
    document), run in slices that resume from the previous slice's fp64 state
    (the same token-by-token arithmetic as one unsplit run), compared slice by
    slice with the GPU outputs.  Returns (o error, worst head's o error, final
    state error, worst head's state error)."""
    T, H = d["q"].shape[0], d["q"].shape[1]
    num = np.zeros(H)
    den = np.zeros(H)
    S = None
    for a in range(0, T, slice_len):
        b = min(T, a + slice_len)
        sl = lambda x: x[a:b].cpu()
        o_ref, S = oracle.recurrent(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["z"]), d["A"].cpu(),
                                    sl(d["beta"]), init_state=S)
        diff = o_gpu[a:b].double().cpu().numpy() - o_ref
        num += np.sum(diff * diff, axis=(0, 2))
        den += np.sum(o_ref * o_ref, axis=(0, 2))
    eo = float(np.sqrt(num.sum() / den.sum()))
    wo = float(np.max(np.sqrt(num / den)))
    fin = fin_gpu.double().cpu().numpy()
    ef = rel_fro(fin, S)
    wf = max(rel_fro(fin[0, h], S[0, h]) for h in range(H))
    return eo, wo, ef, wf


def test_segscan_1m_h8_full_size():
    """B=1, H=8, T=1,048,576, bf16, 148 segments, against one independent fp64
    oracle run over the whole stream (o and the final state at the stated
    tolerances); the pairs of sampled segments against the oracle's own pairs
    over the same token ranges; and equal to the unsplit chunkwise run."""
    w = kda_synth.WORKLOADS["segscan_1m_h8"]
    inp = kda_synth.workload_inputs("segscan_1m_h8", device=DEV)
    o, fin, pm, ps = kda.segment_scan(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                      w.n_segments, return_pairs=True)
    torch.cuda.synchronize()
    eo, wo, ef, wf = oracle_sliced(inp, o, fin)
    print(f"segscan_1m_h8 vs oracle: o {eo:.3e} (worst head {wo:.3e}), final state {ef:.3e} (worst head {wf:.3e})")
    assert eo <= TOL["bf16"][0], f"o rel err {eo:.3e} (worst head {wo:.3e})"
    assert ef <= TOL["bf16"][1], f"final state rel err {ef:.3e} (worst head {wf:.3e})"
    # sampled pairs against the oracle's pairs over the same tokens: segment 0
    # starts the document (the pair resets to (0, S~ from the zero init))
    rng = segment_token_ranges(w.T, None, w.n_segments)
    for h, i in [(0, 0), (3, 57), (5, 100), (7, 147)]:
        a, b = rng[i]
        sl = lambda x: x[a:b].cpu()
        M_ref, St_ref = oracle.pair(sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"].cpu(), sl(inp["beta"]),
                                    0, b - a, h, reset_at_begin=(a == 0))
        e_m, e_s = rel_fro(pm[h, i], M_ref), rel_fro(ps[h, i], St_ref)
        assert e_m <= 1e-2 and e_s <= 1e-2, f"pair ({h}, {i}): M {e_m:.3e}, S~ {e_s:.3e}"
    # the unsplit run: kda_chunk_fwd given a workspace with room for one segment
    # only keeps its single chain per head (its planner would take segments)
    del pm, ps
    one_doc = torch.tensor([0, w.T], dtype=torch.int32, device=DEV)
    assert kda.chunk_fwd_plan_segments(w.T, w.H, 1, varlen=True) >= 2
    ws = torch.empty(kda.segment_scan_workspace_size(w.T, w.H, 1, 1), dtype=torch.uint8, device=DEV)
    kda.profile_enable(True)
    kda.profile_collect()
    o_u, fin_u = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], cu_seqlens=one_doc,
                               workspace=ws)
    torch.cuda.synchronize()
    names = [n for n, _ in kda.profile_collect()]
    kda.profile_enable(False)
    assert "compose" not in names, names
    assert rel_fro(o, o_u) <= 1e-3 and rel_fro(fin, fin_u) <= 1e-3


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_148_segments_slow_decay_non_vacuous(dtype):
    """148 segments of two chunks each under slow decay (z ~ N(-10,1), small
    beta, large initial state): every segment's pair is compared with the
    oracle's pair over the same tokens, every composed entering state carries
    more than a tenth of the segment's exit state (the composition is not
    vacuous), and o and the final state match the oracle."""
    n_seg, H = 148, 2
    T = n_seg * 128
    inp = kda_synth.prefill_inputs(T, H, dtype, seed=41, z_mean=-10.0, beta_mean=-4.0, init_std=0.5)
    o, fin, pm, ps = run(inp, n_seg)
    torch.cuda.synchronize()
    k64, v64, z64, b64 = (inp[n].double().numpy() for n in ("k", "v", "z", "beta"))
    tol_pair = 1e-4 if dtype == "f32" else 1e-2
    pm, ps = pm.double().cpu().numpy(), ps.double().cpu().numpy()
    for h in range(H):
        S = None
        for i in range(n_seg):
            a, b = 128 * i, 128 * (i + 1)
            M_ref, St_ref = oracle.pair(k64, v64, z64, inp["A"], b64, a, b, h, reset_at_begin=(i == 0),
                                        init_state=inp["init_state"])
            e_m, e_s = rel_fro(pm[h, i], M_ref), rel_fro(ps[h, i], St_ref)
            assert e_m <= tol_pair and e_s <= tol_pair, f"pair ({h}, {i}): M {e_m:.3e}, S~ {e_s:.3e}"
            if i > 0:
                carried = np.linalg.norm(M_ref @ S) / np.linalg.norm(M_ref @ S + St_ref)
                assert carried > 0.1, f"segment {i}: carried share {carried:.3f}"
            S = St_ref if i == 0 else M_ref @ S + St_ref
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    init_state=inp["init_state"])
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref)
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= to, f"o: {mo}"
    assert ef <= tf, f"final state: {mf}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_scan_input_options(dtype):
    """The input options through kda_segment_scan (both phases prepare from the
    same records): unnormalised q, k and beta logits in, q scaled by d_k^-1/2,
    oracle on the prepared inputs."""
    inp = kda_synth.prefill_inputs(1500, 2, dtype, seed=77, z_std=1.5, A_std=0.5, init_std=0.05)
    g = torch.Generator().manual_seed(77)
    t = inp["q"].dtype
    inp["q"] = (inp["q"].float() * (0.5 + 2.5 * torch.rand((1500, 2, 1), generator=g))).to(t)
    inp["k"] = (inp["k"].float() * (0.5 + 2.5 * torch.rand((1500, 2, 1), generator=g))).to(t)
    inp["beta"] = torch.randn((1500, 2), generator=g)
    d = to_dev(inp, DEV)
    o, fin = kda.segment_scan(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], 5,
                              init_state=d["init_state"], qk_l2norm=True, beta_sigmoid=True, q_scale=True)
    torch.cuda.synchronize()
    qn, kn, bn = oracle.input_prep(inp["q"], inp["k"], inp["beta"], qk_l2norm=True, beta_sigmoid=True,
                                   q_scale=True)
    o_ref, f_ref = oracle.recurrent(qn, kn, inp["v"], inp["z"], inp["A"], bn, init_state=inp["init_state"])
    to, tf = TOL[dtype]
    eo, mo = err_report(o, o_ref, "tokens", inp.get("cu_seqlens"))
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= to, f"o: {mo}"
    assert ef <= tf, f"final state: {mf}"


def test_segment_scan_automatic_count():
    """n_segments = 0 takes kda_segment_scan_auto_segments' count (pairs of that
    many segments come back) and matches the oracle."""
    T, H = 6000, 2
    n = kda.segment_scan_auto_segments(T, H, 1)
    assert 1 <= n <= 64
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=42, z_std=1.5, A_std=0.5, init_std=0.05)
    o, fin, pm, ps = run(inp, 0)
    torch.cuda.synchronize()
    assert pm.shape[1] == n
    o_ref, f_ref = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                    init_state=inp["init_state"])
    eo, mo = err_report(o, o_ref)
    ef, mf = err_report(fin, f_ref, "state")
    assert eo <= TOL["bf16"][0], f"o: {mo}"
    assert ef <= TOL["bf16"][1], f"final state: {mf}"
