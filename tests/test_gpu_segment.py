"""Parity of kda_segment_scan (CUDA, through the C ABI) with the fp64 oracle and
with the unsplit kda_chunk_fwd."""
import numpy as np
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import oracle
from kda_testutil import TOL, rel_fro, to_dev

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
    assert rel_fro(o, o_ref) <= to and rel_fro(fin, f_ref) <= tf


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
    assert rel_fro(o, o_ref) <= to and rel_fro(fin, f_ref) <= tf


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
    assert rel_fro(o, o_ref) <= to and rel_fro(fin, f_ref) <= tf


def test_segscan_1m_h8_full_size():
    """B=1, H=8, T=1,048,576, bf16, 148 segments: equals the unsplit chunkwise run,
    and sampled segments rerun by the oracle from the composed entering state
    reproduce o and the next entering state."""
    w = kda_synth.WORKLOADS["segscan_1m_h8"]
    inp = kda_synth.workload_inputs("segscan_1m_h8", device=DEV)
    o, fin, pm, ps = kda.segment_scan(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                                      w.n_segments, return_pairs=True)
    # the unsplit run: a one-document cu_seqlens keeps kda_chunk_fwd on its single
    # chain per head (its planner segments only equal-length batches)
    one_doc = torch.tensor([0, w.T], dtype=torch.int32, device=DEV)
    assert kda.chunk_fwd_plan_segments(w.T, w.H, 1, varlen=True) == 0
    o_u, fin_u = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"], cu_seqlens=one_doc)
    torch.cuda.synchronize()
    assert rel_fro(o, o_u) <= 1e-3 and rel_fro(fin, fin_u) <= 1e-3
    T = w.T
    rng = segment_token_ranges(T, None, w.n_segments)
    for h, i in [(0, 0), (3, 57), (7, 147)]:
        a, b = rng[i]
        # entering state of segment i from the library's pairs, composed in fp64
        S = np.zeros((128, 128))
        for j in range(i):
            S = pm[h, j].double().cpu().numpy() @ S + ps[h, j].double().cpu().numpy()
        sl = lambda x: x[a:b, h:h + 1].cpu()
        o_ref, f_ref = oracle.recurrent(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]),
                                        inp["A"][h:h + 1].cpu(), inp["beta"][a:b, h:h + 1].cpu(),
                                        init_state=S[None, None])
        assert rel_fro(o[a:b, h:h + 1], o_ref) <= TOL["bf16"][0]
        S_next = pm[h, i].double().cpu().numpy() @ S + ps[h, i].double().cpu().numpy()
        assert rel_fro(S_next, f_ref[0, 0]) <= TOL["bf16"][1]
    # the last segment's exit state is the final state
    a, b = rng[-1]
    assert rel_fro(fin[0, 7], torch.from_numpy(S_next)) <= TOL["bf16"][1]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_scan_input_options(dtype):
    """The input options through kda_segment_scan (both phases prepare from the
    same records): unnormalised q, k and beta logits in, oracle on the prepared inputs."""
    inp = kda_synth.prefill_inputs(1500, 2, dtype, seed=77, z_std=1.5, A_std=0.5, init_std=0.05)
    g = torch.Generator().manual_seed(77)
    t = inp["q"].dtype
    inp["q"] = (inp["q"].float() * (0.5 + 2.5 * torch.rand((1500, 2, 1), generator=g))).to(t)
    inp["k"] = (inp["k"].float() * (0.5 + 2.5 * torch.rand((1500, 2, 1), generator=g))).to(t)
    inp["beta"] = torch.randn((1500, 2), generator=g)
    d = to_dev(inp, DEV)
    o, fin = kda.segment_scan(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], 5,
                              init_state=d["init_state"], qk_l2norm=True, beta_sigmoid=True)
    torch.cuda.synchronize()
    qn, kn, bn = oracle.input_prep(inp["q"], inp["k"], inp["beta"], qk_l2norm=True, beta_sigmoid=True)
    o_ref, f_ref = oracle.recurrent(qn, kn, inp["v"], inp["z"], inp["A"], bn, init_state=inp["init_state"])
    to, tf = TOL[dtype]
    assert rel_fro(o, o_ref) <= to and rel_fro(fin, f_ref) <= tf
