"""Guard bytes around every buffer the library writes.

No memory checker is available on this pool, so each output, state, cache,
pair array and workspace is placed inside a larger allocation whose bytes
before and after it hold a known pattern.  A call must leave that pattern and
its inputs untouched, and must give bit for bit the result of the same call on
plain buffers (the kernels are deterministic).  The shapes are ragged on
purpose: documents of 1 and 63 tokens, chunk tails, a segment split that does
not divide the chunks, decode windows with replays.  Every path the calls
choose between is taken: the fused launch and its input-option
instantiation, the three-kernel path of many chains, the automatic segments,
the fp32 path, the checkpoint pages, the segment scan with its pairs, and
both decode steps."""
import pytest
import torch

import kda_synth
import linear_attention_serving_gb300 as kda
import linear_attention_serving_gb300.kda as kmod
from kda_testutil import to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096  # bytes of pattern on each side of a buffer
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside an allocation with GUARD pattern
    bytes on each side (its own bytes start as the pattern too, unless `init`
    is given)."""

    def __init__(self, shape, dtype, init=None):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= int(s)
        g = GUARD // es
        self.buf = torch.empty(n + 2 * g, dtype=dtype, device=DEV)
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[g:g + n].view(tuple(shape))
        if init is not None:
            self.t.copy_(init)

    def intact(self) -> bool:
        raw = self.buf.view(torch.uint8)
        return bool((raw[:GUARD] == PATTERN).all()) and bool((raw[-GUARD:] == PATTERN).all())


def _inputs_unchanged(before: dict, after: dict):
    for name, t in before.items():
        if t is not None:
            assert torch.equal(t, after[name]), f"input {name} was written"


def _snapshot(d: dict) -> dict:
    return {k: (v.clone() if isinstance(v, torch.Tensor) else None) for k, v in d.items()}


def _prefill_case(name):
    if name == "fused":  # few chains: the single cooperative launch
        lens, H, dtype = [1, 63, 65, 200], 3, "bf16"
    elif name == "many_chains":  # too many chains for the fused launch
        lens, H, dtype = kda_synth.draw_doc_lengths(2600, 1, 140, seed=77), 2, "bf16"
    elif name == "segmented":  # one long document: the planner takes segments
        lens, H, dtype = [8192 + 37], 1, "bf16"
    else:  # fp32 inputs: the exact CUDA-core path
        lens, H, dtype = [5, 130], 2, "f32"
    cu = kda_synth.cu_from_lengths(lens)
    T = int(cu[-1])
    inp = kda_synth.prefill_inputs(T, H, dtype, seed=len(lens) + H, cu_seqlens=cu, init_std=0.05)
    return inp, len(lens)


@pytest.mark.parametrize("path", ["fused", "many_chains", "segmented", "fp32"])
def test_chunk_fwd_writes_only_its_buffers(path):
    inp, n = _prefill_case(path)
    d = to_dev(inp, DEV)
    T, H, Dm = d["q"].shape
    if path == "segmented":
        assert kda.chunk_fwd_plan_segments(T, H, n, varlen=True) > 0
    before = _snapshot(d)
    ws_bytes = kda.chunk_fwd_workspace_size(T, H, n, d["q"].dtype)
    o = Guarded(d["q"].shape, d["q"].dtype)
    fin = Guarded((n, H, Dm, Dm), torch.float32)
    ws = Guarded((ws_bytes,), torch.uint8)
    lib = kda.load()
    p = kmod._p
    rc = lib.kda_chunk_fwd(p(d["q"]), p(d["k"]), p(d["v"]), p(d["z"]), p(d["A"]), p(d["beta"]),
                           p(d["cu_seqlens"]), n, T, H, Dm, kmod._dtype_code(d["q"]), float(kmod.G_MIN),
                           p(d["init_state"]), p(o.t), p(fin.t), p(ws.t), ws_bytes, 0, kmod._stream(d["q"].device))
    assert rc == 0
    torch.cuda.synchronize()
    assert kda.read_device_error(ws.t) == 0
    assert o.intact() and fin.intact() and ws.intact()
    _inputs_unchanged(before, d)
    o_ref, f_ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"],
                                 init_state=d["init_state"])
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_ref) and torch.equal(fin.t, f_ref)


def test_segment_scan_writes_only_its_buffers():
    cu = kda_synth.cu_from_lengths([300, 1000, 1])
    n, T, H = 3, 1301, 2
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=5, cu_seqlens=cu, init_std=0.05)
    d = to_dev(inp, DEV)
    Dm = d["q"].shape[2]
    n_seg = 5  # 22 chunks in 5 segments, documents starting inside segments
    before = _snapshot(d)
    ws_bytes = kda.segment_scan_workspace_size(T, H, n, n_seg)
    o = Guarded(d["q"].shape, d["q"].dtype)
    fin = Guarded((n, H, Dm, Dm), torch.float32)
    pm = Guarded((H, n_seg, Dm, Dm), torch.float32)
    ps = Guarded((H, n_seg, Dm, Dm), torch.float32)
    ws = Guarded((ws_bytes,), torch.uint8)
    lib = kda.load()
    p = kmod._p
    rc = lib.kda_segment_scan(p(d["q"]), p(d["k"]), p(d["v"]), p(d["z"]), p(d["A"]), p(d["beta"]),
                              p(d["cu_seqlens"]), n, T, H, Dm, kmod._dtype_code(d["q"]), float(kmod.G_MIN),
                              p(d["init_state"]), n_seg, p(pm.t), p(ps.t), p(o.t), p(fin.t), p(ws.t), ws_bytes, 0,
                              kmod._stream(d["q"].device))
    assert rc == 0
    torch.cuda.synchronize()
    assert kda.read_device_error(ws.t) == 0
    assert all(g.intact() for g in (o, fin, pm, ps, ws))
    _inputs_unchanged(before, d)
    o_r, f_r, pm_r, ps_r = kda.segment_scan(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], n_seg,
                                            cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], return_pairs=True)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_r) and torch.equal(fin.t, f_r) and torch.equal(pm.t, pm_r) and torch.equal(ps.t, ps_r)


def _decode_setup(fused, dtype):
    N, W, H, seed = 7, 5, 3, 12
    state = kda_synth.decode_state(N, H, seed, device=DEV)
    A = kda_synth.decode_A(H, seed, A_std=0.5, device=DEV)
    if fused:
        w = kda_synth.decode_fused_window(N, W, H, 1, seed, dtype, device=DEV)
    else:
        w = kda_synth.decode_window(N, W, H, 1, seed, dtype, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(seed)
    tdt = w["q"].dtype
    # a cache holding the previous window's drafts, so that accepted drafts replay
    cache = tuple(torch.randn((N, W - 1, H, 128), generator=g, device=DEV).to(t)
                  for t in (tdt, tdt, tdt, torch.float32))
    cache = cache + (torch.sigmoid(torch.randn((N, W - 1, H), generator=g, device=DEV)),)
    return N, W, H, state, A, w, cache


@pytest.mark.parametrize("fused", [False, True])
def test_decode_writes_only_its_buffers(fused):
    N, W, H, state0, A, w, cache0 = _decode_setup(fused, "bf16")
    Dm = 128
    prm = kda_synth.decode_fused_params(H, 12, device=DEV) if fused else None
    cs0 = kda_synth.decode_conv_state(N, H, 12, device=DEV) if fused else None
    inputs = dict(q=w["q"], k=w["k"], v=w["v"], z=w["z"], beta=w["beta"], A=A, nacc=w["num_accepted"])
    if fused:
        inputs.update(o_gate=w["o_gate"], conv_w=prm["conv_w"], o_norm_w=prm["o_norm_w"])
    before = _snapshot(inputs)
    st = Guarded(state0.shape, torch.float32, state0)
    cg = [Guarded(c.shape, c.dtype, c) for c in cache0]
    o = Guarded(w["q"].shape, w["q"].dtype)
    err = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32))
    cs = Guarded(cs0.shape, torch.float32, cs0) if fused else None
    lib = kda.load()
    p = kmod._p
    dt = kmod._dtype_code(w["q"])
    stream = kmod._stream(w["q"].device)
    if fused:
        flags = kmod.KDA_FLAG_QK_L2NORM | kmod.KDA_FLAG_BETA_SIGMOID | kmod.KDA_FLAG_CONV_SILU
        rc = lib.kda_decode_step_fused(p(st.t), p(w["q"]), p(w["k"]), p(w["v"]), p(w["z"]), p(w["beta"]), p(A),
                                       p(prm["conv_w"]), p(cs.t), p(w["o_gate"]), p(prm["o_norm_w"]), 1e-6,
                                       *[p(c.t) for c in cg], p(w["num_accepted"]), N, H, Dm, W, dt,
                                       float(kmod.G_MIN), p(o.t), p(err.t), flags, stream)
    else:
        rc = lib.kda_decode_step(p(st.t), p(w["q"]), p(w["k"]), p(w["v"]), p(w["z"]), p(w["beta"]), p(A),
                                 *[p(c.t) for c in cg], p(w["num_accepted"]), N, H, Dm, W, dt, float(kmod.G_MIN),
                                 p(o.t), p(err.t), 0, stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.t.item()) == 0
    guards = [st, o, err] + cg + ([cs] if fused else [])
    assert all(g.intact() for g in guards)
    _inputs_unchanged(before, inputs)
    # the same step on plain buffers
    state_r = state0.clone()
    cache_r = tuple(c.clone() for c in cache0)
    if fused:
        cs_r = cs0.clone()
        o_r = kda.decode_step_fused(state_r, w["q"], w["k"], w["v"], w["z"], w["beta"], A, prm["conv_w"], cs_r,
                                    w["o_gate"], prm["o_norm_w"], cache_r, num_accepted=w["num_accepted"],
                                    qk_l2norm=True, beta_sigmoid=True, conv_silu=True)
    else:
        o_r = kda.decode_step(state_r, w["q"], w["k"], w["v"], w["z"], w["beta"], A, cache_r,
                              num_accepted=w["num_accepted"])
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_r) and torch.equal(st.t, state_r)
    assert all(torch.equal(g.t, c) for g, c in zip(cg, cache_r))
    if fused:
        assert torch.equal(cs.t, cs_r)


def test_chunk_fwd_ckpt_writes_only_its_buffers():
    """Checkpoint pages: the marked ones written, the skipped ones (-1, and
    positions past a document's end) left as they were, nothing outside."""
    lens, H, interval = [100, 700], 2, 128
    cu = kda_synth.cu_from_lengths(lens)
    n, T = len(lens), int(cu[-1])
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=31, cu_seqlens=cu, init_std=0.05)
    d = to_dev(inp, DEV)
    Dm = d["q"].shape[2]
    per_seq = max(lens) // interval + 1
    slot = torch.full((n, per_seq), -1, dtype=torch.int32)
    nxt = 0
    for doc in range(n):
        for j in range(per_seq):
            if j % 3 != 1:
                slot[doc, j] = nxt
                nxt += 1
    slot = slot.to(DEV)
    before = _snapshot(dict(d, slot=slot))
    ws_bytes = kda.chunk_fwd_workspace_size(T, H, n)
    o = Guarded(d["q"].shape, d["q"].dtype)
    fin = Guarded((n, H, Dm, Dm), torch.float32)
    ck = Guarded((nxt, H, Dm, Dm), torch.float32)
    ws = Guarded((ws_bytes,), torch.uint8)
    lib = kda.load()
    p = kmod._p
    rc = lib.kda_chunk_fwd_ckpt(p(d["q"]), p(d["k"]), p(d["v"]), p(d["z"]), p(d["A"]), p(d["beta"]),
                                p(d["cu_seqlens"]), n, T, H, Dm, kmod._dtype_code(d["q"]), float(kmod.G_MIN),
                                p(d["init_state"]), p(o.t), p(fin.t), interval, p(slot), per_seq, p(ck.t), nxt,
                                p(ws.t), ws_bytes, 0, kmod._stream(d["q"].device))
    assert rc == 0
    torch.cuda.synchronize()
    assert kda.read_device_error(ws.t) == 0
    assert all(g.intact() for g in (o, fin, ck, ws))
    _inputs_unchanged(before, dict(d, slot=slot))
    ck_r = torch.empty_like(ck.t)
    ck_r.view(torch.uint8).fill_(PATTERN)
    o_r, f_r = kda.chunk_fwd_ckpt(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], interval, slot, ck_r,
                                  cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], n_seqs=n)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_r) and torch.equal(fin.t, f_r)
    assert torch.equal(ck.t.view(torch.uint8), ck_r.view(torch.uint8))


def test_chunk_fwd_input_options_writes_only_its_buffers():
    """The input-option instantiation (L2 norm of q and k, beta's sigmoid, the q
    scale) on raw inputs, on the fused launch."""
    lens, H = [1, 63, 65, 200], 3
    cu = kda_synth.cu_from_lengths(lens)
    n, T = len(lens), int(cu[-1])
    inp = kda_synth.prefill_inputs(T, H, "bf16", seed=41, cu_seqlens=cu, init_std=0.05)
    d = to_dev(inp, DEV)
    g = torch.Generator(device=DEV).manual_seed(41)
    d["q"] = (d["q"].float() * (0.5 + torch.rand(T, H, 1, generator=g, device=DEV) * 4)).to(torch.bfloat16)
    d["k"] = (d["k"].float() * (0.5 + torch.rand(T, H, 1, generator=g, device=DEV) * 4)).to(torch.bfloat16)
    d["beta"] = torch.randn(T, H, generator=g, device=DEV)  # logits
    Dm = d["q"].shape[2]
    flags = kmod.KDA_FLAG_QK_L2NORM | kmod.KDA_FLAG_BETA_SIGMOID | kmod.KDA_FLAG_Q_SCALE
    before = _snapshot(d)
    ws_bytes = kda.chunk_fwd_workspace_size(T, H, n)
    o = Guarded(d["q"].shape, d["q"].dtype)
    fin = Guarded((n, H, Dm, Dm), torch.float32)
    ws = Guarded((ws_bytes,), torch.uint8)
    lib = kda.load()
    p = kmod._p
    rc = lib.kda_chunk_fwd(p(d["q"]), p(d["k"]), p(d["v"]), p(d["z"]), p(d["A"]), p(d["beta"]),
                           p(d["cu_seqlens"]), n, T, H, Dm, kmod._dtype_code(d["q"]), float(kmod.G_MIN),
                           p(d["init_state"]), p(o.t), p(fin.t), p(ws.t), ws_bytes, flags,
                           kmod._stream(d["q"].device))
    assert rc == 0
    torch.cuda.synchronize()
    assert kda.read_device_error(ws.t) == 0
    assert o.intact() and fin.intact() and ws.intact()
    _inputs_unchanged(before, d)
    o_r, f_r = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu_seqlens=d["cu_seqlens"],
                             init_state=d["init_state"], qk_l2norm=True, beta_sigmoid=True, q_scale=True)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_r) and torch.equal(fin.t, f_r)
