"""Benchmark of the KDA forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one kda_chunk_fwd over the prefill workload B=1, H=16, T=8192,
d=128, bf16 (synthetic inputs, seeded), timed with CUDA events on the launch
stream; L2 is flushed (a 256 MB write) before every step, outside the step's
events.  Rank 0 prints one JSON line.  The line also carries the decode step
(N=256, H=96, 1 + 4 drafts, fp32 state) measured the same way, the dominant
kernel's roofline, the end-to-end number through the public API with
host-resident inputs, the clocks seen during the timed region, and the fp64
oracle's throughput on the host cores.

Under torchrun every rank runs its own copy of the workload on its own GPU
(independent problems, no data-path collective: weak scaling); the step time
is the maximum over ranks.

--impl reference times the fp64 CPU oracle (the only reference this path has)
on a bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
METRIC = "KDA prefill tokens/s (H=16,T=8K) & decode tokens/s (B=256); % of roofline"
_CSRC = "linear_attention_serving_gb300/csrc/"
# every source file a kernel is compiled from (its .cu and the headers it includes)
KERNEL_SOURCES = {
    "prep_simt": [_CSRC + f for f in ("kda_prep_simt.cu", "kda_internal.cuh")],
    "scan_simt": [_CSRC + f for f in ("kda_scan_simt.cu", "kda_internal.cuh")],
    "prep_tc": [_CSRC + f for f in ("kda_prep_tc.cu", "kda_prep_body.cuh", "kda_tri.cuh", "kda_tc.cuh", "kda_internal.cuh")],
    "scan_tc": [_CSRC + f for f in ("kda_scan_tc.cu", "kda_scan_body.cuh", "kda_tc.cuh", "kda_internal.cuh")],
    "fused_tc": [_CSRC + f for f in ("kda_fused_tc.cu", "kda_prep_body.cuh", "kda_scan_body.cuh", "kda_tri.cuh",
                                     "kda_tc.cuh", "kda_internal.cuh")],
    "out_tc": [_CSRC + f for f in ("kda_out_tc.cu", "kda_tc.cuh", "kda_internal.cuh")],
    "decode": [_CSRC + f for f in ("kda_decode.cu", "kda_tc.cuh", "kda_internal.cuh")],
    "decode_fused": [_CSRC + f for f in ("kda_decode.cu", "kda_tc.cuh", "kda_internal.cuh")],
}


# About 200 us of device spin ahead of each timed step's first event, while the
# host enqueues the step: the events then time the device's work only.
HOST_COVER_CYCLES = 400_000


# ---------------------------------------------------------------- environment

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def src_sha(paths):
    h = hashlib.sha256()
    for path in paths:
        full = os.path.join(ROOT, path)
        if not os.path.exists(full):
            return None
        h.update(open(full, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel):
    """dram bytes per launch from a committed ncu summary, or None when absent
    or when the kernel source changed since the counters were taken."""
    try:
        t = json.load(open(TRAFFIC_FILE))[kernel]
    except Exception:
        return None
    if t.get("src_sha") != src_sha(KERNEL_SOURCES.get(kernel, [])):
        return None
    return t.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks sampled every 200 ms from the start of the timed region
    until --clock-window seconds of the same load have run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join("/tmp", f"kda_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- timing helpers

def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x, ws, dev):
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def kernel_times(marks):
    by = {}
    for name, ms in marks:
        by.setdefault(name, []).append(ms)
    return by


# ---------------------------------------------------------------- prefill

def bench_prefill(args, dev, ws, kda):
    w = kda_synth.WORKLOADS[args.workload]
    inp = kda_synth.workload_inputs(args.workload, device=dev)
    q, k, v, z, A, beta = (inp[n] for n in ("q", "k", "v", "z", "A", "beta"))
    cu, init = inp["cu_seqlens"], inp["init_state"]
    if cu is not None:
        cu = cu.to(dev)
    n_seqs = 1 if cu is None else cu.numel() - 1
    T, H = w.T, w.H
    wsp = torch.empty(kda.chunk_fwd_workspace_size(T, H, n_seqs, q.dtype), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        return kda.chunk_fwd(q, k, v, z, A, beta, cu_seqlens=cu, init_state=init, workspace=wsp, out=o)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    kda.profile_enable(True)
    launches0 = kda.launch_count()
    clocks.start()
    t_clk = time.time()
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        # the device spins while the host enqueues the step, so the events time
        # the device's work, not the host's launch latency
        torch.cuda._sleep(HOST_COVER_CYCLES)
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize()
    barrier(ws)
    launches = kda.launch_count() - launches0
    marks = kda.profile_collect()
    kda.profile_enable(False)
    # the timed steps last milliseconds, the clock samples come every 200 ms: the
    # same step keeps running (untimed, after the marks are taken) until the
    # samples cover --clock-window seconds of this load
    while time.time() - t_clk < getattr(args, "clock_window", 0.0):
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    return dict(T=T, H=H, n_seqs=n_seqs, total_ms=total_ms, step_ms=step_ms, marks=marks,
                launches=launches, clocks=clk, inputs=(q, k, v, z, A, beta, cu, init), workload=w)


def bench_prefill_variants(dev, kda, inputs, steps=10, warmup=3):
    """The same prefill workload through the optional paths: the in-kernel input
    options (q, k L2 norm and beta sigmoid), and state checkpoints every 512 tokens
    into 16 pages.  Device time per call with an L2 flush before each, as the main
    step; kernel names from the library's launch marks."""
    q, k, v, z, A, beta, cu, init = inputs
    T, H = q.shape[0], q.shape[1]
    n_seqs = 1 if cu is None else cu.numel() - 1
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    wsp = torch.empty(kda.chunk_fwd_workspace_size(T, H, n_seqs, q.dtype), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    per_seq = T // 512
    slots = torch.arange(n_seqs * per_seq, dtype=torch.int32, device=dev).reshape(n_seqs, per_seq)
    pages = torch.empty((n_seqs * per_seq, H, 128, 128), dtype=torch.float32, device=dev)
    calls = {
        "input_options": lambda: kda.chunk_fwd(q, k, v, z, A, beta, cu_seqlens=cu, init_state=init, workspace=wsp,
                                               out=o, qk_l2norm=True, beta_sigmoid=True),
        "checkpoints_every_512": lambda: kda.chunk_fwd_ckpt(q, k, v, z, A, beta, 512, slots, pages, cu_seqlens=cu,
                                                            init_state=init, workspace=wsp, out=o),
    }
    out = {}
    for name, fn in calls.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        kda.profile_enable(True)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            torch.cuda._sleep(HOST_COVER_CYCLES)
            evs[i][0].record()
            fn()
            evs[i][1].record()
        torch.cuda.synchronize()
        marks = kda.profile_collect()
        kda.profile_enable(False)
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        out[name] = {"ms_per_step": ms, "kernels": sorted(kernel_times(marks))}
    return out


def e2e_prefill(args, dev, kda, inputs):
    """Through the public API with inputs in pinned host memory: every step copies
    its inputs host -> device, runs kda_chunk_fwd, and reads o and the final state
    back.  Steps are pipelined the way a serving loop runs them: two device input
    sets, the host -> device copy of step i on one stream while step i - 1 computes
    on another, and the device -> host read of step i on a third."""
    q, k, v, z, A, beta, cu, init = inputs
    host = [t.cpu().pin_memory() for t in (q, k, v, z, A, beta)]
    devb = [[torch.empty_like(t) for t in (q, k, v, z, A, beta)] for _ in range(2)]
    T, H = q.shape[0], q.shape[1]
    n_seqs = 1 if cu is None else cu.numel() - 1
    o_d = [torch.empty_like(q) for _ in range(2)]
    o_h = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(2)]
    f_h = [torch.empty((n_seqs, H, 128, 128), dtype=torch.float32).pin_memory() for _ in range(2)]
    wsp = [torch.empty(kda.chunk_fwd_workspace_size(T, H, n_seqs, q.dtype), dtype=torch.uint8, device=dev)
           for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = o_h[0].numel() * o_h[0].element_size() + f_h[0].numel() * f_h[0].element_size()
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    fins = [None, None]

    def step(i):
        b_ = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_run[b_])  # step i - 2 is done reading this input set
            for d_, h_ in zip(devb[b_], host):
                d_.copy_(h_, non_blocking=True)
            ev_in[b_].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b_])
            s_run.wait_event(ev_out[b_])  # step i - 2's outputs have been read back
            _, fins[b_] = kda.chunk_fwd(*devb[b_], cu_seqlens=cu, init_state=init, workspace=wsp[b_], out=o_d[b_])
            ev_run[b_].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b_])
            fins[b_].record_stream(s_out)  # allocated on s_run, read here
            o_h[b_].copy_(o_d[b_], non_blocking=True)
            f_h[b_].copy_(fins[b_], non_blocking=True)
            ev_out[b_].record(s_out)

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    n = max(4, args.steps // 2)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for st in (s_in, s_run, s_out):
        st.wait_event(a)
    for i in range(n):
        step(i)
    cur = torch.cuda.current_stream()
    for st in (s_in, s_run, s_out):
        cur.wait_stream(st)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    return ms, h2d, d2h


# ---------------------------------------------------------------- the other prefill configurations

def timed_calls(fn, kda, flush, steps, warmup):
    """Device time of `fn` per call (CUDA events on the current stream, an L2
    flush and a host-cover spin before each call, outside its events), and the
    library's kernel marks of the timed calls."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    kda.profile_enable(True)
    launches0 = kda.launch_count()
    for i in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        evs[i][0].record()
        fn()
        evs[i][1].record()
    torch.cuda.synchronize()
    launches = kda.launch_count() - launches0
    marks = kda.profile_collect()
    kda.profile_enable(False)
    ms = [a.elapsed_time(b) for a, b in evs]
    kt = {n: sum(v) for n, v in kernel_times(marks).items()}
    tot = sum(kt.values()) or 1.0
    return {"ms_per_call": statistics.mean(ms), "ms_min": min(ms), "calls": steps,
            "launches_per_call": launches / steps,
            "kernel_ms_per_call": {n: v / steps for n, v in kt.items()},
            "kernel_share": {n: v / tot for n, v in kt.items()}}


def bench_other_configs(dev, kda, roofline, hbm, steps=6, warmup=3):
    """The workloads other than the headline, each through the public calls with
    device-resident inputs: tiny_fp32 (kda_chunk_fwd, exact fp32 path),
    varlen_32k_h32 (kda_chunk_fwd over packed documents) and segscan_1m_h8
    (kda_chunk_fwd, which picks its own segments, and kda_segment_scan with the
    configuration's 148 segments).  Throughput is workload tokens per second;
    roofline_frac divides the pages' kernel-level byte count (pro-rated by tokens,
    per-document states included) by the call time and the HBM peak."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    for name in ("tiny_fp32", "varlen_32k_h32", "segscan_1m_h8"):
        w = kda_synth.WORKLOADS[name]
        inp = kda_synth.workload_inputs(name, device=dev)
        q, k, v, z, A, beta = (inp[n] for n in ("q", "k", "v", "z", "A", "beta"))
        cu, init = inp["cu_seqlens"], inp["init_state"]
        n_seqs = 1 if cu is None else cu.numel() - 1
        if cu is not None:
            cu = cu.to(dev)
        T, H = w.T, w.H
        bytes_call = roofline.prefill_kernel_bytes(T, H, n_seqs)

        def entry(r, what):
            r["path"] = what
            r["tokens_per_s"] = T / (r["ms_per_call"] / 1e3)
            r["algorithmic_bytes"] = bytes_call
            r["roofline_frac"] = bytes_call / (r["ms_per_call"] / 1e3) / 1e9 / hbm
            return r

        res = {"T": T, "H": H, "n_seqs": n_seqs, "dtype": w.dtype}
        wsp = torch.empty(kda.chunk_fwd_workspace_size(T, H, n_seqs, q.dtype), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        fn = lambda: kda.chunk_fwd(q, k, v, z, A, beta, cu_seqlens=cu, init_state=init, workspace=wsp, out=o)
        nseg = kda.chunk_fwd_plan_segments(T, H, n_seqs, q.dtype, varlen=cu is not None)
        res["chunk_fwd"] = entry(timed_calls(fn, kda, flush, steps, warmup),
                                 f"kda_chunk_fwd ({nseg} automatic segments)" if nseg else "kda_chunk_fwd")
        del wsp
        if w.n_segments:
            torch.cuda.empty_cache()
            wsp = torch.empty(kda.segment_scan_workspace_size(T, H, n_seqs, w.n_segments, q.dtype),
                              dtype=torch.uint8, device=dev)
            fn = lambda: kda.segment_scan(q, k, v, z, A, beta, w.n_segments, cu_seqlens=cu, init_state=init,
                                          workspace=wsp)
            res["segment_scan"] = entry(timed_calls(fn, kda, flush, steps, warmup),
                                        f"kda_segment_scan ({w.n_segments} segments)")
            del wsp
        if w.dtype == "f32":
            res["note"] = "latency-bound: the byte count takes well under a microsecond at the HBM peak"
        out[name] = res
        del inp, q, k, v, z, A, beta, o
        torch.cuda.empty_cache()
    clk = clocks.stop()
    return out, clk


# ---------------------------------------------------------------- decode

def bench_decode(args, dev, kda, steps=20, warmup=3, fused=False):
    """The decode step over decode_mtp_b256_h96 (state 1.6 GB, larger than L2); with
    fused, kda_decode_step_fused on the same shapes (short convolution, all input
    options, gated output norm)."""
    w = kda_synth.WORKLOADS["decode_mtp_b256_h96"]
    N, H, W = w.N, w.H, w.W
    state = kda_synth.decode_state(N, H, w.seed, std=w.init_std, device=dev)
    A = kda_synth.decode_A(H, w.seed, device=dev)
    t = torch.float32
    cache = (torch.zeros((N, W - 1, H, 128), dtype=t, device=dev), torch.zeros((N, W - 1, H, 128), dtype=t, device=dev),
             torch.zeros((N, W - 1, H, 128), dtype=t, device=dev), torch.zeros((N, W - 1, H, 128), device=dev),
             torch.zeros((N, W - 1, H), device=dev))
    if fused:
        prm = kda_synth.decode_fused_params(H, w.seed, device=dev)
        cs = kda_synth.decode_conv_state(N, H, w.seed, device=dev)
        windows = [kda_synth.decode_fused_window(N, W, H, s, w.seed, "f32", device=dev) for s in range(4)]

        def step(wi, nacc):
            kda.decode_step_fused(state, *(wi[n] for n in ("q", "k", "v", "z", "beta")), A, prm["conv_w"], cs,
                                  wi["o_gate"], prm["o_norm_w"], cache, num_accepted=nacc, out=o,
                                  qk_l2norm=True, beta_sigmoid=True, conv_silu=True)
    else:
        windows = [kda_synth.decode_window(N, W, H, s, w.seed, "f32", device=dev) for s in range(4)]

        def step(wi, nacc):
            kda.decode_step(state, *(wi[n] for n in ("q", "k", "v", "z", "beta")), A, cache,
                            num_accepted=nacc, out=o)
    o = torch.empty_like(windows[0]["q"])
    step(windows[0], None)
    for i in range(warmup):
        wi = windows[(i + 1) % 4]
        step(wi, wi["num_accepted"])
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    committed = 0
    acc_total = 0
    kda.profile_enable(True)
    for i in range(steps):
        wi = windows[(i + warmup + 1) % 4]
        torch.cuda._sleep(HOST_COVER_CYCLES)
        evs[i][0].record()
        step(wi, wi["num_accepted"])
        evs[i][1].record()
    torch.cuda.synchronize()
    kda.profile_collect()
    kda.profile_enable(False)
    for i in range(steps):
        na = windows[(i + warmup + 1) % 4]["num_accepted"]
        acc_total += int(na.sum().item())
        committed += int((na + 1).sum().item())
    ms = [a.elapsed_time(b) for a, b in evs]
    return dict(N=N, H=H, W=W, step_ms=ms, committed=committed, accepted_total=acc_total, steps=steps)


# ---------------------------------------------------------------- oracle timing

def cpu_oracle_prefill(workload, heads=None, min_seconds=0.0):
    """The fp64 oracle on the host cores over `heads` heads of the workload (all by
    default), repeated until min_seconds have passed; tokens/s of the workload."""
    import oracle
    w = kda_synth.WORKLOADS[workload]
    inp = kda_synth.workload_inputs(workload)
    hs = heads or w.H
    sl = lambda x: x[:, :hs].contiguous()
    args = (sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["z"]), inp["A"][:hs].contiguous(), sl(inp["beta"]))
    reps, t0, used = 0, time.time(), 1
    while True:
        _, _, used = oracle.recurrent(*args, return_threads=True)
        reps += 1
        if time.time() - t0 >= min_seconds:
            break
    dt = (time.time() - t0) / reps
    tok_s = w.T * hs / w.H / dt
    return tok_s, used, f"{workload}: {hs} of {w.H} heads x {w.T} tokens, {reps} pass(es), {dt:.2f} s each"


def workload_config(workload, ws):
    """The `config` object of both arms' JSON lines."""
    w = kda_synth.WORKLOADS[workload]
    return {"workload": workload, "B": 1, "H": w.H, "T": w.T, "d": 128, "C": 64,
            "l2": "flushed before every step (256 MB write), outside the step's events",
            "host_launch": "hidden: a device spin precedes each step's first event",
            "parallelism": f"independent copy per GPU x{ws}"}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = kda_synth.WORKLOADS[args.workload]
    heads = w.H  # every head: the oracle threads over (sequence, head), so all host cores work
    for _ in range(args.warmup if args.warmup < 2 else 1):
        cpu_oracle_prefill(args.workload, heads)
    vals = []
    t0 = time.time()
    used = 1
    for _ in range(args.steps):
        v, used, sample = cpu_oracle_prefill(args.workload, heads)
        vals.append(v)
    total = time.time() - t0
    value = len(vals) / sum(1.0 / x for x in vals)  # harmonic mean = total tokens / total time
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args.workload, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"each step: {sample}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_h16_t8k")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the tiny, packed-varlen and 1M-token segment-scan configurations")
    ap.add_argument("--clock-window", type=float, default=0.6,
                    help="seconds of the prefill step the clock samples cover (0: the timed steps only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.warmup < 3:
        args.warmup = 3
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import linear_attention_serving_gb300 as kda_pkg
    from linear_attention_serving_gb300 import kda, roofline

    kda.load()
    hbm, peak_kind = peaks()
    pf = bench_prefill(args, dev, ws, kda)
    T, H = pf["T"], pf["H"]
    steps = args.steps
    tokens = T * steps * ws
    value = tokens / (pf["total_ms"] / 1e3)
    ms_per_step = pf["total_ms"] / steps
    kt = kernel_times(pf["marks"])
    tot = {n: sum(v) for n, v in kt.items()}
    dom = max(tot, key=tot.get) if tot else None
    chunk_heads = H * ((T + 63) // 64)
    algo = {"prep_simt": roofline.prep_bytes_per_chunk_head(), "prep_tc": roofline.prep_bytes_per_chunk_head(),
            "scan_simt": roofline.scan_bytes_per_chunk_head(), "scan_tc": roofline.scan_bytes_per_chunk_head(),
            "out_tc": roofline.out_bytes_per_chunk_head(),
            "fused_tc": roofline.prep_bytes_per_chunk_head() + roofline.scan_bytes_per_chunk_head()}
    roof = None
    if dom is not None:
        avg_ms = statistics.mean(kt[dom])
        bytes_launch = algo.get(dom, 0) * chunk_heads
        achieved = bytes_launch / (avg_ms / 1e3) / 1e9
        tr = traffic_for(dom)
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": tr, "peak_kind": f"{peak_kind} (copy bandwidth)",
                "algorithmic_bytes_per_launch": bytes_launch, "avg_launch_ms": avg_ms,
                "kernel_share": {n: tot[n] / sum(tot.values()) for n in tot}}
    path_bytes = roofline.prefill_kernel_bytes(T, H, pf["n_seqs"])
    path_frac = path_bytes / (ms_per_step / 1e3) / 1e9 / hbm

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.workload, ws),
        "roofline": roof,
        "path_roofline": {"bytes_per_step": path_bytes, "frac": path_frac, "peak": hbm,
                          "note": "pages' kernel-level count T/C(8C^2+22CD)+8D^2 per head"},
        "gpu_launches": pf["launches"],
        "clocks": pf["clocks"],
    }
    if rank == 0 and not args.no_e2e:
        pv = bench_prefill_variants(dev, kda, pf["inputs"])
        ckpt_bytes = (T // 512) * pf["n_seqs"] * H * 128 * 128 * 4
        for name, r in pv.items():
            b_ = path_bytes + (ckpt_bytes if name.startswith("checkpoints") else 0)
            r["tokens_per_s"] = T / (r["ms_per_step"] / 1e3)
            r["roofline_frac"] = b_ / (r["ms_per_step"] / 1e3) / 1e9 / hbm
        line["prefill_variants"] = pv
        ms, h2d, d2h = e2e_prefill(args, dev, kda, pf["inputs"])
        line["e2e"] = {"value": T * ws / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": ms}
    if rank == 0 and not args.no_configs:
        cfgs, cclk = bench_other_configs(dev, kda, roofline, hbm)
        line["other_configs"] = cfgs
        line["other_configs_clocks"] = cclk
    if not args.no_decode:
        dc = bench_decode(args, dev, kda)
        dms = sum(dc["step_ms"])
        dms = max_over_ranks(dms, ws, dev)
        step_bytes = roofline.decode_step_bytes(dc["N"], dc["H"], dc["W"], dc["accepted_total"] // dc["steps"])
        avg = dms / dc["steps"]
        line["decode"] = {
            "workload": "decode_mtp_b256_h96", "value": dc["committed"] * ws / (dms / 1e3), "unit": "tokens/s",
            "seq_steps_per_s": dc["N"] * dc["steps"] * ws / (dms / 1e3), "ms_per_step": avg,
            "roofline": {"kernel": "decode", "bound": "hbm",
                         "achieved": step_bytes / (avg / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": step_bytes / (avg / 1e3) / 1e9 / hbm, "traffic": traffic_for("decode"),
                         "algorithmic_bytes_per_launch": step_bytes},
        }
        fc = bench_decode(args, dev, kda, fused=True)
        fms = max_over_ranks(sum(fc["step_ms"]), ws, dev)
        f_bytes = roofline.decode_fused_step_bytes(fc["N"], fc["H"], fc["W"], fc["accepted_total"] // fc["steps"])
        favg = fms / fc["steps"]
        line["decode_fused"] = {
            "workload": "decode_mtp_b256_h96, short conv + L2 norm + beta sigmoid + gated output norm",
            "value": fc["committed"] * ws / (fms / 1e3), "unit": "tokens/s", "ms_per_step": favg,
            "roofline": {"kernel": "decode_fused", "bound": "hbm",
                         "achieved": f_bytes / (favg / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": f_bytes / (favg / 1e3) / 1e9 / hbm, "traffic": traffic_for("decode_fused"),
                         "algorithmic_bytes_per_launch": f_bytes},
        }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, used, sample = cpu_oracle_prefill(args.workload)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
