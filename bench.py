#!/usr/bin/env python3
"""Benchmark of the band-attention forward on B300.

One step = one forward call (band kernel + global-row kernels) over one batch
of seeded synthetic inputs that are already resident in HBM.  Default
workload: bf16 encoder pattern B2 H12 n4096 d64, w=512, one global token.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints one JSON line (rank 0).  Under torchrun each rank runs its own copy of
the workload (weak scaling; the path needs no collective) and the reported
time is the maximum over ranks.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "band-attn fwd useful TFLOP/s & % bf16 tensor peak; tokens/s vs n"
L2_FLUSH_BYTES = 256 << 20
# fp32 FMA rate of the CUDA cores (the backward's bound): 148 SMs x 128 lanes
# x 2 flops x 2.032 GHz maximum SM clock
FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        j = json.load(open(path))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# The sources of the forward kernels (device code); host planning lives in
# lf_attn.cu, and the entry's kernel name is checked against the one that ran.
FWD_KERNEL_FILES = ("lf_internal.cuh", "band_ring.cuh", "band_duo.cuh", "band_pair.cuh", "band_simt.cuh",
                    "global_rows.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "long_sequence_sliding_longformer_b300", "csrc")
    for f in FWD_KERNEL_FILES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str, kernel: str):
    """DRAM bytes per band-kernel launch from a committed ncu summary, if it was
    taken on the current kernel sources, for this workload and this kernel;
    else None."""
    path = os.path.join(ROOT, "profiles", "band_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        j = json.load(open(path))
        e = j.get(workload)
        if e and e.get("source_hash") == kernel_source_hash() and e.get("kernel") == kernel:
            return e.get("bytes_per_launch_full")
    except (ValueError, OSError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if not dist.is_initialized():
        dist.init_process_group(backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def useful_work(wl):
    import long_sequence_sliding_longformer_b300 as lf
    pairs, flops = lf.count_pairs(B=wl.B, H=wl.H, n=wl.n, d=wl.d, w=wl.w, dilation=wl.dilation,
                                  causal=wl.causal, pad_len=wl.pad_len, global_idx=wl.global_idx)
    # split: pairs on the global tokens' own rows (global-row kernels) vs the rest (band kernel)
    gpairs = 0
    for b in range(wl.B):
        L = wl.valid_len(b)
        for g in wl.global_idx:
            if g < L:
                gpairs += (g + 1 if wl.causal else L) * wl.H
    return pairs, flops, gpairs * 4 * wl.d


def pct(xs, p):
    """p-th percentile (nearest rank) of xs."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(p / 100.0 * (len(ys) - 1)))))]


def band_bytes(wl) -> int:
    """Algorithmic HBM bytes of the band kernel: q, k, v read once, out written
    once, over all rows (8*d bytes per token-head in bf16)."""
    return 4 * wl.B * wl.H * wl.n * wl.d * wl.elem_bytes


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_sample(wl, inp, target_s: float = 12.0, threads: int = 0):
    """Time the oracle on whole (batch, head) slices of the workload until about
    target_s seconds of work; returns (seconds, useful flops, threads, description).
    Useful work is counted by the oracle itself (no product code is loaded)."""
    import numpy as np
    import oracle
    host = workloads.Inputs(*[None if t is None else t.cpu() for t in
                              (inp.q, inp.k, inp.v, inp.qg, inp.kg, inp.vg)])
    n = wl.n
    slices = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    done, secs, flops = 0, 0.0, 0.0
    while done < len(slices):
        take = 1 if done == 0 else max(1, min(len(slices) - done,
                                              int(done * (target_s - secs) / max(secs, 1e-3))))
        if done > 0 and secs >= target_s:
            break
        chunk = slices[done:done + take]
        rows = np.concatenate([np.arange(n, dtype=np.int64) + (b * wl.H + h) * n for b, h in chunk])
        t0 = time.perf_counter()
        oracle.wl_fwd(wl, host, rows=rows, threads=threads)
        secs += time.perf_counter() - t0
        for b, h in chunk:
            pad = None if wl.pad_len is None else [wl.pad_len[b]]
            p, _ = oracle.count_pairs(B=1, H=1, n=n, w=wl.w, dilation=[wl.dilation[h]],
                                      causal=wl.causal, pad_len=pad, global_idx=wl.global_idx)
            flops += 4.0 * wl.d * p
        done += take
    desc = "%d of %d (batch, head) slices, all %d rows each (every row of the sample)" % (
        done, len(slices), n)
    return secs, flops, threads if threads > 0 else oracle.max_threads(), desc


def run_reference(args, wl):
    rank, ws, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    inp = workloads.make_inputs(wl, "cpu", seed=wl.seed)
    times, flops_tot = [], 0.0
    threads, desc = 0, ""
    per_step_target = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for it in range(args.warmup + args.steps):
        secs, flops, threads, desc = cpu_sample(wl, inp, target_s=per_step_target)
        if it >= args.warmup:
            times.append(secs)
            flops_tot += flops
    value = flops_tot / sum(times) / 1e12
    tok = wl.tokens()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (N(0,1), CPU generator seed %d)" % wl.seed,
        "config": dict(wl.describe(), sample="bounded per step"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_per_s": value * 1e12 * tok / (4.0 * wl.d * oracle.wl_count_pairs(wl)[0]),
    }
    print(json.dumps(line), flush=True)


def run_gpu(args, wl):
    import long_sequence_sliding_longformer_b300 as lf
    rank, ws, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lf.load()
    # the same CPU generator and seed as the reference arm (rank r: seed + r)
    inp_host = workloads.make_inputs(wl, "cpu", seed=wl.seed + rank)
    inp = workloads.Inputs(*[None if t is None else t.to(dev) for t in
                             (inp_host.q, inp_host.k, inp_host.v, inp_host.qg, inp_host.kg, inp_host.vg)])
    del inp_host
    out = torch.empty_like(inp.q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(o=out):
        lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, out=o)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    # One step (every kernel of one call) captured once as a CUDA graph and
    # replayed, so that host-side argument checking and launch overhead stay
    # out of the device time; the library records the band kernel's own
    # events inside the graph.
    band_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in band_ev:  # torch creates the underlying CUDA events on first record
        e.record(stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    launches0 = lf.launch_count()
    lf.set_band_events(*band_ev)
    with torch.cuda.graph(graph):
        step()
    lf.set_band_events(None, None)
    launches_per_step = lf.launch_count() - launches0
    band_kernel = lf.last_band_kernel()
    for _ in range(3):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    band_ms = []
    with ClockSampler(dev.index) as clocks:
        barrier(ws)
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(K):
            flush.zero_()  # evict L2 so every step reads its inputs from HBM
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
            ev[i][1].synchronize()  # the band events inside the graph are reused by the next replay
            band_ms.append(band_ev[0].elapsed_time(band_ev[1]))
        torch.cuda.synchronize(dev)
        barrier(ws)
        wall = time.perf_counter() - wall0
    launches = launches_per_step * K
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    ms_per_step = total_ms / K

    # ---- hot L2: the same replay with no flush between steps (inputs that
    # fit in L2 then stay there); reported beside the flushed number
    Kh = min(K, 200)
    evh = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kh)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    for i in range(Kh):
        evh[i][0].record(stream)
        graph.replay()
        evh[i][1].record(stream)
    torch.cuda.synchronize(dev)
    hot_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evh) / Kh, ws, dev)

    # ---- end to end through the public API: pinned host in, host out.  Every
    # step copies its inputs in and its output back; consecutive steps are
    # pipelined over two buffer sets (inputs of step i+1 travel while step i
    # computes and step i-1's output travels back: the copy engines of both
    # directions and the SMs work at once).
    host_in = [t.cpu().pin_memory() for t in inp.tensors()]
    host_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    dev_in = [[torch.empty_like(t) for t in inp.tensors()] for _ in range(2)]
    dev_out = [torch.empty_like(out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    e2e_k = max(3, min(K, 50))
    s_h2ds = [torch.cuda.Stream(dev) for _ in range(2)]  # the inputs split over two copy streams
    s_d2h = torch.cuda.Stream(dev)
    names = ["q", "k", "v", "qg", "kg", "vg"]
    freed = [None, None]  # per buffer set: event after the step that last read it (inputs and output)

    def e2e_step(i):
        j = i % 2
        for c, s_h2d in enumerate(s_h2ds):
            with torch.cuda.stream(s_h2d):
                if freed[j] is not None:
                    s_h2d.wait_event(freed[j])
                for d_, h_ in list(zip(dev_in[j], host_in))[c::len(s_h2ds)]:
                    d_.copy_(h_, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_h2d)
            stream.wait_event(landed)
        t = dict(zip(names, dev_in[j]))
        lf.attn(t["q"], t["k"], t["v"], w=wl.w, dilation=wl.dilation, causal=wl.causal,
                pad_len=wl.pad_len, qg=t.get("qg"), kg=t.get("kg"), vg=t.get("vg"),
                global_idx=wl.global_idx, out=dev_out[j])
        done = torch.cuda.Event()
        done.record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(done)
            host_out[j].copy_(dev_out[j], non_blocking=True)
            back = torch.cuda.Event()
            back.record(s_d2h)
        freed[j] = back

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    freed = [None, None]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(stream)
    for s_h2d in s_h2ds:
        s_h2d.wait_stream(stream)
    for i in range(e2e_k):
        e2e_step(i)
    stream.wait_stream(s_d2h)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_k, ws, dev)
    host_out = host_out[(e2e_k - 1) % 2]

    # ---- backward (the gradients of sum(dout * out)) on the same inputs, one
    # call per step, L2 flushed before each; events on the launching stream
    gen = torch.Generator(device="cpu").manual_seed(wl.seed + 1000 + rank)
    dout = torch.randn(tuple(inp.q.shape), generator=gen).to(inp.q.dtype).to(dev)
    grads = lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                        pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx)
    Kb = max(3, min(K, 30))
    for _ in range(2):
        lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                    pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, grads=grads)
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kb)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    for i in range(Kb):
        flush.zero_()
        evb[i][0].record(stream)
        lf.attn_bwd(inp.q, inp.k, inp.v, dout, w=wl.w, dilation=wl.dilation, causal=wl.causal,
                    pad_len=wl.pad_len, qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, grads=grads)
        evb[i][1].record(stream)
    torch.cuda.synchronize(dev)
    bwd_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evb) / Kb, ws, dev)
    del grads, dout

    # ---- the same forward with a relative position bias table [H, w + 1] on
    # the band scores (its own kernel instantiation); L2 flushed before each
    genb = torch.Generator(device="cpu").manual_seed(wl.seed + 4000 + rank)
    table = torch.randn(wl.H, wl.w + 1, generator=genb).to(dev)
    bout = torch.empty_like(out)

    def bias_call():
        lf.attn(inp.q, inp.k, inp.v, w=wl.w, dilation=wl.dilation, causal=wl.causal, pad_len=wl.pad_len,
                qg=inp.qg, kg=inp.kg, vg=inp.vg, global_idx=wl.global_idx, out=bout, rel_bias=table)

    for _ in range(3):
        bias_call()
    bias_kernel = lf.last_band_kernel()
    Kr = max(3, min(K, 100))
    evr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kr)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    for i in range(Kr):
        flush.zero_()
        evr[i][0].record(stream)
        bias_call()
        evr[i][1].record(stream)
    torch.cuda.synchronize(dev)
    bias_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evr) / Kr, ws, dev)
    del table, bout

    # ---- the projections that produce this workload's inputs from hidden
    # states [B, n, H*d] (q, k, v, and kg, vg with global tokens: one call),
    # bf16 workloads only; L2 flushed before each call
    proj = None
    if wl.dtype == "bf16":
        Kh = wl.H * wl.d
        n_out = 5 if wl.G > 0 else 3
        genp = torch.Generator(device="cpu").manual_seed(wl.seed + 2000 + rank)
        xh = torch.randn(wl.B, wl.n, Kh, generator=genp).to(torch.bfloat16).to(dev)
        wh = (torch.randn(n_out * Kh, Kh, generator=genp) / Kh ** 0.5).to(torch.bfloat16).to(dev)
        yh = lf.proj_heads(xh, wh, H=wl.H, d=wl.d)
        for _ in range(2):
            lf.proj_heads(xh, wh, H=wl.H, d=wl.d, out=yh)
        Kp = max(3, min(K, 100))
        evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kp)]
        barrier(ws)
        torch.cuda.synchronize(dev)
        for i in range(Kp):
            flush.zero_()
            evp[i][0].record(stream)
            lf.proj_heads(xh, wh, H=wl.H, d=wl.d, out=yh)
            evp[i][1].record(stream)
        torch.cuda.synchronize(dev)
        proj_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evp) / Kp, ws, dev)
        pflops = 2.0 * wl.B * wl.n * Kh * n_out * Kh
        pk0 = peaks()
        proj = {"ms_per_call": proj_ms, "steps": Kp, "unit": "TFLOP/s",
                "value": ws * pflops / (proj_ms * 1e-3) / 1e12, "flops_per_call": pflops,
                "shape": {"M": wl.B * wl.n, "K": Kh, "N": n_out * Kh, "outputs": n_out},
                "kernel": "proj_gemm_kernel (tcgen05)",
                "roofline": {"bound": "tensor", "peak": pk0["bf16_tflops"], "unit": "TFLOP/s",
                             "achieved": pflops / (proj_ms * 1e-3) / 1e12,
                             "frac": pflops / (proj_ms * 1e-3) / 1e12 / pk0["bf16_tflops"],
                             "peak_source": pk0["source"] + " (burst)"},
                "l2": "flushed before every call"}
        del xh, wh, yh

    # ---- the Memorizing-Transformer combine on this workload's shape: 32
    # pairs per query retrieved (uniformly at random) from a 65536-entry
    # memory per (b, h), mixed with the band output; HBM-bound gathers
    memc = None
    if wl.dtype == "bf16":
        Mm, km = 65536, 32
        genm = torch.Generator(device="cpu").manual_seed(wl.seed + 3000 + rank)
        mk = torch.randn(wl.B, wl.H, Mm, wl.d, generator=genm).to(torch.bfloat16).to(dev)
        mv = torch.randn(wl.B, wl.H, Mm, wl.d, generator=genm).to(torch.bfloat16).to(dev)
        midx = torch.randint(0, Mm, (wl.B, wl.H, wl.n, km), generator=genm, dtype=torch.int32).to(dev)
        gate = torch.rand(wl.H, generator=genm).to(dev)
        mout = torch.empty_like(out)
        lf.mem_combine(inp.q, out, mk, mv, midx, gate, out=mout)
        Km = max(3, min(K, 100))
        evm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Km)]
        barrier(ws)
        torch.cuda.synchronize(dev)
        for i in range(Km):
            flush.zero_()
            evm[i][0].record(stream)
            lf.mem_combine(inp.q, out, mk, mv, midx, gate, out=mout)
            evm[i][1].record(stream)
        torch.cuda.synchronize(dev)
        mem_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evm) / Km, ws, dev)
        rows_m = wl.B * wl.H * wl.n
        mbytes = rows_m * (3 * wl.d * 2 + km * 4 + km * 2 * wl.d * 2)
        pk1 = peaks()
        memc = {"ms_per_call": mem_ms, "steps": Km, "memory_entries": Mm, "retrieved_per_query": km,
                "bytes_per_call": mbytes,
                "bytes_counted": "q, local, out rows + the indices + the retrieved key and value rows, each once per query",
                "kernel": "mem_combine_kernel (CUDA cores)",
                "roofline": {"bound": "hbm", "peak": pk1["hbm_gbs"], "unit": "GB/s",
                             "achieved": mbytes / (mem_ms * 1e-3) / 1e9,
                             "frac": mbytes / (mem_ms * 1e-3) / 1e9 / pk1["hbm_gbs"],
                             "peak_source": pk1["source"]},
                "l2": "flushed before every call"}
        del mk, mv, midx, mout

    pairs, flops, gflops_part = useful_work(wl)
    band_flops = flops - gflops_part
    pk = peaks()
    value = ws * flops / (ms_per_step * 1e-3) / 1e12
    band_avg_ms = statistics.mean(band_ms)
    band_achieved = band_flops / (band_avg_ms * 1e-3) / 1e12
    hbm_achieved = band_bytes(wl) / (band_avg_ms * 1e-3) / 1e9
    traffic = committed_traffic(wl.name, band_kernel)
    line = None
    if rank == 0:
        cs = clocks.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic (N(0,1), CPU generator seed %d, copied to the device)" % (wl.seed + rank),
            "config": dict(wl.describe(), parallelism="replicas: one workload per GPU" if ws > 1 else "1 GPU",
                           l2="flushed before every step (256 MiB write)"),
            "tokens_per_s": ws * wl.tokens() / (ms_per_step * 1e-3),
            "frac_of_bf16_peak": value / pk["bf16_tflops"],
            "roofline": {"bound": "tensor", "achieved": band_achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": band_achieved / pk["bf16_tflops"],
                         "traffic": traffic, "kernel": band_kernel,
                         "peak_source": pk["source"] + " (burst)",
                         "hbm_achieved_gbs": hbm_achieved, "hbm_frac": hbm_achieved / pk["hbm_gbs"],
                         "band_ms": band_avg_ms, "band_share_of_step": band_avg_ms / statistics.mean(step_ms)},
            "step_ms_p10": pct(step_ms, 10), "step_ms_p50": pct(step_ms, 50), "step_ms_p90": pct(step_ms, 90),
            "band_ms_p10": pct(band_ms, 10), "band_ms_p90": pct(band_ms, 90),
            "hot_l2": {"ms_per_step": hot_ms, "value": ws * flops / (hot_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "steps": Kh, "l2": "not flushed between steps"},
            "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "backward": {
                "ms_per_step": bwd_ms, "steps": Kb, "unit": "TFLOP/s",
                "value": ws * 2.0 * flops / (bwd_ms * 1e-3) / 1e12,
                "flops_per_step": 2.0 * flops,
                "flops_counted": "8*d per attended pair (dP, dV, dQ, dK; the recomputed scores not counted)",
                "kernels": "bwd_rows_tiled + bwd_keys_tiled (+ bwd_grows, bwd_gkeys, bwd_kgvg with global "
                           "tokens; CUDA cores, fp32)",
                "roofline": {"bound": "alu", "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                             "achieved": 2.0 * flops / (bwd_ms * 1e-3) / 1e12,
                             "frac": 2.0 * flops / (bwd_ms * 1e-3) / 1e12 / FP32_PEAK_TFLOPS,
                             "peak_source": "148 SMs x 128 fp32 lanes x 2 flops x 2.032 GHz"},
                "l2": "flushed before every step"},
            "relative_bias": {"ms_per_call": bias_ms, "steps": Kr, "unit": "TFLOP/s",
                              "value": ws * flops / (bias_ms * 1e-3) / 1e12, "band_kernel": bias_kernel,
                              "vs_plain_step": bias_ms / statistics.mean(step_ms),
                              "l2": "flushed before every call"},
            "projection": proj,
            "memory_combine": memc,
            "gpu_launches": launches,
            "clocks": {"sm_mhz": cs["sm_mhz"], "sm_max_mhz": cs["sm_max_mhz"], "reasons": cs["reasons"],
                       "samples": cs["samples"]},
            "wall_s_timed_region": wall,
            "useful_flops_per_step": flops,
        }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        secs, sflops, threads, desc = cpu_sample(wl, inp, target_s=args.cpu_seconds)
        v = sflops / secs / 1e12
        secs1, sflops1, _, desc1 = cpu_sample(wl, inp, target_s=min(3.0, args.cpu_seconds), threads=1)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": secs, "cpu_model": cpu_model(),
                                "one_thread": {"value": sflops1 / secs1 / 1e12, "seconds": secs1,
                                               "sample": desc1}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lf", choices=["lf", "reference"])
    ap.add_argument("--workload", default=workloads.bf16_encoder().name,
                    help="one of: " + ", ".join(w.name for w in workloads.all_workloads()))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = workloads.by_name(args.workload)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl)


if __name__ == "__main__":
    main()
