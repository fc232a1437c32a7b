#!/usr/bin/env python
"""Benchmark of the quantized MoE expert projection on GB300.

One step = the whole hot path over one batch: the gate/up and the down grouped
projections of the prefill workload (256 NVFP4 experts, 4096 tokens top-8 Zipf(1.1);
act_quant fused), each one call of fp4_grouped_expert_gemm. Headline value = expert GEMM
TFLOP/s (algorithmic 2*rows*n*k). The same line carries the decode workload (64 NVFP4
experts, 8 tokens top-8) as weight GB/s, the roofline of the dominant kernel, the CPU
oracle baseline, the end-to-end number with host buffers, and the SM clocks seen.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c4|c3|c5] [--no-decode]

With N > 1 (torchrun, one rank per GPU) every rank runs an independent replica of the
workload (weak scaling; the path has no cross-GPU exchange).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "expert GEMM TFLOP/s (prefill) and weight GB/s (decode) vs GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_NAMES = {"c3": "decode: 64 NVFP4 experts gate/up [3072,4096] + down [4096,1536], "
                        "8 tokens top-8 uniform",
                  "c4": "prefill grouped: 256 NVFP4 experts gate/up [2048,7168] + down "
                        "[7168,2048], 4096 tokens top-8 Zipf(1.1)",
                  "c5": "mixed: 128 NVFP4 + 128 MXFP4 experts [2048,4096], 16384 tokens "
                        "top-8 uniform per recipe"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0 = about 2 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["c3", "c4", "c5"], default="c4")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-mixed", action="store_true",
                    help="skip the mixed-recipe line (128 NVFP4 + 128 MXFP4 experts)")
    ap.add_argument("--no-swiglu", action="store_true",
                    help="skip the SwiGLU + requantisation line (the step after gate/up)")
    ap.add_argument("--no-routing", action="store_true",
                    help="skip the routing front-end line (router, CSR, combine)")
    ap.add_argument("--no-w4a4", action="store_true",
                    help="skip the W4A4 variant (E2M1 activations) on the same workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's expert count")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--path", choices=["auto", "stream", "tc"], default="auto",
                    help="force a kernel path (default: the library's choice by shape)")
    ap.add_argument("--path-sweep", action="store_true",
                    help="instead of the benchmark: time both grouped paths by routed rows per "
                         "expert (the measurement behind the library's path threshold)")
    return ap.parse_args()


# ------------------------------------------------------------------ infrastructure

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.device_index = device_index

    def _target(self):
        import torch
        try:
            p = torch.cuda.get_device_properties(self.device_index)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        tgt = self._target()
        if tgt:
            cmd[1:1] = ["-i", tgt]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# Source files each measured kernel is built from: a traffic figure stays valid only while
# these are unchanged.
KERNEL_SOURCES = {
    "tc_grouped_gemm": ["gemm_tc.cu", "common.cuh", "tcgen05.cuh", "internal.h", "tma_host.h"],
    "mx_grouped_gemm": ["gemm_mx.cu", "common.cuh", "tcgen05.cuh", "internal.h", "tma_host.h"],
    "tc_quantize": ["gemm_tc.cu", "common.cuh", "internal.h"],
    "stream_gemm": ["gemm_stream.cu", "common.cuh", "internal.h"],
    "decode_tma": ["gemm_decode.cu", "common.cuh", "internal.h", "tma_host.h"],
    "w4a4_gemm": ["gemm_w4a4.cu", "common.cuh", "tcgen05.cuh", "internal.h", "tma_host.h"],
}

# The no-workspace path runs the TMA-fed warp-MMA decode kernel for k a multiple of 512 up
# to 28544, which covers each workload here; the FMA streaming kernel takes larger k only.
STREAM_KERNEL = "decode_tma"


def source_hash(kernel=None):
    """Short hash of a kernel's source files (all of csrc/ when kernel is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp4_act_gb300", "csrc")
    names = KERNEL_SOURCES[kernel] if kernel else sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-step DRAM bytes from the committed ncu summary, if it was taken on the current
    sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != source_hash(kernel_key.split("/")[0]):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ workload accounting

def proj_flops(proj):
    return 2.0 * proj.routing.P * proj.bank.n * proj.bank.k


def proj_bytes(proj):
    """Algorithmic bytes: touched experts' nibbles + scales + scale2, activations read
    once, outputs written once."""
    import torch
    b = proj.bank
    gs = 16 if b.recipe == 0 else 32
    touched = int(torch.count_nonzero(torch.diff(proj.routing.offsets)).item())
    weights = touched * (b.n * (b.k // 2) + b.n * (b.k // gs) + 4)
    rows_x = proj.x.shape[0]
    act = rows_x * b.k * 4
    out = proj.routing.P * b.n * 4
    return weights + act + out, weights


def quant_bytes(proj):
    """Algorithmic bytes of the quantise phase: each token's activation row read once (f32),
    the 16-bit workspace row of every routed row written once, plus the row scales. (When
    tokens repeat, the path also writes and re-reads a per-token copy: 2 B per token
    element each way, counted as traffic, not as algorithmic bytes.)"""
    T, k = proj.x.shape
    P = proj.routing.P
    return T * k * 4 + P * k * 2 + P * 4


def launches_per_call(fp4, proj, have_ws):
    """Kernels of ours one grouped call launches: the streaming kernel alone, or the
    tensor-core path's quantise pass(es) (NVFP4: f16 pass, conditional bf16 pass), the
    per-token expand when tokens repeat, and the GEMM."""
    path = fp4.fp4_gemm_path(proj.routing.P, proj.bank.E, proj.bank.n, proj.bank.k,
                             proj.bank.recipe, have_ws)
    if path != fp4.PATH_TC:
        return path, 1
    T = proj.x.shape[0]
    repeats = proj.row_ids_used and T < proj.routing.P  # quantise per token, then expand
    return path, (3 if proj.bank.recipe == fp4.NVFP4 else 2) + (1 if repeats else 0)


# ------------------------------------------------------------------ our arm

def make_calls(fp4, wl, device):
    """One entry per grouped projection. On the tensor-core path the call is run as its
    two halves (fp4_grouped_quantize, then fp4_grouped_gemm_quantized on the same stream:
    exactly the launches fp4_grouped_expert_gemm makes), so that the quantise pass and the
    GEMM kernel are timed apart; the streaming path is one launch."""
    import torch
    calls = []
    for proj in wl.projections:
        T, k = proj.x.shape
        ws = fp4.workspace_for(T, proj.routing.P, proj.bank.n, k, proj.bank.recipe, device=device)
        out = torch.empty(proj.routing.P, proj.bank.n, device=device)
        rid = proj.routing.row_ids if proj.row_ids_used else None
        path, nl = launches_per_call(fp4, proj, ws is not None)

        def call(proj=proj, ws=ws, out=out, rid=rid, x=None):
            fp4.fp4_grouped_expert_gemm(proj.x if x is None else x, rid, proj.routing.offsets,
                                        proj.bank.w, proj.bank.sc, proj.bank.scale2,
                                        proj.bank.recipe, out=out, workspace=ws)
        if path == fp4.PATH_TC:
            def quantize(proj=proj, ws=ws, rid=rid):
                fp4.fp4_grouped_quantize(proj.x, rid, proj.routing.P, proj.bank.recipe, ws)

            def gemm(proj=proj, ws=ws, out=out, rid=rid):
                fp4.fp4_grouped_gemm_quantized(ws, proj.x.shape[0], rid, proj.routing.offsets,
                                               proj.bank.w, proj.bank.sc, proj.bank.scale2,
                                               proj.bank.recipe, out)
            phases = [("quantize", quantize), ("gemm", gemm)]
        else:
            phases = [("gemm", call)]
        calls.append({"proj": proj, "call": call, "phases": phases, "out": out, "ws": ws,
                      "path": path, "launches": nl})
    return calls


def time_steps(calls, steps, flush=None):
    """Run `steps` steps; CUDA events on the launching (current) stream around every phase
    of every call. Returns (elapsed ms of the whole region, per-call list of per-step call
    durations in ms, per-call dict phase -> per-step durations in ms)."""
    import torch
    stream = torch.cuda.current_stream()
    nph = [len(c["phases"]) for c in calls]
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for n in nph]
           for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(steps):
        if flush is not None:
            flush.zero_()
        for i, c in enumerate(calls):
            e = evs[s][i]
            e[0].record(stream)
            for j, (_, fn) in enumerate(c["phases"]):
                fn()
                e[j + 1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    per_call = [[evs[s][i][0].elapsed_time(evs[s][i][-1]) for s in range(steps)]
                for i in range(len(calls))]
    per_phase = [{name: [evs[s][i][j].elapsed_time(evs[s][i][j + 1]) for s in range(steps)]
                  for j, (name, _) in enumerate(c["phases"])} for i, c in enumerate(calls)]
    return t0.elapsed_time(t1), per_call, per_phase


def time_whole_steps(calls, steps, flush=None):
    """Per-step device time (ms) of all calls of a step together: the L2 flush before each
    step stays outside the timed span, and no event is queued between the calls, so a
    kernel may start while the one before it drains (as in a real step)."""
    import torch
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for s in range(steps):
        if flush is not None:
            flush.zero_()
        evs[s][0].record(stream)
        for c in calls:
            c["call"]()
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def pct(v, q):
    """q-quantile of a list (linear interpolation)."""
    import statistics
    v = sorted(v)
    if len(v) == 1:
        return v[0]
    return statistics.quantiles(v, n=100, method="inclusive")[int(q * 100) - 1] if 0 < q < 1 else (
        v[0] if q <= 0 else v[-1])


def stats_ms(v):
    import statistics
    return {"mean": round(sum(v) / len(v), 4), "median": round(statistics.median(v), 4),
            "p10": round(pct(v, 0.10), 4), "p90": round(pct(v, 0.90), 4)}


def run_e2e(fp4, calls, steps):
    """Same step through the public API with host buffers: every step copies its inputs
    in from pinned host memory and its outputs back, inside the timed region. Pipelined as
    a user would run it: host->device copies on one stream, the grouped calls on the
    compute stream, device->host copies on a third, with two sets of device buffers so
    step i+1's inputs arrive and step i-1's outputs leave while step i computes. Events
    order every reuse of a buffer."""
    import torch
    dev = calls[0]["out"].device
    host_in, host_out, dev_in, dev_out = [], [], [[], []], [[], []]
    h2d = d2h = 0
    for c in calls:
        p = c["proj"]
        hx = p.x.cpu().pin_memory()
        hr = p.routing.row_ids.cpu().pin_memory()
        ho = p.routing.offsets.cpu().pin_memory()
        host_in.append((hx, hr, ho))
        for b in range(2):
            dev_in[b].append((torch.empty_like(p.x), torch.empty_like(p.routing.row_ids),
                              torch.empty_like(p.routing.offsets)))
            dev_out[b].append(torch.empty_like(c["out"]))
        host_out.append(torch.empty(c["out"].shape, dtype=torch.float32).pin_memory())
        h2d += hx.numel() * 4 + (hr.numel() * 4 if p.row_ids_used else 0) + ho.numel() * 4
        d2h += c["out"].numel() * 4
    comp = torch.cuda.current_stream()
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    inputs_read = [ev(), ev()]    # compute done with input buffer b
    outputs_read = [ev(), ev()]   # device->host copies done with output buffer b
    for b in range(2):
        inputs_read[b].record(comp)
        outputs_read[b].record(comp)

    def step(i):
        b = i & 1
        arrived = ev()
        with torch.cuda.stream(s_in):
            s_in.wait_event(inputs_read[b])
            for c, (hx, hr, ho), (dx, dr, do) in zip(calls, host_in, dev_in[b]):
                dx.copy_(hx, non_blocking=True)
                do.copy_(ho, non_blocking=True)
                if c["proj"].row_ids_used:
                    dr.copy_(hr, non_blocking=True)
            arrived.record(s_in)
        comp.wait_event(arrived)
        comp.wait_event(outputs_read[b])
        done = []
        for c, (dx, dr, do), dout in zip(calls, dev_in[b], dev_out[b]):
            p = c["proj"]
            fp4.fp4_grouped_expert_gemm(dx, dr if p.row_ids_used else None, do, p.bank.w,
                                        p.bank.sc, p.bank.scale2, p.bank.recipe, out=dout,
                                        workspace=c["ws"])
            e = ev()
            e.record(comp)
            done.append(e)
        inputs_read[b].record(comp)
        with torch.cuda.stream(s_out):
            for e, dout, hout in zip(done, dev_out[b], host_out):
                s_out.wait_event(e)
                hout.copy_(dout, non_blocking=True)
            outputs_read[b].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(steps):
        step(i)
    last = ev()
    last.record(s_out)
    comp.wait_event(last)
    t1.record(comp)
    torch.cuda.synchronize()
    # the host holds the last step's outputs
    ok = all(torch.equal(hout, dout.cpu()) for hout, dout in zip(host_out, dev_out[(steps - 1) & 1]))
    return t0.elapsed_time(t1) / steps, h2d, d2h, ok


def host_cpu():
    """Core count and CPU model of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return os.cpu_count() or 1, model or "unknown"


def cpu_sample_tasks(wl, frac=1.0 / 64, seed=0, rows_per_proj=None):
    """A seeded sample of the workload's routed rows for the CPU oracle: per projection,
    max(1, round(frac * rows)) random rows of every expert that has rows (or, with
    rows_per_proj, that many random routed rows). Each task is one routed row with its
    expert's weights as host arrays; all n columns of the row are computed."""
    import numpy as np
    rng = np.random.default_rng(seed)
    tasks = []
    for proj in wl.projections:
        b = proj.bank
        off = proj.routing.offsets.cpu().numpy().astype(np.int64)
        rid = proj.routing.row_ids.cpu().numpy()
        if rows_per_proj is None:
            picks = []
            for e in range(b.E):
                cnt = int(off[e + 1] - off[e])
                if cnt > 0:
                    m = max(1, int(round(frac * cnt)))
                    picks.extend((off[e] + rng.choice(cnt, size=m, replace=False)).tolist())
        else:
            picks = rng.integers(0, proj.routing.P, size=rows_per_proj).tolist()
        experts = np.searchsorted(off, np.asarray(picks, dtype=np.int64), side="right") - 1
        cache = {}
        for p, e in zip(picks, experts.tolist()):
            if e not in cache:
                cache[e] = (b.w[e].cpu().numpy(), b.sc[e].cpu().numpy(), float(b.scale2[e].item()))
            w, sc, s2 = cache[e]
            t = int(rid[p]) if proj.row_ids_used else int(p)
            tasks.append((proj.x[t:t + 1].cpu().numpy(), w, sc, s2, b.recipe, 2.0 * b.n * b.k))
    return tasks


def run_cpu_tasks(tasks, threads):
    """Time the oracle (as it stands: act_quant + the f64 reference of one routed row, all
    n columns) over the tasks on `threads` host threads. The oracle is C called through
    ctypes, which releases the GIL, so the threads run on separate cores. Returns seconds."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.act_quant(np.zeros((1, 128), dtype=np.float32))  # builds the oracle's tables once

    def one(t):
        x, w, sc, s2, recipe, _ = t
        codes, scales = oracle.act_quant(x)
        oracle.gemm_ref(codes, scales, w, sc, s2, recipe)

    t0 = time.perf_counter()
    if threads <= 1:
        for t in tasks:
            one(t)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, tasks))
    return time.perf_counter() - t0


def cpu_baseline(wl, flops_step, single_budget_s=12.0):
    """The oracle on the host cores over a seeded 1/64 row sample of the workload: all
    cores, and single-threaded on a bounded prefix of the same sample; per-FLOP
    extrapolation to one full step."""
    cores, model = host_cpu()
    tasks = cpu_sample_tasks(wl)
    fl_all = sum(t[-1] for t in tasks)
    secs_all = run_cpu_tasks(tasks, cores)
    rate_all = fl_all / secs_all
    # single thread: the same sample in order until about single_budget_s of work
    per_row_s = secs_all * cores / len(tasks)
    n1 = max(2, min(len(tasks), int(single_budget_s / max(per_row_s, 1e-6))))
    secs_1 = run_cpu_tasks(tasks[:n1], 1)
    rate_1 = sum(t[-1] for t in tasks[:n1]) / secs_1
    names = "+".join(p.name for p in wl.projections)
    return {"value": rate_all / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": model,
            "kind": "oracle",
            "sample": "%d routed rows (1/64 of each expert's rows, at least one per expert with "
                      "rows) x all n columns, act_quant + f64 reference, %s, on %d threads" % (
                          len(tasks), names, cores),
            "seconds": round(secs_all, 2),
            "single_thread": {"value": rate_1 / 1e12, "unit": "TFLOP/s", "rows": n1,
                              "seconds": round(secs_1, 2)},
            "extrapolated_s_per_step": round(flops_step / rate_all, 1),
            "extrapolated_s_per_step_single_thread": round(flops_step / rate_1, 1)}


def run_ours(args, world, rank, local):
    import torch
    import block_scaled_fp4_act_gb300 as fp4
    from block_scaled_fp4_act_gb300 import build as libbuild
    from block_scaled_fp4_act_gb300 import synth

    libbuild.build()
    fp4.lib()
    fp4.fp4_force_path({"auto": fp4.PATH_AUTO, "stream": fp4.PATH_STREAM,
                        "tc": fp4.PATH_TC}[args.path])
    device = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_src = load_peaks()

    kw = {}
    if args.experts:
        kw["E"] = args.experts
    if args.tokens:
        kw["T"] = args.tokens
    wl = synth.workload(args.workload, device=device, **kw)
    calls = make_calls(fp4, wl, device)
    flops_step = sum(proj_flops(c["proj"]) for c in calls)
    bytes_step = sum(proj_bytes(c["proj"])[0] for c in calls)
    for _ in range(max(3, args.warmup)):
        for c in calls:
            c["call"]()
    torch.cuda.synchronize()
    steps = args.steps
    if steps <= 0:
        el, _, _ = time_steps(calls, 3)
        steps = max(10, min(2000, int(2000.0 / max(el / 3, 1e-3))))
    steps = int(max_over_ranks(steps, world))

    barrier(world)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    elapsed, per_call, per_phase = time_steps(calls, steps)
    clk = clocks.stop()
    barrier(world)
    elapsed = max_over_ranks(elapsed, world)
    ms_step = elapsed / steps
    value = world * flops_step / (ms_step * 1e-3) / 1e12
    step_ms = [sum(per_call[i][s] for i in range(len(calls))) for s in range(steps)]

    # roofline of the dominant kernel: on the tensor-core path the GEMM kernel alone (its
    # launches timed apart from the quantise pass), else the streaming kernel
    paths = sorted({c["path"] for c in calls})
    call_ms = [sum(d) / len(d) for d in per_call]
    kflops = sum(proj_flops(c["proj"]) for c in calls)
    tc = all(c["path"] == fp4.PATH_TC for c in calls)
    if tc:
        gemm_ms = sum(sum(ph["gemm"]) / len(ph["gemm"]) for ph in per_phase)
        quant_ms = sum(sum(ph["quantize"]) / len(ph["quantize"]) for ph in per_phase)
        # both recipes run the kind::f16 MMA (16-bit operands, exact): bf16 dense peak
        peak = peaks["bf16_tflops"]
        achieved = kflops / (gemm_ms * 1e-3) / 1e12
        call_level = kflops / (sum(call_ms) * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "kernel": "tc_gemm_kernel",
                    "kernel_ms_per_step": round(gemm_ms, 4),
                    "traffic": ncu_traffic("tc_grouped_gemm/%s" % args.workload),
                    "traffic_basis": "DRAM bytes per step of the tc_gemm_kernel launches (one "
                                     "per projection), without the quantise pass",
                    "peak_source": peak_src + " bf16 dense (burst)",
                    # the FP8 dense rate (2x bf16, nominal ratio) for comparison with an
                    # FP8-MMA design; this path's exact products need 16-bit operands
                    "fp8_peak": round(2 * peak, 1), "frac_of_fp8": round(achieved / (2 * peak), 4),
                    "call_level": {"achieved": round(call_level, 2),
                                   "frac": round(call_level / peak, 4),
                                   "ms_per_step": round(sum(call_ms), 4),
                                   "what": "quantise pass + GEMM per grouped call"}}
        qbytes = sum(quant_bytes(c["proj"]) for c in calls)
        qgbs = qbytes / (quant_ms * 1e-3) / 1e9
        result_quant = {"kernel": "quant_ws_kernel", "ms_per_step": round(quant_ms, 4),
                        "bytes_per_step": qbytes,
                        "roofline": {"bound": "hbm", "achieved": round(qgbs, 1),
                                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": round(qgbs / peaks["hbm_gbs"], 4),
                                     "traffic": ncu_traffic("tc_quantize/%s" % args.workload),
                                     "peak_source": peak_src + " HBM copy bandwidth"},
                        "bytes_basis": "activation rows read once per token (f32), the 16-bit "
                                       "workspace row of every routed row written once"}
    else:
        # the streaming path is bound by HBM reads of the weights
        kms = sum(call_ms)
        kbytes = sum(proj_bytes(c["proj"])[0] for c in calls)
        achieved = kbytes / (kms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "kernel": STREAM_KERNEL,
                    "traffic": ncu_traffic("%s/%s" % (STREAM_KERNEL, args.workload)),
                    "traffic_basis": "DRAM bytes per step (all grouped calls)",
                    "peak_source": peak_src + " HBM copy bandwidth"}
        result_quant = None
    roofline["launches"] = steps * sum(c["launches"] for c in calls)
    roofline["per_call_ms"] = [round(m, 4) for m in call_ms]
    roofline["per_phase_ms"] = [{k: round(sum(v) / len(v), 4) for k, v in ph.items()}
                                for ph in per_phase]

    result = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
              "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "e4m3 x e2m1 -> f32 (tensor path: bf16 operands, f32 accumulate)"
              if tc else "e4m3 x e2m1 -> f32 (warp MMA: f16 or bf16 operands, f32 accumulate)",
              "data": "synthetic (seeded; weights, routing and activations as the workload "
                      "recipe states)",
              "config": {"workload": WORKLOAD_NAMES[args.workload] if not kw else
                         "%s with overrides %s" % (WORKLOAD_NAMES[args.workload], kw),
                         "paths": paths,
                         "flops_per_step": flops_step, "bytes_per_step": bytes_step,
                         "l2": "inputs larger than L2 (weights %.2f GB per step)" %
                               (sum(proj_bytes(c["proj"])[1] for c in calls) / 1e9),
                         "parallelism": "replicas x%d" % world},
              "step_ms": stats_ms(step_ms),
              "roofline": roofline, "clocks": clk,
              "gpu_launches": steps * sum(c["launches"] for c in calls)}
    if result_quant is not None:
        result["quantize"] = result_quant

    # the W4A4 variant on the same workload (its own numeric class: E2M1 activations)
    if args.workload == "c4" and not args.no_w4a4:
        result["w4a4"] = measure_w4a4(fp4, wl, result["config"]["workload"], peaks, peak_src,
                                      ms_step)

    # decode workload alongside: weight GB/s against HBM, L2 flushed between steps
    if args.workload == "c4" and not args.no_decode:
        wd = synth.decode_c3(device=device)
        dcalls = make_calls(fp4, wd, device)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        for _ in range(3):
            for c in dcalls:
                c["call"]()
        dsteps = 200
        _, dper, _ = time_steps(dcalls, dsteps, flush=flush)
        dms = [sum(d) / len(d) for d in dper]
        wsteps = time_whole_steps(dcalls, dsteps, flush=flush)
        step_ms = sum(wsteps) / len(wsteps)
        dbytes = sum(proj_bytes(c["proj"])[0] for c in dcalls)
        dweights = sum(proj_bytes(c["proj"])[1] for c in dcalls)
        gbs = dbytes / (step_ms * 1e-3) / 1e9
        result["decode"] = {
            "workload": WORKLOAD_NAMES["c3"], "value": round(world * dweights /
                                                              (step_ms * 1e-3) / 1e9, 1),
            "unit": "weight GB/s", "us_per_step": round(step_ms * 1e3, 2),
            "us_per_step_p10_p50_p90": [round(pct(wsteps, q) * 1e3, 2) for q in (0.1, 0.5, 0.9)],
            "us_per_call_timed_apart": [round(m * 1e3, 2) for m in dms],
            "timing": "events around the whole gate/up + down step; the per-call figures come "
                      "from a separate pass with an event between the calls",
            "steps": dsteps, "l2": "flushed (256 MB write) between steps",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": ncu_traffic(STREAM_KERNEL + "/c3"), "kernel": STREAM_KERNEL,
                         "traffic_basis": "DRAM bytes per step (gate/up + down)",
                         "bytes_per_step": dbytes, "peak_source": peak_src},
            "gpu_launches": dsteps * sum(c["launches"] for c in dcalls)}
        del dcalls, wd, flush

    # the mixed-recipe workload, reported per recipe and combined
    if args.workload == "c4" and not args.no_mixed:
        result["mixed"] = measure_mixed(fp4, synth, device, peaks, peak_src)

    # the step after the gate/up projection: SwiGLU + e4m3 requantisation of its output
    if args.workload == "c4" and not args.no_swiglu:
        result["swiglu_quant"] = measure_swiglu(fp4, device, peaks, peak_src)
        result["moe_chain"] = measure_moe_chain(fp4, device, peaks, peak_src)

    # the routing front-end (before and after the projections)
    if args.workload == "c4" and not args.no_routing:
        result["routing"] = measure_routing(fp4, device, peaks, peak_src)

    # end to end through the public API with host buffers
    if not args.no_e2e:
        e2e_steps = min(steps, 10)
        e2e_ms, h2d, d2h, e2e_ok = run_e2e(fp4, calls, e2e_steps)
        e2e_ms = max_over_ranks(e2e_ms, world)
        result["e2e"] = {"value": round(world * flops_step / (e2e_ms * 1e-3) / 1e12, 3),
                         "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                         "steps": e2e_steps, "outputs_match": e2e_ok,
                         "schedule": "copies in / grouped calls / copies out on three "
                                     "streams, double-buffered device inputs and outputs"}

    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, flops_step)
    return result


def run_reference(args, world, rank):
    """The oracle (as it stands) on all host cores: each step is a bounded sample of the
    same workload (16 random routed rows per projection, all n columns)."""
    import torch
    from block_scaled_fp4_act_gb300 import synth
    import oracle
    oracle.lib_path()
    device = "cuda" if torch.cuda.is_available() else "cpu"
    wl = synth.workload(args.workload, device=device)
    cores, model = host_cpu()
    rows = 16
    for i in range(args.warmup):
        run_cpu_tasks(cpu_sample_tasks(wl, seed=1000 + i, rows_per_proj=rows), cores)
    fl_tot, s_tot, ntasks = 0.0, 0.0, 0
    steps = args.steps if args.steps > 0 else 10
    step_s = []
    for i in range(steps):
        tasks = cpu_sample_tasks(wl, seed=i, rows_per_proj=rows)
        secs = run_cpu_tasks(tasks, cores)
        fl_tot += sum(t[-1] for t in tasks)
        s_tot += secs
        ntasks += len(tasks)
        step_s.append(secs * 1e3)
    value = fl_tot / s_tot / 1e12
    ms = s_tot / steps * 1e3
    desc = "%d random routed rows per projection per step x all n columns (act_quant + f64 " \
           "reference), %s, on %d threads" % (rows, "+".join(p.name for p in wl.projections), cores)
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "step_ms": stats_ms(step_s),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": WORKLOAD_NAMES[args.workload],
                       "sample": "%d random routed rows per projection per step" % rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                             "cpu_model": model, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def measure_mixed(fp4, synth, device, peaks, peak_src, steps=20):
    """The mixed workload: 128 NVFP4 + 128 MXFP4 experts [2048, 4096], 16,384 tokens
    top-8 uniform per recipe, one grouped call per recipe (inputs larger than L2). Both
    recipes run 16-bit kind::f16 MMAs (the exact route); each is shown against the bf16
    dense peak of that kind and against the FP8 dense rate (2x, nominal ratio)."""
    import torch
    wl = synth.mixed_c5(device=device)
    calls = make_calls(fp4, wl, device)
    for _ in range(3):
        for c in calls:
            c["call"]()
    _, per, phases = time_steps(calls, steps)
    ms = [sum(d) / len(d) for d in per]
    bf16 = peaks["bf16_tflops"]
    out = {"workload": WORKLOAD_NAMES["c5"], "steps": steps, "recipes": {}}
    tot_f = 0.0
    for c, m, ph in zip(calls, ms, phases):
        f = proj_flops(c["proj"])
        tot_f += f
        tf = f / (m * 1e-3) / 1e12
        rec = {"ms_per_call": round(m, 4), "tflops": round(tf, 1),
               "frac_bf16": round(tf / bf16, 4), "frac_fp8": round(tf / (2 * bf16), 4),
               "path": c["path"]}
        if "quantize" in ph:
            gm = sum(ph["gemm"]) / len(ph["gemm"])
            kt = f / (gm * 1e-3) / 1e12
            rec["gemm_kernel"] = {"ms": round(gm, 4), "tflops": round(kt, 1),
                                  "frac_bf16": round(kt / bf16, 4),
                                  "frac_fp8": round(kt / (2 * bf16), 4)}
            rec["quantize_ms"] = round(sum(ph["quantize"]) / len(ph["quantize"]), 4)
        out["recipes"][c["proj"].name] = rec
    tf_all = tot_f / (sum(ms) * 1e-3) / 1e12
    out["combined"] = {"ms_per_step": round(sum(ms), 4), "tflops": round(tf_all, 1),
                       "frac_bf16": round(tf_all / bf16, 4), "frac_fp8": round(tf_all / (2 * bf16), 4),
                       "peak_bf16": bf16, "peak_source": peak_src + " bf16 dense (burst); fp8 = 2x"}
    out["gpu_launches"] = steps * sum(c["launches"] for c in calls)
    del calls, wl
    torch.cuda.empty_cache()
    return out


def w4a4_gemm_bytes(proj):
    """Algorithmic bytes of one W4A4 GEMM launch: the touched experts' packed weights and
    e4m3 scales (+ scale2), the routed rows' packed codes, micro-scales and row scales read
    once, the f32 output written once."""
    import torch
    b = proj.bank
    touched = int(torch.count_nonzero(torch.diff(proj.routing.offsets)).item())
    P, k = proj.routing.P, b.k
    return touched * (b.n * (k // 2) + b.n * (k // 16) + 4) + P * (k // 2 + k // 16 + 4) + \
        P * b.n * 4


def w4a4_quant_bytes(proj):
    """Algorithmic bytes of the W4A4 quantise phase: each token row read once (f32), each
    routed row's codes, micro-scales and row scale written once."""
    T, k = proj.x.shape
    P = proj.routing.P
    return T * k * 4 + P * (k // 2 + k // 16 + 4)


def measure_w4a4(fp4, wl, workload_name, peaks, peak_src, w4a8_ms, steps=20):
    """The W4A4 NVFP4 variant (two-level E2M1 activations on the block-scaled 4-bit MMA) on
    the same projections: quantise phase and GEMM timed apart (CUDA events on the current
    stream), inputs larger than L2. The GEMM streams the expert weights once per tile
    column, so its roofline is HBM; its tensor rate is shown against the FP4 dense rate
    (6x the measured bf16 peak, the nominal FP4/bf16 ratio of this GPU)."""
    import torch
    calls = []
    for proj in wl.projections:
        T, k = proj.x.shape
        P = proj.routing.P
        ws = fp4.w4a4_workspace_for(T, P, k, proj.x.device)
        out = torch.empty(P, proj.bank.n, device=proj.x.device)
        rid = proj.routing.row_ids if proj.row_ids_used else None

        def quantize(proj=proj, ws=ws, rid=rid):
            fp4.fp4_w4a4_quantize(proj.x, rid, proj.routing.P, ws)

        def gemm(proj=proj, ws=ws, out=out, rid=rid):
            fp4.fp4_w4a4_gemm_quantized(ws, proj.x.shape[0], rid, proj.routing.offsets,
                                        proj.bank.w, proj.bank.sc, proj.bank.scale2, out)
        repeats = rid is not None and T < P
        calls.append({"proj": proj, "phases": [("quantize", quantize), ("gemm", gemm)],
                      "launches": 3 if repeats else 2, "ws": ws, "out": out})
    for _ in range(3):
        for c in calls:
            for _, fn in c["phases"]:
                fn()
    torch.cuda.synchronize()
    _, per, phases = time_steps(calls, steps)
    assert fp4.fp4_get_device_error() == 0
    ms = sum(sum(d) / len(d) for d in per)
    gemm_ms = sum(sum(ph["gemm"]) / len(ph["gemm"]) for ph in phases)
    quant_ms = sum(sum(ph["quantize"]) / len(ph["quantize"]) for ph in phases)
    flops = sum(proj_flops(c["proj"]) for c in calls)
    gbytes = sum(w4a4_gemm_bytes(c["proj"]) for c in calls)
    qbytes = sum(w4a4_quant_bytes(c["proj"]) for c in calls)
    hbm = peaks["hbm_gbs"]
    fp4_peak = 6 * peaks["bf16_tflops"]
    g_gbs = gbytes / (gemm_ms * 1e-3) / 1e9
    g_tf = flops / (gemm_ms * 1e-3) / 1e12
    q_gbs = qbytes / (quant_ms * 1e-3) / 1e9
    out = {"what": "W4A4 NVFP4 variant: E2M1 activations with a per-token row scale and an "
                   "e4m3 micro-scale per 16 values (kernel_check.rs, NVFP4 W4A4 MMQ GEMM "
                   "section), GEMM on tcgen05 kind::mxf4nvf4 with 4X ue4m3 scales",
           "workload": workload_name, "steps": steps,
           "ms_per_step": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
           "speedup_vs_w4a8_step": round(w4a8_ms / ms, 3),
           "per_call_ms": [round(sum(d) / len(d), 4) for d in per],
           "gemm": {"kernel": "w4a4_gemm_kernel", "ms_per_step": round(gemm_ms, 4),
                    "tflops": round(g_tf, 1), "frac_of_fp4": round(g_tf / fp4_peak, 4),
                    "fp4_peak": round(fp4_peak, 1),
                    "roofline": {"bound": "hbm", "achieved": round(g_gbs, 1), "peak": hbm,
                                 "unit": "GB/s", "frac": round(g_gbs / hbm, 4),
                                 "bytes_per_step": gbytes,
                                 "traffic": ncu_traffic("w4a4_gemm/c4"),
                                 "peak_source": peak_src + " HBM copy bandwidth"}},
           "quantize": {"ms_per_step": round(quant_ms, 4), "bytes_per_step": qbytes,
                        "roofline": {"bound": "hbm", "achieved": round(q_gbs, 1), "peak": hbm,
                                     "unit": "GB/s", "frac": round(q_gbs / hbm, 4)}},
           "gpu_launches": steps * sum(c["launches"] for c in calls)}
    del calls
    torch.cuda.empty_cache()
    return out


def measure_swiglu(fp4, device, peaks, peak_src, rows=32768, inter=1024, limit=7.0, iters=50):
    """Time fp4_swiglu_quant on the prefill gate/up output shape (fused [rows, 2*inter]
    layout, inputs 268 MB: larger than L2). HBM-bound: algorithmic bytes = 8 B read +
    1 B of code per element + 4 B of scale per 128."""
    import torch
    gen = torch.Generator(device=device).manual_seed(21)
    gu = torch.randn(rows, 2 * inter, generator=gen, device=device) * 3.0
    gu[::97] *= 50.0
    gate, up = gu[:, :inter], gu[:, inter:]
    codes = torch.empty(rows, inter, dtype=torch.uint8, device=device)
    scales = torch.empty(rows, inter // 128, dtype=torch.float32, device=device)
    call = lambda: fp4.fp4_swiglu_quant(gate, up, limit, codes=codes, scales=scales)
    for _ in range(3):
        call()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / iters
    nbytes = rows * inter * (4 + 4 + 1) + rows * (inter // 128) * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    del gu, codes, scales
    return {"workload": "SwiGLU (swiglu_limit %g) + e4m3 requantisation of the prefill gate/up "
                        "output [%d, 2x%d] f32" % (limit, rows, inter),
            "us_per_call": round(us, 2), "calls": iters,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "bytes_per_call": nbytes, "kernel": "swiglu_quant",
                         "peak_source": peak_src},
            "gpu_launches": iters}


def measure_moe_chain(fp4, device, peaks, peak_src, T=4096, E=256, topk=8, hidden=7168,
                      inter=2048, limit=7.0, steps=10):
    """The prefill MoE layer body on the tensor-core path, gate/up projection -> SwiGLU ->
    down projection (NVFP4, Zipf(1.1) top-8 routing, gate/up bank [2*inter, hidden], down
    bank [hidden, inter]), two ways: unfused (gate/up output [P, 2*inter] written, then
    fp4_swiglu_quant writes h) and fused (fp4_grouped_gate_up_swiglu writes h from the
    gate/up epilogue). The down call quantises h itself (the requantisation)."""
    import torch
    from block_scaled_fp4_act_gb300 import synth
    r = synth.zipf_topk(T, E, topk, 2004, device)
    gen = torch.Generator(device=device).manual_seed(4)
    x = synth.bf16_rounded(torch.randn(T, hidden, generator=gen, device=device))
    gu = synth.make_bank(fp4.NVFP4, E, 2 * inter, hidden, 1104, device)
    dn = synth.make_bank(fp4.NVFP4, E, hidden, inter, 1105, device)
    P = r.P
    ws1 = fp4.workspace_for(T, P, 2 * inter, hidden, fp4.NVFP4, device=device)
    ws2 = fp4.workspace_for(P, P, hidden, inter, fp4.NVFP4, device=device)
    gu_out = torch.empty(P, 2 * inter, device=device)
    h = torch.empty(P, inter, device=device)
    d = torch.empty(P, hidden, device=device)
    codes = torch.empty(P, inter, dtype=torch.uint8, device=device)
    scales = torch.empty(P, inter // 128, dtype=torch.float32, device=device)

    def down():
        fp4.fp4_grouped_expert_gemm(h, None, r.offsets, dn.w, dn.sc, dn.scale2, fp4.NVFP4,
                                    out=d, workspace=ws2)

    def unfused():
        fp4.fp4_grouped_expert_gemm(x, r.row_ids, r.offsets, gu.w, gu.sc, gu.scale2, fp4.NVFP4,
                                    out=gu_out, workspace=ws1)
        fp4.fp4_swiglu_quant(gu_out[:, :inter], gu_out[:, inter:], limit, codes=codes,
                             scales=scales, h_out=h)
        down()

    def fused():
        fp4.fp4_grouped_gate_up_swiglu(x, r.row_ids, r.offsets, gu.w, gu.sc, gu.scale2,
                                       fp4.NVFP4, limit, ws1, h=h)
        down()

    stream = torch.cuda.current_stream()
    res = {}
    for name, fn in (("unfused", unfused), ("fused", fused)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / steps
    h_fused = h.clone()
    unfused()
    torch.cuda.synchronize()
    same = bool(torch.equal(h, h_fused))
    flops = 2.0 * P * (2 * inter) * hidden + 2.0 * P * hidden * inter
    out = {"workload": "prefill MoE layer body, NVFP4: %d experts, %d tokens top-%d Zipf(1.1), "
                       "gate/up [2x%d, %d] -> SwiGLU (swiglu_limit %g) -> down [%d, %d]" % (
                           E, T, topk, inter, hidden, limit, hidden, inter),
           "unfused_ms": round(res["unfused"], 4), "fused_ms": round(res["fused"], 4),
           "saving_ms": round(res["unfused"] - res["fused"], 4),
           "fused_tflops": round(flops / (res["fused"] * 1e-3) / 1e12, 1),
           "h_bit_equal": same, "steps": steps,
           "what": "fused: h from the gate/up epilogue; unfused: gate/up output written, then "
                   "fp4_swiglu_quant"}
    del gu, dn, ws1, ws2, gu_out, h, d, x
    torch.cuda.empty_cache()
    return out


def measure_routing(fp4, device, peaks, peak_src, T=4096, E=256, topk=8, n=7168, iters=50):
    """The routing front-end at the prefill shapes: the router over [T, E] logits, the CSR
    construction of T x topk routed rows, and the weighted combine of the down projection's
    output [T*topk, n] back to [T, n] (HBM-bound: every routed row read once, y written
    once). Not part of the projection step."""
    import torch
    gen = torch.Generator(device=device).manual_seed(33)
    logits = torch.randn(T, E, generator=gen, device=device)
    ids, w = fp4.fp4_route_topk(logits, topk, renormalize=True)
    ws = torch.empty(max(16, int(fp4.lib().fp4_route_csr_workspace_size(T, E))), dtype=torch.uint8,
                     device=device)
    off, rid, prow = fp4.fp4_route_csr(ids, E, workspace=ws)
    out = torch.randn(T * topk, n, generator=gen, device=device)
    y = torch.empty(T, n, device=device)
    calls = {"route_topk": lambda: fp4.fp4_route_topk(logits, topk, renormalize=True, ids=ids,
                                                      weights=w),
             "route_csr": lambda: fp4.fp4_route_csr(ids, E, workspace=ws, offsets=off,
                                                    row_ids=rid, pair_rows=prow),
             "moe_combine": lambda: fp4.fp4_moe_combine(out, prow, w, y=y)}
    res = {"workload": "router over [%d, %d] logits top-%d, CSR of %d routed rows, combine of "
                       "[%d, %d] f32 into [%d, %d]" % (T, E, topk, T * topk, T * topk, n, T, n)}
    stream = torch.cuda.current_stream()
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name + "_us"] = round(e0.elapsed_time(e1) * 1e3 / iters, 2)
    nbytes = T * topk * n * 4 + T * n * 4 + T * topk * 8
    gbs = nbytes / (res["moe_combine_us"] * 1e-6) / 1e9
    res["combine_roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                               "bytes_per_call": nbytes, "kernel": "moe_combine_kernel",
                               "peak_source": peak_src}
    res["gpu_launches"] = iters * (1 + 4 + 1)
    del out, y
    return res


def path_sweep(rows_per_expert=(2, 4, 8, 16, 24, 32, 48, 64), E=64, n=3072, k=4096, iters=20):
    """Both grouped paths (no-workspace and tensor-core) on 64 NVFP4 experts [3072, 4096]
    with exactly r routed rows per expert, L2 flushed before each call; median microseconds.
    One JSON line per r."""
    import torch
    import block_scaled_fp4_act_gb300 as fp4
    from block_scaled_fp4_act_gb300 import synth
    dev = "cuda"
    bank = synth.make_bank(fp4.NVFP4, E, n, k, 77, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for rpe in rows_per_expert:
        T = rpe * E // 8
        # each token picks 8 distinct experts; round-robin blocks give exactly rpe per expert
        choices = torch.stack([torch.arange(8) + 8 * (t % (E // 8)) for t in range(T)])
        r = synth.routing_from_choices(choices, E)
        gen = torch.Generator(device="cpu").manual_seed(rpe)
        x = torch.randn(T, k, generator=gen).to(dev)
        rid, off = r.row_ids.to(dev), r.offsets.to(dev)
        ws = fp4.workspace_for(T, r.P, n, k, fp4.NVFP4, device=dev)
        us = {}
        for name, path in (("no_workspace", fp4.PATH_STREAM), ("tensor_core", fp4.PATH_TC)):
            fp4.fp4_force_path(path)
            try:
                def call():
                    fp4.fp4_grouped_expert_gemm(x, rid, off, bank.w, bank.sc, bank.scale2,
                                                fp4.NVFP4, workspace=ws)
                for _ in range(3):
                    call()
                ts = []
                for _ in range(iters):
                    flush.fill_(1)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    call()
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1000.0)
            finally:
                fp4.fp4_force_path(fp4.PATH_AUTO)
            ts.sort()
            us[name] = round(ts[len(ts) // 2], 1)
        auto = fp4.fp4_gemm_path(r.P, E, n, k, fp4.NVFP4, True)
        print(json.dumps({"rows_per_expert": rpe, "routed_rows": r.P, "us": us,
                          "auto_path": "tensor_core" if auto == fp4.PATH_TC else "no_workspace"}),
              flush=True)


def main():
    args = parse_args()
    if args.path_sweep:
        path_sweep()
        return
    if args.impl == "reference":
        # the oracle arm runs on rank 0 only; other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    world, rank, local = dist_setup()
    result = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
