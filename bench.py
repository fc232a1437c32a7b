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
    "tc_grouped_gemm": ["gemm_tc.cu", "common.cuh", "internal.h", "tma_host.h"],
    "stream_gemm": ["gemm_stream.cu", "common.cuh", "internal.h"],
    "decode_mma": ["gemm_decode.cu", "common.cuh", "internal.h"],
}

# The no-workspace path runs the warp-MMA decode kernel for every k up to 28544, which
# covers each workload here; the FMA streaming kernel takes larger k only.
STREAM_KERNEL = "decode_mma"


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


def launches_per_call(fp4, proj, have_ws):
    """Kernels of ours one grouped call launches: the streaming kernel alone, or the
    tensor-core path's quantise pass(es) + GEMM (NVFP4: f16 pass, conditional bf16 pass)."""
    path = fp4.fp4_gemm_path(proj.routing.P, proj.bank.E, proj.bank.n, proj.bank.k,
                             proj.bank.recipe, have_ws)
    if path != fp4.PATH_TC:
        return path, 1
    return path, (3 if proj.bank.recipe == fp4.NVFP4 else 2)


# ------------------------------------------------------------------ our arm

def make_calls(fp4, wl, device):
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
        calls.append({"proj": proj, "call": call, "out": out, "ws": ws, "path": path,
                      "launches": nl})
    return calls


def time_steps(calls, steps, flush=None):
    """Run `steps` steps; per call, CUDA events on the launching (current) stream.
    Returns (elapsed ms of the whole region, per-call list of durations in ms)."""
    import torch
    stream = torch.cuda.current_stream()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in calls] for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(steps):
        if flush is not None:
            flush.zero_()
        for i, c in enumerate(calls):
            evs[s][i][0].record(stream)
            c["call"]()
            evs[s][i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    per_call = [[evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(steps)]
                for i in range(len(calls))]
    return t0.elapsed_time(t1), per_call


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


def cpu_oracle_sample(wl, budget_s, rows_cap=None, seed=0):
    """Time the CPU oracle (as it stands, single-threaded C) on a bounded sample of the
    workload's routed rows, all n columns each. Returns (flops, seconds, description)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    flops = 0.0
    secs = 0.0
    rows_done = 0
    per_proj = budget_s / len(wl.projections)
    for proj in wl.projections:
        b = proj.bank
        off = proj.routing.offsets.cpu().numpy().astype(np.int64)
        rid = proj.routing.row_ids.cpu().numpy()
        P = proj.routing.P
        t_start = time.perf_counter()
        done_here = 0
        while True:
            p = int(rng.integers(0, P))
            e = int(np.searchsorted(off, p, side="right") - 1)
            t = int(rid[p]) if proj.row_ids_used else p
            x = proj.x[t:t + 1].cpu().numpy()
            w = b.w[e].cpu().numpy()
            sc = b.sc[e].cpu().numpy()
            s2 = float(b.scale2[e].item())
            t1 = time.perf_counter()
            codes, scales = oracle.act_quant(x)
            oracle.gemm_ref(codes, scales, w, sc, s2, b.recipe)
            secs += time.perf_counter() - t1
            flops += 2.0 * b.n * b.k
            done_here += 1
            rows_done += 1
            if rows_cap is not None and done_here >= rows_cap:
                break
            if time.perf_counter() - t_start >= per_proj and done_here >= 2:
                break
    desc = "%d random routed rows x all n columns (act_quant + f64 reference), %s" % (
        rows_done, "+".join(p.name for p in wl.projections))
    return flops, secs, desc


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
        el, _ = time_steps(calls, 3)
        steps = max(10, min(2000, int(2000.0 / max(el / 3, 1e-3))))
    steps = int(max_over_ranks(steps, world))

    barrier(world)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    elapsed, per_call = time_steps(calls, steps)
    clk = clocks.stop()
    barrier(world)
    elapsed = max_over_ranks(elapsed, world)
    ms_step = elapsed / steps
    value = world * flops_step / (ms_step * 1e-3) / 1e12

    # roofline of the dominant kernel: the grouped GEMM call (all launches of it)
    paths = sorted({c["path"] for c in calls})
    call_ms = [sum(d) / len(d) for d in per_call]
    kflops = sum(proj_flops(c["proj"]) for c in calls)
    kms = sum(call_ms)
    tc = all(c["path"] == fp4.PATH_TC for c in calls)
    if tc:
        # both recipes run the bf16 kind::f16 MMA (operands bf16, exact): bf16 dense peak
        peak = peaks["bf16_tflops"]
        achieved = kflops / (kms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "kernel": "tc_grouped_gemm",
                    "traffic": ncu_traffic("tc_grouped_gemm/%s" % args.workload),
                    "traffic_basis": "DRAM bytes per step (all grouped calls)",
                    "peak_source": peak_src + " bf16 dense (burst)",
                    # the FP8 dense rate (2x bf16, nominal ratio) for comparison with an
                    # FP8-MMA design; this path's exact products need 16-bit operands
                    "fp8_peak": round(2 * peak, 1), "frac_of_fp8": round(achieved / (2 * peak), 4)}
    else:
        # the streaming path is bound by HBM reads of the weights
        kbytes = sum(proj_bytes(c["proj"])[0] for c in calls)
        achieved = kbytes / (kms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "kernel": STREAM_KERNEL,
                    "traffic": ncu_traffic("%s/%s" % (STREAM_KERNEL, args.workload)),
                    "traffic_basis": "DRAM bytes per step (all grouped calls)",
                    "peak_source": peak_src + " HBM copy bandwidth"}
    roofline["launches"] = steps * sum(c["launches"] for c in calls)
    roofline["per_call_ms"] = [round(m, 4) for m in call_ms]

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
              "roofline": roofline, "clocks": clk,
              "gpu_launches": steps * sum(c["launches"] for c in calls)}

    # decode workload alongside: weight GB/s against HBM, L2 flushed between steps
    if args.workload == "c4" and not args.no_decode:
        wd = synth.decode_c3(device=device)
        dcalls = make_calls(fp4, wd, device)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        for _ in range(3):
            for c in dcalls:
                c["call"]()
        dsteps = 200
        _, dper = time_steps(dcalls, dsteps, flush=flush)
        dms = [sum(d) / len(d) for d in dper]
        dbytes = sum(proj_bytes(c["proj"])[0] for c in dcalls)
        dweights = sum(proj_bytes(c["proj"])[1] for c in dcalls)
        gbs = dbytes / (sum(dms) * 1e-3) / 1e9
        result["decode"] = {
            "workload": WORKLOAD_NAMES["c3"], "value": round(world * dweights /
                                                              (sum(dms) * 1e-3) / 1e9, 1),
            "unit": "weight GB/s", "us_per_step": round(sum(dms) * 1e3, 2),
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
        fl, secs, desc = cpu_oracle_sample(wl, 12.0)
        result["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": 1,
                                  "kind": "oracle", "sample": desc,
                                  "seconds": round(secs, 2)}
    return result


def run_reference(args, world, rank):
    """The oracle (as it stands) on the host cores: each step is a bounded sample of the
    same workload (16 random routed rows per projection, all n columns)."""
    import torch
    from block_scaled_fp4_act_gb300 import synth
    import oracle
    oracle.lib_path()
    device = "cuda" if torch.cuda.is_available() else "cpu"
    wl = synth.workload(args.workload, device=device)
    rows = 16
    for i in range(args.warmup):
        cpu_oracle_sample(wl, 1e9, rows_cap=rows, seed=1000 + i)
    fl_tot, s_tot = 0.0, 0.0
    steps = args.steps if args.steps > 0 else 10
    for i in range(steps):
        fl, secs, desc = cpu_oracle_sample(wl, 1e9, rows_cap=rows, seed=i)
        fl_tot += fl
        s_tot += secs
    value = fl_tot / s_tot / 1e12
    ms = s_tot / steps * 1e3
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": WORKLOAD_NAMES[args.workload],
                       "sample": "%d random routed rows per projection per step" % rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
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
    _, per = time_steps(calls, steps)
    ms = [sum(d) / len(d) for d in per]
    bf16 = peaks["bf16_tflops"]
    out = {"workload": WORKLOAD_NAMES["c5"], "steps": steps, "recipes": {}}
    tot_f = 0.0
    for c, m in zip(calls, ms):
        f = proj_flops(c["proj"])
        tot_f += f
        tf = f / (m * 1e-3) / 1e12
        out["recipes"][c["proj"].name] = {
            "ms_per_call": round(m, 4), "tflops": round(tf, 1),
            "frac_bf16": round(tf / bf16, 4), "frac_fp8": round(tf / (2 * bf16), 4),
            "path": c["path"]}
    tf_all = tot_f / (sum(ms) * 1e-3) / 1e12
    out["combined"] = {"ms_per_step": round(sum(ms), 4), "tflops": round(tf_all, 1),
                       "frac_bf16": round(tf_all / bf16, 4), "frac_fp8": round(tf_all / (2 * bf16), 4),
                       "peak_bf16": bf16, "peak_source": peak_src + " bf16 dense (burst); fp8 = 2x"}
    out["gpu_launches"] = steps * sum(c["launches"] for c in calls)
    del calls, wl
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
