"""Benchmark of the fused shifted-window attention on GB300.

A step is one pass of the hot path over the Swin-L 224 stage sweep at batch 64: the
fused forward of each of the four stages (56x56 C=192 nH=6 s=3; 28x28 C=384 nH=12 s=3;
14x14 C=768 nH=24 s=3; 7x7 C=1536 nH=48 s=0; window 7, bf16), with the dense bias and
shift mask built once per plan. The line also reports the Swin-B 224 training step (bias
re-expansion + forward + backward of its four stages) as `train_step`, and the whole
attention sub-block of the same sweep (LayerNorm + qkv projection, the attention, output
projection + bias + residual), captured as one CUDA graph, as `block_sweep`.

Prints one JSON line (rank 0). `value` is tokens/s over the whole job with inputs
resident in HBM; `e2e` is the same metric through the host-buffer entry point, with the
host<->device copies inside the timed region. `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from swin_window_attention_gb300 import dp, inputs  # noqa: E402

METRIC = "fused SW-MSA fwd/bwd tokens/s on 1 GB300; achieved HBM GB/s as % of roofline"
SWEEP = ["swin_l224_s1", "swin_l224_s2", "swin_l224_s3", "swin_l224_s4"]
TRAIN = ["swin_b224_s1", "swin_b224_s2", "swin_b224_s3", "swin_b224_s4"]
L384 = ["swin_l384_s1", "swin_l384_s2", "swin_l384_s3", "swin_l384_s4"]
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---- algorithmic work per launch --------------------------------------------------------

def fwd_bytes(wl) -> int:
    """qkv read + output write + dense bias + shift mask (s > 0)."""
    esz = 2 if wl.dtype == "bf16" else 4
    nn = wl.N * wl.N
    return (wl.tokens * 4 * wl.C * esz + wl.nH * nn * 4 + (wl.nW * nn * 4 if wl.s > 0 else 0))


def fwd_fp8_bytes(wl) -> int:
    """8-bit forward: qkv read at 3C bytes per token, bf16 output write, bias and mask."""
    nn = wl.N * wl.N
    return wl.tokens * 5 * wl.C + wl.nH * nn * 4 + (wl.nW * nn * 4 if wl.s > 0 else 0)


def bwd_bytes(wl) -> int:
    """qkv (3C) + dO (C) read, dqkv (3C) write, dense bias, mask, table gradient write."""
    esz = 2 if wl.dtype == "bf16" else 4
    nn = wl.N * wl.N
    return (wl.tokens * 7 * wl.C * esz + wl.nH * nn * 4 + (wl.nW * nn * 4 if wl.s > 0 else 0)
            + (2 * wl.M - 1) ** 2 * wl.nH * 4)


def fwd_flops(wl) -> int:
    return 4 * wl.N * wl.N * wl.hd * wl.window_heads


def bwd_flops(wl) -> int:
    return 10 * wl.N * wl.N * wl.hd * wl.window_heads


def qkv_bytes(wl) -> int:
    """Producer: x read, qkv written, W read (bf16)."""
    return 2 * (wl.tokens * wl.C + wl.tokens * 3 * wl.C + 3 * wl.C * wl.C)


def qkv_flops(wl) -> int:
    return 2 * wl.tokens * wl.C * 3 * wl.C


def proj_bytes(wl) -> int:
    """Consumer: attention output and residual read, y written, Wp read (bf16)."""
    return 2 * (3 * wl.tokens * wl.C + wl.C * wl.C)


def proj_flops(wl) -> int:
    return 2 * wl.tokens * wl.C * wl.C


def gemm_roofline(nbytes, flops, ms, peaks):
    """The binding roofline of a GEMM step timed alone: the larger of its HBM time
    (measured copy bandwidth) and its tensor time (measured bf16 burst rate)."""
    t_hbm = nbytes / (float(peaks["hbm_gbs"]) * 1e9)
    t_tc = flops / (float(peaks["bf16_tflops"]) * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {"us": round(ms * 1e3, 2), "bound": bound,
            "frac": round(max(t_hbm, t_tc) / (ms / 1e3), 4),
            "GBps": round(nbytes / (ms / 1e3) / 1e9, 1),
            "tflops": round(flops / (ms / 1e3) / 1e12, 1)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The files the forward kernel is compiled from: its DRAM traffic recorded by ncu stays
# valid while these are unchanged.
FWD_KERNEL_FILES = ("common.cuh", "fwd.cu", "tc.cuh")


def kernel_source_hash(files=FWD_KERNEL_FILES) -> str:
    """Short hash of the named csrc files (None: every file under csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "swin_window_attention_gb300", "csrc")
    for name in sorted(os.listdir(csrc) if files is None else files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_hash: str):
    """Per-launch DRAM bytes of the forward kernel on the first sweep stage, from the
    committed ncu summary, if it was captured on the forward kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "fwd_swin_l224_s1_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_launch")


# ---- clocks -----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; only samples taken while the
    timed region ran (by wall clock) count."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.1 <= r[0] <= self.t1 + 0.1]
        if not inside and rows and self.t0 is not None:
            inside = [min(rows, key=lambda r: abs(r[0] - self.t0))]
        reasons = set()
        for r in inside:
            for n, v in zip(self.NAMES, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": inside[0][2] if inside else None, "reasons": sorted(reasons),
                "samples": len(inside), "timed_region_s": round((self.t1 or 0) - (self.t0 or 0), 3)}


# ---- GPU arm ----------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(wls, target_s: float = 12.0):
    """The fp64 oracle, as it stands, on host cores: images of the sweep one at a time,
    round-robin over the stages, until about `target_s` seconds have been spent."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    data = []
    for wl in wls:
        one = wl.with_batch(1)
        q = inputs.act_f64(inputs.make_qkv(one))
        t = inputs.make_table(wl).double().numpy()
        data.append((wl, q, t))
    tokens, images, t0 = 0, 0, time.perf_counter()
    while True:
        for wl, q, t in data:
            oracle.fwd(q, t, wl.nH, wl.M, wl.s)
            tokens += wl.H * wl.W
            images += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": tokens / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{images} images ({images // len(data)} per stage) of the sweep, "
                      f"batch 1 each, {el:.1f} s wall"}


def run_gpu(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from swin_window_attention_gb300 import build, capi
    if rank == 0 or ws == 1:
        build.build()
    barrier(ws)
    lib = capi.load()
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream

    # ---- inference sweep: plans and resident inputs ------------------------------------
    sweep = [inputs.BY_NAME[n] for n in (args.workload or SWEEP)]
    plans, qkvs, outs, hosts = [], [], [], []
    with torch.cuda.stream(stream):
        for wl in sweep:
            q = inputs.make_qkv(wl)
            tab = inputs.make_table(wl).to(dev)
            h = make_plan(capi, wl, tab, sh, args)
            plans.append(h)
            qkvs.append(q.to(dev))
            outs.append(torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16, device=dev))
            hosts.append((q.pin_memory(),
                          torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16).pin_memory()))
    torch.cuda.synchronize()

    def step(events=None):
        for k, (h, q, o) in enumerate(zip(plans, qkvs, outs)):
            if events is not None:
                events[k][0].record(stream)
            rc = lib.swin_wattn_fwd(h, q.data_ptr(), o.data_ptr(), sh)
            if events is not None:
                events[k][1].record(stream)
            if rc != capi.OK:
                raise capi.SwinWAttnError("swin_wattn_fwd", rc)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The step as one CUDA graph (four forward launches), replayed for the headline
    # number: no host launch gaps between the stages.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize()

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in sweep]
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(args.steps):
            graph.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, ws)
    launches = len(sweep) * args.steps  # kernels inside the replayed graphs

    # Second timed region, same steps launched one by one with CUDA events around every
    # launch: per-stage durations for the roofline of each kernel.
    capi.swin_wattn_launch_count(reset=True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    eager_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    eager_launches = capi.swin_wattn_launch_count()
    clk = clocks.stop()

    # Third timed region: the same graph replayed for at least a second, so that the step
    # time is also known at the clock the GPU settles to under sustained load (the kernels
    # are paced by instruction issue, so their speed follows the SM clock).
    step_s = total_ms / args.steps / 1e3
    sus_steps = args.steps if args.skip_sustained else max(args.steps, int(math.ceil(1.0 / max(step_s, 1e-9))))
    clocks2 = ClockSampler(local)
    clocks2.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks2.mark(True)
    with torch.cuda.stream(stream):
        s0.record(stream)
        for _ in range(sus_steps):
            graph.replay()
        s1.record(stream)
    torch.cuda.synchronize()
    clocks2.mark(False)
    barrier(ws)
    sus_ms = max_over_ranks(s0.elapsed_time(s1), ws)
    clk2 = clocks2.stop()
    # per-stage launch times: the median over the timed steps
    per_stage_ms = [statistics.median(ev[i][k][0].elapsed_time(ev[i][k][1])
                                      for i in range(args.steps)) for k in range(len(sweep))]

    tokens_step = sum(wl.tokens for wl in sweep)
    value = ws * tokens_step * args.steps / (total_ms / 1e3)
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])

    stages = []
    for wl, ms in zip(sweep, per_stage_ms):
        gbs = fwd_bytes(wl) / (ms / 1e3) / 1e9
        stages.append({"workload": wl.name, "us": round(ms * 1e3, 2),
                       "tokens_per_s": wl.tokens / (ms / 1e3),
                       "window_heads_per_s": wl.window_heads / (ms / 1e3), "GBps": round(gbs, 1),
                       "frac_of_measured_hbm": round(gbs / hbm, 4),
                       "tflops": round(fwd_flops(wl) / (ms / 1e3) / 1e12, 1)})
    sweep_bytes = sum(fwd_bytes(wl) for wl in sweep)
    sweep_ms = sum(per_stage_ms)

    # dominant kernel: the largest share of the step
    kdom = max(range(len(sweep)), key=lambda k: per_stage_ms[k])
    wdom = sweep[kdom]
    ach = fwd_bytes(wdom) / (per_stage_ms[kdom] / 1e3) / 1e9
    khash = kernel_source_hash()
    roofline = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": ncu_traffic(khash) if wdom.name == "swin_l224_s1" else None,
                "kernel": f"{kernel_name(capi, plans[kdom])} on {wdom.name}",
                "bytes_per_launch": fwd_bytes(wdom), "peak_source": peak_src + " hbm_gbs",
                "kernel_source_hash": khash}

    # ---- end to end through the host-buffer entry point --------------------------------
    e2e_steps = max(3, min(args.steps, 20))
    h2d = sum(q.numel() * q.element_size() for q, _ in hosts)
    d2h = sum(o.numel() * o.element_size() for _, o in hosts)

    def e2e_step():
        for h, q, o, (qh, oh) in zip(plans, qkvs, outs, hosts):
            rc = lib.swin_wattn_fwd_host(h, qh.data_ptr(), oh.data_ptr(), q.data_ptr(),
                                         o.data_ptr(), sh)
            if rc != capi.OK:
                raise capi.SwinWAttnError("swin_wattn_fwd_host", rc)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    e2e = {"value": ws * tokens_step * e2e_steps / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "entry_point": "swin_wattn_fwd_host (pinned host buffers)", "steps": e2e_steps}

    for h in plans:
        capi.swin_wattn_destroy(h)
    del qkvs, outs, hosts
    torch.cuda.empty_cache()

    train = run_train_step(args, dev, stream, lib, capi, hbm, ws) if not args.skip_train else None
    l384 = run_fwd_sweep(L384, args, dev, stream, lib, capi, hbm, ws) if not args.skip_train else None
    block = run_block_sweep(SWEEP, args, dev, stream, lib, capi, peaks, ws) if not args.skip_train else None
    fp8 = run_fp8_sweep(SWEEP, args, dev, stream, lib, capi, hbm, ws) if not args.skip_train else None
    block8 = (run_block_sweep(SWEEP, args, dev, stream, lib, capi, peaks, ws, fp8=True)
              if not args.skip_train else None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) qkv, trunc-normal table)",
            "config": {"workload": "swin_l224_sweep_fwd", "batch_per_gpu": 64, "window": 7,
                       "stages": [f"{w.H}x{w.W} C={w.C} nH={w.nH} s={w.s}" for w in sweep],
                       "tokens_per_step_per_gpu": tokens_step,
                       "algorithmic_bytes_per_step": sweep_bytes,
                       "l2": f"step working set {sweep_bytes / 1e6:.0f} MB > 129 MB L2 "
                             "(stages run in turn; each stage's inputs are evicted by the "
                             "others' before they are read again); no flush",
                       "parallelism": f"dp{ws} (independent batch shards, no collective)",
                       "fwd_kernel": kernel_name(capi, plans[0])},
            "roofline": roofline,
            "sweep": {"us": round(sweep_ms * 1e3, 2),
                      "window_heads_per_s": sum(wl.window_heads for wl in sweep) / (sweep_ms / 1e3),
                      "GBps": round(sweep_bytes / (sweep_ms / 1e3) / 1e9, 1),
                      "frac_of_measured_hbm": round(sweep_bytes / (sweep_ms / 1e3) / 1e9 / hbm, 4),
                      "stages": stages},
            "e2e": e2e,
            "gpu_launches": int(launches),
            "timing": {"value_from": "CUDA-graph replays of the step (4 forward launches each)",
                       "eager_ms_per_step": eager_ms / args.steps,
                       "eager_launches": int(eager_launches),
                       "per_stage_from": "CUDA events around each launch in a second, eager "
                                         "timed region of the same steps (median per stage)"},
            "clocks": clk,
            "sustained": {
                "what": "the same graph replayed for at least 1 s in a third timed region, with "
                        "its own clock samples (reported beside the driver-length headline)",
                "steps": sus_steps, "seconds": round(sus_ms / 1e3, 3),
                "us_per_step": round(sus_ms / sus_steps * 1e3, 2),
                "tokens_per_s": ws * tokens_step * sus_steps / (sus_ms / 1e3),
                "frac_of_measured_hbm": round(sweep_bytes / (sus_ms / sus_steps / 1e3) / 1e9 / hbm, 4),
                "clocks": clk2,
                "us_x_median_sm_mhz": (round(sus_ms / sus_steps * 1e3 * clk2["sm_mhz"], 1)
                                       if clk2.get("sm_mhz") else None),
                "headline_us_x_median_sm_mhz": (round(total_ms / args.steps * 1e3 * clk["sm_mhz"], 1)
                                                if clk.get("sm_mhz") else None)},
            "train_step": train,
            "l384_sweep": l384,
            "block_sweep": block,
            "fp8_sweep": fp8,
            "fp8_block_sweep": block8,
        }
        if ws == 1 and not args.skip_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(sweep)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_fwd_sweep(names, args, dev, stream, lib, capi, hbm, ws):
    """Forward of another stage sweep (context for the line: the 12x12-window Swin-L 384
    sweep), per stage with CUDA events."""
    sh = stream.cuda_stream
    wls = [inputs.BY_NAME[n] for n in names]
    st = []
    with torch.cuda.stream(stream):
        for wl in wls:
            tab = inputs.make_table(wl).to(dev)
            h = make_plan(capi, wl, tab, sh, args)
            q = inputs.make_qkv(wl).to(dev)
            st.append(dict(wl=wl, h=h, q=q, o=torch.empty(wl.B, wl.H, wl.W, wl.C,
                                                         dtype=torch.bfloat16, device=dev)))
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 200))
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in st] for _ in range(steps + 3)]
    for i in range(steps + 3):
        for k, x in enumerate(st):
            ev[i][k][0].record(stream)
            if lib.swin_wattn_fwd(x["h"], x["q"].data_ptr(), x["o"].data_ptr(), sh) != capi.OK:
                raise RuntimeError("forward failed")
            ev[i][k][1].record(stream)
    torch.cuda.synchronize()
    out, tot_b, tot_ms = [], 0, 0.0
    for k, x in enumerate(st):
        wl = x["wl"]
        ms = statistics.mean(ev[i][k][0].elapsed_time(ev[i][k][1]) for i in range(3, steps + 3))
        tot_b += fwd_bytes(wl)
        tot_ms += ms
        out.append({"workload": wl.name, "us": round(ms * 1e3, 2),
                    "frac_of_measured_hbm": round(fwd_bytes(wl) / (ms / 1e3) / 1e9 / hbm, 4),
                    "tflops": round(fwd_flops(wl) / (ms / 1e3) / 1e12, 1),
                    "fwd_kernel": "tcgen05" if capi.swin_wattn_fwd_kernel(x["h"]) == capi.KERNEL_TCGEN05
                    else "mma.sync"})
        capi.swin_wattn_destroy(x["h"])
    return {"workload": "swin_l384_sweep_fwd (B=16, 12x12 windows)", "us": round(tot_ms * 1e3, 2),
            "tokens_per_s": sum(x["wl"].tokens for x in st) / (tot_ms / 1e3),
            "frac_of_measured_hbm": round(tot_b / (tot_ms / 1e3) / 1e9 / hbm, 4), "stages": out}


def run_fp8_sweep(names, args, dev, stream, lib, capi, hbm, ws):
    """The same sweep's forward on 8-bit operands (OCP FP8 E4M3 q, k, v with per-tensor
    scales, bf16 output), captured as one CUDA graph and replayed; per-stage times from an
    eager region with CUDA events around every launch. Context for the line, not the
    headline (which is the bf16 forward)."""
    sh = stream.cuda_stream
    st = []
    with torch.cuda.stream(stream):
        for name in names:
            wl = inputs.BY_NAME[name]
            q8, scales = inputs.make_qkv_fp8(wl)
            h = make_plan(capi, wl, inputs.make_table(wl).to(dev), sh, args)
            st.append(dict(wl=wl, h=h, q=q8.to(dev), sc=scales,
                           o=torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16, device=dev)))
    torch.cuda.synchronize()

    def one(events=None):
        for k, z in enumerate(st):
            if events is not None:
                events[k][0].record(stream)
            rc = lib.swin_wattn_fwd_fp8(z["h"], z["q"].data_ptr(), z["sc"][0], z["sc"][1], z["sc"][2],
                                        z["o"].data_ptr(), sh)
            if events is not None:
                events[k][1].record(stream)
            if rc != capi.OK:
                raise capi.SwinWAttnError("swin_wattn_fwd_fp8", rc)

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        one()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 2000))
    for _ in range(3):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(a.elapsed_time(b), ws) / steps
    esteps = max(3, min(args.steps, 200))
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in st] for _ in range(esteps)]
    for i in range(esteps):
        one(ev[i])
    torch.cuda.synchronize()
    stages, tot_b = [], 0
    for k, z in enumerate(st):
        wl = z["wl"]
        ms = statistics.mean(ev[i][k][0].elapsed_time(ev[i][k][1]) for i in range(esteps))
        tot_b += fwd_fp8_bytes(wl)
        stages.append({"workload": wl.name, "us": round(ms * 1e3, 2),
                       "frac_of_measured_hbm": round(fwd_fp8_bytes(wl) / (ms / 1e3) / 1e9 / hbm, 4),
                       "speedup_vs_bf16_bytes": round(fwd_bytes(wl) / fwd_fp8_bytes(wl), 3)})
    for z in st:
        capi.swin_wattn_destroy(z["h"])
    tokens = sum(z["wl"].tokens for z in st)
    return {"workload": "swin_l224_sweep_fwd on OCP FP8 E4M3 q, k, v (per-tensor scales), bf16 out",
            "steps": steps, "graph_us_per_step": round(graph_ms * 1e3, 2),
            "tokens_per_s": ws * tokens / (graph_ms / 1e3),
            "frac_of_measured_hbm": round(tot_b / (graph_ms / 1e3) / 1e9 / hbm, 4),
            "bytes_per_token": "5C (qkv 3C as E4M3, out 2C as bf16) + bias + mask per launch",
            "stages": stages}


def run_block_sweep(names, args, dev, stream, lib, capi, peaks, ws, fp8=False):
    """The attention sub-block of each stage, x -> LayerNorm + qkv projection -> shifted-
    window attention -> output projection + bias + residual x, captured as one CUDA graph
    and replayed; per-call times from a second, eager region with CUDA events around every
    call. The qkv weights are prepared once per stage (the fold of gamma into W and the
    bias vectors), as an inference deployment does with fixed weights; the dense bias and
    mask of each attention plan are likewise built once. With fp8, the producer writes
    OCP FP8 E4M3 qkv (per-tensor scales from the max |qkv| of one earlier pass: delayed
    scaling) and the attention runs on those 8-bit operands."""
    sh = stream.cuda_stream
    st = []
    with torch.cuda.stream(stream):
        for name in names:
            wl = inputs.BY_NAME[name]
            x, g, be, w, b = [t.to(dev) for t in inputs.make_producer(wl)]
            _, wp, bp, _ = [t.to(dev) for t in inputs.make_consumer(wl)]
            h = make_plan(capi, wl, inputs.make_table(wl).to(dev), sh, args)
            T = wl.tokens
            proj = capi.QkvProjection(g, be, w, b, stream=stream)
            nws = capi.swin_wattn_qkv_stats_bytes(T)
            sc = (1.0, 1.0, 1.0)
            if fp8:
                amax = torch.zeros(3, dtype=torch.float32, device=dev)
                proj.fp8(x, sc, amax=amax, stream=stream)
                torch.cuda.synchronize()
                sc = tuple(float(a) / 448.0 for a in amax.cpu())
            st.append(dict(wl=wl, x=x, wp=wp, bp=bp, h=h, T=T, nws=nws, prep=proj.prepared, sc=sc,
                           ws=torch.empty(nws, dtype=torch.uint8, device=dev),
                           qkv=torch.empty(wl.B, wl.H, wl.W, 3 * wl.C, dtype=torch.uint8 if fp8 else torch.bfloat16,
                                           device=dev),
                           o=torch.empty_like(x), y=torch.empty_like(x)))
    torch.cuda.synchronize()

    def one(events=None):
        for k, z in enumerate(st):
            wl = z["wl"]
            if events is not None:
                events[k][0].record(stream)
            if fp8:
                sq, sk, sv = z["sc"]
                ok = lib.swin_wattn_qkv_proj_prepared_fp8(z["x"].data_ptr(), z["prep"].data_ptr(),
                                                          z["qkv"].data_ptr(), z["T"], wl.C, 1e-5, sq, sk, sv, None,
                                                          z["ws"].data_ptr(), z["nws"], None, sh) == capi.OK
            else:
                ok = lib.swin_wattn_qkv_proj_prepared(z["x"].data_ptr(), z["prep"].data_ptr(), z["qkv"].data_ptr(),
                                                      z["T"], wl.C, 1e-5, z["ws"].data_ptr(), z["nws"], None,
                                                      sh) == capi.OK
            if events is not None:
                events[k][1].record(stream)
            if fp8:
                ok &= lib.swin_wattn_fwd_fp8(z["h"], z["qkv"].data_ptr(), sq, sk, sv, z["o"].data_ptr(),
                                             sh) == capi.OK
            else:
                ok &= lib.swin_wattn_fwd(z["h"], z["qkv"].data_ptr(), z["o"].data_ptr(), sh) == capi.OK
            if events is not None:
                events[k][2].record(stream)
            ok &= lib.swin_wattn_proj_residual(z["o"].data_ptr(), z["wp"].data_ptr(), z["bp"].data_ptr(),
                                               z["x"].data_ptr(), z["y"].data_ptr(), z["T"], wl.C, None,
                                               sh) == capi.OK
            if events is not None:
                events[k][3].record(stream)
            if not ok:
                raise RuntimeError("block step call failed")

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    capi.swin_wattn_launch_count(reset=True)
    one()
    launches_per_step = capi.swin_wattn_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        one()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 200))
    for _ in range(3):
        with torch.cuda.stream(stream):
            graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(a.elapsed_time(b), ws) / steps
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in st] for _ in range(steps)]
    a.record(stream)
    for i in range(steps):
        one(ev[i])
    b.record(stream)
    torch.cuda.synchronize()
    eager_ms = a.elapsed_time(b) / steps
    hbm = float(peaks["hbm_gbs"])
    stages = []
    for k, z in enumerate(st):
        wl = z["wl"]
        q_ms, f_ms, p_ms = (statistics.mean(ev[i][k][j].elapsed_time(ev[i][k][j + 1]) for i in range(steps))
                            for j in range(3))
        qb = qkv_bytes(wl) - (3 * wl.C * wl.tokens if fp8 else 0)  # 8-bit qkv written
        fb = fwd_fp8_bytes(wl) if fp8 else fwd_bytes(wl)
        stages.append({"workload": wl.name,
                       "producer": gemm_roofline(qb, qkv_flops(wl), q_ms, peaks),
                       "attention": {"us": round(f_ms * 1e3, 2),
                                     "frac_of_measured_hbm": round(fb / (f_ms / 1e3) / 1e9 / hbm, 4)},
                       "consumer": gemm_roofline(proj_bytes(wl), proj_flops(wl), p_ms, peaks)})
    for z in st:
        capi.swin_wattn_destroy(z["h"])
    tokens = sum(z["T"] for z in st)
    return {"workload": "swin_l224 attention sub-block sweep (B=64 per GPU; per stage LayerNorm + qkv "
                        "projection, SW-MSA, output projection + bias + residual)"
                        + (" with qkv as OCP FP8 E4M3 between the producer and the attention" if fp8 else ""),
            "steps": steps, "graph_us_per_step": round(graph_ms * 1e3, 2),
            "eager_us_per_step": round(eager_ms * 1e3, 2), "tokens_per_s": ws * tokens / (graph_ms / 1e3),
            "launches_per_step": int(launches_per_step),
            "roofline_note": "GEMM steps: bound = the larger of bytes / measured HBM and flops / measured "
                             "bf16 burst rate; frac = that time / measured time",
            "stages": stages}


def run_train_step(args, dev, stream, lib, capi, hbm, ws):
    """Swin-B 224 training step of the path: per stage, bias re-expansion from the
    (updated) table, forward, and backward with the table gradient."""
    sh = stream.cuda_stream
    wls = [inputs.BY_NAME[n] for n in TRAIN]
    st = []
    with torch.cuda.stream(stream):
        for wl in wls:
            tab = inputs.make_table(wl).to(dev)
            h = make_plan(capi, wl, tab, sh, args)
            q = inputs.make_qkv(wl).to(dev)
            d = inputs.make_dout(wl).to(dev)
            st.append(dict(wl=wl, h=h, tab=tab, q=q, d=d, o=torch.empty_like(d),
                           dq=torch.empty_like(q), dt=torch.empty_like(tab)))
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 50))

    def one(events=None):
        for k, x in enumerate(st):
            if events is not None:
                events[k][0].record(stream)
            ok = lib.swin_wattn_set_bias(x["h"], x["tab"].data_ptr(), sh) == capi.OK
            if events is not None:
                events[k][1].record(stream)
            ok &= lib.swin_wattn_fwd(x["h"], x["q"].data_ptr(), x["o"].data_ptr(), sh) == capi.OK
            if events is not None:
                events[k][2].record(stream)
            ok &= lib.swin_wattn_bwd(x["h"], x["q"].data_ptr(), x["d"].data_ptr(),
                                     x["dq"].data_ptr(), x["dt"].data_ptr(), sh) == capi.OK
            if ws > 1:
                # the one exchange of the path: the bias-table gradient summed over ranks
                with torch.cuda.stream(stream):
                    dp.allreduce_table_grad(x["dt"])
            if events is not None:
                events[k][3].record(stream)
            if not ok:
                raise RuntimeError("training step call failed")

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in st] for _ in range(steps)]
    barrier(ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        one(ev[i])
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), ws) / steps
    tokens = sum(x["wl"].tokens for x in st)
    stages = []
    for k, x in enumerate(st):
        wl = x["wl"]
        f_ms = statistics.mean(ev[i][k][1].elapsed_time(ev[i][k][2]) for i in range(steps))
        b_ms = statistics.mean(ev[i][k][2].elapsed_time(ev[i][k][3]) for i in range(steps))
        s_ms = statistics.mean(ev[i][k][0].elapsed_time(ev[i][k][1]) for i in range(steps))
        stages.append({"workload": wl.name, "set_bias_us": round(s_ms * 1e3, 2),
                       "window_heads_per_s_fwd_bwd": wl.window_heads / ((f_ms + b_ms) / 1e3),
                       "fwd_us": round(f_ms * 1e3, 2), "bwd_us": round(b_ms * 1e3, 2),
                       "fwd_frac_of_measured_hbm": round(fwd_bytes(wl) / (f_ms / 1e3) / 1e9 / hbm, 4),
                       "bwd_frac_of_measured_hbm": round(bwd_bytes(wl) / (b_ms / 1e3) / 1e9 / hbm, 4),
                       "bwd_tflops": round(bwd_flops(wl) / (b_ms / 1e3) / 1e12, 1)})
    for x in st:
        capi.swin_wattn_destroy(x["h"])
    return {"workload": "swin_b224_train_step (B=128 per GPU, 4 stages: set_bias + fwd + bwd"
                        + (", table-gradient all-reduce" if ws > 1 else "") + ")",
            "steps": steps, "ms_per_step": ms, "tokens_per_s": ws * tokens / (ms / 1e3),
            "stages": stages}


FWD_KERNELS = {"auto": 0, "mma_sync": 1, "tcgen05": 2}


def kernel_name(capi, h):
    """The forward kernel a plan launches, as named in the library's sources."""
    return ("fwd_tc_kernel (tcgen05)" if capi.swin_wattn_fwd_kernel(h) == capi.KERNEL_TCGEN05
            else "fwd_kernel<7,bf16,3> (mma.sync)")


def make_plan(capi, wl, tab, sh, args):
    """A bf16 plan for the workload, with the forward (and, for a training workload, the
    backward) kernel that --fwd-kernel / --bwd-kernel ask for."""
    rc, h = capi.swin_wattn_plan(wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s, capi.BF16,
                                 tab.data_ptr(), sh)
    if rc != capi.OK:
        raise capi.SwinWAttnError("swin_wattn_plan", rc)
    kernel = FWD_KERNELS[args.fwd_kernel]
    if kernel != 0:
        rc = capi.swin_wattn_set_fwd_kernel(h, kernel)
        if rc != capi.OK:
            raise capi.SwinWAttnError("swin_wattn_set_fwd_kernel", rc)
    kernel = FWD_KERNELS[getattr(args, "bwd_kernel", "auto")]
    if kernel != 0 and wl.bwd:
        rc = capi.swin_wattn_set_bwd_kernel(h, kernel)
        if rc != capi.OK:
            raise capi.SwinWAttnError("swin_wattn_set_bwd_kernel", rc)
    return h


def run_gemm_only(args):
    """Producer and consumer launches of one workload (warm-up + timed), for kernel
    profiling: after one swin_wattn_qkv_prepare, each iteration is
    swin_wattn_qkv_proj_prepared then swin_wattn_proj_residual."""
    from swin_window_attention_gb300 import build, capi
    build.build()
    wl = inputs.BY_NAME[args.gemm_workload]
    dev = torch.device("cuda", 0)
    x, g, be, w, b = [t.to(dev) for t in inputs.make_producer(wl)]
    o, wp, bp, r = [t.to(dev) for t in inputs.make_consumer(wl)]
    qkv = torch.empty(x.shape[:-1] + (3 * wl.C,), dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(o)
    proj = capi.QkvProjection(g, be, w, b)  # the weights prepared once
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup + args.steps):
        ev[i][0].record()
        proj(x, qkv)
        ev[i][1].record()
        capi.proj_residual(o, wp, bp, r, y)
        ev[i][2].record()
    torch.cuda.synchronize()
    peaks, _ = load_peaks()
    q_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev[args.warmup:])
    p_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev[args.warmup:])
    print(json.dumps({"workload": wl.name,
                      "producer": gemm_roofline(qkv_bytes(wl), qkv_flops(wl), q_ms, peaks),
                      "consumer": gemm_roofline(proj_bytes(wl), proj_flops(wl), p_ms, peaks)}))


def run_fp8_only(args):
    """Forward launches on FP8 operands for one workload (warm-up + timed), for kernel
    profiling."""
    from swin_window_attention_gb300 import build, capi
    build.build()
    wl = inputs.BY_NAME[args.fp8_workload]
    dev = torch.device("cuda", 0)
    q8, scales = inputs.make_qkv_fp8(wl)
    att = capi.WindowAttention(wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s, inputs.make_table(wl).to(dev))
    q = q8.to(dev)
    for _ in range(args.warmup):
        att.fwd_fp8(q, scales)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        att.fwd_fp8(q, scales)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    print(json.dumps({"workload": wl.name, "fp8_fwd_us": ms * 1e3,
                      "frac_of_measured_hbm": fwd_fp8_bytes(wl) / (ms / 1e3) / 1e9 / load_peaks()[0]["hbm_gbs"]}))
    att.close()


def run_bwd_only(args):
    """Backward launches of one workload (warm-up + timed), for kernel profiling."""
    from swin_window_attention_gb300 import build, capi
    build.build()
    wl = inputs.BY_NAME[args.bwd_workload]
    dev = torch.device("cuda", 0)
    att = capi.WindowAttention(wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s,
                               inputs.make_table(wl).to(dev))
    att.set_bwd_kernel(FWD_KERNELS[args.bwd_kernel])
    q, d = inputs.make_qkv(wl).to(dev), inputs.make_dout(wl).to(dev)
    dq, dt = torch.empty_like(q), torch.empty((2 * wl.M - 1) ** 2, wl.nH, device=dev)
    for _ in range(args.warmup):
        att.bwd(q, d, dq, dt)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        att.bwd(q, d, dq, dt)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    print(json.dumps({"workload": wl.name, "bwd_us": ms * 1e3, "bwd_kernel": att.bwd_kernel,
                      "frac_of_measured_hbm": bwd_bytes(wl) / (ms / 1e3) / 1e9 / load_peaks()[0]["hbm_gbs"]}))
    att.close()


# ---- reference arm: the oracle --------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return
    import oracle
    oracle.build()
    sweep = [inputs.BY_NAME[n] for n in SWEEP]
    data = []
    for wl in sweep:
        one = wl.with_batch(1)
        data.append((wl, inputs.act_f64(inputs.make_qkv(one)), inputs.make_table(wl).double().numpy()))

    def step():
        for wl, q, t in data:
            oracle.fwd(q, t, wl.nH, wl.M, wl.s)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    tokens = sum(wl.H * wl.W for wl in sweep)
    value = tokens * args.steps / el
    cores = oracle.max_threads()
    sample = "one image per stage of the Swin-L 224 sweep per step (batch 1 of 64)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "swin_l224_sweep_fwd", "batch_per_step": 1, "window": 7},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", action="append", choices=sorted(inputs.BY_NAME),
                    help="time only these forward workloads instead of the Swin-L 224 sweep "
                         "(profiling runs)")
    ap.add_argument("--bwd-workload", choices=sorted(n for n, w in inputs.BY_NAME.items() if w.bwd),
                    help="profiling run: only the backward of this workload, a few launches")
    ap.add_argument("--fp8-workload", choices=sorted(n for n, w in inputs.BY_NAME.items() if w.M == 7),
                    help="profiling run: only the forward on FP8 operands of this workload, a few launches")
    ap.add_argument("--gemm-workload", choices=sorted(inputs.BY_NAME),
                    help="profiling run: only the producer and consumer of this workload, a few launches")
    ap.add_argument("--bwd-kernel", default="auto", choices=sorted(FWD_KERNELS),
                    help="backward kernel of the plans (training step and --bwd-workload runs)")
    ap.add_argument("--fwd-kernel", default="auto", choices=sorted(FWD_KERNELS),
                    help="forward kernel of every plan (auto: the library's default)")
    ap.add_argument("--skip-train", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-sustained", action="store_true",
                    help="no seconds-long timed region (kernel profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.bwd_workload:
        run_bwd_only(args)
    elif args.gemm_workload:
        run_gemm_only(args)
    elif args.fp8_workload:
        run_fp8_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
