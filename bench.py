"""Benchmark of the NVFP4 MoE expert path on GB300.

One step = one prefill pass of 4096 tokens through a 384-expert MoE layer
(hidden 7168, intermediate 2048, top-8 Zipf(1.1) routing, one shared expert),
fed as 32 sequential chunks of 128 tokens.  Each chunk runs the whole hot path:
routing + global scale + quantise/permute (dispatch), the w13 grouped GEMM with
SiLU*up and NVFP4 re-quantisation, the w2 grouped GEMM with the weighted
scatter-add, and the bf16 conversion.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE tokens/s; TFLOPS & HBM GB/s as % of 1×GB300 FP4/HBM roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio
TIMED_EVERY = 4  # chunks between the ones whose GEMM launches carry CUDA events


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-secondary", action="store_true")
    # internal: the oracle timing of the CPU baseline, run in a child process whose BLAS is
    # pinned to one thread before numpy loads
    p.add_argument("--cpu-baseline-child", nargs=3, type=int, metavar=("TOKENS", "REPEATS", "THREADS"),
                   help=argparse.SUPPRESS)
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def strip_comments(src: str) -> str:
    """C++ source without comments and with whitespace runs collapsed (string literals in
    these files hold no comment markers)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash() -> str:
    """Hash of the GEMM kernel's code (comments and layout excluded), which keys the ncu traffic."""
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "internal.h"):
        with open(os.path.join(ROOT, "nvfp4_block_scaled_quant_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples go to NVFP4_BENCH_LOG_DIR when set (kept), else to the temp directory
        out_dir = os.environ.get("NVFP4_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"nvfp4_clocks_gpu{index}_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pmax = max(power) if power else 0.0
        loaded = [c for c, p in zip(sm, power) if p >= 0.5 * pmax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- workload accounting

def chunk_accounting(ids_cpu, cfg):
    """Algorithmic bytes and flops of one chunk, from its routing."""
    T, H, I, k = cfg.T, cfg.H, cfg.I, cfg.topk
    groups = len(set(ids_cpu.flatten().tolist())) + (1 if cfg.shared else 0)
    rows = T * k + (T if cfg.shared else 0)
    nvfp4 = 0.5 + 1.0 / 16.0  # bytes per element incl. scales
    w13 = groups * 2 * I * H * nvfp4
    w2 = groups * H * I * nvfp4
    w13_bytes = w13 + rows * H * nvfp4 + rows * I * nvfp4          # weights + A rows + hq written
    w2_bytes = w2 + rows * I * nvfp4 + T * H * 4 * 2                  # weights + hq rows + fp32 accumulator r/w
    dispatch_bytes = T * H * 2 * 2 + rows * H * nvfp4 + T * H * 4     # x read twice, xq rows, zeroing y_acc
    flops = 2.0 * rows * (2 * I * H + H * I)
    return dict(groups=groups, rows=rows, w13_bytes=w13_bytes, w2_bytes=w2_bytes,
                step_bytes=w13_bytes + w2_bytes + dispatch_bytes + T * H * (4 + 2), flops=flops)


# --------------------------------------------------------------------------- native arm

def run_native(args, rank: int, world: int, local_rank: int):
    import torch

    from nvfp4_block_scaled_quant_gb300 import build as B
    B.build()
    from nvfp4_block_scaled_quant_gb300 import model, ops, replicas, workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = workloads.PREFILL
    T, H, I, E, k, C = cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk, cfg.chunks

    W = model.make_moe_weights(E, H, I, workloads.BENCH_WEIGHT_SEED, dev, shared=True)
    chunks = []
    acct = []
    for c in range(C):
        x, ids, w = workloads.prefill_chunk(c, device="cpu")
        acct.append(chunk_accounting(ids.numpy(), cfg))
        chunks.append((x.to(dev), ids.to(dev), w.to(dev)))
    L = ops.moe_workspace_layout(T, H, I, E, k, True)
    ws = torch.empty(L.total, dtype=torch.uint8, device=dev)
    a1 = torch.empty(1, dtype=torch.float32, device=dev)
    ys = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(C)]

    # warm-up calibration of the static scale of the intermediate (page 3: gs from a warm-up pass)
    h_dbg = torch.empty(L.rows_capacity, I, dtype=torch.float32, device=dev)
    ones = torch.ones(E + 1, dtype=torch.float32, device=dev)
    amax = 0.0
    for c in range(2):
        x, ids, w = chunks[c]
        ops.moe_dispatch(x, ids, W, a1, True, ws)
        h_dbg.zero_()
        ops.moe_w13(T, k, W, a1, ones, ws, h_debug=h_dbg)
        amax = max(amax, float(h_dbg.abs().amax().item()))
    a2 = torch.full((E + 1,), amax / 2688.0, dtype=torch.float32, device=dev)
    del h_dbg

    stream = torch.cuda.current_stream(dev)
    # w13 and w2 launch durations, live in the timed region, on every TIMED_EVERY-th chunk: an
    # event recorded between two launches ends the programmatic overlap of the second with
    # the first, so the other chunks run the chain unperturbed
    timed = [c for c in range(C) if c % TIMED_EVERY == 0]
    ev = [{c: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for c in timed} for _ in range(args.steps)]

    def step(evs):
        for c in range(C):
            x, ids, w = chunks[c]
            e = evs.get(c) if evs is not None else None
            ops.moe_dispatch(x, ids, W, a1, True, ws)
            if e is not None:
                e[0].record(stream)
            ops.moe_w13(T, k, W, a1, a2, ws)
            if e is not None:
                e[1].record(stream)
            ops.moe_w2(T, k, w, W, a2, ws)
            if e is not None:
                e[2].record(stream)
            ops.moe_finalize(T, k, W, ys[c], ws)

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    st, flags = ops.device_error()
    if st != 0:
        raise RuntimeError(f"device fault flags {flags:#x} after warm-up")

    dist = None
    if world > 1:
        import torch.distributed as dist
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.5)  # let the sampler start before the timed region
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    start.record(stream)
    for s in range(args.steps):
        step(ev[s])
    stop.record(stream)
    stop.synchronize()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed_ms = start.elapsed_time(stop)
    clk = clocks.stop()
    n_timed = args.steps * len(timed)  # timed launches of each GEMM
    t_w13 = sum(ev[s][c][0].elapsed_time(ev[s][c][1]) for s in range(args.steps) for c in timed)
    t_w2 = sum(ev[s][c][1].elapsed_time(ev[s][c][2]) for s in range(args.steps) for c in timed)
    st, flags = ops.device_error()
    if st != 0:
        raise RuntimeError(f"device fault flags {flags:#x} in the timed region")

    # independent replicas: all ranks' tokens over the slowest rank's time
    tokens_per_step = T * C
    value, elapsed_ms, _ = replicas.replica_throughput(elapsed_ms, tokens_per_step * args.steps, device=dev)
    ms_per_step = elapsed_ms / args.steps
    hbm, bf16, bf16_sus, peak_kind = peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    w13_bytes = sum(a["w13_bytes"] for a in acct)  # per step (one launch per chunk)
    step_bytes = sum(a["step_bytes"] for a in acct)
    flops = sum(a["flops"] for a in acct)
    w13_avg_ms = t_w13 / n_timed
    # the timed chunks' own algorithmic bytes
    w13_timed_bytes = sum(acct[c]["w13_bytes"] for c in timed) / len(timed)
    w2_timed_bytes = sum(acct[c]["w2_bytes"] for c in timed) / len(timed)
    achieved = w13_timed_bytes / (w13_avg_ms / 1e3) / 1e9
    traffic = measured_traffic("w13", cfg.name)  # mean launch of the step
    if traffic is not None:  # the same traffic / algorithmic ratio, per timed launch
        traffic *= w13_timed_bytes / (w13_bytes / C)

    # ---------------------------------------------------------------- end to end through the public API
    xh = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(C)]
    idh = [torch.empty(T, k, dtype=torch.int32).pin_memory() for _ in range(C)]
    wh = [torch.empty(T, k, dtype=torch.float32).pin_memory() for _ in range(C)]
    yh = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(C)]
    for c in range(C):
        xh[c].copy_(chunks[c][0].cpu())
        idh[c].copy_(chunks[c][1].cpu())
        wh[c].copy_(chunks[c][2].cpu())
    # Double-buffered pipeline: chunk c + 1's inputs go up on one copy stream and chunk c's
    # output comes back on another while chunk c computes; events order each buffer's reuse.
    xd = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    idd = [torch.empty(T, k, dtype=torch.int32, device=dev) for _ in range(2)]
    wd = [torch.empty(T, k, dtype=torch.float32, device=dev) for _ in range(2)]
    yd = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, in_free = [ev() for _ in range(2)], [ev() for _ in range(2)]
    out_ready, out_free = [ev() for _ in range(2)], [ev() for _ in range(2)]
    for b in range(2):  # every buffer starts free
        in_free[b].record(stream)
        out_free[b].record(stream)

    def e2e_step():
        for c in range(C):
            b = c % 2
            with torch.cuda.stream(up):
                up.wait_event(in_free[b])
                xd[b].copy_(xh[c], non_blocking=True)
                idd[b].copy_(idh[c], non_blocking=True)
                wd[b].copy_(wh[c], non_blocking=True)
                in_ready[b].record(up)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            ops.moe_forward(xd[b], idd[b], wd[b], W, a2, workspace=ws, out=yd[b], stream=stream)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                yh[c].copy_(yd[b], non_blocking=True)
                out_free[b].record(down)

    def e2e_drain():  # the compute stream waits for the last output copies
        for b in range(2):
            stream.wait_event(out_free[b])

    for _ in range(args.warmup):
        e2e_step()
    e2e_drain()
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    up.wait_event(e_start)
    down.wait_event(e_start)
    for _ in range(args.steps):
        e2e_step()
    e2e_drain()
    e_stop.record(stream)
    e_stop.synchronize()
    e_ms = e_start.elapsed_time(e_stop)
    if dist:
        tt = torch.tensor([e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e_ms = float(tt.item())
    # every output arrived: spot-check the last step's host copies against a device recompute
    last = C - 1
    yref = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ops.moe_forward(chunks[last][0], chunks[last][1], chunks[last][2], W, a2, workspace=ws, out=yref, stream=stream)
    torch.cuda.synchronize()
    e2e_check = float((yh[last].to(dev).float() - yref.float()).abs().max() / yref.float().abs().max().clamp_min(1e-30))
    h2d = C * (T * H * 2 + T * k * 4 * 2)
    d2h = C * T * H * 2
    e2e = {"value": world * tokens_per_step * args.steps / (e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "api": "nvfp4_moe_forward (one call per chunk), pinned host buffers; inputs of chunk c+1 uploaded and "
                  "outputs of chunk c downloaded on two copy streams while chunk c computes",
           "check_max_rel_diff_last_chunk": e2e_check}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block scales) -> f32 acc",
        "data": "synthetic (seeded; bf16 N(0,0.02) weights quantised to NVFP4, N(0,1) activations with 1% x20 "
                "outlier channels, Zipf(1.1) top-8 routing)",
        "config": {"workload": cfg.name, "tokens_per_step": tokens_per_step, "chunks": C, "chunk_tokens": T,
                   "hidden": H, "intermediate": I, "experts": E, "topk": k, "shared_expert": True,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "working set of ~5.6 GB of expert weights per chunk (> 129 MB L2); no flush needed",
                   "a1_gs": "dynamic per chunk", "a2_gs": "static, warm-up calibrated"},
        "roofline": {"bound": "hbm", "kernel": "w13 grouped GEMM + SiLU*up + requant",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": w13_timed_bytes, "avg_launch_ms": w13_avg_ms,
                     "launches_timed": n_timed,
                     "timed_chunks": f"every {TIMED_EVERY}th chunk of each step ({len(timed)} of {C})"},
        "step_roofline": {"hbm_gbs": step_bytes / (ms_per_step / 1e3) / 1e9,
                          "hbm_frac": step_bytes / (ms_per_step / 1e3) / 1e9 / hbm,
                          "tflops": flops / (ms_per_step / 1e3) / 1e12,
                          "tensor_frac_fp4": flops / (ms_per_step / 1e3) / 1e12 / fp4_peak,
                          "fp4_peak_tflops": fp4_peak, "fp4_peak_source": f"{peak_kind} bf16 x {FP4_OVER_BF16}",
                          "w2_avg_ms": t_w2 / n_timed,
                          "w2_gbs": w2_timed_bytes / (t_w2 / n_timed / 1e3) / 1e9,
                          "groups_per_chunk_mean": sum(a["groups"] for a in acct) / C},
        "e2e": e2e,
        "gpu_launches": args.steps * C * 5,
        "clocks": clk,
    }
    return result, (W, chunks, a2, ws, a1, dev)


# --------------------------------------------------------------------------- secondary workloads

def run_secondary(state, args):
    """Decode steps and the dense linear / GEMM workloads, one line each in 'secondary'."""
    import numpy as np
    import torch

    from nvfp4_block_scaled_quant_gb300 import model, ops, workloads
    W, _, a2, _, _, dev = state
    hbm, bf16, _, _ = peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    out = []
    stream = torch.cuda.current_stream(dev)

    def time_fn(fn, iters):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(iters):
            fn()
        e.record(stream)
        e.synchronize()
        return s.elapsed_time(e) / iters

    cap = torch.cuda.Stream(dev)

    def graph_time_fn(body, calls, reps):
        """Device time per call from CUDA-graph replay: body(stream) enqueues `calls` calls;
        the graph of one body is replayed `reps` times between two events."""
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            body(cap)  # warm-up outside the capture (per-device set-up, kernel attributes)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            body(cap)
        with torch.cuda.stream(cap):
            for _ in range(2):
                g.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cap):  # replay() launches on the current stream
            s.record(cap)
            for _ in range(reps):
                g.replay()
            e.record(cap)
        e.synchronize()
        stream.wait_stream(cap)
        del g
        return s.elapsed_time(e) / (reps * calls)

    for T in (1, 8, 64):
        cfg = workloads.DECODE[T]
        steps = [workloads.decode_step(T, step=i, device="cpu") for i in range(16)]
        acct = [chunk_accounting(s[1].numpy(), cfg) for s in steps]
        dev_steps = [(x.to(dev), i.to(dev), w.to(dev)) for x, i, w in steps]
        ws = ops.moe_workspace(T, cfg.H, cfg.I, cfg.E, cfg.topk, True, dev)
        y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
        it = [0]

        def fwd():
            x, i, w = dev_steps[it[0] % 16]
            it[0] += 1
            ops.moe_forward(x, i, w, W, a2, workspace=ws, out=y)

        def fwd16(st):
            for x, i, w in dev_steps:
                ops.moe_forward(x, i, w, W, a2, workspace=ws, out=y, stream=st)

        eager_ms = time_fn(fwd, 64)
        ms = graph_time_fn(fwd16, 16, 8)
        b = sum(a["step_bytes"] for a in acct) / 16
        out.append({"workload": cfg.name, "tokens_per_s": T / (ms / 1e3), "ms_per_step": ms,
                    "hbm_gbs": b / (ms / 1e3) / 1e9, "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                    "eager_ms_per_step": eager_ms, "groups_mean": sum(a["groups"] for a in acct) / 16,
                    "note": "16 seeded routings cycled, replayed as one CUDA graph (eager_ms_per_step: plain calls); "
                            "weights streamed from HBM (> L2)"})
    # whole prefill in one call: the 32 chunks' 4096 tokens at once (hot experts span many m tiles)
    cfg = workloads.PREFILL_WHOLE
    x, ids, w = workloads.prefill_whole(device="cpu")
    acct = chunk_accounting(ids.numpy(), cfg)
    xd, idd, wd = x.to(dev), ids.to(dev), w.to(dev)
    wsw = ops.moe_workspace(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk, True, dev)
    yw = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    ms = time_fn(lambda: ops.moe_forward(xd, idd, wd, W, a2, workspace=wsw, out=yw), 10)
    out.append({"workload": cfg.name, "tokens_per_s": cfg.T / (ms / 1e3), "ms_per_call": ms,
                "hbm_gbs": acct["step_bytes"] / (ms / 1e3) / 1e9,
                "hbm_frac": acct["step_bytes"] / (ms / 1e3) / 1e9 / hbm,
                "tflops": acct["flops"] / (ms / 1e3) / 1e12,
                "tensor_frac_fp4": acct["flops"] / (ms / 1e3) / 1e12 / fp4_peak, "groups": acct["groups"],
                "note": "one call over the same 4096 tokens as the 32-chunk step"})
    # The same call's hot-expert tiles alone: groups of >= 1000 rows (the popular experts and the
    # shared expert).  Every other slot of the routing gets an out-of-range id, which the routing
    # drops (it raises the bad-id flag, read and cleared here), so the GEMMs run exactly the hot
    # groups' tiles; w13 and w2 are timed with events around their launches.
    idn = ids.numpy()
    counts = np.bincount(idn.reshape(-1), minlength=cfg.E)
    hot = counts >= 1000
    ids_hot = np.where(hot[idn], idn, cfg.E).astype(np.int32)
    rows_hot = int(counts[hot].sum()) + cfg.T
    idh = torch.from_numpy(ids_hot).to(dev)
    a1 = torch.empty(1, dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t13 = t2 = 0.0
    for rep in range(6):
        ops.moe_dispatch(xd, idh, W, a1, True, wsw)
        ev[0].record()
        ops.moe_w13(cfg.T, cfg.topk, W, a1, a2, wsw)
        ev[1].record()
        ops.moe_w2(cfg.T, cfg.topk, wd, W, a2, wsw)
        ev[2].record()
        ev[2].synchronize()
        if rep >= 2:
            t13 += ev[0].elapsed_time(ev[1]) / 4
            t2 += ev[1].elapsed_time(ev[2]) / 4
    flag = ops.device_error()
    f13 = 2.0 * rows_hot * 2 * cfg.I * cfg.H
    f2 = 2.0 * rows_hot * cfg.H * cfg.I
    out.append({"workload": "prefill_whole_hot_expert_tiles_rows_ge_1000", "groups": int(hot.sum()) + 1,
                "rows": rows_hot, "w13_ms": t13, "w2_ms": t2,
                "w13_tflops": f13 / (t13 / 1e3) / 1e12, "w2_tflops": f2 / (t2 / 1e3) / 1e12,
                "tflops": (f13 + f2) / ((t13 + t2) / 1e3) / 1e12,
                "tensor_frac_fp4": (f13 + f2) / ((t13 + t2) / 1e3) / 1e12 / fp4_peak,
                "w13_tensor_frac_fp4": f13 / (t13 / 1e3) / 1e12 / fp4_peak,
                "bad_id_flag_expected": list(flag),
                "note": "the 4096-token call's groups with >= 1000 rows and the shared expert, the other slots "
                        "dropped; 128-row m tiles on the one-SM grouped GEMM; CUDA events around each launch"})
    del wsw, xd, idd, wd, yw, idh
    # dense linear K=1536 N=16384: 14 MB of weights fit in L2, so rotate 16 weight copies (> L2)
    K, N = 1536, 16384
    dws = [model.make_dense_weight(N, K, seed=50 + i, device=dev) for i in range(16)]
    for M in (1, 32, 128):
        x = workloads.activations(M, K, seed=60 + M, device=dev, outliers=True)
        wsl = torch.empty(int(ops.lib().nvfp4_linear_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        gs = torch.empty(1, dtype=torch.float32, device=dev)
        it = [0]
        # gs_mode 0: the activation global scale from x's amax on every call; 1: a static scale,
        # read (the dynamic call's value, as a warm-up calibration leaves it)
        for gs_mode in (0, 1):

            def lin(st=stream, d=None, gs_mode=gs_mode):
                if d is None:
                    d = dws[it[0] % 16]
                    it[0] += 1
                ops.call("nvfp4_linear", x.data_ptr(), M, K, N, d.w.data_ptr(), d.sf.data_ptr(), d.ws2.data_ptr(),
                         gs_mode, gs.data_ptr(), y.data_ptr(), wsl.data_ptr(), wsl.numel(), st.cuda_stream)

            def lin16(st, lin=lin):
                for d in dws:
                    lin(st, d)

            eager_ms = time_fn(lin, 160)
            ms = graph_time_fn(lin16, 16, 10)
            b = N * K * (0.5 + 1 / 16) + M * K * 2 + M * N * 2
            out.append({"workload": f"dense_linear_M{M}_K{K}_N{N}" + ("_static_gs" if gs_mode else ""),
                        "us_per_call": ms * 1e3,
                        "hbm_gbs": b / (ms / 1e3) / 1e9, "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                        "tflops": 2 * M * N * K / (ms / 1e3) / 1e12, "eager_us_per_call": eager_ms * 1e3,
                        "note": ("quantise (static, calibrated gs) + GEMM" if gs_mode else "amax + quantise + GEMM")
                                + "; 16 weight copies rotated (230 MB > L2), replayed as one CUDA graph "
                                  "(eager_us_per_call: plain calls, bounded by the host)"})
    del dws
    # fixed-group linear (grouped o-projection): 8 x (4096 -> 1024); 16 weight copies rotated (> L2)
    for M in sorted(workloads.GROUPED_LINEAR):
        _, G, K, N = workloads.GROUPED_LINEAR[M]
        gws = [model.make_grouped_weight(G, N, K, seed=90 + i, device=dev) for i in range(16)]
        x = workloads.activations(M, G * K, seed=95 + M, device=dev, outliers=True)
        wsg = torch.empty(int(ops.lib().nvfp4_grouped_linear_workspace_bytes(M, G, K)), dtype=torch.uint8, device=dev)
        y = torch.empty(M, G * N, dtype=torch.bfloat16, device=dev)
        gs = torch.empty(1, dtype=torch.float32, device=dev)
        it = [0]
        for gs_mode in (0, 1):  # dynamic, then the static (calibrated) scale as for the dense linear

            def grp(st=stream, d=None, gs_mode=gs_mode):
                if d is None:
                    d = gws[it[0] % 16]
                    it[0] += 1
                ops.call("nvfp4_grouped_linear", x.data_ptr(), M, G, K, N, d.w.data_ptr(), d.sf.data_ptr(),
                         d.ws2.data_ptr(), gs_mode, gs.data_ptr(), y.data_ptr(), wsg.data_ptr(), wsg.numel(),
                         st.cuda_stream)

            def grp16(st, grp=grp):
                for d in gws:
                    grp(st, d)

            eager_ms = time_fn(grp, 160)
            ms = graph_time_fn(grp16, 16, 10)
            b = G * N * K * (0.5 + 1 / 16) + M * G * K * 2 + M * G * N * 2
            out.append({"workload": f"grouped_linear_M{M}_G{G}_K{K}_N{N}" + ("_static_gs" if gs_mode else ""),
                        "us_per_call": ms * 1e3,
                        "hbm_gbs": b / (ms / 1e3) / 1e9, "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                        "tflops": 2 * M * G * N * K / (ms / 1e3) / 1e12, "eager_us_per_call": eager_ms * 1e3,
                        "note": ("quantise (static, calibrated gs) + grouped GEMM" if gs_mode
                                 else "amax + quantise + grouped GEMM")
                                + "; 16 weight copies rotated (300 MB > L2), replayed as one CUDA graph "
                                  "(eager_us_per_call: plain calls, bounded by the host)"})
        del gws
    # routing + dispatch (stages a and b): latency-bound at small T, reported in microseconds
    for T in (1, 8, 64, 128, 4096):
        cfg = workloads.DECODE.get(T) or (workloads.PREFILL if T == 128 else workloads.PREFILL_WHOLE)
        if T in workloads.DECODE:
            ins = [workloads.decode_step(T, step=i, device=dev)[:2] for i in range(16)]
        elif T == 128:
            ins = [workloads.prefill_chunk(c, device=dev)[:2] for c in range(16)]
        else:
            x, ids, _ = workloads.prefill_whole(device="cpu")
            ins = [(x.to(dev), ids.to(dev))]
        wsr = ops.moe_workspace(T, cfg.H, cfg.I, cfg.E, cfg.topk, True, dev)
        g1 = torch.empty(1, dtype=torch.float32, device=dev)

        def disp(st, ins=ins, wsr=wsr, g1=g1):
            for x, ids in ins:
                ops.moe_dispatch(x, ids, W, g1, True, wsr, stream=st)

        ms = graph_time_fn(disp, len(ins), 16 if len(ins) > 1 else 64)
        rows = T * cfg.topk + T
        b = T * cfg.H * 2 * 2 + rows * cfg.H * (0.5 + 1 / 16) + T * cfg.H * 4
        out.append({"workload": f"route_dispatch_T{T}", "us_per_call": ms * 1e3, "hbm_gbs": b / (ms / 1e3) / 1e9,
                    "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                    "note": "nvfp4_moe_dispatch: routing (histogram, scans, stable ranks, tile table) + amax + "
                            "quantise/permute of x into the k+1 segments + zeroing of the fp32 accumulator; "
                            "CUDA-graph replay over rotated inputs"})
        del wsr
    # fused RMSNorm -> NVFP4 (the quantiser's producer): 2 B read + 0.5625 B written per element
    K = 7168
    gamma = workloads.norm_weight(K, seed=5, device=dev)
    for M in (1, 128, 4096):
        nin = 16 if M < 4096 else 4  # > L2 in total
        xs = [workloads.activations(M, K, seed=500 + i, device=dev, outliers=True) for i in range(nin)]
        q = torch.empty(M, K // 2, dtype=torch.uint8, device=dev)
        sfq = torch.empty(int(ops.sf_bytes(M, K)), dtype=torch.uint8, device=dev)
        gq = torch.empty(1, dtype=torch.float32, device=dev)
        wsn = torch.empty(int(ops.lib().nvfp4_rmsnorm_quantize_workspace_bytes(M, K)), dtype=torch.uint8,
                          device=dev)

        def norm(st, xs=xs, q=q, sfq=sfq, gq=gq, wsn=wsn, M=M):
            for x in xs:
                ops.call("nvfp4_rmsnorm_quantize", x.data_ptr(), M, K, K, gamma.data_ptr(), workloads.RMSNORM_EPS,
                         0, gq.data_ptr(), q.data_ptr(), sfq.data_ptr(), 0, None, wsn.data_ptr(), wsn.numel(),
                         st.cuda_stream)

        ms = graph_time_fn(norm, nin, 16)
        b = M * K * (2 + 0.5 + 1 / 16) + K * 2
        out.append({"workload": f"rmsnorm_quantize_M{M}_K{K}", "us_per_call": ms * 1e3,
                    "hbm_gbs": b / (ms / 1e3) / 1e9, "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                    "note": "fused RMSNorm -> NVFP4 with dynamic gs (statistics + encode launches); rotated inputs, "
                            "CUDA-graph replay"})
        del xs
    # router gate: logits over E experts, softmax, top-k; 32 rotated gate weights (176 MB > L2)
    for T in sorted(workloads.ROUTER):
        _, Hr, Er, kr = workloads.ROUTER[T]
        gates = []
        for i in range(32):
            q, sfw, ws2 = model.quantize_weight(workloads.weight(Er, Hr, workloads.ROUTER_WEIGHT_SEED + i, dev))
            gates.append(ops.router_prepare(q, sfw, ws2, Er, Hr))
        x = workloads.activations(T, Hr, seed=40 + T, device=dev)
        ids = torch.empty(T, kr, dtype=torch.int32, device=dev)
        wts = torch.empty(T, kr, dtype=torch.float32, device=dev)
        lg = torch.empty(T, Er, dtype=torch.float32, device=dev)
        wsr = torch.empty(max(256, int(ops.lib().nvfp4_router_workspace_bytes(T, Er))), dtype=torch.uint8, device=dev)

        def route(st, gates=gates, x=x, ids=ids, wts=wts, lg=lg, wsr=wsr, T=T, Hr=Hr, Er=Er, kr=kr):
            for wg in gates:
                ops.call("nvfp4_router", x.data_ptr(), T, Hr, wg.data_ptr(), Er, kr, ids.data_ptr(), wts.data_ptr(),
                         lg.data_ptr(), wsr.data_ptr(), wsr.numel(), st.cuda_stream)

        ms = graph_time_fn(route, 32, 8)
        b = Er * Hr * 2 + T * Hr * 2 + T * Er * 4
        out.append({"workload": f"router_T{T}_H{Hr}_E{Er}_k{kr}", "us_per_call": ms * 1e3,
                    "hbm_gbs": b / (ms / 1e3) / 1e9, "hbm_frac": b / (ms / 1e3) / 1e9 / hbm,
                    "tflops": 2 * T * Er * Hr / (ms / 1e3) / 1e12,
                    "note": "bf16 gate (FP8 round trip applied once at load) x activations -> fp32 logits on the "
                            "tensor cores (split over H), softmax, top-k; 32 rotated gate copies, CUDA-graph replay"})
        del gates
    K = N = 7168
    dw = model.make_dense_weight(N, K, seed=70, device=dev)
    for M in (1024, 4096, 16384):
        x = workloads.activations(M, K, seed=80 + M, device=dev)
        q, sf, gs = ops.quantize_act(x)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ms = time_fn(lambda: ops.gemm(q, sf, gs, K, dw.w, dw.sf, dw.ws2, N, out=y), 10)
        fl = 2.0 * M * N * K
        out.append({"workload": f"dense_gemm_M{M}_K{K}_N{N}", "ms_per_call": ms, "tflops": fl / (ms / 1e3) / 1e12,
                    "tensor_frac_fp4": fl / (ms / 1e3) / 1e12 / fp4_peak,
                    "note": "GEMM alone on quantised activations; operands (<= 170 MB) re-read across calls"})
    return out


# --------------------------------------------------------------------------- CPU oracle

def oracle_sample(n_tokens: int, chunk: int = 0, device="cpu"):
    """Inputs of a bounded sample of the workload for the oracle: n tokens of one prefill chunk."""
    import numpy as np
    import torch

    from nvfp4_block_scaled_quant_gb300 import workloads
    from oracle import nvfp4_oracle as O
    cfg = workloads.PREFILL
    x, ids, w = workloads.prefill_chunk(chunk, device="cpu")
    tokens = list(range(n_tokens))
    needed = sorted(set(ids[:n_tokens].flatten().tolist()))
    gdev = device if device != "cpu" and torch.cuda.is_available() else "cpu"
    experts = {}
    for e in needed + [cfg.E]:
        s13, s2 = workloads.expert_seeds(workloads.BENCH_WEIGHT_SEED, e)
        q13 = O.quantize(workloads.weight(2 * cfg.I, cfg.H, s13, gdev).float().cpu().numpy())
        q2 = O.quantize(workloads.weight(cfg.H, cfg.I, s2, gdev).float().cpu().numpy())
        experts[e] = O.Expert(q13.codes, q13.sf, q13.gs, q2.codes, q2.sf, q2.gs)
    a2 = np.full(cfg.E + 1, np.float32(0.01), dtype=np.float32)
    return cfg, x.float().numpy(), ids.numpy(), w.numpy(), experts, a2, tokens


def thread_mapper(threads: int):
    """The oracle's per-expert jobs on a pool of host threads (numpy releases the GIL in its
    array loops and contractions)."""
    from concurrent.futures import ThreadPoolExecutor
    ex = ThreadPoolExecutor(max_workers=threads)
    return (lambda fn, jobs: ex.map(fn, jobs)), ex


def time_oracle(n_tokens: int, reps: int, device="cpu", threads: int = 1):
    """Seconds per oracle MoE forward of n tokens (experts prepared beforehand, untimed), ``reps``
    times; threads > 1 runs the per-expert jobs on that many host threads."""
    from oracle import nvfp4_oracle as O
    cfg, x, ids, w, experts, a2, tokens = oracle_sample(n_tokens, device=device)
    mapper, ex = thread_mapper(threads) if threads > 1 else (map, None)
    times = []
    try:
        for _ in range(reps):
            t0 = time.perf_counter()
            O.moe_forward(x, ids, w, experts.__getitem__, cfg.E, a2, shared=experts[cfg.E], tokens=tokens,
                          mapper=mapper)
            times.append(time.perf_counter() - t0)
    finally:
        if ex is not None:
            ex.shutdown()
    return cfg, times


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


CPU_BASELINE_TOKENS = 2
CPU_BASELINE_REPEATS = 3
SINGLE_THREAD_ENV = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}


def cpu_baseline_child(n_tokens: int, reps: int, threads: int):
    """Child process (BLAS pinned to one thread by its environment): the oracle on one thread
    (the builtin map) and on ``threads`` host threads, ``reps`` times each; prints one JSON line."""
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"
    _, t1 = time_oracle(n_tokens, reps, device=device, threads=1)
    _, tn = time_oracle(n_tokens, reps, device=device, threads=threads)
    print(json.dumps({"t1": t1, "tn": tn, "weights_drawn_on": device}), flush=True)


def cpu_baseline():
    """The oracle as it stands, on this host's cores: a bounded sample of the workload (the
    first tokens of prefill chunk 0), 1 thread and all cores, several repeats each."""
    cores = cpu_cores()
    env = dict(os.environ, **SINGLE_THREAD_ENV)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", str(CPU_BASELINE_TOKENS),
                        str(CPU_BASELINE_REPEATS), str(cores)], env=env, capture_output=True, text=True,
                       timeout=1800)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": cores, "kind": "oracle",
                "error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    t1, tn = statistics.median(d["t1"]), statistics.median(d["tn"])
    n = CPU_BASELINE_TOKENS
    return {"value": n / tn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1t": n / t1, "value_nt": n / tn, "threads_nt": cores, "repeats": CPU_BASELINE_REPEATS,
            "seconds_1t": d["t1"], "seconds_nt": d["tn"],
            "sample": f"{n} tokens of prefill chunk 0 (8 routed experts each + the shared expert), the full oracle "
                      f"MoE forward (fp64 dequantisation and contractions), experts prepared beforehand; "
                      f"median of {CPU_BASELINE_REPEATS} runs on 1 thread (BLAS pinned to 1) and on {cores} host "
                      f"threads (per-expert jobs split over the cores); value = the {cores}-thread figure"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return None
    import torch
    cores = cpu_cores()
    # the weights are drawn on the GPU, like the native arm's; the oracle itself runs on the host cores
    cfg, times = time_oracle(1, args.warmup + args.steps, device="cuda" if torch.cuda.is_available() else "cpu",
                             threads=cores)
    timed = times[args.warmup:]
    total = sum(timed)
    value = len(timed) / total
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded), same workload", "config": {"workload": cfg.name, "oracle_tokens_per_step": 1},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: 1 token of prefill chunk 0 through the full oracle MoE forward, "
                                       f"per-expert jobs on {cores} host threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def relaunch(n: int) -> int:
    """Start n local ranks of this benchmark (one per GPU) and return their exit status."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def main():
    args = parse()
    if args.cpu_baseline_child:
        cpu_baseline_child(*args.cpu_baseline_child)
        return
    from nvfp4_block_scaled_quant_gb300 import replicas
    action, why = replicas.launch_plan(args.gpus, os.environ)
    if action == "error":
        print(f"bench.py: {why}", file=sys.stderr)
        sys.exit(2)
    if action == "relaunch":
        sys.exit(relaunch(args.gpus))
    rank, world, local_rank = replicas.env_ranks()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result, state = run_native(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_secondary:
            result["secondary"] = run_secondary(state, args)
        if not args.no_cpu_baseline and world == 1:
            del state
            torch.cuda.empty_cache()
            result["cpu_baseline"] = cpu_baseline()
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
