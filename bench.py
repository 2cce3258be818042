"""Benchmark of the fused Hadamard + FP4 quantizer and block-scaled FP4 GEMM.

One step = the whole hot path for one linear layer of a Llama-3.1-8B-class
model (synthetic, seeded): the fused rotation + MXFP4 quantization of X
[16384, 4096], W [4096, 4096] and dY [16384, 4096], both orientations each,
then the Fprop, Dgrad and Wgrad block-scaled GEMMs (E2M1 recipe: random H16
with signs shared along each contraction axis, RTNE on X and W, SR on dY).

  value        fused quantize throughput, GB/s of algorithmic bytes (read bf16,
               write codes + scales of both copies) over the quantize phase
  gemm.tflops  block-scaled GEMM throughput over the GEMM phase
  e2e          the same two metrics through the C ABI from pinned host
               buffers: inputs copied host->device inside the quantize phase,
               GEMM outputs copied device->host inside the GEMM phase, the
               copies on a second stream overlapping the compute that does
               not depend on them

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torch.distributed.run: every rank runs the same per-rank
workload on its own GPU (replicas, weak scaling); the time is the max over
ranks and value counts the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TOKENS, D_IN, D_OUT = 16384, 4096, 4096
SEED = 1005
MX_BYTES_PER_ELEM = 2 + 2 * (0.5 + 1 / 32)     # bf16 in, two copies of codes + E8M0 scales
WORKLOAD = ("one linear layer, bf16 X[16384,4096] W[4096,4096] dY[16384,4096]: fused random-H16 + "
            "MXFP4 E2M1 quantization of all three (row+col copies; RTNE X/W, Philox SR dY), then "
            "Fprop Y=XW^T, Dgrad dX=dY W, Wgrad dW=dY^T X block-scaled FP4 GEMMs (bf16 out; Dgrad and Wgrad in "
            "one grouped launch)")


# ------------------------------------------------------------------ ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def allreduce_max(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_rank: float, seconds_per_rank: float, world: int, device=None) -> float:
    """Whole-job throughput: bytes of all ranks over the slowest rank's time."""
    return bytes_per_rank * world / allreduce_max(seconds_per_rank, world, device)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        # raw samples; the summary goes into the JSON line
        log_dir = os.environ.get("FP4Q_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"fp4q_clocks_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = [l.split(",") for l in open(self.path) if l.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    from fp4_microscaled_quantization_gb300 import fp4q, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    bf16_peak = peaks.get("bf16_tflops", 1900.0)
    fp4_peak = bf16_peak * (13.5 / 2.25)     # nominal dense FP4 : BF16 ratio on GB300
    peak_src = "measured" if peaks else "fallback"

    # ---------------- inputs (bf16, resident)
    Xb, Wb, dYb = synth.layer(TOKENS, D_IN, D_OUT, SEED)
    X, W, dY = (synth.as_torch(a).to(dev) for a in (Xb, Wb, dYb))
    mK = fp4q.sign_mask_from_seed(SEED, 16)
    mN = fp4q.sign_mask_from_seed(SEED + 1, 16)
    mM = fp4q.sign_mask_from_seed(SEED + 2, 16)
    cfg_x = fp4q.Config(grid=fp4q.GRID_E2M1, rot=16, sign_mask_row=mK, sign_mask_col=mM, sf_layout=fp4q.SF_MMA)
    cfg_w = fp4q.Config(grid=fp4q.GRID_E2M1, rot=16, sign_mask_row=mK, sign_mask_col=mN, sf_layout=fp4q.SF_MMA)
    cfg_g = fp4q.Config(grid=fp4q.GRID_E2M1, rot=16, sign_mask_row=mN, sign_mask_col=mM, round=fp4q.SR,
                        sr_seed=SEED + 3, sf_layout=fp4q.SF_MMA)
    Xr, Xc = fp4q.alloc_operand(TOKENS, D_IN, cfg_x, dev), fp4q.alloc_operand(D_IN, TOKENS, cfg_x, dev)
    Wr, Wc = fp4q.alloc_operand(D_OUT, D_IN, cfg_w, dev), fp4q.alloc_operand(D_IN, D_OUT, cfg_w, dev)
    Gr, Gc = fp4q.alloc_operand(TOKENS, D_OUT, cfg_g, dev), fp4q.alloc_operand(D_OUT, TOKENS, cfg_g, dev)
    Y = torch.empty((TOKENS, D_OUT), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((TOKENS, D_IN), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((D_OUT, D_IN), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2

    q_bytes = MX_BYTES_PER_ELEM * (TOKENS * D_IN + D_OUT * D_IN + TOKENS * D_OUT)
    flops = 3 * 2.0 * TOKENS * D_IN * D_OUT
    launches_per_step = 5      # 3 quantizer launches, Fprop, the grouped Dgrad + Wgrad

    ev = lambda: torch.cuda.Event(enable_timing=True)
    kq = {"x": [], "w": [], "g": []}
    kg = {"fprop": [], "dgrad_wgrad": []}

    def quantize_phase(rec=None):
        e = [ev() for _ in range(4)] if rec is not None else None
        if e: e[0].record(stream)
        fp4q.rht_quantize(X, cfg_x, Xr, Xc, status=status, stream=stream)
        if e: e[1].record(stream)
        fp4q.rht_quantize(W, cfg_w, Wr, Wc, status=status, stream=stream)
        if e: e[2].record(stream)
        fp4q.rht_quantize(dY, cfg_g, Gr, Gc, status=status, stream=stream)
        if e: e[3].record(stream)
        if rec is not None:
            rec.append(("q", e))

    def gemm_phase(rec=None):
        # Fprop, then the backward GEMMs (Dgrad, Wgrad) in one grouped launch
        e = [ev() for _ in range(3)] if rec is not None else None
        if e: e[0].record(stream)
        fp4q.gemm(Xr, Wr, fp4q.GRID_E2M1, fp4q.SCALE_MX, want_f32=False, D_bf16=Y, status=status, stream=stream)
        if e: e[1].record(stream)
        fp4q.gemm_group([(Gr, Wc), (Gc, Xc)], fp4q.GRID_E2M1, fp4q.SCALE_MX, want_bf16=True, want_f32=False,
                        outs=[(dX, None), (dW, None)], status=status, stream=stream)
        if e: e[2].record(stream)
        if rec is not None:
            rec.append(("g", e))

    for _ in range(args.warmup):
        flush.zero_()
        quantize_phase()
        gemm_phase()
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} during warm-up")

    bus = None
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        pass
    clocks = ClockSampler(bus)
    clocks.start()
    time.sleep(0.3)
    recs = []
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()        # outside the events: evict the previous step from L2
        quantize_phase(recs)
        gemm_phase(recs)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the timed region")

    q_times, g_times = [], []
    for kind, e in recs:
        per = [e[i].elapsed_time(e[i + 1]) * 1e-3 for i in range(len(e) - 1)]
        (q_times if kind == "q" else g_times).append(sum(per))
        for key, t in zip(("x", "w", "g") if kind == "q" else ("fprop", "dgrad_wgrad"), per):
            (kq if kind == "q" else kg)[key].append(t)
    q_s = sum(q_times) / len(q_times)
    g_s = sum(g_times) / len(g_times)

    def pct(v):
        v = sorted(v)
        return {"p10_us": round(v[len(v) // 10] * 1e6, 2), "median_us": round(v[len(v) // 2] * 1e6, 2),
                "p90_us": round(v[(9 * len(v)) // 10] * 1e6, 2)}
    value = aggregate(q_bytes, q_s, world, dev) / 1e9
    gemm_tflops = aggregate(flops, g_s, world, dev) / 1e12

    # ---------------- end to end through the C ABI from pinned host buffers
    hX, hW, hdY = (t.cpu().pin_memory() for t in (X, W, dY))
    hY, hdX, hdW = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (Y, dX, dW))
    h2d = sum(t.numel() * t.element_size() for t in (hX, hW, hdY))
    d2h = sum(t.numel() * t.element_size() for t in (hY, hdX, hdW))
    # host<->device copies run on a copy stream (one copy engine's worth of link
    # bandwidth: splitting a copy over more streams measured no faster).  The
    # uploads go in the order dY, X, W so that the longest quantization (dY,
    # stochastic rounding) overlaps the uploads after it and only W's short one
    # is left at the end; the download of each GEMM's output overlaps the GEMMs
    # after it; every compute step waits for its own input's upload
    copy_stream = torch.cuda.Stream(dev)
    e2e_q, e2e_g = [], []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        copy_stream.wait_event(e0)
        up = [ev() for _ in range(3)]
        with torch.cuda.stream(copy_stream):
            for dst, src, u in ((dY, hdY, up[0]), (X, hX, up[1]), (W, hW, up[2])):
                dst.copy_(src, non_blocking=True)
                u.record(copy_stream)
        for u, (x, cfg, ro, co) in zip(up, ((dY, cfg_g, Gr, Gc), (X, cfg_x, Xr, Xc), (W, cfg_w, Wr, Wc))):
            stream.wait_event(u)
            fp4q.rht_quantize(x, cfg, ro, co, status=status, stream=stream)
        e1.record(stream)
        fp4q.gemm(Xr, Wr, fp4q.GRID_E2M1, fp4q.SCALE_MX, want_f32=False, D_bf16=Y, status=status, stream=stream)
        g = ev()
        g.record(stream)
        copy_stream.wait_event(g)
        with torch.cuda.stream(copy_stream):
            hY.copy_(Y, non_blocking=True)
        fp4q.gemm_group([(Gr, Wc), (Gc, Xc)], fp4q.GRID_E2M1, fp4q.SCALE_MX, want_bf16=True, want_f32=False,
                        outs=[(dX, None), (dW, None)], status=status, stream=stream)
        g = ev()
        g.record(stream)
        copy_stream.wait_event(g)
        with torch.cuda.stream(copy_stream):
            hdX.copy_(dX, non_blocking=True)
            hdW.copy_(dW, non_blocking=True)
        down = ev()
        down.record(copy_stream)
        stream.wait_event(down)
        e2.record(stream)
        e2.synchronize()
        if it >= args.warmup:
            e2e_q.append(e0.elapsed_time(e1) * 1e-3)
            e2e_g.append(e1.elapsed_time(e2) * 1e-3)
    e2e_value = aggregate(q_bytes, sum(e2e_q) / len(e2e_q), world, dev) / 1e9
    e2e_gemm = aggregate(flops, sum(e2e_g) / len(e2e_g), world, dev) / 1e12
    # the link alone: the same uploads and downloads with no compute (median of 5)
    link = {}
    for name, pairs in (("h2d", ((dY, hdY), (X, hX), (W, hW))), ("d2h", ((hY, Y), (hdX, dX), (hdW, dW)))):
        ts = []
        for _ in range(5):
            a, b = ev(), ev()
            a.record(copy_stream)
            with torch.cuda.stream(copy_stream):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            b.record(copy_stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e-3)
        link[name] = (h2d if name == "h2d" else d2h) / sorted(ts)[2] / 1e9

    # ---------------- rooflines of the two kernels (per-launch averages).  The
    # GEMM kernel runs twice a step (Fprop; Dgrad + Wgrad grouped): achieved =
    # the step's GEMM flops / the two launches' summed durations, traffic = the
    # mean of the two launches' measured DRAM bytes
    g_achieved = flops / (statistics.mean(kg["fprop"]) + statistics.mean(kg["dgrad_wgrad"])) / 1e12
    x_launch = statistics.mean(kq["x"])
    x_bytes = MX_BYTES_PER_ELEM * TOKENS * D_IN
    x_achieved = x_bytes / x_launch / 1e9
    traffic = read_traffic()
    dominant_gemm = sum(g_times) >= sum(q_times)
    g_traffic = None
    if "gemm_mxf4_fprop_bytes" in traffic and "gemm_mxf4_group_dgrad_wgrad_bytes" in traffic:
        g_traffic = (traffic["gemm_mxf4_fprop_bytes"] + traffic["gemm_mxf4_group_dgrad_wgrad_bytes"]) // 2
    roof_gemm = {"kernel": "bs_gemm_kernel<mxf4> (tcgen05): Fprop launch + grouped Dgrad/Wgrad launch",
                 "bound": "tensor", "achieved": round(g_achieved, 1),
                 "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(g_achieved / fp4_peak, 4),
                 "traffic": g_traffic,
                 "peak_source": f"{peak_src} bf16 burst x 6 (nominal FP4:BF16 dense ratio)"}
    roof_q = {"kernel": "rht_quant_kernel (X, both copies)", "bound": "hbm", "achieved": round(x_achieved, 1),
              "peak": hbm_peak, "unit": "GB/s", "frac": round(x_achieved / hbm_peak, 4),
              "traffic": traffic.get("quant_x_bytes"), "peak_source": f"{peak_src} HBM copy"}

    line = {
        "metric": "fused RHT+FP4 quantize GB/s and % of HBM peak; block-scaled FP4 GEMM TFLOPS",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((q_s + g_s) * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp4-e2m1 (fp32 quantizer arithmetic, fp32 accumulate)",
        "data": "synthetic (seeded; shapes of Llama-3.1-8B hidden 4096, 16384 tokens)",
        "config": {"workload": WORKLOAD, "global_batch_tokens": TOKENS * world, "per_rank": "replica",
                   "l2": "flushed (256 MiB write) before every timed step", "recipe": "E2M1 MXFP4 H16"},
        "hbm_frac": round(value / world / hbm_peak, 4),
        "inputs_sha256": {"X": synth.sha256(Xb), "W": synth.sha256(Wb), "dY": synth.sha256(dYb)},
        "quantize": {"us_per_step": round(q_s * 1e6, 2), "gb_s": round(value, 1), "spread": pct(q_times),
                     "bytes_per_step": q_bytes, "per_tensor_us": {k: round(statistics.mean(v) * 1e6, 2)
                                                                  for k, v in kq.items()}},
        "gemm": {"tflops": round(gemm_tflops, 1), "us_per_step": round(g_s * 1e6, 2), "flops_per_step": flops,
                 "spread": pct(g_times),
                 "per_gemm_us": {k: round(statistics.mean(v) * 1e6, 2) for k, v in kg.items()}},
        "roofline": roof_gemm if dominant_gemm else roof_q,
        "roofline_other": roof_q if dominant_gemm else roof_gemm,
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "gemm_tflops": round(e2e_gemm, 1),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "link_h2d_gb_s": round(link["h2d"], 1), "link_d2h_gb_s": round(link["d2h"], 1),
                "note": "H2D of dY/X/W (in that order) inside the quantize phase, D2H of Y/dX/dW inside the GEMM "
                        "phase; copies on a second stream overlap the compute that does not depend on them; "
                        "link_*: the same copies alone"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 4),
    }
    if not args.no_configs:
        del hX, hW, hdY, hY, hdX, hdW
        line["quantizer_configs"] = quant_configs(dev, stream, flush)
        line["epilogue_fusion"] = epilogue_fusion(dev, stream, flush, X, W, cfg_x, cfg_w)
        line["recipe_quality"] = recipe_quality(X, W, dY)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    return line


def read_traffic() -> dict:
    """DRAM bytes per launch measured by ncu (profiles/dram_traffic.txt: 'key bytes' lines)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if os.path.exists(path):
        for line in open(path):
            parts = line.split()
            if len(parts) == 2 and not line.startswith("#"):
                out[parts[0]] = int(parts[1])
    return out


# ------------------------------------------------------------------ quantizer configurations
def quant_configs(dev, stream, flush, reps: int = 20) -> dict:
    """The quantizer alone on each workload shape: microseconds per call (median
    of `reps`, L2 flushed before each, outside the events) and GB/s of
    algorithmic bytes; the fused call against the same call without rotation
    (plain) and against a separate rotation kernel followed by plain
    quantization of each rotated copy (unfused)."""
    import torch

    from fp4_microscaled_quantization_gb300 import fp4q, synth

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            if i >= 2:
                ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    out = {}

    def entry(name, us, nbytes):
        out[name] = {"us": round(us, 2), "gb_s": round(nbytes / us / 1e3, 1) if nbytes else None}

    def q_bytes(R, C, b, copies):
        return 2.0 * R * C + copies * R * C * (0.5 + 1.0 / b)

    # tiny: X 256x512, row-wise copy only, random H16 (launch-bound; microseconds only)
    x = synth.as_torch(synth.tiny_x()).to(dev)
    m = fp4q.sign_mask_from_seed(1001, 16)
    for g, gname in ((0, "e2m1"), (1, "e1m2")):
        cfg = fp4q.Config(grid=g, rot=16, sign_mask_row=m, want_col=False)
        ro, _ = fp4q.rht_quantize(x, cfg, stream=stream)
        entry(f"tiny_256x512_row_{gname}", timed(lambda: fp4q.rht_quantize(x, cfg, ro, stream=stream)), 0)
    # activations: X 8192x4096 both copies, deterministic H16, MX; plain and unfused arms
    x = synth.as_torch(synth.act_x()).to(dev)
    R, C = x.shape
    for g, gname in ((0, "e2m1"), (1, "e1m2"), (2, "e2m1_cap4")):
        cfg = fp4q.Config(grid=g, rot=16)
        ro, co = fp4q.rht_quantize(x, cfg, stream=stream)
        entry(f"act_8192x4096_{gname}_h16", timed(lambda: fp4q.rht_quantize(x, cfg, ro, co, stream=stream)),
              q_bytes(R, C, 32, 2))
    cfg = fp4q.Config(grid=0, rot=0)
    ro, co = fp4q.rht_quantize(x, cfg, stream=stream)
    plain = timed(lambda: fp4q.rht_quantize(x, cfg, ro, co, stream=stream))
    entry("act_8192x4096_e2m1_plain", plain, q_bytes(R, C, 32, 2))
    yr = torch.empty_like(x)
    yc = torch.empty_like(x)
    cr = fp4q.Config(grid=0, rot=0, want_col=False)
    cc = fp4q.Config(grid=0, rot=0, want_row=False)

    def unfused():
        fp4q.hadamard_rotate_bf16(x, 16, 0, 0, y_row=yr, y_col=yc, stream=stream)
        fp4q.rht_quantize(yr, cr, ro, None, stream=stream)
        fp4q.rht_quantize(yc, cc, None, co, stream=stream)
    unf = timed(unfused)
    entry("act_8192x4096_e2m1_unfused", unf, q_bytes(R, C, 32, 2))
    fused = out["act_8192x4096_e2m1_h16"]["us"]
    out["fusion_ratio_fused_over_plain"] = round(fused / plain, 3)
    out["fusion_ratio_unfused_over_plain"] = round(unf / plain, 3)
    del x, yr, yc
    # gradients: dY 8192x14336, E1M2, random H16, stochastic rounding, both copies
    x = synth.as_torch(synth.grad_dy()).to(dev)
    R, C = x.shape
    cfg = fp4q.Config(grid=1, rot=16, round=fp4q.SR, sign_mask_row=fp4q.sign_mask_from_seed(1003, 16),
                      sign_mask_col=fp4q.sign_mask_from_seed(1004, 16), sr_seed=1004)
    ro, co = fp4q.rht_quantize(x, cfg, stream=stream)
    entry("grad_8192x14336_e1m2_sr_h16", timed(lambda: fp4q.rht_quantize(x, cfg, ro, co, stream=stream)),
          q_bytes(R, C, 32, 2))
    del x, ro, co
    # weights: W 14336x4096, deterministic H32, NVFP4-style scales, one and two passes
    x = synth.as_torch(synth.weight_w()).to(dev)
    R, C = x.shape
    for g, gname in ((0, "e2m1"), (1, "e1m2")):
        cfg = fp4q.Config(grid=g, scale=fp4q.SCALE_NV, rot=32)
        ro, co = fp4q.rht_quantize(x, cfg, stream=stream)
        ws = torch.empty(max(1, fp4q.workspace_bytes(R, C, cfg)), dtype=torch.uint8, device=dev)
        entry(f"weight_14336x4096_{gname}_nv_h32_two_pass",
              timed(lambda: fp4q.rht_quantize(x, cfg, ro, co, workspace=ws, stream=stream)),
              q_bytes(R, C, 16, 2) + 2.0 * R * C)
        amax = fp4q.rotated_amax(x, cfg, stream=stream)
        cfg1 = fp4q.Config(grid=g, scale=fp4q.SCALE_NV, rot=32, global_amax=amax)
        entry(f"weight_14336x4096_{gname}_nv_h32_one_pass",
              timed(lambda: fp4q.rht_quantize(x, cfg1, ro, co, stream=stream)), q_bytes(R, C, 16, 2))
    torch.cuda.synchronize(dev)
    return out


def epilogue_fusion(dev, stream, flush, X, W, cfg_x, cfg_w, reps: int = 20) -> dict:
    """Fprop followed by the quantization of its bf16 output for the next layer
    (row-wise copy, random H16, MX E2M1): the two calls against the GEMM that
    quantizes in its epilogue (no bf16 output)."""
    import torch

    from fp4_microscaled_quantization_gb300 import fp4q

    Xr, _ = fp4q.rht_quantize(X, fp4q.Config(grid=cfg_x.grid, rot=16, sign_mask_row=cfg_x.sign_mask_row,
                                             want_col=False, sf_layout=fp4q.SF_MMA), stream=stream)
    Wr, _ = fp4q.rht_quantize(W, fp4q.Config(grid=cfg_w.grid, rot=16, sign_mask_row=cfg_w.sign_mask_row,
                                             want_col=False, sf_layout=fp4q.SF_MMA), stream=stream)
    M, N = Xr.rows, Wr.rows
    ocfg = fp4q.Config(rot=16, sign_mask_row=fp4q.sign_mask_from_seed(SEED + 7, 16), want_col=False,
                       sf_layout=fp4q.SF_MMA)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    q1 = fp4q.alloc_operand(M, N, ocfg, dev)
    q2 = fp4q.alloc_operand(M, N, ocfg, dev)

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            if i >= 2:
                ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    def two_calls():
        fp4q.gemm(Xr, Wr, fp4q.GRID_E2M1, fp4q.SCALE_MX, want_f32=False, D_bf16=Y, stream=stream)
        fp4q.rht_quantize(Y, ocfg, q1, stream=stream)

    t2 = timed(two_calls)
    t1 = timed(lambda: fp4q.gemm_quantize(Xr, Wr, fp4q.GRID_E2M1, fp4q.SCALE_MX, ocfg, out=q2, stream=stream))
    torch.cuda.synchronize(dev)
    same = bool(torch.equal(q1.codes, q2.codes) and torch.equal(q1.scales, q2.scales))
    return {"shape": f"{M}x{N}x{Xr.cols}", "gemm_then_quantize_us": round(t2, 2), "fused_us": round(t1, 2),
            "fused_over_two_calls": round(t1 / t2, 3), "identical_copies": same}


def recipe_quality(X, W, dY) -> dict:
    """Output SQNR (dB), attenuation alpha and shrinkage of Fprop, Dgrad and Wgrad
    under the UFP4 and E2M1 recipes, against fp32 GEMMs of the bf16 originals."""
    from fp4_microscaled_quantization_gb300 import linear

    ref = linear.reference_gemms(X, W, dY)
    out = {}
    for recipe in linear.RECIPES:
        res = linear.Fp4Linear(recipe, seed=SEED, out_f32=True)(X, W, dY)
        q = linear.output_quality(res, ref)
        out[recipe] = {k: {m: round(v[m], 5) for m in ("sqnr_db", "alpha", "shrinkage")} for k, v in q.items()}
    return out


# ------------------------------------------------------------------ oracle arm
def _oracle_sample(rows: int):
    from fp4_microscaled_quantization_gb300 import synth
    Xb, Wb, dYb = synth.layer(TOKENS, D_IN, D_OUT, SEED)
    return Xb[:rows].copy(), Wb[: max(128, rows // 4)].copy(), dYb[:rows].copy()


def _oracle_step(orc, Xs, Ws, Gs, mK, mN, mM):
    orc.quantize(Xs, 0, 0, 0, 16, mK)
    orc.quantize(Xs, 1, 0, 0, 16, mM)
    orc.quantize(Ws, 0, 0, 0, 16, mK)
    orc.quantize(Ws, 1, 0, 0, 16, mN)
    orc.quantize(Gs, 0, 0, 0, 16, mN, orc.SR, SEED + 3)
    orc.quantize(Gs, 1, 0, 0, 16, mM, orc.SR, SEED + 3)


def cpu_baseline(args, rows: int = 1024, min_s: float = 10.0) -> dict:
    """The CPU oracle (single-threaded C) on a bounded sample of the same step."""
    import oracle
    orc = oracle
    orc.build()
    Xs, Ws, Gs = _oracle_sample(rows)
    mK, mN, mM = (orc.sign_mask_from_seed(SEED + i, 16) for i in range(3))
    nbytes = MX_BYTES_PER_ELEM * (Xs.size + Ws.size + Gs.size)
    t0 = time.perf_counter()
    n = 0
    while True:
        _oracle_step(orc, Xs, Ws, Gs, mK, mN, mM)
        n += 1
        if time.perf_counter() - t0 >= min_s:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"quantize (both copies) of rows 0..{rows - 1} of X and dY and rows 0..{Ws.shape[0] - 1} "
                      f"of W of the same workload, {n} repetitions, {dt:.2f} s each; GEMMs not included"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    rows = 256
    Xs, Ws, Gs = _oracle_sample(rows)
    mK, mN, mM = (oracle.sign_mask_from_seed(SEED + i, 16) for i in range(3))
    nbytes = MX_BYTES_PER_ELEM * (Xs.size + Ws.size + Gs.size)
    for _ in range(args.warmup):
        _oracle_step(oracle, Xs, Ws, Gs, mK, mN, mM)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, Xs, Ws, Gs, mK, mN, mM)
    dt = (time.perf_counter() - t0) / args.steps
    v = round(nbytes / dt / 1e9, 4)
    sample = (f"quantize (both copies) of rows 0..{rows - 1} of X and dY and rows 0..{Ws.shape[0] - 1} of W "
              f"per step; GEMMs not included")
    return {"impl": "reference", "metric": "fused RHT+FP4 quantize GB/s and % of HBM peak; block-scaled FP4 GEMM TFLOPS",
            "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp32 quantizer arithmetic (CPU oracle)", "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-shape quantizer timings")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
