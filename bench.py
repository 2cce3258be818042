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

import numpy as np

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
# The two recipes of one linear layer's step ("Repensando o Vies de
# Encolhimento", Metodologia 2): E2M1 GEMMs on kind::mxf4; UFP4 = the uniform
# E1M2 grid, whose GEMMs run kind::mxf8f6f4 on the exact E4M3 bytes of the
# codes (one more byte per element and copy written by the quantizer).
RECIPES = {"e2m1": {"grid": 0, "e4m3": False, "mma": "kind::mxf4 (FP4)", "flop_ratio": 13.5 / 2.25,
                    "mma_flop_clk_sm": 32768},
           "ufp4": {"grid": 1, "e4m3": True, "mma": "kind::mxf8f6f4 (FP8 E4M3 bytes of E1M2 codes)",
                    "flop_ratio": 4.5 / 2.25, "mma_flop_clk_sm": 16384}}


def recipe_buffers(fp4q, recipe, dev):
    """Configs (random H16 with signs shared along each contraction axis, RTNE on
    X and W, Philox SR on dY, MMA scale layout) and the six copies and three
    outputs of one recipe."""
    grid, e4 = RECIPES[recipe]["grid"], RECIPES[recipe]["e4m3"]
    mK = fp4q.sign_mask_from_seed(SEED, 16)
    mN = fp4q.sign_mask_from_seed(SEED + 1, 16)
    mM = fp4q.sign_mask_from_seed(SEED + 2, 16)
    cx = fp4q.Config(grid=grid, rot=16, sign_mask_row=mK, sign_mask_col=mM, sf_layout=fp4q.SF_MMA, emit_e4m3=e4)
    cw = fp4q.Config(grid=grid, rot=16, sign_mask_row=mK, sign_mask_col=mN, sf_layout=fp4q.SF_MMA, emit_e4m3=e4)
    cg = fp4q.Config(grid=grid, rot=16, sign_mask_row=mN, sign_mask_col=mM, round=fp4q.SR, sr_seed=SEED + 3,
                     sf_layout=fp4q.SF_MMA, emit_e4m3=e4)
    import torch
    b = {"grid": grid, "cfg": (cx, cw, cg),
         "Xr": fp4q.alloc_operand(TOKENS, D_IN, cx, dev), "Xc": fp4q.alloc_operand(D_IN, TOKENS, cx, dev),
         "Wr": fp4q.alloc_operand(D_OUT, D_IN, cw, dev), "Wc": fp4q.alloc_operand(D_IN, D_OUT, cw, dev),
         "Gr": fp4q.alloc_operand(TOKENS, D_OUT, cg, dev), "Gc": fp4q.alloc_operand(D_OUT, TOKENS, cg, dev),
         "Y": torch.empty((TOKENS, D_OUT), dtype=torch.bfloat16, device=dev),
         "dX": torch.empty((TOKENS, D_IN), dtype=torch.bfloat16, device=dev),
         "dW": torch.empty((D_OUT, D_IN), dtype=torch.bfloat16, device=dev)}
    b["bytes_per_elem"] = MX_BYTES_PER_ELEM + (2.0 if e4 else 0.0)
    return b


def pct(v):
    v = sorted(v)
    return {"p10_us": round(v[len(v) // 10] * 1e6, 2), "median_us": round(v[len(v) // 2] * 1e6, 2),
            "p90_us": round(v[(9 * len(v)) // 10] * 1e6, 2)}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_ours(args, world, rank, local):
    import torch

    from fp4_microscaled_quantization_gb300 import fp4q, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    bf16_peak = peaks.get("bf16_tflops", 1900.0)
    peak_src = "measured" if peaks else "fallback"
    props = torch.cuda.get_device_properties(dev)
    n_sm = props.multi_processor_count
    sm_max_mhz = peaks.get("sm_max_mhz", 2070.0)

    # ---------------- inputs (bf16, resident)
    Xb, Wb, dYb = synth.layer(TOKENS, D_IN, D_OUT, SEED)
    X, W, dY = (synth.as_torch(a).to(dev) for a in (Xb, Wb, dYb))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2
    elems = TOKENS * D_IN + D_OUT * D_IN + TOKENS * D_OUT
    flops = 3 * 2.0 * TOKENS * D_IN * D_OUT
    launches_per_step = 5      # 3 quantizer launches, Fprop, the grouped Dgrad + Wgrad
    rb = {r: recipe_buffers(fp4q, r, dev) for r in RECIPES}

    ev = lambda: torch.cuda.Event(enable_timing=True)

    def quantize_phase(b, e=None):
        cx, cw, cg = b["cfg"]
        if e: e[0].record(stream)
        fp4q.rht_quantize(X, cx, b["Xr"], b["Xc"], status=status, stream=stream)
        if e: e[1].record(stream)
        fp4q.rht_quantize(W, cw, b["Wr"], b["Wc"], status=status, stream=stream)
        if e: e[2].record(stream)
        fp4q.rht_quantize(dY, cg, b["Gr"], b["Gc"], status=status, stream=stream)
        if e: e[3].record(stream)

    def gemm_phase(b, e=None):
        # Fprop, then the backward GEMMs (Dgrad, Wgrad) in one grouped launch
        if e: e[0].record(stream)
        fp4q.gemm(b["Xr"], b["Wr"], b["grid"], fp4q.SCALE_MX, want_f32=False, D_bf16=b["Y"], status=status,
                  stream=stream)
        if e: e[1].record(stream)
        fp4q.gemm_group([(b["Gr"], b["Wc"]), (b["Gc"], b["Xc"])], b["grid"], fp4q.SCALE_MX, want_bf16=True,
                        want_f32=False, outs=[(b["dX"], None), (b["dW"], None)], status=status, stream=stream)
        if e: e[2].record(stream)

    # The timed steps record events at the phase boundaries only, so that each
    # kernel's launch overlaps the tail of the one before it (programmatic
    # dependent launch).  The per-launch split comes from separate steps with
    # an event between every launch, which serialises them.
    def timed_steps(b, steps):
        recs = []
        for _ in range(steps):
            flush.zero_()        # outside the events: evict the previous step from L2
            e = [ev() for _ in range(3)]
            e[0].record(stream)
            quantize_phase(b)
            e[1].record(stream)
            gemm_phase(b)
            e[2].record(stream)
            recs.append(e)
        return recs

    def split_steps(b, steps):
        recs = []
        for _ in range(steps):
            flush.zero_()
            eq, eg = [ev() for _ in range(4)], [ev() for _ in range(3)]
            quantize_phase(b, eq)
            gemm_phase(b, eg)
            recs.append((eq, eg))
        return recs

    def summarize(recs):
        q_times = [e[0].elapsed_time(e[1]) * 1e-3 for e in recs]
        g_times = [e[1].elapsed_time(e[2]) * 1e-3 for e in recs]
        return q_times, g_times

    def summarize_split(recs):
        kq = {"x": [], "w": [], "g": []}
        kg = {"fprop": [], "dgrad_wgrad": []}
        for eq, eg in recs:
            for i, k in enumerate(kq):
                kq[k].append(eq[i].elapsed_time(eq[i + 1]) * 1e-3)
            for i, k in enumerate(kg):
                kg[k].append(eg[i].elapsed_time(eg[i + 1]) * 1e-3)
        return kq, kg

    for _ in range(args.warmup):
        for r in RECIPES:
            flush.zero_()
            quantize_phase(rb[r])
            gemm_phase(rb[r])
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} during warm-up")

    bus = None
    try:
        bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except AttributeError:
        pass
    clocks = ClockSampler(bus)
    clocks.start()
    time.sleep(0.3)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    recs = timed_steps(rb["e2m1"], args.steps)          # the timed region of the headline metric
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    wall = time.perf_counter() - wall0
    recs_u = timed_steps(rb["ufp4"], args.steps)        # the second recipe, same step, same sizes
    n_split = min(args.steps, 200)
    split = {r: split_steps(rb[r], n_split) for r in RECIPES}   # per-launch split, outside the timed region
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item():#x} in the timed region")

    q_times, g_times = summarize(recs)
    kq, kg = summarize_split(split["e2m1"])
    q_s = sum(q_times) / len(q_times)
    g_s = sum(g_times) / len(g_times)
    q_bytes = MX_BYTES_PER_ELEM * elems
    value = aggregate(q_bytes, q_s, world, dev) / 1e9
    gemm_tflops = aggregate(flops, g_s, world, dev) / 1e12
    clock_mhz = clk.get("sm_mhz") or sm_max_mhz

    # ---------------- rooflines.  The GEMM kernel runs twice a step (Fprop; the
    # grouped Dgrad + Wgrad): achieved = the step's GEMM flops / the mean time
    # of the GEMM phase (the two launches back to back) in the timed steps.  Denominators: the measured bf16 GEMM
    # rate x the nominal dense ratio of the kind (the recipe's rule), and, for
    # reference, ncu's FP4 peak (49152 flop/clk/SM) and the rate of the MMA
    # instruction this kernel issues (128 cycles per 128 x 256 x 64 FP4 MMA per
    # SM, measured), both at the maximum SM clock.
    traffic = read_traffic()

    def gemm_roof(r, g_phase, peak_bf16):
        achieved = flops / statistics.mean(g_phase) / 1e12
        peak = peak_bf16 * RECIPES[r]["flop_ratio"]
        mma_peak = RECIPES[r]["mma_flop_clk_sm"] * n_sm * sm_max_mhz * 1e6 / 1e12
        out = {"kernel": f"bs_gemm_kernel ({RECIPES[r]['mma']}, cta_group::2): Fprop launch + grouped "
                         "Dgrad/Wgrad launch",
               "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
               "frac": round(achieved / peak, 4),
               "peak_source": f"{peak_src} bf16 burst x {RECIPES[r]['flop_ratio']:.0f} (nominal dense ratio)",
               "mma_instruction_peak": round(mma_peak, 1), "frac_of_mma_instruction_peak": round(achieved / mma_peak, 4)}
        if r == "e2m1":
            ncu_peak = 49152 * n_sm * sm_max_mhz * 1e6 / 1e12
            out["ncu_fp4_peak"] = round(ncu_peak, 1)
            out["frac_of_ncu_fp4_peak"] = round(achieved / ncu_peak, 4)
        key = "gemm_mxf4" if r == "e2m1" else "gemm_mxf8f6f4"
        g_traffic = traffic.get(f"{key}_fprop_bytes"), traffic.get(f"{key}_group_dgrad_wgrad_bytes")
        out["traffic"] = (g_traffic[0] + g_traffic[1]) // 2 if all(g_traffic) else None
        out["traffic_source"] = "ncu capture summarised in profiles/dram_traffic.txt (per launch, mean of the two)"
        return out

    roof_gemm = gemm_roof("e2m1", g_times, bf16_peak)
    q_achieved = q_bytes / q_s / 1e9
    roof_q = {"kernel": "rht_quant_kernel: the step's three launches (X, W RTNE; dY SR), both copies each",
              "bound": "hbm", "achieved": round(q_achieved, 1), "peak": hbm_peak, "unit": "GB/s",
              "frac": round(q_achieved / hbm_peak, 4), "traffic": traffic.get("quant_step_bytes"),
              "peak_source": f"{peak_src} HBM copy",
              "per_launch_frac": {k: round(MX_BYTES_PER_ELEM * n / statistics.mean(kq[k]) / 1e9 / hbm_peak, 4)
                                  for k, n in (("x", TOKENS * D_IN), ("w", D_OUT * D_IN), ("g", TOKENS * D_OUT))},
              "per_launch_source": f"{n_split} separate steps with an event between every launch"}
    dominant_gemm = sum(g_times) >= sum(q_times)

    # ---------------- the UFP4 recipe's step
    uq, ug = summarize(recs_u)
    ukq, ukg = summarize_split(split["ufp4"])
    u_bytes = rb["ufp4"]["bytes_per_elem"] * elems
    ufp4 = {"recipe": "UFP4: E1M2 grid, MX b32, random H16 on all three GEMMs, RTNE X/W, SR dY; "
                      "GEMMs on kind::mxf8f6f4 over the E4M3 bytes of the E1M2 codes",
            "quantize": {"gb_s": round(u_bytes / statistics.mean(uq) / 1e9, 1), "spread": pct(uq),
                         "bytes_per_step": u_bytes, "bytes_per_elem": rb["ufp4"]["bytes_per_elem"],
                         "frac_of_hbm": round(u_bytes / statistics.mean(uq) / 1e9 / hbm_peak, 4),
                         "per_tensor_us": {k: round(statistics.mean(v) * 1e6, 2) for k, v in ukq.items()}},
            "gemm": {"tflops": round(flops / statistics.mean(ug) / 1e12, 1), "spread": pct(ug),
                     "per_gemm_us": {k: round(statistics.mean(v) * 1e6, 2) for k, v in ukg.items()}},
            "roofline": gemm_roof("ufp4", ug, bf16_peak),
            "ms_per_step": round((statistics.mean(uq) + statistics.mean(ug)) * 1e3, 4)}

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
        "per_launch_split": f"per_tensor_us / per_gemm_us: {n_split} separate steps with an event between every "
                            "launch (serialised launches); the phase times come from the timed steps, events at "
                            "the phase boundaries only",
        "gemm": {"tflops": round(gemm_tflops, 1), "us_per_step": round(g_s * 1e6, 2), "flops_per_step": flops,
                 "spread": pct(g_times),
                 "per_gemm_us": {k: round(statistics.mean(v) * 1e6, 2) for k, v in kg.items()}},
        "roofline": roof_gemm if dominant_gemm else roof_q,
        "roofline_other": roof_q if dominant_gemm else roof_gemm,
        "ufp4": ufp4,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 4),
    }
    line["e2e"] = end_to_end(args, fp4q, rb["e2m1"], X, W, dY, status, stream, flush, q_bytes, flops, world, dev)
    if not args.no_configs:
        line["tiny_config"] = tiny_config(dev, stream)
        line["quantizer_configs"] = quant_configs(dev, stream, flush)
        b = rb["e2m1"]
        line["epilogue_fusion"] = epilogue_fusion(dev, stream, flush, X, W, b["cfg"][0], b["cfg"][1])
        line["recipe_quality"] = recipe_quality(X, W, dY)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    return line


def end_to_end(args, fp4q, b, X, W, dY, status, stream, flush, q_bytes, flops, world, dev):
    """The E2M1 step through the C ABI from pinned host buffers: the H2D copies
    of dY, X, W inside the quantize phase, the D2H copies of Y, dX, dW inside
    the GEMM phase, on a copy stream that overlaps the compute not waiting for
    them.  Median (and p10/p90) over the timed steps, after at least ten
    untimed ones (the first uploads into freshly pinned buffers are slow)."""
    import torch
    ev = lambda: torch.cuda.Event(enable_timing=True)
    cx, cw, cg = b["cfg"]
    hX, hW, hdY = (t.cpu().pin_memory() for t in (X, W, dY))
    hY, hdX, hdW = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (b["Y"], b["dX"], b["dW"]))
    h2d = sum(t.numel() * t.element_size() for t in (hX, hW, hdY))
    d2h = sum(t.numel() * t.element_size() for t in (hY, hdX, hdW))
    # uploads in the order dY, X, W: the longest quantization (dY, stochastic
    # rounding) overlaps the uploads after it; each compute step waits for its
    # own input's upload; each GEMM's download overlaps the GEMMs after it
    copy_stream = torch.cuda.Stream(dev)
    e2e_q, e2e_g = [], []
    warm = max(args.warmup, 10)
    for it in range(warm + args.steps):
        flush.zero_()
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        copy_stream.wait_event(e0)
        up = [ev() for _ in range(3)]
        with torch.cuda.stream(copy_stream):
            for dst, src, u in ((dY, hdY, up[0]), (X, hX, up[1]), (W, hW, up[2])):
                dst.copy_(src, non_blocking=True)
                u.record(copy_stream)
        for u, (x, cfg, ro, co) in zip(up, ((dY, cg, b["Gr"], b["Gc"]), (X, cx, b["Xr"], b["Xc"]),
                                            (W, cw, b["Wr"], b["Wc"]))):
            stream.wait_event(u)
            fp4q.rht_quantize(x, cfg, ro, co, status=status, stream=stream)
        e1.record(stream)
        fp4q.gemm(b["Xr"], b["Wr"], b["grid"], fp4q.SCALE_MX, want_f32=False, D_bf16=b["Y"], status=status,
                  stream=stream)
        g = ev()
        g.record(stream)
        copy_stream.wait_event(g)
        with torch.cuda.stream(copy_stream):
            hY.copy_(b["Y"], non_blocking=True)
        fp4q.gemm_group([(b["Gr"], b["Wc"]), (b["Gc"], b["Xc"])], b["grid"], fp4q.SCALE_MX, want_bf16=True,
                        want_f32=False, outs=[(b["dX"], None), (b["dW"], None)], status=status, stream=stream)
        g = ev()
        g.record(stream)
        copy_stream.wait_event(g)
        with torch.cuda.stream(copy_stream):
            hdX.copy_(b["dX"], non_blocking=True)
            hdW.copy_(b["dW"], non_blocking=True)
        down = ev()
        down.record(copy_stream)
        stream.wait_event(down)
        e2.record(stream)
        e2.synchronize()
        if it >= warm:
            e2e_q.append(e0.elapsed_time(e1) * 1e-3)
            e2e_g.append(e1.elapsed_time(e2) * 1e-3)
    q_med, g_med = statistics.median(e2e_q), statistics.median(e2e_g)
    e2e_value = aggregate(q_bytes, q_med, world, dev) / 1e9
    e2e_gemm = aggregate(flops, g_med, world, dev) / 1e12
    # the link alone: the same uploads and downloads with no compute (median of 5)
    link = {}
    for name, pairs in (("h2d", ((dY, hdY), (X, hX), (W, hW))), ("d2h", ((hY, b["Y"]), (hdX, b["dX"]),
                                                                      (hdW, b["dW"])))):
        ts = []
        for _ in range(5):
            a, z = ev(), ev()
            a.record(copy_stream)
            with torch.cuda.stream(copy_stream):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            z.record(copy_stream)
            z.synchronize()
            ts.append(a.elapsed_time(z) * 1e-3)
        link[name] = (h2d if name == "h2d" else d2h) / sorted(ts)[2] / 1e9
    return {"value": round(e2e_value, 1), "unit": "GB/s", "gemm_tflops": round(e2e_gemm, 1),
            "statistic": f"median of {args.steps} steps after {warm} untimed ones",
            "quantize_spread": pct(e2e_q), "gemm_spread": pct(e2e_g),
            "quantize_mean_us": round(statistics.mean(e2e_q) * 1e6, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "link_h2d_gb_s": round(link["h2d"], 1), "link_d2h_gb_s": round(link["d2h"], 1),
            "note": "H2D of dY/X/W (in that order) inside the quantize phase, D2H of Y/dX/dW inside the GEMM "
                    "phase; copies on a second stream overlap the compute that does not depend on them; "
                    "link_*: the same copies alone"}


def tiny_config(dev, stream) -> dict:
    """The tiny single-tensor workload (X 256x512, N(0,1) with 1% of positions
    x50; row-wise copy, H16 with seeded signs, MX E2M1 and E1M2, RTNE): the
    codes and scales (SHA-256 and code histogram), and the reconstruction's
    SQNR, attenuation alpha and shrinkage against X in the original domain,
    the per-element mean signed relative error beside that aggregate, and the
    rounding error in grid units, overall and per level."""
    import torch

    from fp4_microscaled_quantization_gb300 import fp4q, synth
    bits = synth.tiny_x()
    x = synth.as_torch(bits).to(dev)
    xf = x.float()
    mask = fp4q.sign_mask_from_seed(1001, 16)
    out = {"shape": "256x512", "rot": "H16", "sign_mask": f"{mask:#06x}"}
    for g, name in ((0, "e2m1"), (1, "e1m2")):
        cfg = fp4q.Config(grid=g, rot=16, sign_mask_row=mask, want_col=False)
        ro, _ = fp4q.rht_quantize(x, cfg, stream=stream)
        deq = fp4q.dequantize(ro, cfg, orient=0, unrotate=True)
        st = fp4q.bias_stats(xf, deq, ro.codes)
        rel = fp4q.rel_error(xf.reshape(-1), deq.reshape(-1), stream=stream)
        ge = fp4q.grid_error(x, cfg, ro, stream=stream)
        torch.cuda.synchronize(dev)
        codes = ro.codes.cpu().numpy()
        scales = ro.scales.cpu().numpy()
        out[name] = {"codes_sha256": synth.sha256(codes), "scales_sha256": synth.sha256(scales),
                     "code_histogram": [int(v) for v in st["hist"]],
                     "sqnr_db": round(st["sqnr_db"], 4), "alpha": round(st["alpha"], 6),
                     "shrinkage": round(st["shrinkage"], 6),
                     "mean_rel_error": round(rel["mean"], 6),
                     "grid_error_mean": round(ge["mean"], 6),
                     "grid_error_per_level": [round(float(sm / c), 4) if c else None
                                              for sm, c in zip(ge["sums"], ge["counts"])]}
    return out


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
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "cpu_model": cpu_model(),
            "host_threads": os.cpu_count(), "kind": "oracle",
            "sample": f"quantize (both copies) of rows 0..{rows - 1} of X and dY and rows 0..{Ws.shape[0] - 1} "
                      f"of W of the same workload, {n} repetitions, {dt:.2f} s each; the GEMMs in `gemm`",
            "gemm": cpu_gemm_sample(orc, Xs, Ws, mK)}


def cpu_gemm_sample(orc, Xs, Ws, mK, entries: int = 65536, min_s: float = 3.0) -> dict:
    """The oracle's GEMM (one fp64 dot per output entry, single-threaded C) on
    sampled Fprop outputs of the same workload: the rows of X and W that the
    quantize sample holds, quantized and dequantized by the oracle, and
    `entries` seeded (row, column) pairs with K = 4096."""
    qa = orc.quantize(Xs, 0, 0, orc.SCALE_MX, 16, mK)
    qb = orc.quantize(Ws, 0, 0, orc.SCALE_MX, 16, mK)
    A = orc.dequantize(qa["codes"], qa["scales"], 0.0, 0, orc.SCALE_MX)
    B = orc.dequantize(qb["codes"], qb["scales"], 0.0, 0, orc.SCALE_MX)
    g = np.random.Generator(np.random.PCG64(SEED))
    ii = g.integers(0, A.shape[0], entries)
    jj = g.integers(0, B.shape[0], entries)
    t0 = time.perf_counter()
    n = 0
    while True:
        orc.gemm_entries(A, B, ii, jj)
        n += 1
        if time.perf_counter() - t0 >= min_s:
            break
    dt = (time.perf_counter() - t0) / n
    flops = 2.0 * entries * A.shape[1]
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "sample": f"{entries} sampled Fprop outputs (K = {A.shape[1]}) of the oracle-quantized rows 0..{A.shape[0] - 1} "
                      f"of X and 0..{B.shape[0] - 1} of W, {n} repetitions, {dt:.2f} s each"}


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
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
                             "sample": sample},
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
