#!/usr/bin/env python3
"""Benchmark of libfusedconv on the three full-size workloads.

One step = one pass of the whole fused path over the three full-size
workloads, back to back on one stream:
  * conv2d 3x3 (x [128,8,128,128]) + bias -> ReLU -> HardSwish,
  * conv3d 3x3x3 (x [128,8,16,64,64]) + bias -> LeakyReLU(0.2) -> + s[64]
    -> clamp[-1,1] -> exact GELU,
  * transposed conv 3x3 s1 p1 (x [128,64,256,256]) + bias -> maxpool 2x2 ->
    hardtanh[-1,1] -> mean(H,W) -> tanh.
Metric: effective GFLOP/s = 2 * MACs / device time, MACs counted from the
shapes (no epilogue ops counted).  Inputs are seeded synthetic tensors with
the workloads' distributions, resident in HBM before the timed region; L2 is
flushed (a 256 MiB write) before every workload call, outside its events.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded sample of the same workloads.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from convolution_epilogue_gb300 import synth  # noqa: E402

METRIC = "effective GFLOP/s (2*MACs/device time) and % of roofline per config, 1 GB300"
UNIT = "GFLOP/s"
WORKLOADS = (3, 4, 5)
CHAIN_RH = (("relu",), ("hardswish",))
SMS = 152


def macs_of(wid: int) -> int:
    """MAC count of a workload from its shapes (stride 1)."""
    if wid in (1, 3):
        N, C, H, W = synth.WORKLOADS[wid]["x"]
        return N * 64 * (H - 2) * (W - 2) * C * 9
    if wid == 4:
        N, C, D, H, W = synth.WORKLOADS[wid]["x"]
        return N * 64 * (D - 2) * (H - 2) * (W - 2) * C * 27
    N, C, H, W = synth.WORKLOADS[wid]["x"]
    return N * 64 * H * W * C * 9


def algorithmic_bytes(wid: int) -> int:
    """x + W + b (+ s) + y, each counted once, fp32."""
    spec = synth.WORKLOADS[wid]
    xs = spec["x"]
    nx = int(np.prod(xs))
    if wid in (1, 3):
        N, C, H, W = xs
        nw, ny = 64 * C * 9, N * 64 * (H - 2) * (W - 2)
        extra = 64
    elif wid == 4:
        N, C, D, H, W = xs
        nw, ny = 64 * C * 27, N * 64 * (D - 2) * (H - 2) * (W - 2)
        extra = 128
    else:
        N, C, H, W = xs
        nw, ny = C * 64 * 9, N * 64
        extra = 64
    return 4 * (nx + nw + extra + ny)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of each
# workload's main kernel from one ncu capture, scaled to one full launch.
# An entry is used only while the kernel sources hash to `src`; after any
# change to them the roofline's traffic is reported as null until the kernel
# is captured again.
NCU_TRAFFIC = {
    # batch-32 capture (542.5088 MB read + write, CTA-pair kernel) x 4 for
    # the 128-image launch
    (5, "tc_f16x3"): {"src": "b12c46aaf68ff92f", "bytes": 2170035200},
    # full-size capture; the tail of y is still in L2 when the launch ends
    (3, "tc_f16x3"): {"src": "b12c46aaf68ff92f", "bytes": 527528960},
}

KERNEL_SOURCES = ("fc_tc.cu", "fc_tc_ptx.cuh", "fc_epi.cuh", "fc_internal.h")


def kernel_src_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "convolution_epilogue_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(wid: int, variant: str):
    e = NCU_TRAFFIC.get((wid, variant))
    if e is None or e["src"] != kernel_src_digest():
        return None
    return e["bytes"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0,
                source="fallback")


def pipe_peak_tflops(variant: str, peaks, basis: str = "burst") -> tuple[float, str, str]:
    """Peak of the pipe a variant uses, in useful fp32-accurate TFLOP/s.

    tc_f16x3: fp16 tensor rate (= the measured bf16 rate) / 3 products.
    tc_tf32x3: tf32 rate (measured bf16 x nominal 1.1/2.25) / 3 products.
    ffma: 152 SMs x 128 FMA/clk x 2 FLOP x max SM clock.
    `basis` "burst" takes the bf16 GEMM measured alone (the kernels here are
    timed one call at a time, between L2 flushes); "sustained" the rate of
    a seconds-long GEMM loop under the power cap."""
    bf16 = peaks["bf16"] if basis == "burst" else peaks["bf16_sus"]
    if variant == "tc_f16x3":
        return bf16 / 3.0, "tensor", f"fp16 tensor (measured bf16 {basis}) / 3"
    if variant == "tc_tf32x3":
        return (bf16 * 1.1 / 2.25 / 3.0, "tensor",
                f"tf32 tensor (measured bf16 {basis} x 1.1/2.25) / 3")
    return (SMS * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12, "alu",
            "fp32 FFMA: 152 SMs x 128 lanes x 2 x max SM clock")


# nominal HBM3e bandwidth of a GB300 (~8 TB/s), reported beside the
# measured copy bandwidth
NOMINAL_HBM_GBS = 8000.0


def roofline_ms(flops, nbytes, variant, peaks, basis="burst", hbm_gbs=None):
    """Roofline time = the slower of FLOPs at the used pipe's peak and bytes
    at HBM bandwidth (ms), and which of the two binds."""
    pk, kind, _ = pipe_peak_tflops(variant, peaks, basis)
    t_f = flops / (pk * 1e12)
    t_b = nbytes / ((hbm_gbs or peaks["hbm_gbs"]) * 1e9)
    return (max(t_f, t_b) * 1e3, "hbm" if t_b > t_f else kind)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the
    timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU side
def cpu_sample(scale: int):
    """A bounded sample of the three workloads for the CPU oracle:
    `scale` images of the conv2d and conv3d workloads (full planes) and
    16*scale (n, c_out) outputs of the pooled workload.  Returns a callable
    that runs it and the MACs it covers."""
    import oracle
    scale = max(1, min(int(scale), 128))
    inp3 = synth.make_inputs(3, first_images=scale)
    inp4 = synth.make_inputs(4, first_images=scale)
    inp5 = synth.make_inputs(5, first_images=math.ceil(16 * scale / 64))
    x5, w5, b5 = inp5["x"], inp5["w"], inp5["b"]
    s4 = inp4["s"].reshape(-1)
    x3 = inp3["x"]
    x4 = inp4["x"]
    pairs = [(i // 64, i % 64) for i in range(16 * scale)]
    chain4 = (("leaky_relu", 0.2), ("add_channel", s4), ("clamp", -1.0, 1.0), ("gelu_erf",))

    def run():
        oracle.conv_epi(x3, inp3["w"], inp3["b"], CHAIN_RH)
        oracle.conv_epi(x4, inp4["w"], inp4["b"], chain4)
        oracle.convT_pool_mean_points(x5, w5, b5, pairs)

    macs = (macs_of(3) // 128 * scale + macs_of(4) // 128 * scale
            + 256 * 256 * 64 * 9 * len(pairs))
    desc = (f"{scale} image(s) of the conv2d and conv3d workloads (all outputs) + "
            f"{len(pairs)} (n, c_out) outputs of the pooled transposed-conv workload")
    return run, macs, desc


def cpu_baseline(scale: int):
    import oracle
    oracle.build()
    run, macs, desc = cpu_sample(scale)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": 2.0 * macs / dt / 1e9, "unit": UNIT,
            "cores": int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)),
            "kind": "oracle", "sample": desc, "seconds": round(dt, 3)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    run, macs, desc = cpu_sample(args.ref_scale)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2.0 * macs * args.steps / total / 1e9
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "CPU oracle (plain C, fp64) on a bounded sample of the "
                                   "three full-size workloads", "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def aggregate_replicas(my_ms, world, steps, flops_step, max_over_ranks=None):
    """Whole-job throughput of `world` independent replicas (weak scaling):
    every rank runs the same `steps` steps of `flops_step` FLOPs; the job
    takes as long as its slowest rank, so the time is the max over ranks of
    each rank's summed step time (ms) and the value counts every rank's work.
    Returns (job ms, GFLOP/s)."""
    tot_ms = max_over_ranks(my_ms) if (world > 1 and max_over_ranks is not None) else my_ms
    return tot_ms, world * flops_step * steps / (tot_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ GPU side
def run_ours(args):
    import torch
    import convolution_epilogue_gb300 as fc
    from convolution_epilogue_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device() if world == 1 else local)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    fc.lib()
    fc.set_variant(args.variant)
    fc.set_staging(args.staging)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)

    # inputs resident in HBM, outputs and workspaces preallocated
    host = {w: synth.make_inputs(w) for w in WORKLOADS}
    d = {}
    for w in WORKLOADS:
        d[w] = {k: torch.from_numpy(v).to(dev) for k, v in host[w].items()}
    y3 = torch.empty((128, 64, 126, 126), device=dev)
    y4 = torch.empty((128, 64, 14, 62, 62), device=dev)
    y5 = torch.empty((128, 64, 1, 1), device=dev)
    ws = {3: torch.empty(fc.workspace_bytes(0, (128, 8, 128, 128, 64, 3, 0)), dtype=torch.uint8, device=dev),
          4: torch.empty(fc.workspace_bytes(1, (128, 8, 16, 64, 64, 64, 3, 0)), dtype=torch.uint8, device=dev),
          5: torch.empty(fc.workspace_bytes(2, (128, 64, 256, 256, 64, 3, 1)), dtype=torch.uint8, device=dev)}
    s4 = d[4]["s"].reshape(-1)
    chain4 = (("leaky_relu", 0.2), ("add_channel", s4), ("clamp", -1.0, 1.0), ("gelu_erf",))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    calls = {
        3: lambda: fc.fc_conv2d_epi(d[3]["x"], d[3]["w"], d[3]["b"], CHAIN_RH, y=y3, ws=ws[3]),
        4: lambda: fc.fc_conv3d_epi(d[4]["x"], d[4]["w"], d[4]["b"], chain4, y=y4, ws=ws[4]),
        5: lambda: fc.fc_convT2d_pool_mean(d[5]["x"], d[5]["w"], d[5]["b"], y=y5, ws=ws[5]),
    }
    variants, launches_per_step = {}, 0
    for w in WORKLOADS:
        calls[w]()
        variants[w] = fc.last_variant()
        launches_per_step += fc.last_launch_count()
    torch.cuda.synchronize()
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set during warm-up")

    for _ in range(args.warmup):
        for w in WORKLOADS:
            flush.zero_()
            calls[w]()
    ev = {w: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for w in WORKLOADS}
    fc.profile_reset()
    fc.profile_enable(True)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    n_launch = 0
    for k in range(args.steps):
        for w in WORKLOADS:
            flush.zero_()
            ev[w][k][0].record(stream)
            calls[w]()
            ev[w][k][1].record(stream)
            n_launch += fc.last_launch_count()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    fc.profile_enable(False)
    status = fc.get_last_device_error()

    per = {}
    step_ms = [0.0] * args.steps
    for w in WORKLOADS:
        ts = [ev[w][k][0].elapsed_time(ev[w][k][1]) for k in range(args.steps)]
        for k in range(args.steps):
            step_ms[k] += ts[k]
        per[w] = ts
    my_ms = sum(step_ms)

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    flops_step = sum(2 * macs_of(w) for w in WORKLOADS)
    tot_ms, value = aggregate_replicas(my_ms, world, args.steps, flops_step,
                                       max_over_ranks if world > 1 else None)

    # dominant kernel: the main kernel with the largest summed time
    entry_of = {3: 0, 4: 1, 5: 2}
    kern = {}
    for w in WORKLOADS:
        ms, cnt = fc.profile_read(entry_of[w])
        kern[w] = (ms / max(cnt, 1), cnt)
    dom = max(WORKLOADS, key=lambda w: kern[w][0] * kern[w][1])
    avg_ms = kern[dom][0]
    pk_t, bound_kind, pk_desc = pipe_peak_tflops(variants[dom], peaks, "burst")
    t_flop = 2 * macs_of(dom) / (pk_t * 1e12)
    t_byte = algorithmic_bytes(dom) / (peaks["hbm_gbs"] * 1e9)
    if t_byte > t_flop:
        achieved = algorithmic_bytes(dom) / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = 2 * macs_of(dom) / (avg_ms * 1e-3) / 1e12
        roof = {"bound": bound_kind, "achieved": achieved, "peak": pk_t, "unit": "TFLOP/s",
                "frac": achieved / pk_t}
    # the same kernel against the other peak bases: the sustained GEMM rate,
    # and the 8 TB/s HBM figure with the burst tensor rate
    r_sus, _ = roofline_ms(2 * macs_of(dom), algorithmic_bytes(dom), variants[dom], peaks,
                           "sustained")
    r_8tb, _ = roofline_ms(2 * macs_of(dom), algorithmic_bytes(dom), variants[dom], peaks,
                           "burst", NOMINAL_HBM_GBS)
    roof.update({"traffic": ncu_traffic(dom, variants[dom]), "kernel": f"{synth.WORKLOADS[dom]['name']} main kernel "
                 f"[{variants[dom]}]", "avg_ms": avg_ms, "peak_basis": pk_desc + " (of measured)",
                 "peak_source": peaks["source"],
                 "frac_sustained_peak": r_sus / avg_ms, "frac_8tbs_burst": r_8tb / avg_ms})

    per_cfg = {}
    for w in WORKLOADS:
        med = statistics.median(per[w])
        f, nb = 2 * macs_of(w), algorithmic_bytes(w)
        t_roof, bnd = roofline_ms(f, nb, variants[w], peaks, "burst")
        t_sus, _ = roofline_ms(f, nb, variants[w], peaks, "sustained")
        t_8tb, _ = roofline_ms(f, nb, variants[w], peaks, "burst", NOMINAL_HBM_GBS)
        per_cfg[synth.WORKLOADS[w]["name"]] = {
            "variant": variants[w], "ms_median": med,
            "ms_p10": float(np.percentile(per[w], 10)), "ms_p90": float(np.percentile(per[w], 90)),
            "gflops": f / (med * 1e-3) / 1e9,
            "roofline_ms": t_roof, "roofline_bound": bnd, "roofline_frac": t_roof / med,
            "kernel_ms": kern[w][0], "roofline_frac_kernel": t_roof / kern[w][0],
            "roofline_frac_sustained_peak": t_sus / med, "roofline_frac_8tbs_burst": t_8tb / med}

    # the same calls back to back without the L2 flush (inputs may sit in
    # L2 between calls); reported beside the flushed series, not used for
    # the roofline fraction
    for w in WORKLOADS:
        evw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(20)]
        for e0, e1 in evw:
            e0.record(stream)
            calls[w]()
            e1.record(stream)
        torch.cuda.synchronize()
        per_cfg[synth.WORKLOADS[w]["name"]]["ms_median_no_flush"] = statistics.median(
            e0.elapsed_time(e1) for e0, e1 in evw)

    # fusion ablation for the pooled workload: the transposed conv as a
    # materialised conv (swapped, flipped weights, padding 1; 2.15 GB
    # written and read back) followed by the standalone tail kernel
    ablation = None
    if not args.no_ablation:
        ablation = fusion_ablation(fc, d[5], flush, stream, per[5])

    # widened layer parameters beyond the headline workloads, on the conv2d
    # workload's input: stride 2, and dilation 2 with "same" padding
    widened = None
    if not args.no_ablation:
        widened = {
            "conv2d_stride2_relu_hardswish_128x8x128x128": widened_conv(
                fc, d[3], flush, stream, peaks, stride=2, pad=0, dilation=1),
            "conv2d_dilation2_pad2_relu_hardswish_128x8x128x128": widened_conv(
                fc, d[3], flush, stream, peaks, stride=1, pad=2, dilation=2),
            "convT2d_stride2_outpad1_pool_mean_128x64x128x128": widened_convT_s2(
                fc, d[5], flush, stream, peaks),
            "convT2d_maxpool3s2_mean_16x64x256x256": widened_general_pool(
                fc, d[5], flush, stream, peaks),
        }

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, fc, host, dev, stream, chain4_host=host[4]["s"].reshape(-1))

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": " + ".join(synth.WORKLOADS[w]["name"] for w in WORKLOADS),
                       "l2": "flushed by a 256 MiB write before every workload call (outside events)",
                       "variants": {synth.WORKLOADS[w]["name"]: variants[w] for w in WORKLOADS},
                       "staging": args.staging,
                       "per_workload": per_cfg,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof, "clocks": clocks, "gpu_launches": n_launch,
            "device_status": status, "wall_s_timed": t_wall}
    if e2e is not None:
        line["e2e"] = e2e
    if ablation is not None:
        line["fusion_ablation"] = ablation
    if widened is not None:
        line["widened"] = widened
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.cpu_scale)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def fusion_ablation(fc, d5, flush, stream, fused_ms_list, reps=10):
    """Unfused pipeline for the pooled workload, same L2 flushing as the
    fused timing: conv (y_conv materialised) then fc_pool_mean_tail."""
    import torch
    x, w, b = d5["x"], d5["w"], d5["b"]
    w_conv = torch.flip(w.permute(1, 0, 2, 3), dims=(2, 3)).contiguous()
    N, C, H, W = x.shape
    y_conv = torch.empty((N, w.shape[1], H, W), dtype=torch.float32, device=x.device)
    y = torch.empty((N, w.shape[1], 1, 1), dtype=torch.float32, device=x.device)
    ws = torch.empty(fc.workspace_bytes(0, (N, C, H, W, w.shape[1], 3, 1)), dtype=torch.uint8,
                     device=x.device)
    conv = lambda: fc.fc_conv2d_epi(x, w_conv, b, (), pad=1, y=y_conv, ws=ws)
    tail = lambda: fc.fc_pool_mean_tail(y_conv, y=y)
    conv()
    conv_variant = fc.last_variant()
    tail()
    torch.cuda.synchronize()
    t_conv, t_tail = [], []
    for _ in range(reps):
        for fn, out in ((conv, t_conv), (tail, t_tail)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1))
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set in the ablation")
    mc, mt = statistics.median(t_conv), statistics.median(t_tail)
    fused = statistics.median(fused_ms_list)
    tail_bytes = y_conv.numel() * 4
    del y_conv
    return {"workload": "convT2d_pool_mean_128x64x256x256",
            "unfused_conv_ms": mc, "unfused_tail_ms": mt, "unfused_total_ms": mc + mt,
            "fused_ms": fused, "fused_speedup": (mc + mt) / fused,
            "tail_gbs": tail_bytes / (mt * 1e-3) / 1e9, "conv_variant": conv_variant}


def widened_conv(fc, d3, flush, stream, peaks, stride, pad, dilation, reps=20):
    """conv2d + ReLU + HardSwish on x [128,8,128,128] at the given stride,
    padding and dilation (stride 2: y [128,64,63,63]; dilation 2, pad 2:
    y [128,64,128,128]), L2 flushed before each call; roofline = max(FLOPs at
    the used pipe's peak, bytes at HBM bandwidth)."""
    import torch
    x, w, b = d3["x"], d3["w"], d3["b"]
    N, C, H, W = x.shape
    span = 2 * dilation + 1
    Ho, Wo = (H + 2 * pad - span) // stride + 1, (W + 2 * pad - span) // stride + 1
    y = torch.empty((N, w.shape[0], Ho, Wo), dtype=torch.float32, device=x.device)
    call = lambda: fc.fc_conv2d_epi(x, w, b, CHAIN_RH, y=y, stride=stride, pad=pad,
                                    dilation=dilation)
    call()
    variant = fc.last_variant()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set in the widened conv")
    ms = statistics.median(ts)
    flops = 2.0 * N * w.shape[0] * Ho * Wo * C * 9
    nbytes = 4.0 * (x.numel() + w.numel() + b.numel() + y.numel())
    pk, _, basis = pipe_peak_tflops(variant, peaks, "burst")
    t_roof = max(flops / (pk * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    return {"variant": variant, "ms_median": ms, "gflops": flops / (ms * 1e-3) / 1e9,
            "roofline_ms": t_roof * 1e3, "roofline_frac": t_roof * 1e3 / ms, "peak_basis": basis}


def widened_convT_s2(fc, d5, flush, stream, peaks, reps=20):
    """Stride-2 transposed conv (k 3, pad 1, output padding 1) on x
    [128,64,128,128] (every other row and column of the pooled workload's
    input) -> 256 x 256 -> 2x2 max pool -> hardtanh -> mean -> tanh.  Useful
    FLOPs = 2 x N x C_in x C_out x H x W x 9 (each input pixel meets each of
    the 9 taps once); roofline = max(FLOPs at the used pipe's peak, bytes at
    HBM bandwidth)."""
    import torch
    x = d5["x"][:, :, ::2, ::2].contiguous()
    w, b = d5["w"], d5["b"]
    N, C, H, W = x.shape
    CO = w.shape[1]
    y = torch.empty((N, CO, 1, 1), dtype=torch.float32, device=x.device)
    call = lambda: fc.fc_convT2d_pool_mean(x, w, b, y=y, stride=2, out_pad=1)
    call()
    variant = fc.last_variant()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set in the stride-2 transposed conv")
    ms = statistics.median(ts)
    flops = 2.0 * N * C * CO * H * W * 9
    nbytes = 4.0 * (x.numel() + w.numel() + b.numel() + y.numel())
    pk, _, basis = pipe_peak_tflops(variant, peaks, "burst")
    t_roof = max(flops / (pk * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    del x
    return {"variant": variant, "ms_median": ms, "gflops": flops / (ms * 1e-3) / 1e9,
            "roofline_ms": t_roof * 1e3, "roofline_frac": t_roof * 1e3 / ms, "peak_basis": basis}


def widened_general_pool(fc, d5, flush, stream, peaks, reps=10):
    """Transposed conv (stride 1) on 16 images of the pooled workload's input
    [16,64,256,256] -> 3x3 max pool, stride 2 (overlapping, floor extent
    127 x 127) -> hardtanh -> mean -> tanh, fused in the variant the library
    picks (the tensor cores' general-pool units).
    Useful FLOPs = 2 x conv MACs (each conv output counted once; the kernel
    recomputes the outputs shared by overlapping windows, 2.25x here)."""
    import torch
    x = d5["x"][:16]
    w, b = d5["w"], d5["b"]
    N, C, H, W = x.shape
    CO = w.shape[1]
    y = torch.empty((N, CO, 1, 1), dtype=torch.float32, device=x.device)
    call = lambda: fc.fc_convT2d_pool_mean(x, w, b, y=y, pool=(3, 2))
    call()
    variant = fc.last_variant()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set in the general-pool entry")
    ms = statistics.median(ts)
    flops = 2.0 * N * C * CO * H * W * 9
    nbytes = 4.0 * (x.numel() + w.numel() + b.numel() + y.numel())
    pk, _, basis = pipe_peak_tflops(variant, peaks, "burst")
    t_roof = max(flops / (pk * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))
    return {"variant": variant, "ms_median": ms, "gflops": flops / (ms * 1e-3) / 1e9,
            "roofline_ms": t_roof * 1e3, "roofline_frac": t_roof * 1e3 / ms, "peak_basis": basis}


def measure_e2e(args, fc, host, dev, stream, chain4_host, chunk=16):
    """Same metric with host buffers: pinned-host -> device copies of every
    input, the three calls, device -> pinned-host copies of every output, all
    inside the timed region.  Each workload's batch goes through in chunks of
    `chunk` images on three streams (copy in, compute, copy out), so the
    input copy of one chunk, the calls on the previous one and the output
    copy of the one before overlap, as a caller streaming batches would run
    the public API."""
    import torch
    pin = {w: {k: torch.from_numpy(v).pin_memory() for k, v in host[w].items()} for w in WORKLOADS}
    dd = {w: {k: torch.empty(v.shape, dtype=torch.float32, device=dev) for k, v in host[w].items()}
          for w in WORKLOADS}
    outs = {3: torch.empty((128, 64, 126, 126), device=dev),
            4: torch.empty((128, 64, 14, 62, 62), device=dev),
            5: torch.empty((128, 64, 1, 1), device=dev)}
    outs_h = {w: torch.empty(o.shape, dtype=torch.float32).pin_memory() for w, o in outs.items()}
    ws = {3: torch.empty(fc.workspace_bytes(0, (chunk, 8, 128, 128, 64, 3, 0)), dtype=torch.uint8, device=dev),
          4: torch.empty(fc.workspace_bytes(1, (chunk, 8, 16, 64, 64, 64, 3, 0)), dtype=torch.uint8, device=dev),
          5: torch.empty(fc.workspace_bytes(2, (chunk, 64, 256, 256, 64, 3, 1)), dtype=torch.uint8, device=dev)}
    h2d = sum(t.numel() * 4 for w in WORKLOADS for t in pin[w].values())
    d2h = sum(o.numel() * 4 for o in outs.values())
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nchunks = 128 // chunk

    def step():
        for w in WORKLOADS:
            with torch.cuda.stream(s_in):  # weights, bias, addend: once per step
                for k in pin[w]:
                    if k != "x":
                        dd[w][k].copy_(pin[w][k], non_blocking=True)
            for c in range(nchunks):
                sl = slice(c * chunk, (c + 1) * chunk)
                with torch.cuda.stream(s_in):
                    dd[w]["x"][sl].copy_(pin[w]["x"][sl], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                s_cmp.wait_event(ev_in)
                x, wt, b = dd[w]["x"][sl], dd[w]["w"], dd[w]["b"]
                if w == 3:
                    fc.fc_conv2d_epi(x, wt, b, CHAIN_RH, y=outs[3][sl], ws=ws[3], stream=s_cmp)
                elif w == 4:
                    ch4 = (("leaky_relu", 0.2), ("add_channel", dd[4]["s"].reshape(-1)),
                           ("clamp", -1.0, 1.0), ("gelu_erf",))
                    fc.fc_conv3d_epi(x, wt, b, ch4, y=outs[4][sl], ws=ws[4], stream=s_cmp)
                else:
                    fc.fc_convT2d_pool_mean(x, wt, b, y=outs[5][sl], ws=ws[5], stream=s_cmp)
                ev_c = torch.cuda.Event()
                ev_c.record(s_cmp)
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    outs_h[w][sl].copy_(outs[w][sl], non_blocking=True)

    def join():
        for s_ in (s_in, s_cmp, s_out):
            ev = torch.cuda.Event()
            ev.record(s_)
            stream.wait_event(ev)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    join()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in (s_in, s_cmp, s_out):
        s_.wait_event(e0)
    for _ in range(steps):
        step()
    join()
    e1.record(stream)
    torch.cuda.synchronize()
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set in the end-to-end run")
    ms = e0.elapsed_time(e1) / steps
    flops = sum(2 * macs_of(w) for w in WORKLOADS)
    return {"value": flops / (ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipeline": f"chunks of {chunk} images on copy-in / compute / copy-out streams"}


# ------------------------------------------------------- variant table
# (entry, dims) per shape: entry 0 conv2d / 1 conv3d with
# (N, C, [D,] H, W, CO, k, stride, pad, dilation, channels_last), entry 2
# the pooled transposed conv with (N, C, H, W, CO, k, stride, pad, out_pad,
# pool window, pool stride).  The five workloads, smaller and larger
# neighbours, other channel counts, and the widened forms.
TABLE_SHAPES = (
    [(0, (n, c, h, w, co, 3, 1, 0, 1, 0)) for (n, c, h, w, co) in [
        (4, 8, 32, 32, 64), (2, 3, 9, 37, 10), (16, 8, 64, 64, 64), (32, 8, 128, 128, 64),
        (128, 8, 128, 128, 64), (1, 64, 32, 32, 64), (8, 64, 64, 64, 64), (2, 16, 128, 128, 128),
        (1, 256, 16, 16, 256), (64, 32, 64, 64, 64)]]
    + [(0, (n, c, h, w, co, 3, 2, 0, 1, 0)) for (n, c, h, w, co) in [
        (4, 8, 32, 32, 64), (128, 8, 128, 128, 64), (8, 64, 64, 64, 64)]]
    + [(0, (n, c, h, w, co, 3, 1, 2, 2, 0)) for (n, c, h, w, co) in [
        (4, 8, 32, 32, 64), (128, 8, 128, 128, 64)]]
    + [(0, (n, c, h, w, co, 3, 1, 1, 1, 1)) for (n, c, h, w, co) in [
        (4, 8, 32, 32, 64), (128, 8, 128, 128, 64), (8, 64, 64, 64, 64)]]
    + [(1, (n, c, d, h, w, co, 3, 1, 0, 1, 0)) for (n, c, d, h, w, co) in [
        (1, 8, 5, 10, 12, 64), (8, 8, 16, 64, 64, 64), (128, 8, 16, 64, 64, 64),
        (2, 16, 8, 32, 32, 32), (4, 64, 8, 16, 16, 64)]]
    + [(1, (8, 8, 16, 64, 64, 64, 3, 2, 1, 1, 0)), (1, (8, 8, 16, 64, 64, 64, 3, 1, 1, 1, 1))]
    + [(2, (n, c, h, w, co, 3, 1, 1, 0, 2, 2)) for (n, c, h, w, co) in [
        (2, 64, 32, 32, 64), (16, 64, 64, 64, 64), (128, 64, 256, 256, 64), (2, 5, 7, 10, 3),
        (4, 16, 64, 64, 64)]]
    + [(2, (2, 64, 16, 20, 64, 3, 2, 1, 1, 2, 2)), (2, (128, 64, 128, 128, 64, 3, 2, 1, 1, 2, 2))]
    + [(2, (16, 64, 256, 256, 64, 3, 1, 1, 0, 3, 2)), (2, (2, 16, 17, 21, 64, 3, 1, 1, 0, 3, 2))]
)
# candidates in the table's column order
TABLE_COLS = (("ffma", "loads"), ("tc_tf32x3", "loads"), ("tc_tf32x3", "tma"),
              ("tc_f16x3", "loads"), ("tc_f16x3", "tma"))


def _table_case(fc, dev, entry, dims):
    """Device tensors and a call for one table shape; MACs as the library
    counts them for its selection."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(1234)
    rnd = lambda *sh: torch.randn(*sh, generator=g).to(dev)
    if entry in (0, 1):
        if entry == 0:
            N, C, H, W, CO, k, st, pad, dil, cl = dims
            D = 1
        else:
            N, C, D, H, W, CO, k, st, pad, dil, cl = dims
        ext = lambda n: (n + 2 * pad - dil * (k - 1) - 1) // st + 1
        Do = ext(D) if entry == 1 else 1
        Ho, Wo = ext(H), ext(W)
        xs = (N, C, H, W) if entry == 0 else (N, C, D, H, W)
        if cl:
            xs = (xs[0],) + xs[2:] + (C,)
        x = rnd(*xs)
        w = rnd(*((CO, C) + (k,) * (2 if entry == 0 else 3))) * 0.1
        b = rnd(CO) * 0.1
        ops = (("relu",), ("hardswish",)) if entry == 0 else (
            ("leaky_relu", 0.2), ("add_channel", rnd(CO)), ("clamp", -1.0, 1.0), ("gelu_erf",))
        f = {(0, 0): fc.fc_conv2d_epi, (0, 1): fc.fc_conv2d_epi_nhwc,
             (1, 0): fc.fc_conv3d_epi, (1, 1): fc.fc_conv3d_epi_ndhwc}[(entry, cl)]
        call = lambda: f(x, w, b, ops, pad=pad, stride=st, dilation=dil)
        macs = N * CO * Do * Ho * Wo * C * (k ** (2 if entry == 0 else 3))
        key = dict(entry=entry, k=k, stride=st, dil=dil, cl=cl, pool_general=0, C=C, CO=CO)
    else:
        N, C, H, W, CO, k, st, pad, op, pk, ps = dims
        x = rnd(N, C, H, W)
        w = rnd(C, CO, k, k) * 0.05
        b = rnd(CO) * 0.1
        call = lambda: fc.fc_convT2d_pool_mean(x, w, b, stride=st, pad=pad, out_pad=op,
                                               pool=(pk, ps))
        if st == 2 and k == 3 and pad == 1 and (pk, ps) == (2, 2):  # per parity class
            macs = N * C * CO * H * W * k * k
        else:
            Ho, Wo = (H - 1) * st - 2 * pad + k + op, (W - 1) * st - 2 * pad + k + op
            macs = N * CO * Ho * Wo * C * k * k
        key = dict(entry=2, k=k, stride=st, dil=1, cl=0, pool_general=int((pk, ps) != (2, 2)),
                   C=C, CO=CO)
    key["macs"] = float(macs)
    return call, key


def run_variant_table(args):
    """Times every (variant, input staging) pair on TABLE_SHAPES (median
    main-kernel time from the library's own event pairs, L2 flushed before
    each call) and writes the table the automatic choice compiles in."""
    import torch
    import convolution_epilogue_gb300 as fc
    from convolution_epilogue_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    entry_prof = {0: 0, 1: 1, 2: 2}
    rows = []
    for entry, dims in TABLE_SHAPES:
        call, key = _table_case(fc, dev, entry, dims)
        ms = []
        for variant, staging in TABLE_COLS:
            fc.set_variant(variant)
            fc.set_staging(staging)
            try:
                call()
                torch.cuda.synchronize()
            except fc.FcError:
                ms.append(-1.0)
                continue
            if variant != "ffma" and fc.last_staging() != staging:
                ms.append(-1.0)  # this plan cannot stage that way
                continue
            times = []
            for _ in range(args.table_reps):
                flush.zero_()
                fc.profile_reset()
                fc.profile_enable(True)
                call()
                fc.profile_enable(False)
                t, n = fc.profile_read(entry_prof[entry])
                times.append(t / max(n, 1))
            if fc.get_last_device_error() != 0:
                raise RuntimeError(f"device status word set at {dims} [{variant}/{staging}]")
            ms.append(float(statistics.median(times)))
        fc.set_variant("auto")
        fc.set_staging("auto")
        rows.append(dict(key, dims=list(dims), ms=ms))
        print(json.dumps(rows[-1]), flush=True)
    out = {"columns": [f"{v}/{s}" for v, s in TABLE_COLS], "rows": rows,
           "gpu": torch.cuda.get_device_name(0)}
    with open(args.variant_table, "w") as f:
        json.dump(out, f, indent=1)
    with open(os.path.splitext(args.variant_table)[0] + ".h", "w") as f:
        f.write(variant_table_header(out))
    return 0


def variant_table_header(tab) -> str:
    """The C table for fc_variant_table.h from a measured table."""
    lines = []
    for r in tab["rows"]:
        ms = ", ".join(f"{m:.5f}f" if m >= 0 else "-1.f" for m in r["ms"])
        lines.append(f"    {{{r['entry']}, {r['k']}, {r['stride']}, {r['dil']}, {r['cl']}, "
                     f"{r['pool_general']}, {r['macs']:.1f}, {r['C']}, {r['CO']}, {{{ms}}}}},"
                     f"  // {r['dims']}")
    return "\n".join(lines) + "\n"


def install_variant_table(src_json: str, csrc: str | None = None) -> int:
    """Copy a table measured by --variant-table into the library's sources:
    the JSON beside the header, and the header's rows and GPU name.  The
    rest of fc_variant_table.h (row type, lookup) is kept.  Returns the
    number of rows."""
    import re
    csrc = csrc or os.path.join(ROOT, "convolution_epilogue_gb300", "csrc")
    with open(src_json) as f:
        tab = json.load(f)
    with open(os.path.join(csrc, "fc_variant_table.json"), "w") as f:
        json.dump(tab, f, indent=1)
    hp = os.path.join(csrc, "fc_variant_table.h")
    with open(hp) as f:
        h = f.read()
    head = "static const VariantRow kVariantTable[] = {\n"
    a = h.index(head) + len(head)
    b = h.index("};\nstatic const char kVariantTableSource[]")
    h = h[:a] + variant_table_header(tab) + h[b:]
    h = re.sub(r"// Measured on .* \(fc_variant_table.json",
               lambda m: f"// Measured on {tab['gpu']} (fc_variant_table.json", h)
    with open(hp, "w") as f:
        f.write(h)
    return len(tab["rows"])


def parse_pool(text: str) -> tuple[int, int]:
    """`K,S` of --profile-pool: max-pool window and stride, each 1..4."""
    try:
        pool = tuple(int(v) for v in text.split(","))
    except ValueError:
        pool = ()
    if len(pool) != 2 or not all(1 <= v <= 4 for v in pool):
        raise ValueError(f"--profile-pool takes K,S with 1 <= K, S <= 4, not {text!r}")
    return pool


def run_profile_case(args):
    """Run one workload (optionally at a smaller batch) `--profile-reps`
    times through the public API and exit: the command profilers wrap."""
    import torch
    import convolution_epilogue_gb300 as fc
    from convolution_epilogue_gb300 import _build
    _build.build()
    wid = args.profile_workload
    spec = synth.WORKLOADS[wid]
    nb = args.profile_batch or spec["x"][0]
    inp = synth.make_inputs(wid, first_images=nb)
    d = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    pool = parse_pool(args.profile_pool)
    fc.set_variant(args.variant)
    fc.set_staging(args.staging)
    for _ in range(args.profile_reps):
        if spec["kind"] == "conv2d":
            y = fc.fc_conv2d_epi(d["x"], d["w"], d["b"], CHAIN_RH)
        elif spec["kind"] == "conv3d":
            ops = (("leaky_relu", 0.2), ("add_channel", d["s"].reshape(-1)), ("clamp", -1.0, 1.0),
                   ("gelu_erf",))
            y = fc.fc_conv3d_epi(d["x"], d["w"], d["b"], ops)
        else:
            y = fc.fc_convT2d_pool_mean(d["x"], d["w"], d["b"], pool=pool)
    torch.cuda.synchronize()
    if fc.get_last_device_error() != 0:
        raise RuntimeError("device status word set")
    print(f"profile case: workload {wid} batch {nb} variant {fc.last_variant()} "
          f"pool {pool} out {tuple(y.shape)}")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="auto", choices=["auto", "ffma", "tc_tf32x3", "tc_f16x3"])
    ap.add_argument("--staging", default="auto", choices=["auto", "tma", "loads"],
                    help="input staging of the tensor-core variants")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--cpu-scale", type=int, default=128)
    ap.add_argument("--ref-scale", type=int, default=2)
    ap.add_argument("--variant-table", default="",
                    help="time every variant / staging on the table's shapes; write JSON and .h here")
    ap.add_argument("--table-reps", type=int, default=7)
    ap.add_argument("--install-variant-table", default="",
                    help="copy a table measured by --variant-table into the library's sources")
    ap.add_argument("--profile-workload", type=int, default=0,
                    help="run only this workload (1..5) --profile-reps times, for profilers")
    ap.add_argument("--profile-batch", type=int, default=0)
    ap.add_argument("--profile-reps", type=int, default=2)
    ap.add_argument("--profile-pool", default="2,2",
                    help="max-pool window,stride of the pooled workload's profile case")
    args = ap.parse_args()
    parse_pool(args.profile_pool)  # refuse a bad window before any build or device work
    if args.install_variant_table:
        print(f"installed {install_variant_table(args.install_variant_table)} rows")
        return 0
    if args.profile_workload:
        return run_profile_case(args)
    if args.variant_table:
        return run_variant_table(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
