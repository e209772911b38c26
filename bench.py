#!/usr/bin/env python3
"""Benchmark of the chunked SSD forward scan on GB300.

One step = one ssd_chunked_forward call (the whole K1..K5 path) over one batch of the
Mamba-2-shape SISO workload (batch 4, T 4096, 32 heads, P 64, N 128, chunk 256, bf16 x/B/C,
B/C shared by all heads), inputs already resident in HBM.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the problems are
independent; there is no collective on the data path); the time is the max over ranks and the
value counts the tokens of all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "SSD forward tokens/s and % of roofline (HBM GB/s / tensor-pipe) at 1 GB300"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# Dense tf32 tensor-core throughput of this GPU, measured the way the bf16 figure of
# MEASURED_PEAKS.json is: torch.matmul of two 8192 x 8192 fp32 matrices with TF32 allowed, best
# of 10 timed with CUDA events, 2 N^3 FLOP (`python bench.py --measure-peak tf32`;
# profiles/peaks_tf32.md).  The roofline of an fp32-input workload takes its contraction FLOPs at
# this rate.
MEASURED_TF32_TFLOPS = 1043.5
FALLBACK_TF32_TFLOPS = 1100.0   # nominal dense tf32, used only while no measurement is recorded
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz (maximum SM clock).
ALU_FP32_TFLOPS = round(152 * 128 * 2 * 2.07e9 / 1e12, 1)

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant kernel, from one
# ncu capture of the same workload and the current kernel (profiles/dram_traffic.md); writes
# still held in L2 when the kernel ends are not counted.  Workloads without a capture report
# null.
NCU_TRAFFIC_BYTES = {
    "mamba2_siso_bf16": 77_669_632 + 27_295_744,           # ssd_fused_bf16_kernel<false>
    "mamba3_mimo_bf16": 1_441_407_232 + 253_506_816,       # ssd_fused_bf16_kernel<false>
    # tc32_scan_kernel, captured at T = 16384 and scaled by 8 (its traffic grows with T)
    "long_rotation_f32": (407_122_688 + 79_207_168) * 8,
    "selective_scan_f32": 77_815_552 + 8_036_864,          # ss_lookback_kernel
    # bwd_chunk_grad_kernel, captured at batch 1 and scaled by 4 (traffic grows with the batch)
    "mamba2_backward_bf16": (191_560_192 + 22_935_552) * 4,
}


def metric_name(cfg, is_ss):
    if is_ss:
        return "selective scan tokens/s at 1 GB300"
    if getattr(cfg, "backward", False):
        return "SSD backward tokens/s and % of roofline (fp32 CUDA-core FLOP/s) at 1 GB300"
    return METRIC


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mamba2_siso_bf16")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    # smaller cases of a workload's shape, for profiler captures (not bench lines)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch")
    ap.add_argument("--seqlen", type=int, default=0, help="override the workload's seqlen")
    ap.add_argument("--tf32", action="store_true",
                    help="fp32 workloads with P = N = 64: run ssd_chunked_forward_tf32 (the chunk "
                         "scan on the tensor core) instead of ssd_chunked_forward")
    ap.add_argument("--measure-peak", choices=["tf32"], default=None,
                    help="measure a tensor-core peak (torch.matmul) and print it instead")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def tf32_peak():
    if MEASURED_TF32_TFLOPS:
        return MEASURED_TF32_TFLOPS, "measured (torch.matmul 8192^3, TF32 allowed, best of 10)"
    return FALLBACK_TF32_TFLOPS, "nominal (no measurement recorded)"


def measure_matmul_peak(kind: str):
    """Dense tensor-core throughput as torch.matmul of two 8192 x 8192 matrices achieves it:
    best of 10 launches timed with CUDA events, 2 N^3 FLOP each (the method of the bf16 figure
    in MEASURED_PEAKS.json)."""
    n = 8192
    torch.backends.cuda.matmul.allow_tf32 = kind == "tf32"
    a = torch.randn(n, n, device="cuda", dtype=torch.float32)
    b = torch.randn(n, n, device="cuda", dtype=torch.float32)
    for _ in range(3):
        torch.matmul(a, b)
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return {"peak": kind, "tflops": round(2 * n ** 3 / (best * 1e-3) / 1e12, 1), "ms": round(best, 4),
            "how": "torch.matmul fp32 8192^3 with allow_tf32, best of 10, CUDA events",
            "gpu": torch.cuda.get_device_name(0)}


def workload(name, batch=0, seqlen=0):
    cfg = _named_workload(name)
    kw = {}
    if batch:
        kw["batch"] = batch
    if seqlen:
        kw["seqlen"] = seqlen
    return cfg.with_(**kw) if kw else cfg


def _named_workload(name):
    from chunked_ssd_scan_gb300 import workloads as wl
    for c in wl.SSD_CONFIGS:
        if c.name == name:
            return c
    if name == wl.SELECTIVE_SCAN_F32.name:
        return wl.SELECTIVE_SCAN_F32
    if name == wl.TRAP_MIMO_ROT_F32.name:
        return wl.TRAP_MIMO_ROT_F32
    if name == wl.ROT_VARIANT_F32.name:
        return wl.ROT_VARIANT_F32
    if name == wl.MAMBA2_BWD_BF16.name:
        return wl.MAMBA2_BWD_BF16
    if name == wl.LONG_ROT_BWD_F32.name:
        return wl.LONG_ROT_BWD_F32
    if name == wl.TRAP_BWD_F32.name:
        return wl.TRAP_BWD_F32
    raise SystemExit(f"unknown workload {name}")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def timed_steps(fn, steps, warmup, stream, flush):
    """Warm up, then time each step with CUDA events on `stream`, flushing L2 between steps."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.fill_(1)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        times.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in times]


def slowest_replica_ms(ms: float, world: int, device) -> float:
    """Mean step time of the slowest rank: every rank runs its own replica of the workload, and
    the job's step time is the max over ranks (one all-reduce, host-side bookkeeping only)."""
    if world > 1:
        t = torch.tensor([ms], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms


def job_tokens(tokens_per_replica: int, world: int) -> int:
    """Tokens the whole job processes per step (one replica per rank)."""
    return tokens_per_replica * world


def kernel_chunk(pkg, shape, R, chunk_len, variant=None):
    """Steps per chunk the kernels actually tile by: the fp32 path with the tf32 chunk scan uses
    128 fused rows (128 / R steps) whatever chunk_len says; every other path tiles by chunk_len
    (the fused bf16 kernel's FLOPs are not its bound, so its count keeps chunk_len)."""
    v = variant or pkg.ssd_chunked_variant(shape)
    return 128 // R if v == "tc_tf32" else chunk_len


def run_ours(args, rank, world, local):
    import chunked_ssd_scan_gb300 as pkg
    from chunked_ssd_scan_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = workload(args.workload, args.batch, args.seqlen)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    is_ss = isinstance(cfg, wl.SelectiveScanConfig)

    if is_ss:
        host = wl.make_selective_scan_inputs(cfg, seed=0)
        d = {k: v.to(dev) for k, v in host.items()}
        y = torch.empty_like(d["u"])
        ws = torch.zeros(pkg.selective_scan_workspace_bytes(cfg.batch, cfg.seqlen, cfg.d_model,
                                                            cfg.d_state), dtype=torch.uint8,
                         device=dev)
        # validated once; each step is only the C-ABI call
        fn = pkg.SelectiveScanPlan(d["u"], d["delta"], d["A"], d["B"], d["C"], d["skip"], y=y,
                                   workspace=ws, stream=stream)
        launches_per_call = 3
        variant = "selective_scan"
        dtype = "f32"
        io_bytes = cfg.io_bytes()
        flops = 0
    elif cfg.backward and cfg.trapezoidal:
        host = wl.make_trap_bwd_inputs(cfg, seed=0)
        d = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        wsb = torch.zeros(pkg.ssd_trapezoidal_backward_workspace_bytes(
            pkg.shape_of(d["x"], d["B"], 64, cfg.theta)), dtype=torch.uint8, device=dev)

        tgrads = pkg.ssd_trapezoidal_backward(
            d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"], d["dy"], theta=d["theta"],
            prev_x=d["prev_x"], prev_B=d["prev_B"], init_state=d["init_state"],
            dfinal=d["dfinal"], workspace=wsb, stream=stream)

        def fn():
            pkg.ssd_trapezoidal_backward(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                         d["dy"], theta=d["theta"], prev_x=d["prev_x"],
                                         prev_B=d["prev_B"], init_state=d["init_state"],
                                         dfinal=d["dfinal"], grads=tgrads, workspace=wsb,
                                         stream=stream)
        ws = wsb
        variant = "backward"
        # the expansion (2), dy^, the rotated backward of the expanded problem (8), the two
        # chain kernels
        launches_per_call = 2 + 1 + (8 if cfg.theta else 3) + 2
        dtype = cfg.dtype
        io_bytes = cfg.io_bytes()
        flops = cfg.with_(mimo_rank=2 * cfg.mimo_rank,
                          ngroups=cfg.nheads if cfg.theta else cfg.ngroups).backward_flops()
    elif cfg.backward:
        host = wl.make_bwd_inputs(cfg, seed=0)
        d = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        fn = pkg.SSDBackwardPlan(d["x"], d["dA"], d["B"], d["C"], d["dy"], theta=d["theta"],
                                 init_state=d["init_state"], dfinal=d["dfinal"], stream=stream)
        ws = fn.workspace
        variant = "backward"
        # chunk products (S_c, D_c), the two-way carry across chunks, the chunk gradients; with
        # theta also the chunk and step angles, B~/C~, dL/dg_{T-1}, the turn back of dB~/dC~ and
        # the two dtheta passes
        launches_per_call = 3 + (8 if cfg.theta else 0)
        dtype = cfg.dtype
        io_bytes = cfg.io_bytes()
        flops = cfg.backward_flops()
    elif cfg.trapezoidal:
        host = wl.make_trap_inputs(cfg, seed=0)
        d = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        y = torch.empty_like(d["x"])
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), dtype=torch.float32,
                          device=dev)
        shape = pkg.shape_of(d["x"], d["B"], cfg.chunk_len, cfg.theta)
        ws = torch.zeros(pkg.ssd_trapezoidal_workspace_bytes(shape), dtype=torch.uint8,
                         device=dev)
        fn = pkg.SSDTrapezoidalPlan(d["x"], d["dA"], d["B"], d["C"], d["gamma"], d["beta"],
                                    chunk_len=cfg.chunk_len, theta=d["theta"],
                                    prev_x=d["prev_x"], prev_B=d["prev_B"],
                                    init_state=d["init_state"], y=y, final_state=fin,
                                    workspace=ws, stream=stream)
        variant = "trapezoidal"
        # two expansion kernels, the chunk pipeline on 2R write channels, the output compaction
        launches_per_call = 2 + 3 + (2 if cfg.theta else 0) + 1
        dtype = cfg.dtype
        io_bytes = cfg.io_bytes()
        exp = pkg.make_shape(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                             cfg.nheads if cfg.theta else cfg.ngroups, 2 * cfg.mimo_rank,
                             cfg.chunk_len, "f32", cfg.theta)
        flops = cfg.with_(mimo_rank=2 * cfg.mimo_rank,
                          chunk_len=kernel_chunk(pkg, exp, 2 * cfg.mimo_rank, cfg.chunk_len)
                          ).causal_flops()
    elif cfg.rope_dim or cfg.halves:
        import ctypes
        host = wl.make_ssd_inputs(cfg, seed=0)
        d = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        y = torch.empty_like(d["x"])
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), dtype=torch.float32,
                          device=dev)
        shape = pkg.shape_of(d["x"], d["B"], cfg.chunk_len, True)
        ws = torch.zeros(pkg.load_library().ssd_rotation_variant_workspace_bytes(
            ctypes.byref(shape), cfg.rope_dim, int(cfg.halves)), dtype=torch.uint8, device=dev)

        def fn():
            pkg.ssd_rotation_variant_forward(d["x"], d["dA"], d["B"], d["C"], d["theta"],
                                             chunk_len=cfg.chunk_len, rope_dim=cfg.rope_dim,
                                             halves=cfg.halves, init_state=d["init_state"], y=y,
                                             final_state=fin, workspace=ws, stream=stream)
        variant = "rotation_variant"
        # B/C reorder (+ final-state reorder) for split halves, theta padding, the chunked call
        launches_per_call = (pkg.ssd_chunked_launches(shape) + (2 if cfg.halves else 0)
                             + (1 if cfg.rope_dim and cfg.rope_dim < cfg.dstate else 0))
        dtype = cfg.dtype
        io_bytes = cfg.io_bytes()
        flops = cfg.with_(chunk_len=kernel_chunk(pkg, shape, cfg.mimo_rank,
                                                 cfg.chunk_len)).causal_flops()
    else:
        host = wl.make_ssd_inputs(cfg, seed=0)
        d = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
        y = torch.empty_like(d["x"])
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), dtype=torch.float32,
                          device=dev)
        shape = pkg.shape_of(d["x"], d["B"], cfg.chunk_len, cfg.theta)
        ws = torch.zeros(pkg.ssd_chunked_workspace_bytes(shape), dtype=torch.uint8, device=dev)
        # validated once; each step is only the C-ABI call
        fn = pkg.SSDForwardPlan(d["x"], d["dA"], d["B"], d["C"], chunk_len=cfg.chunk_len,
                                theta=d["theta"], init_state=d["init_state"], y=y,
                                final_state=fin, workspace=ws, stream=stream, tf32=args.tf32)
        variant = "tc_tf32" if args.tf32 else pkg.ssd_chunked_variant(shape)
        launches_per_call = pkg.ssd_chunked_launches(shape)
        dtype = cfg.dtype
        io_bytes = cfg.io_bytes()
        flops = cfg.with_(chunk_len=kernel_chunk(pkg, shape, cfg.mimo_rank, cfg.chunk_len,
                                                 variant)).causal_flops()

    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if clocks:
        clocks.start()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = timed_steps(fn, args.steps, args.warmup, stream, flush)
    status = pkg.workspace_status(ws, stream)   # a bounded device wait that gave up shows here
    if status != ("SSD_OK", 0):
        raise RuntimeError(f"device-side error word after the timed steps: {status}")
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    ms = slowest_replica_ms(sum(step_ms) / len(step_ms), world, dev)
    tokens = job_tokens(cfg.tokens, world)
    hbm, tf, peak_src = measured_peaks()
    # the capture's bytes belong to the workload's own shape, not to an overridden one
    traffic = None if (args.batch or args.seqlen) else NCU_TRAFFIC_BYTES.get(cfg.name)
    kernel = ("selective_scan_forward" if is_ss
              else ("ssd_trapezoidal_backward" if cfg.trapezoidal else "ssd_chunked_backward")
              if variant == "backward"
              else "ssd_trapezoidal_forward" if variant == "trapezoidal"
              else "ssd_rotation_variant_forward" if variant == "rotation_variant"
              else f"ssd_chunked_forward[{variant}]")
    roof = roofline(io_bytes, flops, ms * 1e-3, hbm, tf, peak_src, bf16_inputs=dtype == "bf16",
                    tensor_path=variant in ("tc_bf16", "tc_tf32"))
    roof.update({"traffic": traffic, "kernel": kernel, "algorithmic_bytes_per_launch": io_bytes})
    if flops:
        roof["algorithmic_flops_per_launch"] = flops

    out = {
        "metric": metric_name(cfg, is_ss),
        "value": round(tokens / (ms * 1e-3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic (seeded; distributions of the workload definition)",
        "config": config_dict(cfg, is_ss),
        "roofline": roof,
        "gpu_launches": launches_per_call * args.steps,
        "variant": variant,
        "step_ms_min": round(min(step_ms), 5),
        "step_ms_median": round(statistics.median(step_ms), 5),
    }
    if clk:
        out["clocks"] = clk
    if not args.no_e2e:
        try:
            out["e2e"] = e2e_measure(args, cfg, is_ss, host, dev, stream)
        except Exception as ex:  # pragma: no cover
            out["e2e"] = {"error": repr(ex)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            out["cpu_baseline"] = cpu_baseline(cfg, is_ss, host)
        except Exception as ex:  # pragma: no cover
            out["cpu_baseline"] = {"error": repr(ex)}
    return out


def roofline(io_bytes, flops, sec, hbm, tf_bf16, peak_src, bf16_inputs, tensor_path):
    """The roofline of one call: the slower of the algorithmic bytes at the measured HBM
    bandwidth and the contraction FLOPs at the tensor-core peak (bf16 for bf16 inputs, tf32 for
    fp32 inputs), over the measured time.  `bound` names the slower one; `frac` is that
    roofline time over the measured time.  Paths that run their contractions on the CUDA cores
    (fp32 FMA) also report the fraction of the fp32-lane peak (`alu_frac`), as a second figure."""
    t_hbm = io_bytes / (hbm * 1e9)
    if bf16_inputs:
        tc, tc_src = tf_bf16, f"bf16, {peak_src}"
    else:
        tc, tc_src = tf32_peak()
        tc_src = "tf32, " + tc_src
    t_tc = flops / (tc * 1e12) if flops else 0.0
    gbs = io_bytes / sec / 1e9
    if t_tc > t_hbm:
        roof = {"bound": "tensor", "achieved": round(flops / sec / 1e12, 2), "peak": tc,
                "unit": "TFLOP/s", "frac": round(t_tc / sec, 4), "peak_source": tc_src,
                "hbm_gbs": round(gbs, 1), "hbm_frac": round(t_hbm / sec, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(t_hbm / sec, 4), "peak_source": peak_src}
    if flops:
        roof["tensor_peak"] = tc
        roof["tensor_peak_source"] = tc_src
        roof["tensor_tflops"] = round(flops / sec / 1e12, 2)
        roof["tensor_frac"] = round(t_tc / sec, 4)
        if not tensor_path:
            a_tf = flops / sec / 1e12
            roof["alu_tflops"] = round(a_tf, 2)
            roof["alu_frac"] = round(a_tf / ALU_FP32_TFLOPS, 4)
            roof["alu_peak_source"] = "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz"
    roof["roofline_frac"] = roof["frac"]
    return roof


def config_dict(cfg, is_ss):
    if is_ss:
        c = {"workload": cfg.name, "batch": cfg.batch, "seq_len": cfg.seqlen,
             "d_model": cfg.d_model, "d_state": cfg.d_state}
    else:
        c = {"workload": cfg.name, "batch": cfg.batch, "seq_len": cfg.seqlen,
             "nheads": cfg.nheads, "headdim": cfg.headdim, "dstate": cfg.dstate,
             "chunk_len": cfg.chunk_len, "mimo_rank": cfg.mimo_rank, "ngroups": cfg.ngroups,
             "io_dtype": cfg.dtype, "theta": cfg.theta}
        if cfg.trapezoidal:
            c["trapezoidal"] = True
        if cfg.rope_dim or cfg.halves:
            c["rope_dim"], c["halves"] = cfg.rope_dim, cfg.halves
        if cfg.backward:
            c["backward"] = True
            c["chunk_len"] = max(1, 64 // cfg.mimo_rank)   # the backward tiles by 64 fused rows
    c["l2"] = "flushed between timed steps (256 MiB write, outside the timed events)"
    c["cuda_graph"] = False
    return c


def e2e_measure(args, cfg, is_ss, host, dev, stream):
    """Same metric through the public API with pinned host buffers: every step copies the
    step's inputs host->device, runs the call, and reads the outputs back device->host."""
    import chunked_ssd_scan_gb300 as pkg

    pin = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    dbuf = {k: (torch.empty_like(v, device=dev) if v is not None else None)
            for k, v in host.items()}
    if is_ss:
        y = torch.empty_like(dbuf["u"])
        y_h = torch.empty_like(pin["u"]).pin_memory()
        outs = [(y, y_h)]

        def call():
            pkg.selective_scan_forward(dbuf["u"], dbuf["delta"], dbuf["A"], dbuf["B"],
                                       dbuf["C"], dbuf["skip"], y=y)
    elif cfg.backward and cfg.trapezoidal:
        ws = torch.zeros(pkg.ssd_trapezoidal_backward_workspace_bytes(
            pkg.shape_of(dbuf["x"], dbuf["B"], 64, cfg.theta)), dtype=torch.uint8, device=dev)
        grads = pkg.ssd_trapezoidal_backward(
            dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"], dbuf["gamma"], dbuf["beta"], dbuf["dy"],
            theta=dbuf["theta"], prev_x=dbuf["prev_x"], prev_B=dbuf["prev_B"],
            init_state=dbuf["init_state"], dfinal=dbuf["dfinal"], workspace=ws)
        grads.pop("workspace")
        outs = [(v, torch.empty(v.shape, dtype=v.dtype).pin_memory())
                for v in grads.values() if v is not None]

        def call():
            pkg.ssd_trapezoidal_backward(
                dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"], dbuf["gamma"], dbuf["beta"],
                dbuf["dy"], theta=dbuf["theta"], prev_x=dbuf["prev_x"], prev_B=dbuf["prev_B"],
                init_state=dbuf["init_state"], dfinal=dbuf["dfinal"], grads=grads, workspace=ws)
    elif cfg.backward:
        plan = pkg.SSDBackwardPlan(dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"], dbuf["dy"],
                                   theta=dbuf["theta"], init_state=dbuf["init_state"],
                                   dfinal=dbuf["dfinal"])
        ws = plan.workspace
        outs = [(v, torch.empty(v.shape, dtype=v.dtype).pin_memory())
                for v in plan.grads.values() if v is not None]

        def call():
            plan()
    else:
        y = torch.empty_like(dbuf["x"])
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate),
                          dtype=torch.float32, device=dev)
        outs = [(y, torch.empty(y.shape, dtype=y.dtype).pin_memory()),
                (fin, torch.empty(fin.shape, dtype=fin.dtype).pin_memory())]
        shape = pkg.shape_of(dbuf["x"], dbuf["B"], cfg.chunk_len, cfg.theta)
        if cfg.rope_dim or cfg.halves:
            import ctypes
            shape = pkg.shape_of(dbuf["x"], dbuf["B"], cfg.chunk_len, True)
            ws = torch.zeros(pkg.load_library().ssd_rotation_variant_workspace_bytes(
                ctypes.byref(shape), cfg.rope_dim, int(cfg.halves)), dtype=torch.uint8,
                device=dev)

            def call():
                pkg.ssd_rotation_variant_forward(dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"],
                                                 dbuf["theta"], chunk_len=cfg.chunk_len,
                                                 rope_dim=cfg.rope_dim, halves=cfg.halves,
                                                 init_state=dbuf["init_state"], y=y,
                                                 final_state=fin, workspace=ws)
        elif cfg.trapezoidal:
            ws = torch.zeros(pkg.ssd_trapezoidal_workspace_bytes(shape), dtype=torch.uint8,
                             device=dev)

            def call():
                pkg.ssd_trapezoidal_forward(dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"],
                                            dbuf["gamma"], dbuf["beta"], chunk_len=cfg.chunk_len,
                                            theta=dbuf["theta"], prev_x=dbuf["prev_x"],
                                            prev_B=dbuf["prev_B"], init_state=dbuf["init_state"],
                                            y=y, final_state=fin, workspace=ws)
        else:
            ws = torch.zeros(pkg.ssd_chunked_workspace_bytes(shape), dtype=torch.uint8,
                             device=dev)

            def call():
                pkg.ssd_chunked_forward(dbuf["x"], dbuf["dA"], dbuf["B"], dbuf["C"],
                                        chunk_len=cfg.chunk_len, theta=dbuf["theta"],
                                        init_state=dbuf["init_state"], y=y, final_state=fin,
                                        workspace=ws, tf32=args.tf32)

    h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
    d2h = sum(o.numel() * o.element_size() for o, _ in outs)

    def step():
        for k, v in pin.items():
            if v is not None:
                dbuf[k].copy_(v, non_blocking=True)
        call()
        for o, oh in outs:
            oh.copy_(o, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    n = max(1, min(args.steps, 10))
    s.record(stream)
    for _ in range(n):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    if not is_ss:
        status = pkg.workspace_status(ws, stream)
        if status != ("SSD_OK", 0):
            raise RuntimeError(f"device-side error word after the end-to-end steps: {status}")
    # the copies run in series with the call on one stream: their effective bandwidth shows how
    # much of the end-to-end time is the host link rather than the kernels
    return {"value": round(cfg.tokens / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n,
            "copy_gbs_effective": round((h2d + d2h) / (ms * 1e-3) / 1e9, 1)}


def _ssd_sample(cfg, host, heads, batches=1):
    """Batches 0..batches-1, heads 0..heads-1 of the workload as fp64 arrays (independent
    (batch, head) problems; a sub-problem of the workload with the same per-problem size)."""
    import numpy as np

    hpg = cfg.nheads // cfg.ngroups
    if cfg.ngroups > 1 and hpg > 1:
        heads = max(hpg, heads // hpg * hpg)
    groups = 1 if cfg.ngroups == 1 else -(-heads // hpg)
    f = lambda v: None if v is None else v.to(torch.float64).numpy()
    a = {k: f(v) for k, v in host.items()}
    nb = batches
    sub = {
        "x": a["x"][:nb, :, :, :heads], "dA": a["dA"][:nb, :, :heads],
        "B": a["B"][:nb, :, :, :groups], "C": a["C"][:nb, :, :, :groups],
        "theta": None if a["theta"] is None else a["theta"][:nb, :, :heads],
        "init_state": None if a["init_state"] is None else a["init_state"][:nb, :heads],
    }
    if cfg.rope_dim or cfg.halves:
        sub["rope_dim"], sub["halves"] = cfg.rope_dim, cfg.halves
    if "dy" in a:   # backward
        sub["dy"], sub["dfinal"] = a["dy"][:nb, :, :, :heads], a["dfinal"][:nb, :heads]
    if "gamma" in a:   # trapezoidal form
        sub["gamma"], sub["beta"] = a["gamma"][:nb, :, :heads], a["beta"][:nb, :, :heads]
        sub["prev_x"] = None if a["prev_x"] is None else a["prev_x"][:nb, :, :heads]
        sub["prev_B"] = None if a["prev_B"] is None else a["prev_B"][:nb, :, :groups]
    sub = {k: (np.ascontiguousarray(v) if isinstance(v, np.ndarray) else v)
           for k, v in sub.items()}
    return sub, heads


def _time_oracle_ssd(sub, nthr):
    import oracle

    t0 = time.perf_counter()
    if "dy" in sub and "gamma" in sub:
        oracle.ssd_trap_backward(sub["x"], sub["dA"], sub["B"], sub["C"], sub["gamma"],
                                 sub["beta"], sub["dy"], theta=sub["theta"],
                                 init_state=sub["init_state"], prev_x=sub["prev_x"],
                                 prev_B=sub["prev_B"], dfinal=sub["dfinal"], nthreads=nthr)
    elif "dy" in sub:
        oracle.ssd_backward(sub["x"], sub["dA"], sub["B"], sub["C"], sub["dy"],
                            init_state=sub["init_state"], dfinal=sub["dfinal"],
                            theta=sub["theta"], nthreads=nthr)
    elif "rope_dim" in sub:
        oracle.ssd_rotation_variant(sub["x"], sub["dA"], sub["B"], sub["C"], sub["theta"],
                                    sub["init_state"], rope_dim=sub["rope_dim"],
                                    halves=sub["halves"], nthreads=nthr)
    elif "gamma" in sub:
        oracle.ssd_trapezoidal(sub["x"], sub["dA"], sub["B"], sub["C"], sub["gamma"],
                               sub["beta"], sub["theta"], sub["init_state"], sub["prev_x"],
                               sub["prev_B"], nthreads=nthr)
    else:
        oracle.ssd(sub["x"], sub["dA"], sub["B"], sub["C"], sub["theta"], sub["init_state"],
                   nthreads=nthr)
    return time.perf_counter() - t0


def _time_oracle_ss(cfg, host, nthr, channels):
    import oracle

    f = lambda v: v.to(torch.float64).numpy()
    u, dl = f(host["u"])[0:1, :, :channels], f(host["delta"])[0:1, :, :channels]
    A, sk = f(host["A"])[:channels], f(host["skip"])[:channels]
    B, C = f(host["B"])[0:1], f(host["C"])[0:1]
    import numpy as np
    u, dl, A, sk = (np.ascontiguousarray(v) for v in (u, dl, A, sk))
    t0 = time.perf_counter()
    oracle.selective_scan(u, dl, A, B, C, sk, nthreads=nthr)
    return time.perf_counter() - t0


def oracle_single_thread(cfg, is_ss, host):
    """The oracle on one host thread: (tokens/s scaled to the full workload, description)."""
    if is_ss:
        ch = min(cfg.d_model, 64)
        t = _time_oracle_ss(cfg, host, 1, ch)
        frac = ch / (cfg.d_model * cfg.batch)
        desc = f"one thread, batch 0, channels 0..{ch - 1}, full T"
    else:
        sub1, _ = _ssd_sample(cfg, host, 1)
        t = _time_oracle_ssd(sub1, 1)
        frac = 1.0 / (cfg.nheads * cfg.batch)
        desc = "one thread, the (batch 0, head 0) problem, full T"
    return round(cfg.tokens * frac / t, 1), desc + f"; {t:.2f} s wall"


def oracle_sampler(cfg, is_ss, host, target_s):
    """Returns (step callable -> seconds, sampled fraction of the workload, cores, description):
    the oracle as it stands over whole independent problems of batch 0, sized to ~target_s."""
    import oracle

    nthr = oracle.default_threads()
    if is_ss:
        D = cfg.d_model
        t1 = _time_oracle_ss(cfg, host, nthr, min(D, 64))
        per_ch = t1 / min(D, 64)
        ch = int(max(1, min(D, target_s / max(per_ch, 1e-9))))
        frac = ch / (D * cfg.batch)
        desc = f"batch 0, channels 0..{ch - 1} of {D}, full T (independent problems)"
        return (lambda: _time_oracle_ss(cfg, host, nthr, ch)), frac, min(nthr, ch), desc
    sub1, _ = _ssd_sample(cfg, host, 1)
    t1 = _time_oracle_ssd(sub1, nthr)                # one (batch, head) problem, one thread
    problems = int(max(1, (target_s * nthr) / max(t1, 1e-9)))
    if problems >= cfg.nheads:
        batches, heads = int(min(cfg.batch, problems // cfg.nheads)), cfg.nheads
    else:
        batches, heads = 1, problems
    sub, heads = _ssd_sample(cfg, host, heads, batches)
    frac = heads * batches / (cfg.nheads * cfg.batch)
    desc = (f"batches 0..{batches - 1} of {cfg.batch}, heads 0..{heads - 1} of {cfg.nheads} "
            f"(each a full-T independent (batch, head) problem); value scaled by the sampled "
            f"fraction {frac:.4g}")
    return (lambda: _time_oracle_ssd(sub, nthr)), frac, min(nthr, heads * batches), desc


def cpu_baseline(cfg, is_ss, host, target_s: float = 12.0):
    """The fp64 oracle as it stands, on this host's cores, over a bounded sample of the workload,
    scaled to tokens/s of the full workload."""
    step, frac, cores, desc = oracle_sampler(cfg, is_ss, host, target_s)
    # repeat a sample that ends quickly until about half the target has elapsed (mean time)
    total, reps = 0.0, 0
    while reps == 0 or (total < 0.5 * target_s and reps < 50):
        total += step()
        reps += 1
    dt = total / reps
    st_value, st_desc = oracle_single_thread(cfg, is_ss, host)
    return {"value": round(cfg.tokens * frac / dt, 1), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": desc + f"; {dt:.2f} s wall per repetition, {reps} repetitions",
            "single_thread_value": st_value, "single_thread_sample": st_desc}


def run_reference(args, rank, world):
    """Reference arm: the fp64 oracle on the host cores, W untimed and K timed steps, each step a
    bounded sample of the same workload; same metric and unit as our arm."""
    cfg = workload(args.workload, args.batch, args.seqlen)
    from chunked_ssd_scan_gb300 import workloads as wl
    is_ss = isinstance(cfg, wl.SelectiveScanConfig)
    host = (wl.make_selective_scan_inputs(cfg, seed=0) if is_ss
            else wl.make_trap_bwd_inputs(cfg, 0) if cfg.trapezoidal and cfg.backward
            else wl.make_trap_inputs(cfg, 0) if cfg.trapezoidal
            else wl.make_bwd_inputs(cfg, 0) if cfg.backward else wl.make_ssd_inputs(cfg, 0))
    per_step = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    step, frac, cores, desc = oracle_sampler(cfg, is_ss, host, per_step)
    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    sec = sum(times) / len(times)
    val = round(cfg.tokens * frac / sec, 1)
    return {
        "impl": "reference",
        "metric": metric_name(cfg, is_ss),
        "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(cfg.tokens / val * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(cfg, is_ss),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": desc + f"; {sec:.2f} s wall per step"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.measure_peak:
        print(json.dumps(measure_matmul_peak(args.measure_peak)))
        return
    rank, world, local = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)))
        return
    out = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
