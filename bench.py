"""Benchmark of the dense-product hot path on GB300.

One step = one pass of the hot path over its workload:
  * gemm_bf16  M = N = K = 8192, BF16 operands (normal, sigma = 1/sqrt(K),
    seed 6), FP32 accumulate and output  -- the headline (TFLOP/s);
  * gemv_f32   y = A x with A 4096 x 4096 (uniform [-1, 1), seed 2) -- the
    fully connected layer (HBM GB/s): GEMV_GROUP back-to-back launches at
    batch 1 over distinct copies of A (a stack of layers), then
    GEMV_GROUP launches at batch 8.
Every kernel runs through the C ABI (libgtg.so) on the current torch stream.
`value` is the BF16 GEMM's throughput; the GEMV's is reported beside it with
its own roofline. The remaining workload configurations are measured after
the timed region (`configs`, skipped with --no-sweep).

Prints ONE JSON line on rank 0. `--impl reference` times the FP64 CPU oracle
(the reference arm of this project) on host cores instead.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (% of GB300 peak) and GEMV HBM GB/s (% of peak), 1 GPU"
GEMM_SHAPE = (8192, 8192, 8192)
GEMV_SHAPE = (4096, 4096)
GEMV_GROUP = 8
# convolutional layers of a residual image network: (name, N, H, W, C, CO, KH, KW, stride, pad, timed calls)
CONV_LAYERS = [
    ("f4: bf16 conv 3x3 64->64, 56x56, batch 32, pad 1", 32, 56, 56, 64, 64, 3, 3, 1, 1, 20),
    ("f4: bf16 conv 3x3 256->256, 14x14, batch 64, pad 1", 64, 14, 14, 256, 256, 3, 3, 1, 1, 20),
    ("f4: bf16 conv 3x3 512->512, 7x7, batch 64, pad 1", 64, 7, 7, 512, 512, 3, 3, 1, 1, 20),
    ("f4: bf16 conv 1x1 256->1024, 14x14, batch 64", 64, 14, 14, 256, 1024, 1, 1, 1, 0, 20),
    ("f4: bf16 conv 7x7/2 3->64, 224x224, batch 16, pad 3", 16, 224, 224, 3, 64, 7, 7, 2, 3, 10),
]
# the same network's layers in TF32 (FP32 storage): implicit GEMM from a rounded copy of the image
CONV_LAYERS_TF32 = [
    ("f4: tf32 conv 3x3 256->256, 56x56, batch 16, pad 1", 16, 56, 56, 256, 256, 3, 3, 1, 1, 10),
]
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the part's nominal figures (dense BF16 tensor rate, HBM3e bandwidth), reported
# beside the measured denominators
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 7900.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1500)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["gtg", "reference"], default="gtg")
    p.add_argument("--no-sweep", action="store_true", help="skip the per-configuration sweep")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--only-ablation", action="store_true",
                   help="run only the pages' kernel designs beside the library's (prints their table)")
    p.add_argument("--ablation-iters", type=int, default=0, help="timed launches per ablation kernel (0: default)")
    p.add_argument("--only-gemv", default=None, metavar="PREC:N:BATCH",
                   help="run only an N x N GEMV (prec f32 or bf16) at the given batch, three calls (for profiling)")
    p.add_argument("--only-gemm", default=None, metavar="PREC:M:N:K",
                   help="run only one GEMM (prec bf16, f16, tf32 or f32), three calls (for profiling)")
    p.add_argument("--only-conv", type=int, default=None, metavar="IDX",
                   help="run only convolutional layer IDX of the sweep, three calls (for profiling)")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gemv_tiled_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(key, files):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source
    is unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "counters.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(key)
    if not e or e.get("source_sha") != kernel_source_sha(files):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the GPU works."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "power_cap": parts[8]})
            except ValueError:
                continue
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for k, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                            ("sw_thermal", "sw_thermal_slowdown"), ("power_cap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(loaded), "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------------ ranks

def reduce_max(x: float, world: int, device) -> float:
    """Maximum of `x` over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float, scale: float = 1e12) -> float:
    """Whole-job throughput: every rank processes `units_per_rank` (replicas,
    weak scaling), and the job takes as long as its slowest rank."""
    return world * units_per_rank / max_seconds / scale


# ------------------------------------------------------------------ GPU arm

def gpu_arm(args, rank, world, local_rank):
    import numpy as np
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import gemm_normal_bf16, gemm_uniform_f32, gemv_uniform_f32

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 0
    peaks, peak_src = load_peaks()

    def bf16_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def ok(st, what):
        if st != gtg.GTG_OK:
            raise gtg.GtgError(st, what)

    # ---- inputs (seeded, synthetic, resident in HBM before timing)
    M, N, K = GEMM_SHAPE
    (Ab, Bb), = gemm_normal_bf16(6, [GEMM_SHAPE], lambda k: k ** -0.5)
    dA, dB = bf16_dev(Ab), bf16_dev(Bb)
    dC = torch.empty((M, N), dtype=torch.float32, device=dev)
    gm, gn = GEMV_SHAPE
    Av, xv, Xv = gemv_uniform_f32(2, gm, gn, batch=8)
    # four copies of the GEMV operands at distinct addresses: consecutive
    # launches never find their matrix in L2 (4 x 64 MiB > L2)
    nrot = max(4, math.ceil(3 * l2 / (4 * gm * gn)) if l2 else 4)
    vA = [torch.from_numpy(Av).to(dev) for _ in range(nrot)]
    vx = torch.from_numpy(xv).to(dev)
    vX = torch.from_numpy(Xv).to(dev)
    vy = torch.empty(gn, device=dev)
    vY = torch.empty((8, gm), device=dev)

    def gemm_call():
        ok(gtg.gemm_bf16(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, sh), "gemm_bf16")

    def gemv_call(i, batch):
        A_ = vA[i % nrot]
        if batch == 1:
            ok(gtg.gemv_f32(gm, gn, A_.data_ptr(), gn, vx.data_ptr(), gn, vy.data_ptr(), gm, 1, sh), "gemv_f32")
        else:
            ok(gtg.gemv_f32(gm, gn, A_.data_ptr(), gn, vX.data_ptr(), gn, vY.data_ptr(), gm, batch, sh),
               "gemv_f32")

    plan = gtg.plan_gemm("bf16", M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N)
    vplan = gtg.plan_gemv(gm, gn, vA[0].data_ptr(), gn, vx.data_ptr(), gn, vy.data_ptr(), gm, 1)

    # ---- warm-up
    for i in range(args.warmup):
        gemm_call()
        for g in range(GEMV_GROUP):
            gemv_call(g, 1)
        for g in range(GEMV_GROUP):
            gemv_call(g + 1, 8)
    torch.cuda.synchronize()
    ok(gtg.gtg_sync_status(sh), "device status after warm-up")

    # ---- timed region: K steps; events on the launching stream around the
    # GEMM and around each group of back-to-back GEMV launches
    ev = lambda: torch.cuda.Event(enable_timing=True)
    e_gemm = [(ev(), ev()) for _ in range(args.steps)]
    e_v1 = [(ev(), ev()) for _ in range(args.steps)]
    e_v8 = [(ev(), ev()) for _ in range(args.steps)]
    start, stop = ev(), ev()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start.record(stream)
        for i in range(args.steps):
            e_gemm[i][0].record(stream)
            gemm_call()
            e_gemm[i][1].record(stream)
            e_v1[i][0].record(stream)
            for g in range(GEMV_GROUP):
                gemv_call(i * GEMV_GROUP + g, 1)
            e_v1[i][1].record(stream)
            e_v8[i][0].record(stream)
            for g in range(GEMV_GROUP):
                gemv_call(i * GEMV_GROUP + g + 1, 8)
            e_v8[i][1].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ok(gtg.gtg_sync_status(sh), "device status after timing")
    launches = (1 + 2 * GEMV_GROUP) * args.steps

    total_ms = start.elapsed_time(stop)
    gemm_ms = [a.elapsed_time(b) for a, b in e_gemm]
    v1_ms = [a.elapsed_time(b) / GEMV_GROUP for a, b in e_v1]
    v8_ms = [a.elapsed_time(b) / GEMV_GROUP for a, b in e_v8]

    # max over ranks
    def rank_max(x):
        return reduce_max(x, world, dev)

    total_ms = rank_max(total_ms)
    gemm_avg = rank_max(sum(gemm_ms) / len(gemm_ms))
    v1_avg = rank_max(sum(v1_ms) / len(v1_ms))
    v8_avg = rank_max(sum(v8_ms) / len(v8_ms))

    flops = 2.0 * M * N * K
    gemm_tflops = job_throughput(flops, world, gemm_avg * 1e-3, 1e12)
    v1_bytes = 4.0 * gm * gn + 4.0 * gn + 4.0 * gm
    v8_bytes = 4.0 * gm * gn + 8 * (4.0 * gn + 4.0 * gm)
    v1_gbs = job_throughput(v1_bytes, world, v1_avg * 1e-3, 1e9)
    v8_gbs = job_throughput(v8_bytes, world, v8_avg * 1e-3, 1e9)

    long_region = total_ms > 1000.0
    peak_kind = "sustained" if long_region else "burst"
    bf16_peak = peaks.get("bf16_tflops_sustained" if long_region else "bf16_tflops")
    hbm_peak = peaks.get("hbm_gbs")
    tc_files = ["gemm_tc.cu", "ptx.cuh"]
    gv_files = ["gemv.cu", "gemv_kernels.cuh", "ptx.cuh"]
    gemm_kernel = ("tc_gemm_pair_kernel (CTA pair, 256x256 tile)" if plan.get("cluster") == 2
                   else f"tc_gemm_kernel<bf16, BN={plan.get('bn')}>")
    if vplan.get("bm") == 1 and vplan.get("smem", 0) > 4 * vplan.get("bn", 0):
        gemv_kernel = "gemv_ring_kernel<batch=1>"   # per-warp partial sums beside the staged x
    else:
        gemv_kernel = {1: "gemv_stream_kernel<batch=1>", 4: "gemv_blocks_kernel"}.get(vplan.get("bm"), "gemv_kernel")
    roofline = {"bound": "tensor", "achieved": round(gemm_tflops / world, 1), "peak": bf16_peak,
                "unit": "TFLOP/s", "frac": round(gemm_tflops / world / bf16_peak, 4),
                "traffic": committed_traffic("gemm_bf16_8192", tc_files),
                "peak_source": f"{peak_src} bf16 {peak_kind}",
                "algorithmic_flops_per_launch": flops, "kernel": gemm_kernel,
                "plan": plan, "peak_nominal": NOMINAL["bf16_tflops"],
                "frac_nominal": round(gemm_tflops / world / NOMINAL["bf16_tflops"], 4)}
    gemv_roofline = {"bound": "hbm", "achieved": round(v1_gbs / world, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(v1_gbs / world / hbm_peak, 4),
                     "traffic": committed_traffic("gemv_f32_4096_b1", gv_files),
                     "peak_source": f"{peak_src} hbm copy", "algorithmic_bytes_per_launch": v1_bytes,
                     "kernel": gemv_kernel, "plan": vplan, "peak_nominal": NOMINAL["hbm_gbs"],
                     "frac_nominal": round(v1_gbs / world / NOMINAL["hbm_gbs"], 4)}

    result = {
        "metric": METRIC, "value": round(gemm_tflops, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"bf16 GEMM M=N=K=8192 (FP32 accumulate/output) + {GEMV_GROUP} x fp32 GEMV "
                               f"4096x4096 batch 1 + {GEMV_GROUP} x batch 8", "gemm_seed": 6,
                   "gemm_inputs": "normal(0, 1/sqrt(K)) -> bf16",
                   "gemv_seed": 2, "gemv_inputs": "uniform[-1,1) fp32",
                   "l2": f"GEMM inputs 256 MiB + output 256 MiB exceed L2 ({l2 >> 20} MiB); GEMV rotates "
                         f"{nrot} copies of A ({nrot * 64} MiB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "gemv": {"value": round(v1_gbs, 1), "unit": "GB/s", "batch8_gbs": round(v8_gbs, 1),
                 "batch8_frac": round(v8_gbs / world / hbm_peak, 4), "roofline": gemv_roofline},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }

    # ---- end to end through the public API: pinned host buffers in, host result out
    if args.e2e_steps > 0:
        hA = torch.from_numpy(Ab.view(np.int16)).view(torch.bfloat16).pin_memory()
        hB = torch.from_numpy(Bb.view(np.int16)).view(torch.bfloat16).pin_memory()
        hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
        def host_call():
            # the C ABI on host buffers: copies in, products, copies out, synchronised
            st = gtg.gemm_host("bf16", M, N, K, hA.data_ptr(), K, hB.data_ptr(), N, hC.data_ptr(), N)
            if st != gtg.GTG_OK:
                raise RuntimeError(f"gemm_host: {gtg.status_string(st)}")
        for _ in range(2):
            host_call()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            host_call()
        torch.cuda.synchronize()
        e2e_s = rank_max(time.perf_counter() - t0)
        result["e2e"] = {"value": round(job_throughput(flops * args.e2e_steps, world, e2e_s), 1), "unit": "TFLOP/s",
                         "h2d_bytes_per_step": int(hA.numel() * 2 + hB.numel() * 2),
                         "d2h_bytes_per_step": int(hC.numel() * 4), "steps": args.e2e_steps,
                         "api": "gemm_host (C ABI), pinned host bf16 A and B, host FP32 C"}
        del hA, hB, hC

    del dA, dB, dC
    torch.cuda.empty_cache()
    if not args.no_sweep:
        result["configs"] = sweep(dev, stream, peaks, l2)
    return result


def only_gemv(spec, local_rank):
    """Three gemv_f32 / gemv_bf16 calls on one N x N configuration (seeded inputs)."""
    import numpy as np
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import PCG32

    prec, n, batch = spec.split(":")
    n, batch = int(n), int(batch)
    torch.cuda.set_device(local_rank)
    g = PCG32(2)
    if prec == "bf16":
        A = torch.from_numpy(g.normal_bf16((n, n)).view(np.int16)).cuda()
        fn = gtg.gemv_bf16
    else:
        A = torch.from_numpy(g.uniform_f32((n, n))).cuda()
        fn = gtg.gemv_f32
    X = torch.from_numpy(g.uniform_f32((batch, n))).cuda()
    Y = torch.empty((batch, n), device="cuda")
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(3):
        e0.record(s)
        rc = fn(n, n, A.data_ptr(), n, X.data_ptr(), n, Y.data_ptr(), n, batch, s.cuda_stream)
        e1.record(s)
        assert rc == gtg.GTG_OK, rc
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert gtg.gtg_sync_status(s.cuda_stream) == gtg.GTG_OK
    plan = gtg.plan_gemv(n, n, A.data_ptr(), n, X.data_ptr(), n, Y.data_ptr(), n, batch, precision=prec)
    return {"config": f"{prec} gemv {n}x{n} batch {batch}", "kernel": plan["kernel"],
            "ms_per_call": [round(t, 4) for t in times]}


def only_gemm(spec, local_rank):
    """Three calls of one GEMM configuration (seeded inputs: normal for 16-bit
    operands, uniform [-1, 1) for FP32 ones)."""
    import numpy as np
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import PCG32

    prec, m, n, k = spec.split(":")
    M, N, K = int(m), int(n), int(k)
    torch.cuda.set_device(local_rank)
    g = PCG32(8)
    if prec in ("bf16", "f16"):
        draw = g.normal_bf16 if prec == "bf16" else g.normal_f16
        A = torch.from_numpy(draw((M, K)).view(np.int16)).cuda()
        B = torch.from_numpy(draw((K, N)).view(np.int16)).cuda()
    else:
        A = torch.from_numpy(g.uniform_f32((M, K))).cuda()
        B = torch.from_numpy(g.uniform_f32((K, N))).cuda()
    C = torch.empty((M, N), device="cuda")
    fn = {"bf16": gtg.gemm_bf16, "f16": gtg.gemm_f16, "tf32": gtg.gemm_tf32, "f32": gtg.gemm_f32}[prec]
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(3):
        e0.record(s)
        rc = fn(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, s.cuda_stream)
        e1.record(s)
        assert rc == gtg.GTG_OK, rc
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert gtg.gtg_sync_status(s.cuda_stream) == gtg.GTG_OK
    plan = gtg.plan_gemm(prec, M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N)
    return {"config": f"{prec} gemm {M}x{N}x{K}", "plan": plan, "ms_per_call": [round(t, 4) for t in times]}


def only_conv(idx, local_rank):
    """Three conv2d_nhwc calls on one layer of CONV_LAYERS (BF16, seeded normal inputs)."""
    import numpy as np
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import PCG32

    torch.cuda.set_device(local_rank)
    name, N, H, W, C, CO, KH, KW, st, pd, _ = CONV_LAYERS[idx]
    g = PCG32(20 + C + CO)
    X = torch.from_numpy(g.normal_bf16((N, H, W, C)).view(np.int16)).cuda()
    Wt = torch.from_numpy(g.normal_bf16((KH, KW, C, CO), (KH * KW * C) ** -0.5).view(np.int16)).cuda()
    OH, OW = gtg.conv_out_size(H, W, KH, KW, st, pd)
    Y = torch.empty((N, OH, OW, CO), device="cuda")
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(3):
        e0.record(s)
        rc = gtg.conv2d_nhwc("bf16", N, H, W, C, CO, KH, KW, st, st, pd, pd, 1, 1, X.data_ptr(), Wt.data_ptr(),
                             Y.data_ptr(), None, s.cuda_stream)
        e1.record(s)
        assert rc == gtg.GTG_OK, rc
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert gtg.gtg_sync_status(s.cuda_stream) == gtg.GTG_OK
    return {"config": name, "ms_per_call": [round(t, 4) for t in times]}


def time_launches(fn, iters, stream, groups=5):
    """Mean time per launch (ms) of `groups` groups of about iters / groups
    back-to-back launches, each group between CUDA events on `stream`, after
    three warm-up launches: returns (median over the groups, best group)."""
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    per = max(1, iters // groups)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(groups)]
    i = 0
    for s, e in evs:
        s.record(stream)
        for _ in range(per):
            fn(i)
            i += 1
        e.record(stream)
    torch.cuda.synchronize()
    ts = sorted(s.elapsed_time(e) / per for s, e in evs)
    return ts[len(ts) // 2], ts[0]


def sweep(dev, stream, peaks, l2):
    """Every workload configuration, each timed on its own (back-to-back
    launches; operands rotated where one set would fit in L2)."""
    import numpy as np
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import gemm_normal_bf16, gemm_uniform_f32, gemv_uniform_f32

    sh = int(stream.cuda_stream)
    out = []
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    hbm_peak = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])

    def roofline_of(flops, nbytes, ms, peak, compute_bound):
        # the slower of the two bounds: arithmetic at `peak` TFLOP/s, or the
        # compulsory bytes (operands read once, output written once) at the HBM peak
        t_c = flops / (peak * 1e12)
        t_m = nbytes / (hbm_peak * 1e9)
        return {"compulsory_bytes": int(nbytes), "bound": "hbm" if t_m > t_c else compute_bound,
                "roofline_frac": round(max(t_c, t_m) / (ms * 1e-3), 4)}

    def gemm_cfg(name, prec, M, N, K, A, B, peak, peak_name, iters, bias=None, act="none"):
        esz = 2 if prec in ("bf16", "f16") else 4
        need = (M * K + K * N) * esz + M * N * 4
        nrot = max(1, math.ceil(2 * l2 / need)) if l2 else 1
        if prec in ("bf16", "f16"):
            mk = lambda X: torch.from_numpy(X.view(np.int16)).to(dev)
        else:
            mk = lambda X: torch.from_numpy(X).to(dev)
        sets = [(mk(A), mk(B), torch.empty((M, N), device=dev)) for _ in range(nrot)]
        fn = {"f32": gtg.gemm_f32_ex, "tf32": gtg.gemm_tf32_ex, "bf16": gtg.gemm_bf16_ex,
              "f16": gtg.gemm_f16_ex}[prec]
        dbias = torch.from_numpy(bias).to(dev) if bias is not None else None
        ep = gtg.epilogue(dbias.data_ptr() if dbias is not None else 0, act) if (bias is not None or act != "none") else None

        def call(i):
            a, b, c = sets[i % nrot]
            st = fn(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, ep, sh)
            assert st == gtg.GTG_OK, st

        ms, ms_best = time_launches(call, iters, stream)
        a, b, c = sets[0]
        plan = gtg.plan_gemm(prec, M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out.append({"config": name, "path": prec, "shape": [M, N, K], "ms": round(ms, 4), "ms_best": round(ms_best, 4),
                    "TFLOP/s": round(tf, 2), "peak": peak, "peak_name": peak_name,
                    "frac": round(tf / peak, 4) if peak else None, "kernel": plan["kernel"],
                    "tile": [plan["bm"], plan["bn"], plan["bk"]], "grid": plan["grid"], "buffer_sets": nrot,
                    **roofline_of(2.0 * M * N * K, need, ms, peak, "fp32 alu" if prec == "f32" else "tensor")})
        del sets

    # FP32 SIMT peak: SMs x 128 FP32 lanes x 2 flops x the max SM clock
    f32_peak = sms * 128 * 2 * 2.070e9 / 1e12
    tf32_peak = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) / 2.0
    bf16_peak = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])

    A, B = gemm_uniform_f32(1, 256, 256, 256)
    gemm_cfg("1: f32 256^3", "f32", 256, 256, 256, A, B, f32_peak, "fp32 simt (2070 MHz)", 200)
    A, B = gemm_uniform_f32(3, 1024, 1024, 1024)
    gemm_cfg("3a: f32 1024^3", "f32", 1024, 1024, 1024, A, B, f32_peak, "fp32 simt (2070 MHz)", 50)
    gemm_cfg("3a: tf32 1024^3", "tf32", 1024, 1024, 1024, A, B, tf32_peak, "bf16 burst / 2 (derived)", 100)
    A, B = gemm_uniform_f32(4, 1000, 700, 1500)
    gemm_cfg("3b: f32 1000x700x1500", "f32", 1000, 700, 1500, A, B, f32_peak, "fp32 simt (2070 MHz)", 50)
    gemm_cfg("3b: tf32 1000x700x1500", "tf32", 1000, 700, 1500, A, B, tf32_peak, "bf16 burst / 2 (derived)", 100)
    A, B = gemm_uniform_f32(3, 8192, 8192, 8192)
    gemm_cfg("tf32 8192^3", "tf32", 8192, 8192, 8192, A, B, tf32_peak, "bf16 burst / 2 (derived)", 20)
    del A, B
    (A, B), = gemm_normal_bf16(5, [(4096, 4096, 4096)])
    gemm_cfg("4: bf16 4096^3", "bf16", 4096, 4096, 4096, A, B, bf16_peak, "bf16 burst", 50)
    shapes = [(8192, 8192, 8192), (16384, 4096, 4096)]
    (A1, B1), (A2, B2) = gemm_normal_bf16(6, shapes, lambda k: k ** -0.5)
    gemm_cfg("5a: bf16 8192^3", "bf16", 8192, 8192, 8192, A1, B1, bf16_peak, "bf16 burst", 20)
    gemm_cfg("5b: bf16 16384x4096x4096", "bf16", 16384, 4096, 4096, A2, B2, bf16_peak, "bf16 burst", 20)
    from seeded import PCG32
    layer_bias = PCG32(7).uniform_f32((8192,))
    gemm_cfg("f1: bf16 dense layer 8192^3, bias + ReLU", "bf16", 8192, 8192, 8192, A1, B1, bf16_peak,
             "bf16 burst", 20, bias=layer_bias, act="relu")
    del A1, B1, A2, B2
    g16 = PCG32(9)
    A16, B16 = g16.normal_f16((8192, 8192), 8192 ** -0.25), g16.normal_f16((8192, 8192), 8192 ** -0.25)
    gemm_cfg("f2: f16 8192^3", "f16", 8192, 8192, 8192, A16, B16, bf16_peak, "bf16 burst (same rate)", 20)
    del A16, B16

    def batched_cfg(name, batch, M, N, K, iters, shared_B=False):
        g = PCG32(10 + batch)
        A = torch.from_numpy(g.normal_bf16((batch, M, K), K ** -0.25).view(np.int16)).to(dev)
        B = torch.from_numpy(g.normal_bf16((1 if shared_B else batch, K, N), K ** -0.25).view(np.int16)).to(dev)
        C = torch.empty((batch, M, N), device=dev)
        sB = 0 if shared_B else K * N

        def call(i):
            st = gtg.gemm_strided_batched("bf16", M, N, K, A.data_ptr(), K, M * K, B.data_ptr(), N, sB,
                                          C.data_ptr(), N, M * N, batch, None, sh)
            assert st == gtg.GTG_OK, st

        ms, ms_best = time_launches(call, iters, stream)
        tf = 2.0 * batch * M * N * K / (ms * 1e-3) / 1e12
        out.append({"config": name, "path": "bf16 strided batch", "shape": [M, N, K], "batch": batch,
                    "ms": round(ms, 4), "ms_best": round(ms_best, 4), "TFLOP/s": round(tf, 2), "peak": bf16_peak, "peak_name": "bf16 burst",
                    "frac": round(tf / bf16_peak, 4),
                    **roofline_of(2.0 * batch * M * N * K,
                                  2 * batch * M * K + 2 * (1 if shared_B else batch) * K * N + 4 * batch * M * N,
                                  ms, bf16_peak, "tensor")})

    def conv_cfg(name, N, H, W, C, CO, KH, KW, st, pd, iters, prec="bf16"):
        g = PCG32(20 + C + CO)
        if prec == "tf32":
            X = torch.from_numpy(g.uniform_f32((N, H, W, C))).to(dev)
            Wt = torch.from_numpy(g.uniform_f32((KH, KW, C, CO)) * np.float32((KH * KW * C) ** -0.5)).to(dev)
            esz, peak, peak_name = 4, tf32_peak, "bf16 burst / 2 (derived)"
        else:
            X = torch.from_numpy(g.normal_bf16((N, H, W, C)).view(np.int16)).to(dev)
            Wt = torch.from_numpy(g.normal_bf16((KH, KW, C, CO), (KH * KW * C) ** -0.5).view(np.int16)).to(dev)
            esz, peak, peak_name = 2, bf16_peak, "bf16 burst"
        OH, OW = gtg.conv_out_size(H, W, KH, KW, st, pd)
        Y = torch.empty((N, OH, OW, CO), device=dev)

        def call(i):
            rc = gtg.conv2d_nhwc(prec, N, H, W, C, CO, KH, KW, st, st, pd, pd, 1, 1, X.data_ptr(), Wt.data_ptr(),
                                 Y.data_ptr(), None, sh)
            assert rc == gtg.GTG_OK, rc

        ms, ms_best = time_launches(call, iters, stream)
        M, K = N * OH * OW, KH * KW * C
        tf = 2.0 * M * K * CO / (ms * 1e-3) / 1e12
        direct = KH == 1 and KW == 1 and st == 1 and pd == 0
        # the implicit GEMM takes 16-bit layers with whole 64-channel blocks
        # and TF32 layers with whole 32-channel blocks (the bench's window
        # sizes, strides and paddings are all within its limits)
        implicit = not direct and (C % 32 == 0 if prec == "tf32" else (C % 64 == 0 and CO % 8 == 0))
        plan = gtg.plan_conv2d(prec, N, H, W, C, CO, KH, KW, st, st, pd, pd, 1, 1, X.data_ptr(), Wt.data_ptr(),
                               Y.data_ptr())
        kern = (f"CTA pair {plan['bm']}x{plan['bn']}" if plan["cluster"] == 2 else f"{plan['bm']}x{plan['bn']} tiles")
        kern += f", {plan['splits']} K ranges" if plan["splits"] > 1 else ""
        label = ("implicit GEMM" if implicit else ("GEMM on X" if direct else "im2col + GEMM")) + f"; {kern}"
        out.append({"config": name, "path": f"{prec} conv ({label})",
                    "gemm_shape": [M, CO, K], "ms": round(ms, 4), "ms_best": round(ms_best, 4), "TFLOP/s": round(tf, 2), "peak": peak,
                    "peak_name": peak_name, "frac": round(tf / peak, 4),
                    "im2col_bytes": 0 if (direct or implicit) else M * ((K + 7) // 8 * 8) * esz,
                    **roofline_of(2.0 * M * K * CO, esz * (N * H * W * C + KH * KW * C * CO) + 4 * M * CO, ms, peak,
                                  "tensor")})

    for layer in CONV_LAYERS:
        conv_cfg(*layer)
    for layer in CONV_LAYERS_TF32:
        conv_cfg(*layer, prec="tf32")
    torch.cuda.empty_cache()

    batched_cfg("f2: bf16 strided batch 16 x 2048^3", 16, 2048, 2048, 2048, 20)
    batched_cfg("f2: bf16 strided batch 256 x 512x512x512", 256, 512, 512, 512, 50)
    batched_cfg("f2: bf16 strided batch 64 x 1024x1024x256, shared B", 64, 1024, 1024, 256, 50, shared_B=True)
    torch.cuda.empty_cache()

    out.extend(ablation(dev, stream, f32_peak, peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]), l2))

    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    from seeded import PCG32
    for n in (4096, 8192, 16384):
        Av, xv, Xv = gemv_uniform_f32(2, n, n, batch=8)
        nrot = max(2, math.ceil(3 * l2 / (4 * n * n))) if l2 else 2
        As = [torch.from_numpy(Av).to(dev) for _ in range(nrot)]
        X = torch.from_numpy(Xv).to(dev)
        Y = torch.empty((8, n), device=dev)
        layer_bias = torch.from_numpy(PCG32(8).uniform_f32((n,))).to(dev)
        variants = [(1, None), (8, None)] + ([(1, "relu")] if n == 4096 else [])
        for batch, act in variants:
            ep = gtg.epilogue(layer_bias.data_ptr(), act) if act else None

            def call(i, batch=batch, ep=ep):
                st = gtg.gemv_f32_ex(n, n, As[i % nrot].data_ptr(), n, X.data_ptr(), n, Y.data_ptr(), n, batch,
                                     ep, sh)
                assert st == gtg.GTG_OK, st
            ms, ms_best = time_launches(call, 250, stream)
            byt = 4.0 * n * n + batch * 4.0 * (2 * n) + (4.0 * n if act else 0.0)
            gbs = byt / (ms * 1e-3) / 1e9
            name = (f"f1: f32 dense vector {n}x{n}, bias + ReLU" if act else
                    f"2: f32 gemv {n}x{n} batch {batch}")
            out.append({"config": name, "path": "gemv_f32", "shape": [n, n],
                        "batch": batch, "ms": round(ms, 5), "ms_best": round(ms_best, 5), "GB/s": round(gbs, 1), "peak": hbm,
                        "frac": round(gbs / hbm, 4), "buffer_sets": nrot})
        del As, X, Y
        # the same layer with its weights stored in BF16 (half the bytes)
        from seeded import f64_to_bf16_bits
        Ab = f64_to_bf16_bits(Av.astype(np.float64)).view(np.int16)
        nrot = max(2, math.ceil(3 * l2 / (2 * n * n))) if l2 else 2
        As = [torch.from_numpy(Ab).to(dev) for _ in range(nrot)]
        X = torch.from_numpy(Xv).to(dev)
        Y = torch.empty((8, n), device=dev)
        for batch in (1, 8):
            def call(i, batch=batch):
                st = gtg.gemv_bf16(n, n, As[i % nrot].data_ptr(), n, X.data_ptr(), n, Y.data_ptr(), n, batch, sh)
                assert st == gtg.GTG_OK, st
            ms, ms_best = time_launches(call, 250, stream)
            byt = 2.0 * n * n + batch * 4.0 * (2 * n)
            gbs = byt / (ms * 1e-3) / 1e9
            out.append({"config": f"f2: bf16-matrix gemv {n}x{n} batch {batch}", "path": "gemv_bf16",
                        "shape": [n, n], "batch": batch, "ms": round(ms, 5), "ms_best": round(ms_best, 5), "GB/s": round(gbs, 1), "peak": hbm,
                        "frac": round(gbs / hbm, 4), "buffer_sets": nrot})
        del As, X, Y
    torch.cuda.empty_cache()
    return out


def ablation(dev, stream, f32_peak, hbm, l2, iters=0):
    """The pages' own kernel designs beside the library's kernels on the same
    workloads, to test the pages' speed-up claims on this GPU."""
    import torch

    import gemv_tiled_gemm_gb300 as gtg
    from seeded import gemm_uniform_f32, gemv_uniform_f32

    sh = int(stream.cuda_stream)
    out = []
    M = N = K = 1024
    A, B = gemm_uniform_f32(3, M, N, K)
    nrot = max(1, math.ceil(2 * l2 / (3 * 4 * M * N))) if l2 else 1
    sets = [(torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev), torch.empty((M, N), device=dev))
            for _ in range(nrot)]
    times = {}
    for variant in ("naive16", "naive32", "tiled16", "tiled32", "library"):
        def call(i, variant=variant):
            a, b, c = sets[i % nrot]
            if variant == "library":
                st = gtg.gemm_f32(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, sh)
            else:
                st = gtg.gtg_ablation_gemm_f32(variant, M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(),
                                               N, sh)
            assert st == gtg.GTG_OK, st
        times[variant], best = time_launches(call, iters or (10 if variant.startswith("naive") else 30), stream)
        tf = 2.0 * M * N * K / (times[variant] * 1e-3) / 1e12
        out.append({"config": f"f3: f32 gemm 1024^3, {variant}", "path": "ablation" if variant != "library" else "f32",
                    "shape": [M, N, K], "ms": round(times[variant], 4), "ms_best": round(best, 4), "TFLOP/s": round(tf, 2), "peak": f32_peak,
                    "frac": round(tf / f32_peak, 4),
                    "speedup_vs_naive16": round(times["naive16"] / times[variant], 2)})
    del sets
    M = N = 4096
    Av, xv, _ = gemv_uniform_f32(2, M, N, batch=1)
    nrot = max(2, math.ceil(3 * l2 / (4 * M * N))) if l2 else 2
    As = [torch.from_numpy(Av).to(dev) for _ in range(nrot)]
    x = torch.from_numpy(xv).to(dev)
    y = torch.empty(M, device=dev)
    for variant in ("naive", "shared", "library"):
        def call(i, variant=variant):
            if variant == "library":
                st = gtg.gemv_f32(M, N, As[i % nrot].data_ptr(), N, x.data_ptr(), N, y.data_ptr(), M, 1, sh)
            else:
                st = gtg.gtg_ablation_gemv_f32(variant, M, N, As[i % nrot].data_ptr(), N, x.data_ptr(),
                                               y.data_ptr(), sh)
            assert st == gtg.GTG_OK, st
        times[variant], best = time_launches(call, iters or (20 if variant != "library" else 100), stream)
        gbs = (4.0 * M * N + 8.0 * M) / (times[variant] * 1e-3) / 1e9
        out.append({"config": f"f3: f32 gemv 4096^2, {variant}", "path": "ablation" if variant != "library" else "gemv_f32",
                    "shape": [M, N], "ms": round(times[variant], 5), "ms_best": round(best, 5), "GB/s": round(gbs, 1), "peak": hbm,
                    "frac": round(gbs / hbm, 4), "speedup_vs_naive": round(times["naive"] / times[variant], 2)})
    del As
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle

_ORACLE_INPUTS = {}


def _oracle_inputs(rows: int):
    """The first `rows` rows of A and all of B of the 8192^3 BF16 workload,
    widened exactly to FP64 (generated once per process)."""
    import numpy as np

    from seeded import PCG32, bf16_bits_to_f32

    M, N, K = GEMM_SHAPE
    if "B" not in _ORACLE_INPUTS:
        g = PCG32(6)
        g.next_u32(2 * ((M * K + 1) // 2))        # skip all of A
        _ORACLE_INPUTS["B"] = bf16_bits_to_f32(g.normal_bf16((K, N), K ** -0.5)).astype(np.float64)
    if _ORACLE_INPUTS.get("rows", 0) < rows:
        g = PCG32(6)                              # the first rows of A: same draws as the workload
        _ORACLE_INPUTS["A"] = bf16_bits_to_f32(g.normal_bf16((rows, K), K ** -0.5)).astype(np.float64)
        _ORACLE_INPUTS["rows"] = rows
    return _ORACLE_INPUTS["A"][:rows], _ORACLE_INPUTS["B"]


def oracle_gemm_sample(rows: int, threads: int = 0):
    """The FP64 oracle on `rows` rows of the 8192^3 BF16 workload (full N, K)."""
    import oracle

    M, N, K = GEMM_SHAPE
    Af, Bf = _oracle_inputs(rows)
    t0 = time.perf_counter()
    oracle.gemm(Af, Bf, threads=threads)
    return time.perf_counter() - t0, 2.0 * rows * N * K


def cpu_baseline(target_s: float = 10.0):
    import oracle
    cores = oracle.threads_default()
    dt, fl = oracle_gemm_sample(4)
    rows = max(4, min(8192, int(4 * target_s / max(dt, 1e-3))))
    dt, fl = oracle_gemm_sample(rows)
    # the same oracle on one host thread, a ~3 s sample
    dt1, _ = oracle_gemm_sample(1, threads=1)
    rows1 = max(1, min(64, int(3.0 / max(dt1, 1e-3))))
    dt1, fl1 = oracle_gemm_sample(rows1, threads=1)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} rows x 8192 x 8192 of the 8192^3 BF16 GEMM (FP64, with the error magnitude E), "
                      f"{dt:.1f} s", "seconds": round(dt, 2),
            "one_core": {"value": round(fl1 / dt1 / 1e12, 6), "cores": 1,
                         "sample": f"{rows1} rows x 8192 x 8192, {dt1:.1f} s"}}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    import oracle
    cores = oracle.threads_default()
    # each step: the oracle on a slab of rows sized to ~2 s
    dt, fl = oracle_gemm_sample(2)
    rows = max(2, int(2 * 2.0 / max(dt, 1e-3)))
    for _ in range(max(0, args.warmup)):
        oracle_gemm_sample(rows)
        break  # one warm-up pass is enough for a CPU loop; more only lengthens the run
    t_total, f_total = 0.0, 0.0
    for _ in range(args.steps if args.steps <= 20 else 20):
        dt, fl = oracle_gemm_sample(rows)
        t_total += dt
        f_total += fl
    steps = args.steps if args.steps <= 20 else 20
    v = f_total / t_total / 1e12
    sample = f"{rows} rows x 8192 x 8192 of the 8192^3 BF16 GEMM per step (FP64 oracle with E)"
    return {"metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(1000 * t_total / steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "bf16 GEMM M=N=K=8192 (row slab per step)", "gemm_seed": 6,
                       "parallelism": "host threads"},
            "impl": "reference",
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def summary_of(res: dict) -> dict:
    """One [rate, fraction of peak] pair per configuration of the workload
    list (GEMM TFLOP/s, GEMV GB/s) plus the in-step GEMV fractions, printed
    last on the line so that a reader keeping only its tail still has them."""
    out = {"headline bf16 8192^3 in step": [res.get("value"), res.get("roofline", {}).get("frac")]}
    gv = res.get("gemv", {})
    if gv:
        out["in-step gemv 4096^2 b1 / b8 frac"] = [gv.get("roofline", {}).get("frac"), gv.get("batch8_frac")]
    for row in res.get("configs", []):
        name = row.get("config", "")
        keep = name[:1].isdigit() or name.startswith("f2: bf16-matrix gemv 4096") or name.startswith("tf32 8192")
        if not keep:
            continue
        rate = row.get("TFLOP/s", row.get("GB/s"))
        out[name.replace("x4096x4096", "x4096^2").replace(" gemv", "")] = [rate, row.get("frac")]
    return out


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = reference_arm(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    if args.only_gemv is not None:
        print(json.dumps(only_gemv(args.only_gemv, local_rank)), flush=True)
        return 0
    if args.only_conv is not None:
        print(json.dumps(only_conv(args.only_conv, local_rank)), flush=True)
        return 0
    if args.only_gemm is not None:
        print(json.dumps(only_gemm(args.only_gemm, local_rank)), flush=True)
        return 0

    if args.only_ablation:
        import torch
        torch.cuda.set_device(local_rank)
        dev = torch.device("cuda", local_rank)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peaks, _ = load_peaks()
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0
        rows = ablation(dev, torch.cuda.current_stream(), sms * 128 * 2 * 2.070e9 / 1e12,
                        peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]), l2, args.ablation_iters)
        print(json.dumps({"ablation": rows}), flush=True)
        return 0

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        res["summary"] = summary_of(res)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
