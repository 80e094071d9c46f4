"""Benchmark of the NVFP4 W4A4 linear layer with residual compensation.

One step = the whole hot path on one batch of the prefill-shape dense
workload (X [8192, 4096] bf16 with 41 Student-t outlier channels, W [4096,
4096], k = 128 compensated channels):
  1. online NVFP4 quantization of X with a dynamic tensor scale: one
     cooperative kernel (amax phase, grid barrier, quantize phase reading X
     again mostly from L2) that also writes the bf16 residual slice,
  2. the block-scaled W4A4 GEMM on tcgen05 (256 x 256 tiles on CTA pairs)
     with the compensation term fused into the accumulator, bf16 output.
     The quantizer emits the residual divided by the tensor scale, the
     operand form the GEMM consumes without a rescaling pass.
Weight quantization, the compensation weight columns and the channel
calibration are offline (done once, untimed), as in a rollout engine.

Timing: CUDA events on the launching stream around each kernel of every
step; 4 rotating (X, W) sets of 74 MB each (296 MB > the 129 MB L2) so every
step reads its inputs from HBM.  `value` is the layer's throughput
2*M*N*K / (quantize + GEMM time) in TFLOP/s; the GEMM kernel alone is
reported in `roofline` against the FP4 tensor peak and the quantizer in
`components` against HBM bandwidth.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
layer shards by rows with no exchange step), the step time is the max over
ranks and `value` the sum of all ranks' work over that time.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nvfp4_w4a4_gemm_gb300 import workloads as W  # noqa: E402

WORKLOAD = "prefill"
GEMM_KERNEL = "w4a4_gemm_pair_kernel"  # the 256x256 CTA-pair kernel the library dispatches for dense M > 256
N_SETS = 4
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio on GB300
FALLBACK = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


# ------------------------------------------------------------ helpers ----
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        def pick(*keys):
            for k in keys:
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k])
            return None
        hbm = pick("hbm_gbs", "hbm_GBs", "copy_gbs")
        bf = pick("bf16_tflops", "bf16_tflops_burst")
        bfs = pick("bf16_tflops_sustained")
        if hbm and bf:
            return dict(hbm_gbs=hbm, bf16_tflops=bf, bf16_tflops_sustained=bfs or bf, source="measured")
    return dict(FALLBACK, source="fallback")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.rows = []
        self.proc = None
        self.dev = device

    def start(self):
        sel = []
        try:
            bus = torch.cuda.get_device_properties(self.dev).pci_bus_id
            sel = ["-i", f"{bus}"] if bus else []
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                     reasons=sorted(reasons), samples=len(sm))


def git_blob_hash(path):
    """git's blob id of a file (sha1 of 'blob <size>\\0' + content), computed
    without git so it works where the repository has no .git."""
    import hashlib
    with open(path, "rb") as f:
        data = f.read()
    return hashlib.sha1(b"blob %d\0" % len(data) + data).hexdigest()


def gemm_traffic():
    """DRAM bytes per GEMM launch from the committed ncu capture, or None when
    the kernel source changed since the counters were taken."""
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tr_path):
        return None
    with open(tr_path) as f:
        rec = json.load(f).get(GEMM_KERNEL, {}).get(WORKLOAD)
    src = os.path.join(ROOT, "nvfp4_w4a4_gemm_gb300", "csrc", "gemm.cu")
    if not rec or git_blob_hash(src) != rec.get("gemm_cu_blob"):
        return None
    return rec["bytes"]


def dist_setup():
    """One process per GPU under torchrun (NCCL); without a GPU (the CPU tests
    of this host logic) the same ranks meet over gloo."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
        return dist, rank, ws
    return None, 0, 1


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------- our arm -----
def prepare(nv, rank):
    """Offline part: inputs, weight quantization, calibration, comp weights."""
    s = W.SPECS[WORKLOAD]
    dev = torch.device("cuda")
    xc = W.activations(s.M, s.K, s.n_out, s.outlier, s.seed, s.seed + 1000).to(dev)
    chan = nv.nvfp4_calibrate_channels(xc, s.k)
    del xc
    sets = []
    for i in range(N_SETS):
        x = W.activations(s.M, s.K, s.n_out, s.outlier, s.seed, s.seed + 17 * i + 101 * rank).to(dev)
        wt = W.weights_t(s.N, s.K, s.seed + 500 + i + 101 * rank).to(dev)
        qw = nv.nvfp4_quantize(wt)
        w_sel = nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], chan)
        del wt
        sets.append(dict(x=x, qw=qw, w_sel=w_sel))
    M, K, N, k = s.M, s.K, s.N, s.k
    out = dict(codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
               scales=torch.empty(nv.scale_bytes(M, K), dtype=torch.uint8, device=dev),
               resid=torch.empty((M, k), dtype=torch.bfloat16, device=dev),
               ws=torch.empty(nv.load().nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev))
    g_x = torch.empty(1, dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    return s, chan, sets, out, g_x, y


def step(nv, s, chan, st, out, g_x, y, ev=None):
    if ev is not None:
        ev[0].record()
    qx = nv.nvfp4_quantize(st["x"], chan=chan, out=out, g_out=g_x, resid_scaled=True)
    if ev is not None:
        ev[1].record()
    nv.w4a4_gemm_comp(qx, st["qw"], s.N, resid=qx["resid"], w_sel=st["w_sel"], y=y, weights_ready=True)
    if ev is not None:
        ev[2].record()


def run_ours(args):
    from nvfp4_w4a4_gemm_gb300 import binding as nv
    dist, rank, ws = dist_setup()
    nv.load()
    dev = torch.device("cuda")
    s, chan, sets, out, g_x, y = prepare(nv, rank)
    flops = 2.0 * s.M * s.N * s.K
    for i in range(args.warmup):
        step(nv, s, chan, sets[i % N_SETS], out, g_x, y)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # a spin kernel ahead of the timed steps keeps the device busy while the
    # host enqueues them, so the per-kernel events measure device time only
    torch.cuda._sleep(int(2e6) + 200000 * args.steps)
    for i in range(args.steps):
        step(nv, s, chan, sets[i % N_SETS], out, g_x, y, evs[i])
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    clocks = clk.stop()
    st, _ = nv.check_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    t_q = [e[0].elapsed_time(e[1]) for e in evs]
    t_g = [e[1].elapsed_time(e[2]) for e in evs]
    t_step = [a + b for a, b in zip(t_q, t_g)]
    ms_step = max_over_ranks(dist, statistics.mean(t_step), dev)
    ms_med = max_over_ranks(dist, statistics.median(t_step), dev)
    ms_min = max_over_ranks(dist, min(t_step), dev)
    ms_gemm = max_over_ranks(dist, statistics.mean(t_g), dev)
    ms_quant = max_over_ranks(dist, statistics.mean(t_q), dev)

    # ---- e2e: host buffers through the same public calls ----
    # Every step copies its X in from pinned host memory and its Y back out.
    # As a serving engine would, the copies run on their own streams with two
    # device buffers each, so step i's copy-out and step i+1's copy-in overlap
    # step i's kernels; events order buffer reuse.
    n_buf = 2
    x_hosts = [sets[j % N_SETS]["x"].cpu().pin_memory() for j in range(n_buf)]
    y_hosts = [torch.empty((s.M, s.N), dtype=torch.bfloat16).pin_memory() for _ in range(n_buf)]
    x_devs = [torch.empty_like(sets[0]["x"]) for _ in range(n_buf)]
    y_devs = [torch.empty((s.M, s.N), dtype=torch.bfloat16, device=dev) for _ in range(n_buf)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_buf)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_buf)]
    ev_out = [torch.cuda.Event() for _ in range(n_buf)]

    def e2e_run(n):
        for i in range(n):
            b = i % n_buf
            with torch.cuda.stream(s_in):
                if i >= n_buf:
                    s_in.wait_event(ev_cmp[b])  # the kernels that read x_devs[b] are done
                x_devs[b].copy_(x_hosts[b], non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[b])
                if i >= n_buf:
                    s_cmp.wait_event(ev_out[b])  # y_devs[b] has been copied out
                st_b = dict(sets[0])
                st_b["x"] = x_devs[b]
                step(nv, s, chan, st_b, out, g_x, y_devs[b])
                ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                y_hosts[b].copy_(y_devs[b], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps = max(4, args.steps // 2)
    e2e_run(2 * n_buf)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(e2e_steps)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(dist, e0.elapsed_time(e1) / e2e_steps, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    pk = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    gemm_tflops = flops / (ms_gemm * 1e-3) / 1e12
    q_bytes = s.M * s.K * 2 + s.M * s.K // 2 + nv.scale_bytes(s.M, s.K) + s.M * s.k * 2
    quant_gbs = q_bytes / (ms_quant * 1e-3) / 1e9
    value = ws * flops / (ms_step * 1e-3) / 1e12
    traffic = gemm_traffic()
    res = {
        "metric": "W4A4+comp GEMM TFLOPS (% FP4 peak); NVFP4 quantize GB/s (% HBM)",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4-e2m1 x e4m3 block scales, fp32 accumulate, bf16 compensation/output",
        "data": "synthetic (seeded; N(0,1) activations with 1% Student-t(3)x20 outlier channels, N(0,0.02^2) weights)",
        "config": {"workload": "prefill-shape dense linear: X[8192,4096] bf16, W[4096,4096] NVFP4, k=128 "
                               "compensated channels; dynamic-scale NVFP4 quantize + W4A4 GEMM + fused compensation",
                   "M": s.M, "N": s.N, "K": s.K, "k": s.k,
                   "l2": f"inputs rotate over {N_SETS} (X, W) sets = "
                         f"{N_SETS * (s.M * s.K * 2 + s.N * s.K // 2) / 1e6:.0f} MB > L2 129 MB",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"kernel": GEMM_KERNEL, "bound": "tensor", "achieved": round(gemm_tflops, 1),
                     "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(gemm_tflops / fp4_peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{pk['source']}: bf16 {pk['bf16_tflops']} TFLOP/s x {FP4_OVER_BF16:g} (nominal FP4/BF16)",
                     "algorithmic": "2*M*N*K per launch (compensation FLOPs excluded, its time included)"},
        "components": {
            "gemm_ms": round(ms_gemm, 4), "gemm_tflops": round(gemm_tflops, 1),
            "gemm_tflops_incl_comp": round((flops + 2.0 * s.M * s.N * s.k) / (ms_gemm * 1e-3) / 1e12, 1),
            "step_ms_median": round(ms_med, 4), "step_ms_min": round(ms_min, 4),
            "quantize_ms": round(ms_quant, 4), "quantize_gbs": round(quant_gbs, 1),
            "quantize_frac_hbm": round(quant_gbs / pk["hbm_gbs"], 4),
            "quantize_bytes": q_bytes, "hbm_peak_gbs": pk["hbm_gbs"],
            "quantize_note": "dynamic tensor scale, one cooperative launch (amax phase, grid barrier, quantize "
                             "phase) plus a 4-byte barrier reset; bytes = X read once + codes + scales + residual; "
                             "inside the step the quantizer also absorbs the write-back of the previous GEMM's 64 MB "
                             "bf16 output from L2",
        },
        "e2e": {"value": round(ws * flops / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": s.M * s.K * 2, "d2h_bytes_per_step": s.M * s.N * 2,
                "ms_per_step": round(ms_e2e, 4),
                "pipelining": "X copy-in, the step's kernels and Y copy-out on three streams, two buffers each"},
        "gpu_launches": 2 * args.steps,  # per step: nvfp4_quant_kernel (cooperative) + w4a4_gemm_pair_kernel
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if not args.no_workloads:
        res["components"].update(prefill_components(nv, pk, s, chan, sets))
        res["workloads"] = other_workloads(nv, pk)
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(s, sample_rows=args.cpu_rows or 4096, steps=2)
    print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------- prefill components alone ----
def prefill_components(nv, pk, s, chan, sets, steps=20):
    """The prefill kernels timed one at a time after an L2 flush: the
    quantizer with the dynamic scale (the step's form) and with a static
    scale, and the GEMM on already-quantized operands."""
    dev = torch.device("cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    M, K, N, k = s.M, s.K, s.N, s.k
    out = dict(codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
               scales=torch.empty(nv.scale_bytes(M, K), dtype=torch.uint8, device=dev),
               resid=torch.empty((M, k), dtype=torch.bfloat16, device=dev),
               ws=torch.empty(nv.load().nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev))
    g_out = torch.empty(1, dtype=torch.float32, device=dev)
    g_static = nv.nvfp4_quantize(sets[0]["x"], chan=chan)["g"].clone()   # a calibrated static scale
    q_bytes = M * K * 2 + M * K // 2 + nv.scale_bytes(M, K) + M * k * 2
    it = [0]

    def quant(g):
        def f():
            it[0] += 1
            nv.nvfp4_quantize(sets[it[0] % N_SETS]["x"], g=g, chan=chan, out=out, g_out=g_out, resid_scaled=True)
        return f
    ms_dyn = _time_steps(quant(None), steps, flush, "prefill_quantize_dynamic")
    ms_st = _time_steps(quant(g_static), steps, flush, "prefill_quantize_static")
    qs = [nv.nvfp4_quantize(st["x"], chan=chan, resid_scaled=True) for st in sets]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def gemm():
        it[0] += 1
        i = it[0] % N_SETS
        nv.w4a4_gemm_comp(qs[i], sets[i]["qw"], N, resid=qs[i]["resid"], w_sel=sets[i]["w_sel"], y=y,
                          weights_ready=True)
    ms_g = _time_steps(gemm, steps, flush, "prefill_gemm")
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    tf = 2.0 * M * N * K / (ms_g * 1e-3) / 1e12
    comp8 = comp_fp8_components(nv, pk, s, chan, sets, qs, flush, steps)
    comp8["comp_overhead_bf16"] = round(ms_g / comp8["gemm_k0_ms"] - 1.0, 4)
    return {"comp_fp8": comp8, "alone_clean_l2": {
        "quantize_dynamic_ms": round(ms_dyn, 4),
        "quantize_dynamic_gbs": round(q_bytes / (ms_dyn * 1e-3) / 1e9, 1),
        "quantize_dynamic_frac_hbm": round(q_bytes / (ms_dyn * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
        "quantize_static_ms": round(ms_st, 4),
        "quantize_static_gbs": round(q_bytes / (ms_st * 1e-3) / 1e9, 1),
        "quantize_static_frac_hbm": round(q_bytes / (ms_st * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
        "gemm_ms": round(ms_g, 4), "gemm_tflops": round(tf, 1), "gemm_frac_fp4_peak": round(tf / fp4_peak, 4),
        "note": "each kernel alone after an L2 flush (write + read of 256 MB); static scale = the dynamic "
                "scale of a previous batch passed in (one read of X, no grid barrier)"}}


def comp_fp8_components(nv, pk, s, chan, sets, qs, flush, steps):
    """The quantized-residual (FP8 E4M3) compensation on the prefill
    workload: the dynamic-scale quantizer writing the E4M3 residual, the GEMM
    with the FP8 term, the same GEMM without compensation (k = 0, the
    baseline of both terms' overhead), each alone after an L2 flush; and the
    whole step (quantize + GEMM, inputs rotating, no flush) with the BF16 and
    with the FP8 term, timed the same way."""
    dev = torch.device("cuda")
    M, K, N, k = s.M, s.K, s.N, s.k
    w8 = [nv.nvfp4_prepare_comp_weights(st["qw"]["codes"], st["qw"]["scales"], chan, flags=nv.COMP_W_DEQ_FP8)
          for st in sets]
    out8 = dict(codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                scales=torch.empty(nv.scale_bytes(M, K), dtype=torch.uint8, device=dev),
                resid=torch.empty((M, k), dtype=torch.uint8, device=dev),
                ws=torch.empty(nv.load().nvfp4_quantize_workspace_bytes(), dtype=torch.uint8, device=dev))
    out16 = dict(out8, resid=torch.empty((M, k), dtype=torch.bfloat16, device=dev))
    g_out = torch.empty(1, dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    it = [0]

    def quant8():
        it[0] += 1
        nv.nvfp4_quantize(sets[it[0] % N_SETS]["x"], chan=chan, out=out8, g_out=g_out, resid_fp8=True)
    ms_q8 = _time_steps(quant8, steps, flush, "prefill_quantize_dynamic_fp8")
    q8 = [nv.nvfp4_quantize(st["x"], chan=chan, resid_fp8=True) for st in sets]

    def gemm8():
        it[0] += 1
        i = it[0] % N_SETS
        nv.w4a4_gemm_comp(q8[i], sets[i]["qw"], N, resid=q8[i]["resid"], w_sel=w8[i], y=y, weights_ready=True)
    ms_g8 = _time_steps(gemm8, steps, flush, "prefill_gemm_fp8")

    def gemm0():
        it[0] += 1
        i = it[0] % N_SETS
        nv.w4a4_gemm_comp(qs[i], sets[i]["qw"], N, y=y, weights_ready=True)
    ms_g0 = _time_steps(gemm0, steps, flush, "prefill_gemm_k0")

    def step_with(fp8):
        def f():
            it[0] += 1
            i = it[0] % N_SETS
            qx = nv.nvfp4_quantize(sets[i]["x"], chan=chan, out=out8 if fp8 else out16, g_out=g_out,
                                   resid_scaled=True, resid_fp8=fp8)
            nv.w4a4_gemm_comp(qx, sets[i]["qw"], N, resid=qx["resid"], w_sel=w8[i] if fp8 else sets[i]["w_sel"],
                              y=y, weights_ready=True)
        return f
    ms_s16 = _time_steps(step_with(False), steps, None, "prefill_step_bf16_comp")
    ms_s8 = _time_steps(step_with(True), steps, None, "prefill_step_fp8_comp")
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    flops = 2.0 * M * N * K
    return {
        "quantize_dynamic_fp8_ms": round(ms_q8, 4),
        "gemm_fp8_ms": round(ms_g8, 4),
        "gemm_fp8_tflops": round(flops / (ms_g8 * 1e-3) / 1e12, 1),
        "gemm_fp8_frac_fp4_peak": round(flops / (ms_g8 * 1e-3) / 1e12 / fp4_peak, 4),
        "gemm_k0_ms": round(ms_g0, 4),
        "comp_overhead_fp8": round(ms_g8 / ms_g0 - 1.0, 4),
        "step_bf16_comp_ms": round(ms_s16, 4),
        "step_fp8_comp_ms": round(ms_s8, 4),
        "step_fp8_comp_tflops": round(flops / (ms_s8 * 1e-3) / 1e12, 1),
        "note": "quantized-residual compensation: E4M3 residual (pre-scaled by 1/g_a) and E4M3 weight rows "
                "(x 2^-3), 128-channel tiles on the FP8 tensor-core kinds; GEMMs and the quantizer alone after an "
                "L2 flush; the two steps (quantize + GEMM) on rotating inputs without a flush, timed the same way; "
                "overheads against the same GEMM with k = 0",
    }


# ------------------------------------------- the other four workloads ----
def _time_steps(fn, steps, flush, name=None):
    """Mean device time (ms) of `fn` over `steps` runs.  Between runs, outside
    the timed window, a buffer larger than the L2 is written and then read
    back: the write flushes the L2, the read writes its dirty lines back to
    HBM, so a step does not start behind 129 MB of pending write-backs.
    flush=None: no flush (the step's own inputs are larger than the L2).
    `name` labels the warm-up and timed runs with an NVTX range, so a
    profiler can select one workload's launches (ncu --nvtx --nvtx-include
    "<name>/")."""
    if name is not None:
        torch.cuda.nvtx.range_push(name)
        try:
            return _time_steps(fn, steps, flush)
        finally:
            torch.cuda.nvtx.range_pop()
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
            flush.view(torch.float32).sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2000000)  # keeps the device busy while the host enqueues the step
        e0.record()
        fn()
        e1.record()
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ts)


def other_workloads(nv, pk, steps=10):
    """Decode, MoE and MXFP4 workloads: one step each = the kernels of that
    path on one batch (dynamic-scale quantize + GEMM)."""
    dev = torch.device("cuda")
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}

    # decode: X[16,4096] x W[4096,14336], k=64 (HBM-bound on the weights).
    # Six layers' weights (6 x 35 MB > L2) are used in turn, as successive
    # layers of a model would: every step streams its weights from HBM, with
    # no flush between steps (X, the channel list and the code stay in L2).
    s = W.SPECS["decode"]
    d = W.dense_inputs("decode")
    x = d["x"].to(dev)
    chan = nv.nvfp4_calibrate_channels(W.dense_inputs("decode", True, False)["x"].to(dev), s.k)
    wt0 = d["wt"].to(dev)
    layers = []
    for i in range(6):
        wt = wt0 if i == 0 else torch.roll(wt0, shifts=977 * i, dims=0)
        qw = nv.nvfp4_quantize(wt)
        layers.append((qw, nv.nvfp4_prepare_comp_weights(qw["codes"], qw["scales"], chan)))
        del wt
    del wt0
    y = torch.empty((s.M, s.N), dtype=torch.bfloat16, device=dev)
    step_i = [0]

    def layer():
        step_i[0] += 1
        return layers[step_i[0] % len(layers)]

    def dec():
        qw, ws = layer()
        nv.w4a4_decode_linear(x, qw, s.N, chan=chan, w_sel=ws, y=y, weights_ready=True)

    def dec_two():
        qw, ws = layer()
        qx = nv.nvfp4_quantize(x, chan=chan, resid_scaled=True)
        nv.w4a4_gemm_comp(qx, qw, s.N, resid=qx["resid"], w_sel=ws, y=y, weights_ready=True)
    ms = _time_steps(dec, steps, None, "decode_layer")
    ms_two = _time_steps(dec_two, steps, None, "decode_two_launch")
    ms_flush = _time_steps(dec, steps, flush, "decode_layer_flushed")

    def dec_seq():
        for _ in range(len(layers)):
            dec()
    # the six layers back to back, as a model runs them: each launch still
    # waits for the previous one to finish before it reads X (programmatic
    # dependent launch), only its prologue overlaps the previous layer's tail
    ms_seq = _time_steps(dec_seq, steps, None, "decode_layer_sequence") / len(layers)
    qw, ws = layers[0]
    byts = qw["codes"].numel() + qw["scales"].numel() + ws.numel() * 2 + x.numel() * 2 + y.numel() * 2
    out["decode"] = {"shape": "X[16,4096] x W[4096,14336], k=64", "ms_per_step": round(ms, 4),
                     "tflops": round(2.0 * s.M * s.N * s.K / (ms * 1e-3) / 1e12, 2),
                     "gbs": round(byts / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                     "bytes_per_step": byts, "bound": "hbm",
                     "two_launch_ms": round(ms_two, 4), "after_l2_flush_ms": round(ms_flush, 4),
                     "per_layer_in_sequence_ms": round(ms_seq, 4),
                     "note": "one launch (w4a4_decode_linear): clusters of 4 CTAs quantize X (dynamic scale) "
                             "into shared memory, the swapped-operand GEMM with compensation streams the weights; "
                             "weights of 6 layers used in turn (> L2); two_launch_ms = quantize kernel + GEMM "
                             "kernel on the same rotation; after_l2_flush_ms = the one launch after a 256 MB "
                             "L2 flush (code and X also cold); per_layer_in_sequence_ms = the six layers launched "
                             "back to back between one event pair, divided by six (each layer waits for the "
                             "previous one before reading X; only launch and prologue overlap)"}
    del layers, x, y

    # MoE: 4096 tokens top-8 of 128 experts; gate/up [2048->1536] and down [768->2048], k=32 per expert
    s = W.SPECS["moe"]
    dm = W.moe_inputs()
    dc = W.moe_inputs(calibration=True, with_weights=False)
    offs = dm["offsets"].to(dev)
    E = s.experts
    res = {}
    tot_ms, tot_flops, tot_bytes = 0.0, 0.0, 0
    tok_rows = dm["token_of_row"].to(torch.int32).to(dev)
    for which, xk, wk in (("gate_up", "x_gate_up", "wt_gate_up"), ("down", "x_down", "wt_down")):
        xg = dm[xk].to(dev)
        K = xg.shape[1]
        # gate/up reads its routed rows straight from the token rows; the
        # down input is per routed row already
        x_in = dm["x_tokens"].to(dev) if which == "gate_up" else xg
        # per-expert channel sets by residual variance on the calibration
        # batch's rows routed to each expert
        chan = nv.nvfp4_calibrate_channels(dc[xk].to(dev), s.k, offsets=dc["offsets"].to(dev))
        codes, scales, gs = [], [], []
        for e in range(E):
            q = nv.nvfp4_quantize(dm[wk][e].to(dev))
            codes.append(q["codes"]); scales.append(q["scales"]); gs.append(q["g"])
        b_codes, b_scales, g_b = torch.stack(codes), torch.cat(scales), torch.cat(gs)
        del codes, scales
        N = b_codes.shape[1]
        w_sel = nv.nvfp4_prepare_comp_weights(b_codes, b_scales, chan, E=E)
        yg = torch.empty((xg.shape[0], N), dtype=torch.bfloat16, device=dev)

        def quantize_x():
            if which == "gate_up":
                return nv.nvfp4_quantize_grouped_gather(x_in, tok_rows, offs, chan, resid_scaled=True)
            return nv.nvfp4_quantize_grouped(xg, offs, chan, resid_scaled=True)

        def moe():
            qx = quantize_x()
            nv.w4a4_grouped_gemm_comp(qx, offs, b_codes, b_scales, g_b, N, resid=qx["resid"], w_sel=w_sel, y=yg,
                                      weights_ready=True)
        ms = _time_steps(moe, steps, flush, "moe_" + which)
        qfix = quantize_x()

        def moe_gemm():
            nv.w4a4_grouped_gemm_comp(qfix, offs, b_codes, b_scales, g_b, N, resid=qfix["resid"], w_sel=w_sel,
                                      y=yg, weights_ready=True)
        ms_g = _time_steps(moe_gemm, steps, flush, "moe_" + which + "_gemm")
        flops = 2.0 * xg.shape[0] * N * K
        byts = (b_codes.numel() + b_scales.numel() + w_sel.numel() * 2 + x_in.numel() * 2 + yg.numel() * 2)
        res[which] = {"ms_per_step": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                      "gbs": round(byts / (ms * 1e-3) / 1e9, 1), "gemm_alone_ms": round(ms_g, 4),
                      "quantize_ms": round(ms - ms_g, 4)}
        tot_ms += ms; tot_flops += flops; tot_bytes += byts
        del xg, x_in, b_codes, b_scales, g_b, w_sel, yg
    out["moe"] = {"shape": "4096 tokens x top-8 of 128 experts, hidden 2048, gate/up 1536, down 2048, k=32/expert",
                  "ms_per_step": round(tot_ms, 4), "tflops": round(tot_flops / (tot_ms * 1e-3) / 1e12, 1),
                  "frac_fp4_peak": round(tot_flops / (tot_ms * 1e-3) / 1e12 / fp4_peak, 4),
                  "gbs": round(tot_bytes / (tot_ms * 1e-3) / 1e9, 1),
                  "frac_hbm": round(tot_bytes / (tot_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                  "bytes_per_step": tot_bytes, "per_projection": res,
                  # attainable = min(FP4 peak, arithmetic intensity x HBM bandwidth): these layers sit
                  # below the ridge, so their ceiling is the memory one
                  "attainable_tflops": round(min(fp4_peak, tot_flops / tot_bytes * pk["hbm_gbs"] / 1e3), 1),
                  "frac_attainable": round((tot_flops / (tot_ms * 1e-3) / 1e12)
                                           / min(fp4_peak, tot_flops / tot_bytes * pk["hbm_gbs"] / 1e3), 4),
                  "note": "each projection: grouped dynamic-scale quantize + grouped GEMM with compensation "
                          "(gate/up quantizes its routed rows straight from the 4096 token rows through the "
                          "routing table, so x bytes = the token rows); channel sets calibrated per expert "
                          "(residual variance on the calibration batch's rows routed to that expert)"}
    out["moe"]["fused_layer"] = moe_fused_layer(nv, pk, flush, steps)
    del dm

    # MXFP4: X[8192,5120] x W[5120,5120], 32-blocks, decomposition statistics
    s = W.SPECS["mxfp4"]
    d = W.dense_inputs("mxfp4")
    x, wt = d["x"].to(dev), d["wt"].to(dev)
    qw = nv.mxfp4_quantize(wt)
    y = torch.empty((s.M, s.N), dtype=torch.bfloat16, device=dev)
    box = {}

    def mx():
        qx = nv.mxfp4_quantize(x, stats=True)
        box["q"] = qx
        nv.w4a4_gemm_comp(dict(codes=qx["codes"], scales=qx["scales"]), dict(codes=qw["codes"], scales=qw["scales"]),
                          s.N, fmt=nv.FMT_MXFP4, y=y, weights_ready=True)
    ms = _time_steps(mx, steps, flush, "mxfp4_step")
    ms_q = _time_steps(lambda: nv.mxfp4_quantize(x, stats=True), steps, flush, "mxfp4_quantize")
    qfix = nv.mxfp4_quantize(x)

    def mx_gemm():
        nv.w4a4_gemm_comp(dict(codes=qfix["codes"], scales=qfix["scales"]),
                          dict(codes=qw["codes"], scales=qw["scales"]), s.N, fmt=nv.FMT_MXFP4, y=y,
                          weights_ready=True)
    ms_g = _time_steps(mx_gemm, steps, flush, "mxfp4_gemm")
    n_el, n_blk = s.M * s.K, s.M * s.K // 32
    q_bytes = n_el * 2 + n_el // 2 + nv.mx_scale_bytes(s.M, s.K) + n_blk * 17   # X + codes + E8M0 + stats/dead
    gf = 2.0 * s.M * s.N * s.K
    out["mxfp4"] = {"shape": "X[8192,5120] x W[5120,5120], MXFP4 + per-block decomposition", "ms_per_step": round(ms, 4),
                    "tflops": round(gf / (ms * 1e-3) / 1e12, 1),
                    "frac_fp4_peak": round(gf / (ms * 1e-3) / 1e12 / fp4_peak, 4),
                    "quantize_decomposition_ms": round(ms_q, 4),
                    "quantize_decomposition_gbs": round(q_bytes / (ms_q * 1e-3) / 1e9, 1),
                    "quantize_decomposition_frac_hbm": round(q_bytes / (ms_q * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                    "gemm_ms": round(ms_g, 4), "gemm_tflops": round(gf / (ms_g * 1e-3) / 1e12, 1),
                    "gemm_frac_fp4_peak": round(gf / (ms_g * 1e-3) / 1e12 / fp4_peak, 4)}
    out["mxfp4"]["corrected"] = mxfp4_corrected(nv, s, x, wt, qfix, qw, y, flush, steps, fp4_peak)
    del qw, x, wt, y, box

    # trainer-side fake quantization (asymmetric W4A16 QAT) of a layer's
    # weights, emitting the rollout's packed codes and scales in the same pass
    s = W.SPECS["decode"]
    wq = W.dense_inputs("decode")["wt"].to(dev)
    w_out = torch.empty_like(wq)

    def qdq():
        nv.nvfp4_qdq(wq, with_codes=True, out=w_out)
    ms = _time_steps(qdq, steps, flush, "qdq")
    n_el = wq.numel()
    byts = n_el * 2 + n_el * 2 + n_el // 2 + nv.load().nvfp4_scale_bytes(s.N, s.K)
    out["qdq"] = {"shape": "W^T[14336,4096] bf16 -> bf16 QDQ + NVFP4 codes/scales, dynamic tensor scale",
                  "ms_per_step": round(ms, 4), "gbs": round(byts / (ms * 1e-3) / 1e9, 1),
                  "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4), "bytes_per_step": byts,
                  "bound": "hbm",
                  "note": "bytes = W read once + QDQ written + codes + scales; one cooperative launch whose amax "
                          "phase reads W a second time (not counted)"}
    return out


def mxfp4_corrected(nv, s, x, wt, qx_plain, qw_plain, y, flush, steps, fp4_peak, k=64):
    """The MXFP4 workload with the decomposition paper's two corrections:
    Outlier Fallback on k channels (chosen offline by the channel calibration
    on a calibration batch) and row macro-block scales, on both operands.
    Times the corrected quantize (row-scale pass + quantizer with the
    decomposition statistics), the corrected GEMM (row scales in the
    epilogue, the fallback term as a BF16 MMA stream) and the whole step;
    reports the relative Frobenius error of the plain and the corrected GEMM
    against the fp32 product of the bf16 inputs (a library matmul, outside
    the timed region)."""
    dev = x.device
    xc = W.dense_inputs("mxfp4", calibration=True, with_weights=False)["x"].to(dev)
    ch = torch.sort(nv.nvfp4_calibrate_channels(xc, k)).values.contiguous()
    del xc
    qwc = nv.mxfp4_quantize(wt, chan=ch, macro=True)

    def step():
        qx = nv.mxfp4_quantize(x, stats=True, chan=ch, macro=True)
        nv.w4a4_gemm_comp(qx, qwc, s.N, resid=qx["fb"], w_sel=qwc["fb"], fmt=nv.FMT_MXFP4, y=y, weights_ready=True)
    ms = _time_steps(step, steps, flush, "mxfp4_corrected_step")
    ms_q = _time_steps(lambda: nv.mxfp4_quantize(x, stats=True, chan=ch, macro=True), steps, flush,
                       "mxfp4_corrected_quantize")
    qxc = nv.mxfp4_quantize(x, chan=ch, macro=True)

    def gemm():
        nv.w4a4_gemm_comp(qxc, qwc, s.N, resid=qxc["fb"], w_sel=qwc["fb"], fmt=nv.FMT_MXFP4, y=y, weights_ready=True)
    ms_g = _time_steps(gemm, steps, flush, "mxfp4_corrected_gemm")
    ref = x.float() @ wt.float().t()
    gemm()
    err_c = float((y.float() - ref).norm() / ref.norm())
    nv.w4a4_gemm_comp(dict(codes=qx_plain["codes"], scales=qx_plain["scales"]),
                      dict(codes=qw_plain["codes"], scales=qw_plain["scales"]), s.N, fmt=nv.FMT_MXFP4, y=y)
    err_p = float((y.float() - ref).norm() / ref.norm())
    del ref
    gf = 2.0 * s.M * s.N * s.K
    return {"k_fallback": k, "ms_per_step": round(ms, 4), "tflops": round(gf / (ms * 1e-3) / 1e12, 1),
            "quantize_decomposition_ms": round(ms_q, 4),
            "gemm_ms": round(ms_g, 4), "gemm_tflops": round(gf / (ms_g * 1e-3) / 1e12, 1),
            "gemm_frac_fp4_peak": round(gf / (ms_g * 1e-3) / 1e12 / fp4_peak, 4),
            "rel_error_plain": round(err_p, 5), "rel_error_corrected": round(err_c, 5),
            "note": "Outlier Fallback (k channels leave both FP4 operands, multiplied in BF16) + row macro-block "
                    "scales (m = significand of RN(rowmax/6), applied in the GEMM epilogue); quantize = row-scale "
                    "pass + quantizer with statistics; errors: ||Y - X W||_F / ||X W||_F against the fp32 product "
                    "of the bf16 inputs"}


def moe_fused_layer(nv, pk, flush, steps):
    """The whole MoE FFN on the routed rows with both fused epilogues:
    grouped dynamic-scale quantize of x, gate/up GEMM with SwiGLU and the down
    input's static-scale NVFP4 quantize in its epilogue, down GEMM with the
    routing-weighted combine into fp32 token rows (zeroed first)."""
    dev = torch.device("cuda")
    s = W.SPECS["moe"]
    d = W.moe_inputs()
    dc = W.moe_inputs(calibration=True, with_weights=False)
    E, inter, hidden = s.experts, s.inter, s.hidden
    offs = d["offsets"].to(dev)
    x = d["x_tokens"].to(dev)
    rows = d["x_gate_up"].shape[0]
    chan = nv.nvfp4_calibrate_channels(dc["x_gate_up"].to(dev), s.k, offsets=dc["offsets"].to(dev))
    h_chan = nv.nvfp4_calibrate_channels(dc["x_down"].to(dev), s.k, offsets=dc["offsets"].to(dev))

    def experts(wt):
        qs = [nv.nvfp4_quantize(wt[e].to(dev)) for e in range(E)]
        return torch.stack([q["codes"] for q in qs]), torch.cat([q["scales"] for q in qs]), torch.cat([q["g"] for q in qs])
    gu_codes, gu_scales, gu_g = experts(nv.interleave_gate_up_rows(d["wt_gate_up"]))
    gu_sel = nv.nvfp4_prepare_comp_weights(gu_codes, gu_scales, chan, E=E)
    dn_codes, dn_scales, dn_g = experts(d["wt_down"])
    dn_sel = nv.nvfp4_prepare_comp_weights(dn_codes, dn_scales, h_chan, E=E)
    # static scale of h: the dynamic scale of the calibration batch's h
    qc = nv.nvfp4_quantize_grouped(dc["x_gate_up"].to(dev), dc["offsets"].to(dev), chan, resid_scaled=True)
    hc = nv.w4a4_grouped_gemm_swiglu_quant(qc, dc["offsets"].to(dev), gu_codes, gu_scales, gu_g, 2 * inter,
                                           torch.ones(1, device=dev), h_chan, resid=qc["resid"], w_sel=gu_sel,
                                           with_h=True)["h"]
    g_h = nv.nvfp4_quantize(hc)["g"]
    del qc, hc
    tok = d["token_of_row"].to(torch.int32).to(dev)
    w_row = d["route_weight"].to(dev)
    out = torch.empty((s.tokens, hidden), dtype=torch.float32, device=dev)

    def layer():
        qx = nv.nvfp4_quantize_grouped_gather(x, tok, offs, chan, resid_scaled=True)
        qh = nv.w4a4_grouped_gemm_swiglu_quant(qx, offs, gu_codes, gu_scales, gu_g, 2 * inter, g_h, h_chan,
                                               resid=qx["resid"], w_sel=gu_sel, h_resid_scaled=True,
                                               weights_ready=True)
        out.zero_()
        nv.w4a4_grouped_gemm_combine(qh, offs, dn_codes, dn_scales, dn_g, hidden, tok, w_row, s.tokens,
                                     resid=qh["resid"], w_sel=dn_sel, out=out, weights_ready=True)
    ms = _time_steps(layer, steps, flush, "moe_fused_layer")
    flops = 2.0 * rows * (2 * inter) * hidden + 2.0 * rows * hidden * inter
    byts = (gu_codes.numel() + gu_scales.numel() + gu_sel.numel() * 2 + dn_codes.numel() + dn_scales.numel()
            + dn_sel.numel() * 2 + x.numel() * 2 + out.numel() * 4)
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    att = min(fp4_peak, flops / byts * pk["hbm_gbs"] / 1e3)
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms_per_step": round(ms, 4), "tflops": round(tf, 1), "frac_fp4_peak": round(tf / fp4_peak, 4),
            "gbs": round(byts / (ms * 1e-3) / 1e9, 1), "bytes_per_step": byts,
            "attainable_tflops": round(att, 1), "frac_attainable": round(tf / att, 4),
            "note": "one step = the whole FFN on 32768 routed rows: grouped dynamic-scale quantize of the routed "
                    "rows read from the 4096 token rows x through the routing table; gate/up "
                    "GEMM with SwiGLU + static-scale NVFP4 quantize of h (with its residual slice) in the "
                    "epilogue; zeroing of the fp32 output; down GEMM with the routing-weighted combine into "
                    "token rows in the epilogue (fp32 vector atomics). Bytes = weights + compensation columns + x "
                    "read + fp32 output; the gate/up output and h never reach memory as bf16"}


# ------------------------------------------------------ the oracle arm ----
def cpu_baseline(s, sample_rows=4096, steps=2):
    """Time the CPU oracle (as it stands) on a bounded sample of the workload:
    the per-batch part (quantize `sample_rows` rows of X with the residual
    slice + the fp64 reference GEMM with compensation against all N outputs);
    weight quantization is offline on both arms and not timed."""
    from oracle import calib, gemm as og, nvfp4 as onv
    x = W.activations(sample_rows, s.K, s.n_out, s.outlier, s.seed, s.seed + 2000).float().numpy()
    xc = W.activations(min(s.M, 2048), s.K, s.n_out, s.outlier, s.seed, s.seed + 1000).float().numpy()
    chan = calib.calibrate(xc, s.k).astype(np.int64)
    wt = W.weights_t(s.N, s.K, s.seed + 500).float().numpy()
    qw = onv.quantize(wt)
    b = onv.dequantize(qw["codes"], qw["sigma"], qw["g"])
    w_sel = og.comp_weight_rows(qw, chan)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        qx = onv.quantize(x, chan=chan)
        a = onv.dequantize(qx["codes"], qx["sigma"], qx["g"])
        og.reference(a, b, qx["resid"], w_sel)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    flops = 2.0 * sample_rows * s.N * s.K
    try:
        threads = len(os.sched_getaffinity(0))
    except AttributeError:
        threads = os.cpu_count()
    return {"value": round(flops / t / 1e12, 5), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{sample_rows} of {s.M} rows of the prefill workload: NVFP4 quantize with residual slice "
                      f"+ fp64 reference GEMM with compensation vs all {s.N} outputs (numpy; BLAS threads = "
                      f"host cores); weight quantization offline", "seconds": round(t, 3)}


def run_reference(args):
    dist, rank, ws = dist_setup()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    s = W.SPECS[WORKLOAD]
    rows = args.cpu_rows or 2048
    # the oracle keeps no state between steps, so warm-up steps are not run;
    # every timed step is one bounded sample of the batch
    cb = cpu_baseline(s, sample_rows=rows, steps=max(1, args.steps))
    ms = cb["seconds"] * 1e3   # measured time of one timed step (one sample of `rows` rows)
    res = {
        "impl": "reference",
        "metric": "W4A4+comp GEMM TFLOPS (% FP4 peak); NVFP4 quantize GB/s (% HBM)",
        "value": cb["value"], "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
        "config": {"workload": "prefill-shape dense linear: X[8192,4096] bf16, W[4096,4096] NVFP4, k=128 "
                               "compensated channels", "sample_rows_per_step": rows,
                   "step": f"one step = quantize {rows} of the {s.M} rows + fp64 reference GEMM vs all outputs; "
                           "ms_per_step is that measured sample time, value its TFLOP/s"},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="oracle sample rows (default 4096 for cpu_baseline, 2048 per reference step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the decode / MoE / MXFP4 measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
