"""Benchmark: FP8 prefill linear layer on one GB300 (or N independent replicas).

One step = the hot path over one batch:
  quantize X bf16 [4096 x 4096] -> E4M3 with 1x128 tile scales (dynamic)
  block-scaled GEMM vs W E4M3 [14336 x 4096] with 128x128 block scales
  (weights quantized once, offline, and resident) -> Out bf16 [4096 x 14336].
value = 2*M*N*K / step time (TFLOP/s), summed over ranks. L2 is flushed
(256 MB write, then 256 MB read) between timed steps; the flush is outside the
per-step events.

Besides the headline, the JSON line carries per-kernel measurements of the
other workloads of the same path (quantizer sweep, decode GEMMs, MXFP8 GEMM),
each against its roofline, unless --headline-only is given.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the reference arm of this build: there is no other implementation).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s (% of 4.5 PF); quantize GB/s (% of HBM peak)"
M, N, K = 4096, 14336, 4096
WORKLOAD = ("prefill FP8 linear: X bf16 4096x4096 -> E4M3 1x128 tile scales (dynamic), "
            "W E4M3 14336x4096 128x128 block scales (offline), Out bf16 4096x14336")
NOMINAL_FP8_PFLOPS = 4.5
# FP4 peak over FP8 peak: "Low precision: FP8, FP4, and microscaling" gives 4.5 and
# 9 PFLOPS dense for FP8 and FP4 on B200 (ratio 2); the hardware table for GB300
# lists 13.5 PF dense FP4, which the NVFP4 line reports beside it
FP4_OVER_FP8 = 2.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def code_digest(text: str) -> str:
    """sha256 of a C++/CUDA source with its comments, indentation and blank lines removed:
    it changes whenever the code does, and not when only a comment does."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.strip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's source file has
    the same code (comments aside) as when the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        src = os.path.join(ROOT, "fp8_block_scaled_04_gb300", "csrc", rec["source"])
        with open(src) as f:
            digest = code_digest(f.read())
        return float(rec["bytes_per_launch"]) if digest == rec["code_sha256"] else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


def make_l2_flush(dev):
    """L2 flush between timed steps: write 256 MB (twice the L2), then read
    another 256 MB so the write's dirty lines are written back before the next
    timed kernel (otherwise an HBM-bound kernel pays for the flush's
    write-back). Both run outside the timed events."""
    import torch

    wbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rbuf = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        wbuf.zero_()
        rbuf.sum()

    return flush


def hold_gpu(cycles: int = 200_000):
    """Keep the GPU busy (~0.1 ms spin) so that the launches recorded after this
    are already queued when their start event runs: host launch latency stays
    out of the per-kernel event times (the e2e measurement keeps it)."""
    import torch

    torch.cuda._sleep(cycles)


# --------------------------------------------------------------------- ranks
def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank number over all ranks (identity with one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time (units per second)."""
    return world * units_per_rank / (slowest_ms * 1e-3)


def rank_env():
    """(world, rank, local_rank) from the launcher's environment (1, 0, 0 without one)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def gather_ranks(obj):
    """Every rank's obj, in rank order (a one-element list with one process)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [obj]
    out = [None] * dist.get_world_size()
    dist.all_gather_object(out, obj)
    return out


def free_port() -> int:
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def spawn_replicas(n: int, argv) -> int:
    """Run this script as n ranks of one node (one process per GPU, replicas of the
    step, no data-path collective) under torch.distributed.run, the way a multi-GPU
    launch would; rank 0 prints the JSON line. Returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def run_stub(args):
    """The rank plumbing of the GPU arm with a CPU stand-in for the step (a fixed
    sleep that grows with the rank, so the ranks differ): gloo process group,
    per-rank device choice, barrier-bracketed timing of exactly K steps after W
    warm-up steps, the slowest rank's time and the whole-job rate. Prints the same
    JSON keys, marked "stub"; it measures nothing about the kernels."""
    import torch.distributed as dist

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("gloo")
    step_s = 0.002 * (1 + rank)
    for _ in range(args.warmup):
        time.sleep(step_s)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep(step_s)
    if world > 1:
        dist.barrier()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    slow = max_over_ranks(ms)
    devices = gather_ranks("cpu:%d" % local)
    per_rank_ms = gather_ranks(ms)
    if rank == 0:
        print(json.dumps({"metric": "stub steps/s", "value": whole_job_rate(1.0, world, slow), "unit": "steps/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": slow,
                          "higher_is_better": True, "scaling": "weak", "stub": True, "devices": devices,
                          "per_rank_ms": per_rank_ms}))
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from fp8_block_scaled_04_gb300 import binding as fb
    from fp8_block_scaled_04_gb300 import synth

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    devices = gather_ranks(str(dev))
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # fp8 = 2 x bf16 (nominal 4.5 / 2.25 PF)
    hbm_peak = peaks["hbm_gbs"]

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    flush = make_l2_flush(dev)

    # ---- inputs (seeded, synthetic); weights quantized once, offline
    x_host = synth.prefill_x(M, K)
    w_host = synth.prefill_w(N, K)
    xd = to_dev(x_host)
    wd = to_dev(w_host)
    qw, sw = fb.quantize(wd, fb.E4M3, fb.BLOCK_128x128)
    del wd
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128) * M, dtype=torch.float32, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        fb.quantize(xd, fb.E4M3, fb.TILE_1x128, q=qx, scales=sx)
        fb.gemm_blockscaled(qx, sx, fb.TILE_1x128, qw, sw, fb.BLOCK_128x128, out=out, status=status)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()

    # the step: one event pair around both launches (nothing between them, so
    # the GEMM's dependent launch can overlap its setup with the quantizer)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    n0 = fb.launch_count()
    barrier()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush()
            hold_gpu()
            e0, e2 = ev[i]
            e0.record(stream)
            step()
            e2.record(stream)
        barrier()
    launches = fb.launch_count() - n0
    step_ms = [a.elapsed_time(c) for a, c in ev]
    # each kernel on its own (the roofline's achieved rate is the GEMM alone)

    def timed(fn):
        out_ms = []
        for _ in range(args.steps):
            flush()
            hold_gpu()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            out_ms.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in out_ms]

    gemm_ms = timed(lambda: fb.gemm_blockscaled(qx, sx, fb.TILE_1x128, qw, sw, fb.BLOCK_128x128, out=out,
                                                status=status))
    quant_ms = timed(lambda: fb.quantize(xd, fb.E4M3, fb.TILE_1x128, q=qx, scales=sx))
    ms = max_over_ranks(sum(step_ms) / args.steps, dev)
    assert int(status.item()) == 0, "device status %d" % int(status.item())
    flops = 2.0 * M * N * K
    value = whole_job_rate(flops, world, ms) / 1e12
    gemm_avg = sum(gemm_ms) / len(gemm_ms)
    achieved = flops / (gemm_avg * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host X in, Out back to pinned host.
    # Every step copies its X host->device and its Out device->host; steps are
    # pipelined over three streams (copy-in, compute, copy-out) with two device
    # buffers each, so step i+1's upload and step i-1's download overlap step i's
    # kernels. The timed region runs from the first upload to the last download.
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_pin = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xe = [torch.empty_like(xd) for _ in range(2)]
    oe = [torch.empty_like(out) for _ in range(2)]
    qxe = [torch.empty_like(qx) for _ in range(2)]
    sxe = [torch.empty_like(sx) for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        ev_x_ready = [torch.cuda.Event() for _ in range(2)]
        ev_x_free = [torch.cuda.Event() for _ in range(2)]
        ev_o_ready = [torch.cuda.Event() for _ in range(2)]
        ev_o_free = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(nsteps):
            b = i & 1
            if i >= 2:
                s_in.wait_event(ev_x_free[b])
            with torch.cuda.stream(s_in):
                xe[b].copy_(x_pin, non_blocking=True)
            ev_x_ready[b].record(s_in)
            s_cmp.wait_event(ev_x_ready[b])
            if i >= 2:
                s_cmp.wait_event(ev_o_free[b])
            fb.quantize(xe[b], fb.E4M3, fb.TILE_1x128, q=qxe[b], scales=sxe[b], stream=s_cmp)
            fb.gemm_blockscaled(qxe[b], sxe[b], fb.TILE_1x128, qw, sw, fb.BLOCK_128x128, out=oe[b], status=status,
                                stream=s_cmp)
            ev_x_free[b].record(s_cmp)
            ev_o_ready[b].record(s_cmp)
            s_out.wait_event(ev_o_ready[b])
            with torch.cuda.stream(s_out):
                out_pin[b].copy_(oe[b], non_blocking=True)
            ev_o_free[b].record(s_out)
        s_in.wait_stream(s_out)
        t1.record(s_in)
        t1.synchronize()
        return t0.elapsed_time(t1) / nsteps

    torch.cuda.synchronize()
    e2e_run(args.warmup)
    torch.cuda.synchronize()
    e2e = max_over_ranks(e2e_run(args.steps), dev)

    extra = {}
    if not args.headline_only and rank == 0:
        extra = measure_other_workloads(args, fb, synth, dev, stream, flush, fp8_peak, hbm_peak)

    cpu = cpu_baseline_sample(x_host, w_host) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if extra and rank == 0 and world == 1 and not args.no_cpu:
        cpu_baselines_other(extra, synth)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate)",
            "data": "synthetic: seeded SplitMix64/Box-Muller N(0,1) X with 1% outlier channels x30, N(0,0.02) W",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "parallelism": "replicas" if world > 1 else "1gpu",
                       "l2": "flushed between steps (256 MB write, then 256 MB read to clean it; outside the step events)",
                       "host_latency": "a 0.1 ms GPU spin precedes each step's events, so launches are queued when timing starts",
                       "kernel_ms_quantize": round(sum(quant_ms) / len(quant_ms), 5),
                       "kernel_ms_gemm": round(gemm_avg, 5),
                       "kernel_timing": "each kernel alone between its own events; the step times both together"},
            "roofline": {"bound": "tensor", "kernel": "gemm_fold_kernel", "achieved": round(achieved, 1),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                         "peak_src": "%s bf16 burst x2 (fp8/bf16 nominal ratio)" % peaks["src"],
                         "frac_of_nominal_4.5PF": round(achieved / (NOMINAL_FP8_PFLOPS * 1000.0), 4),
                         "traffic": kernel_traffic("gemm_fold_kernel"),
                         # the GEMM's compulsory bytes: fp8 X and W read once, bf16 Out written once, scales
                         "algorithmic_bytes": M * K + N * K + 2 * M * N + 4 * (K // 128) * (M + (N // 128)),
                         "algorithmic_flops": 2 * M * N * K,
                         # the whole step adds the 1x128 quantize of X (bf16 read, codes and scales written)
                         # and the GEMM's re-read of the codes (already counted above)
                         "step_algorithmic_bytes": (2 * M * K + M * K + 4 * (K // 128) * M) + M * K + N * K
                                                   + 2 * M * N + 4 * (K // 128) * (M + (N // 128))},
            "e2e": {"value": round(whole_job_rate(flops, world, e2e) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2, "ms_per_step": round(e2e, 4),
                    "pipelining": "3 streams (upload / compute / download), 2 buffers each, across steps"},
            "gpu_launches": int(launches),
            "devices": devices,
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
        }
        if extra:
            line["other_workloads"] = extra
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def _time_kernel(fn, flush, stream, reps, launches=1):
    """Median event time of fn() (which enqueues `launches` kernels) after an L2
    flush; the GPU hold before the start event scales with the number of
    launches so that all of them are queued before it ends."""
    import torch

    for _ in range(3):
        flush()
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        hold_gpu(200_000 * launches)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


NOMINAL_HBM_GBS = 8000.0  # "~8 TB/s" HBM3e, the quantizers' stated target is 80 % of it


def hbm_fracs(byts, t_ms, hbm_peak):
    gbs = byts / (t_ms * 1e-3) / 1e9
    return {"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 4),
            "frac_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4)}


def measure_sweep(args, fb, synth, dev, stream, flush, hbm_peak):
    """Quantizer sweep: 16384 x 8192, E4M3/E5M2 x {tensor (two-pass), token, 1x128, MX-32}.
    frac_hbm is against the measured copy bandwidth, frac_nominal_8TBs against 8 TB/s."""
    import numpy as np
    import torch

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    reps = max(10, args.steps)
    R, C = 16384, 8192
    x = to_dev(synth.sweep_x(R, C))
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    sweep = {}
    for fname, fmt in (("e4m3", fb.E4M3), ("e5m2", fb.E5M2)):
        for gname, gran, lay in (("tensor", fb.TENSOR, fb.SF_LINEAR), ("token", fb.TOKEN, fb.SF_LINEAR),
                                 ("tile1x128", fb.TILE_1x128, fb.SF_LINEAR), ("mx32", fb.MX32, fb.SF_LINEAR),
                                 ("mx32_tiled", fb.MX32, fb.SF_TCGEN05)):
            nb = fb.scales_bytes(R, C, gran, lay)
            sc = torch.empty(max(nb, 4), dtype=torch.uint8, device=dev)
            scv = sc if gran == fb.MX32 else sc.view(torch.float32)
            t = _time_kernel(lambda: fb.quantize(x, fmt, gran, lay, q=q, scales=scv, workspace=ws), flush, stream,
                             reps)
            byts = R * C * 3 + nb + (R * C * 2 if gran == fb.TENSOR else 0)
            e = {"ms": round(t, 5), "algorithmic_bytes": byts}
            e.update(hbm_fracs(byts, t, hbm_peak))
            if gran == fb.TENSOR:
                # the same time against one pass's bytes (read 2 B, write 1 B per element)
                e["single_pass_equivalent"] = hbm_fracs(R * C * 3 + nb, t, hbm_peak)
            sweep["%s_%s" % (fname, gname)] = e
    return sweep


def measure_next_rows(args, fb, synth, dev, stream, flush, fp8_peak, hbm_peak):
    """The rows built after the hot path, each against its roofline:
    - the fold GEMM with 1x128 quantization fused into its epilogue, against the
      GEMM's bf16 output followed by a separate 1x128 quantize of it ("Low
      precision", practice 4: the separate pass costs two trips to HBM), on the
      prefill shape 4096 x 14336 x 4096;
    - per-tensor quantization with delayed scaling (one pass, scale from an amax
      history) against current scaling (two passes) on the sweep tensor 16384 x 8192;
    - per-channel quantization of a KV-cache-shaped tensor, 65536 tokens x 1024
      channels (8 heads x 128 dims)."""
    import numpy as np
    import torch

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    reps = max(10, args.steps)
    res = {}
    # ---- fused quantize-in-epilogue (f1)
    qx, sx = fb.quantize(to_dev(synth.prefill_x(M, K)), fb.E4M3, fb.TILE_1x128)
    qw, sw = fb.quantize(to_dev(synth.prefill_w(N, K)), fb.E4M3, fb.BLOCK_128x128)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    qo = torch.empty((M, N), dtype=torch.uint8, device=dev)
    so = torch.empty((N // 128) * M, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    t_fused = _time_kernel(lambda: fb.gemm_blockscaled_quantized_out(qx, sx, qw, sw, q_out=qo, q_scales=so, status=st),
                           flush, stream, reps)

    def unfused():
        fb.gemm_blockscaled(qx, sx, fb.TILE_1x128, qw, sw, fb.BLOCK_128x128, out=out, status=st)
        fb.quantize(out, fb.E4M3, fb.TILE_1x128, q=qo, scales=so)

    t_unfused = _time_kernel(unfused, flush, stream, reps, launches=2)
    flops = 2.0 * M * N * K
    gemm_in = M * K + N * K + 4 * (K // 128) * (M + N // 128)
    fused_bytes = gemm_in + M * N + 4 * (N // 128) * M
    unfused_bytes = gemm_in + 2 * M * N + (2 * M * N + M * N + 4 * (N // 128) * M)
    res["fused_quantized_out_prefill"] = {
        "fused": {"ms": round(t_fused, 5), "TFLOP/s": round(flops / (t_fused * 1e-3) / 1e12, 1),
                  "frac_fp8_peak": round(flops / (t_fused * 1e-3) / 1e12 / fp8_peak, 4), "algorithmic_bytes": fused_bytes},
        "gemm_then_quantize": {"ms": round(t_unfused, 5), "TFLOP/s": round(flops / (t_unfused * 1e-3) / 1e12, 1),
                               "algorithmic_bytes": unfused_bytes},
        "hbm_bytes_saved": unfused_bytes - fused_bytes, "speedup": round(t_unfused / t_fused, 4),
        "output": "E4M3 codes + 1x128 scales of the bf16-rounded GEMM output (the next layer's activation)"}
    del qx, sx, qw, sw, out, qo, so
    # ---- delayed vs current per-tensor scaling (f3)
    R, C = 16384, 8192
    x = to_dev(synth.sweep_x(R, C))
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    scale = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    hist = torch.zeros(16, dtype=torch.float32, device=dev)
    fb.quantize_delayed(x, fb.E4M3, hist, 0)  # a history with this tensor's amax in it
    slot = [0]

    def delayed():
        slot[0] = (slot[0] + 1) % 16
        fb.quantize_delayed(x, fb.E4M3, hist, slot[0], q=q, scale=scale)

    t_del = _time_kernel(delayed, flush, stream, reps, launches=2)
    t_cur = _time_kernel(lambda: fb.quantize(x, fb.E4M3, fb.TENSOR, q=q, scales=scale, workspace=ws), flush, stream,
                         reps, launches=2)
    one_pass = R * C * 3 + 4
    res["delayed_vs_current_per_tensor_16384x8192"] = {
        "delayed_one_pass": dict({"ms": round(t_del, 5), "algorithmic_bytes": one_pass}, **hbm_fracs(one_pass, t_del, hbm_peak)),
        "current_two_pass": dict({"ms": round(t_cur, 5), "algorithmic_bytes": R * C * 5 + 4},
                                 **hbm_fracs(R * C * 5 + 4, t_cur, hbm_peak)),
        "speedup": round(t_cur / t_del, 4), "history_len": 16}
    del x, q
    # ---- per-channel KV-cache quantizer (f4)
    T, Ch = 65536, 1024
    kv = to_dev(synth.bf16_matrix(T, Ch, 1.0, 41, 42, 0.01, 20.0))
    qk = torch.empty((T, Ch), dtype=torch.uint8, device=dev)
    sk = torch.empty(Ch, dtype=torch.float32, device=dev)
    wk = torch.empty(fb.workspace_bytes(T, Ch, fb.CHANNEL), dtype=torch.uint8, device=dev)
    res_kv = {}
    for fname, fmt in (("e4m3", fb.E4M3), ("e5m2", fb.E5M2)):
        t_kv = _time_kernel(lambda: fb.quantize(kv, fmt, fb.CHANNEL, q=qk, scales=sk, workspace=wk), flush, stream,
                            reps, launches=3)
        byts = T * Ch * 5 + 4 * Ch  # column maxima pass (2 B) + encode pass (2 B read, 1 B written)
        res_kv[fname] = dict({"ms": round(t_kv, 5), "algorithmic_bytes": byts,
                              "single_pass_equivalent": hbm_fracs(T * Ch * 3 + 4 * Ch, t_kv, hbm_peak)},
                             **hbm_fracs(byts, t_kv, hbm_peak))
    res["kv_cache_per_channel_65536x1024"] = res_kv
    return res


def measure_decode(args, fb, synth, dev, stream, flush, hbm_peak):
    """Decode-shaped GEMMs: W 18432 x 7168 (132 MB) streamed once per call, M = 16 and 64."""
    import numpy as np
    import torch

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    reps = max(10, args.steps)
    res = {}
    Nd, Kd = 18432, 7168
    wd = to_dev(synth.decode_w(Nd, Kd))
    qw, sw = fb.quantize(wd, fb.E4M3, fb.BLOCK_128x128)
    del wd
    # back to back: one launch per weight copy (a decode step runs many GEMMs in a
    # row); every copy is larger than L2, so each launch streams its W from HBM
    n_copies = 8
    copies = [(qw.clone(), sw.clone()) for _ in range(n_copies)]
    for m in (16, 64):
        xq, xs = fb.quantize(to_dev(synth.decode_x(m, Kd)), fb.E4M3, fb.TILE_1x128)
        o = torch.empty((m, Nd), dtype=torch.bfloat16, device=dev)
        t = _time_kernel(lambda: fb.gemm_blockscaled(xq, xs, fb.TILE_1x128, qw, sw, fb.BLOCK_128x128, out=o),
                         flush, stream, reps)

        def seq():
            for cw, cs in copies:
                fb.gemm_blockscaled(xq, xs, fb.TILE_1x128, cw, cs, fb.BLOCK_128x128, out=o)

        t_seq = _time_kernel(seq, flush, stream, max(5, reps // 2), launches=n_copies) / n_copies
        byts = Nd * Kd + m * Kd + m * Nd * 2 + 4 * (Kd // 128) * (m + Nd // 128)
        res["decode_gemm_m%d" % m] = {
            "ms": round(t, 5), "GB/s": round(byts / (t * 1e-3) / 1e9, 1),
            "frac_hbm": round(byts / (t * 1e-3) / 1e9 / hbm_peak, 4),
            "TFLOP/s": round(2.0 * m * Nd * Kd / (t * 1e-3) / 1e12, 2), "algorithmic_bytes": byts,
            "single_launch_note": "one launch between its own events (includes ~2.4 us of event-pair latency and the launch)",
            "back_to_back": {"launches": n_copies, "weight_copies": n_copies, "ms_per_launch": round(t_seq, 5),
                             "GB/s": round(byts / (t_seq * 1e-3) / 1e9, 1),
                             "frac_hbm": round(byts / (t_seq * 1e-3) / 1e9 / hbm_peak, 4)}}
    del copies
    return res


def measure_mx(args, fb, synth, dev, stream, flush, fp8_peak):
    """MXFP8 GEMM 8192^3 with UE8M0 scales per 32 K (tensor-core block scaling)."""
    import numpy as np
    import torch

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    reps = max(10, args.steps)
    S = 8192
    x, w = to_dev(synth.mx_x(S, S)), to_dev(synth.mx_w(S, S))
    # the library's fast path: scales quantized straight into the staged-four-times
    # layout (fp8_gemm_mx_x4); the tiled layout's kernel is timed beside it
    xa, sfa4 = fb.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    wb, sfb4 = fb.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05_X4)
    _, sfa = fb.quantize(x, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    _, sfb = fb.quantize(w, fb.E4M3, fb.MX32, fb.SF_TCGEN05)
    del x, w
    o = torch.empty((S, S), dtype=torch.bfloat16, device=dev)
    t = _time_kernel(lambda: fb.gemm_mx(xa, sfa4, wb, sfb4, out=o, sf_layout=fb.SF_TCGEN05_X4), flush, stream, reps)
    t_tiled = _time_kernel(lambda: fb.gemm_mx(xa, sfa, wb, sfb, out=o), flush, stream, reps)
    tf = 2.0 * S ** 3 / (t * 1e-3) / 1e12
    tf_tiled = 2.0 * S ** 3 / (t_tiled * 1e-3) / 1e12
    return {"mx_gemm_8192": {"ms": round(t, 5), "TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 4),
                             "frac_nominal_4.5PF": round(tf / 4500.0, 4), "scale_layout": "tcgen05 tiled, staged x4",
                             "tiled_layout": {"ms": round(t_tiled, 5), "TFLOP/s": round(tf_tiled, 1),
                                              "frac_nominal_4.5PF": round(tf_tiled / 4500.0, 4)}}}


def measure_nvfp4(args, fb, synth, dev, stream, flush, hbm_peak, fp4_peak):
    """NVFP4 ("Low precision", NVFP4 paragraph): the quantizer on the sweep tensor
    16384 x 8192 (two passes with the tensor's own amax, and one pass with a
    static tensor scale) and the block-scaled GEMM 8192^3 on the MX inputs."""
    import numpy as np
    import torch

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    reps = max(10, args.steps)
    res = {}
    R, C = 16384, 8192
    x = to_dev(synth.sweep_x(R, C))
    q, sf, ts = fb.quantize_nvfp4(x)
    out_bytes = R * C // 2 + R * C // 16
    t2 = _time_kernel(lambda: fb.quantize_nvfp4(x, q=q, sf=sf, tensor_scale=ts), flush, stream, reps)
    b2 = 2 * (2 * R * C) + out_bytes  # amax pass reads X, the encode pass reads it again
    static = torch.tensor([0.01], dtype=torch.float32, device=dev)
    t1 = _time_kernel(lambda: fb.quantize_nvfp4(x, static_tensor_scale=static, q=q, sf=sf, tensor_scale=ts),
                      flush, stream, reps)
    b1 = 2 * R * C + out_bytes
    res["nvfp4_quantize_16384x8192"] = {
        "two_pass": {"ms": round(t2, 5), "GB/s": round(b2 / (t2 * 1e-3) / 1e9, 1),
                     "frac_hbm": round(b2 / (t2 * 1e-3) / 1e9 / hbm_peak, 4), "algorithmic_bytes": b2},
        "static_scale": {"ms": round(t1, 5), "GB/s": round(b1 / (t1 * 1e-3) / 1e9, 1),
                         "frac_hbm": round(b1 / (t1 * 1e-3) / 1e9 / hbm_peak, 4), "algorithmic_bytes": b1}}
    del x, q, sf
    S = 8192
    qa, sfa, ta = fb.quantize_nvfp4(to_dev(synth.mx_x(S, S)))
    qb, sfb, tb = fb.quantize_nvfp4(to_dev(synth.mx_w(S, S)))
    o = torch.empty((S, S), dtype=torch.bfloat16, device=dev)
    t = _time_kernel(lambda: fb.gemm_nvfp4(qa, sfa, ta, qb, sfb, tb, out=o), flush, stream, reps)
    tf = 2.0 * S ** 3 / (t * 1e-3) / 1e12
    res["nvfp4_gemm_8192"] = {"ms": round(t, 5), "TFLOP/s": round(tf, 1), "frac_fp4_peak": round(tf / fp4_peak, 4),
                              "fp4_peak": round(fp4_peak, 1),
                              "fp4_peak_src": "measured bf16 burst x 2 (fp8) x 2 (fp4 = 2 x fp8, the pages' 9 vs 4.5 PF)",
                              "frac_nominal_13.5PF": round(tf / 13500.0, 4)}
    return res


def run_workload(args):
    """One non-headline workload on its own (for profiling): prints one JSON line."""
    import torch

    from fp8_block_scaled_04_gb300 import binding as fb
    from fp8_block_scaled_04_gb300 import synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    flush = make_l2_flush(dev)
    if args.workload == "sweep":
        res = {"quantize_sweep_16384x8192": measure_sweep(args, fb, synth, dev, stream, flush, peaks["hbm_gbs"])}
    elif args.workload == "decode":
        res = measure_decode(args, fb, synth, dev, stream, flush, peaks["hbm_gbs"])
    elif args.workload == "nvfp4":
        res = measure_nvfp4(args, fb, synth, dev, stream, flush, peaks["hbm_gbs"],
                            FP4_OVER_FP8 * 2.0 * peaks["bf16_tflops"])
    elif args.workload == "next":
        res = measure_next_rows(args, fb, synth, dev, stream, flush, 2.0 * peaks["bf16_tflops"], peaks["hbm_gbs"])
    else:
        res = measure_mx(args, fb, synth, dev, stream, flush, 2.0 * peaks["bf16_tflops"])
    print(json.dumps({"workload": args.workload, "peaks": peaks["src"], "results": res}))


def measure_other_workloads(args, fb, synth, dev, stream, flush, fp8_peak, hbm_peak):
    """Per-kernel numbers for the other workloads of the path, each against its roofline."""
    res = {"quantize_sweep_16384x8192": measure_sweep(args, fb, synth, dev, stream, flush, hbm_peak)}
    res.update(measure_decode(args, fb, synth, dev, stream, flush, hbm_peak))
    res.update(measure_mx(args, fb, synth, dev, stream, flush, fp8_peak))
    res.update(measure_nvfp4(args, fb, synth, dev, stream, flush, hbm_peak, FP4_OVER_FP8 * fp8_peak))
    res.update(measure_next_rows(args, fb, synth, dev, stream, flush, fp8_peak, hbm_peak))
    return res


# --------------------------------------------------------------------- CPU oracle
def cpu_baselines_other(extra, synth, rows_sweep: int = 512, rows_mx: int = 16):
    """The oracle, as it stands, on bounded samples of the other workloads (the first
    rows of each input; the generator is counter-based, so those rows are the full
    input's): the quantizer sweep on rows_sweep of its 16384 rows, both decode GEMMs in
    full, the MXFP8 GEMM on rows_mx of its 8192 rows. Attached to each workload's entry
    as "cpu_baseline"; the units match the GPU figure beside it."""
    import oracle

    threads = oracle.default_threads()
    C = 8192
    xs = synth.sweep_x(rows_sweep, C)
    sw = extra.get("quantize_sweep_16384x8192", {})
    for fname, fmt in (("e4m3", oracle.E4M3), ("e5m2", oracle.E5M2)):
        for gname, gran, lay in (("tensor", oracle.TENSOR, 0), ("token", oracle.TOKEN, 0),
                                 ("tile1x128", oracle.TILE_1x128, 0), ("mx32", oracle.MX32, 0),
                                 ("mx32_tiled", oracle.MX32, 1)):
            key = "%s_%s" % (fname, gname)
            if key not in sw:
                continue
            t0 = time.perf_counter()
            oracle.quantize(xs, fmt, gran, lay)
            dt = time.perf_counter() - t0
            byts = sw[key]["algorithmic_bytes"] * rows_sweep / 16384.0
            sw[key]["cpu_baseline"] = {"value": round(byts / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
                                       "kind": "oracle", "sample": "first %d of 16384 rows" % rows_sweep}
    Nd, Kd = 18432, 7168
    wq, wsc = oracle.quantize(synth.decode_w(Nd, Kd), oracle.E4M3, oracle.BLOCK_128x128)
    for m in (16, 64):
        key = "decode_gemm_m%d" % m
        if key not in extra:
            continue
        xq, xsc = oracle.quantize(synth.decode_x(m, Kd), oracle.E4M3, oracle.TILE_1x128)
        t0 = time.perf_counter()
        oracle.gemm(xq, xsc, oracle.TILE_1x128, wq, wsc, oracle.BLOCK_128x128)
        dt = time.perf_counter() - t0
        extra[key]["cpu_baseline"] = {"value": round(extra[key]["algorithmic_bytes"] / dt / 1e9, 3), "unit": "GB/s",
                                      "TFLOP/s": round(2.0 * m * Nd * Kd / dt / 1e12, 5), "cores": threads,
                                      "kind": "oracle", "sample": "the whole GEMM (fp64 sums), W quantized beforehand"}
    del wq, wsc
    if "mx_gemm_8192" in extra:
        S = 8192
        xq, xsf = oracle.quantize(synth.mx_x(rows_mx, S), oracle.E4M3, oracle.MX32, 1)
        wq, wsf = oracle.quantize(synth.mx_w(S, S), oracle.E4M3, oracle.MX32, 1)
        t0 = time.perf_counter()
        oracle.gemm(xq, xsf, oracle.MX32, wq, wsf, oracle.MX32, a_sf=1, b_sf=1)
        dt = time.perf_counter() - t0
        extra["mx_gemm_8192"]["cpu_baseline"] = {"value": round(2.0 * rows_mx * S * S / dt / 1e12, 5),
                                                 "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                                 "sample": "first %d of 8192 rows of X, all of W, fp64 sums" % rows_mx}
    nq = extra.get("nvfp4_quantize_16384x8192")
    if nq is not None:
        # the NVFP4 quantizer: both modes on the sample rows (two passes: the
        # sample's own tensor amax, then the encode)
        xs4 = synth.sweep_x(rows_sweep, C)
        for mode, static in (("two_pass", None), ("static_scale", 0.01)):
            if mode not in nq:
                continue
            t0 = time.perf_counter()
            oracle.quantize_nvfp4(xs4, oracle.SF_TILED, static)
            dt = time.perf_counter() - t0
            byts = nq[mode]["algorithmic_bytes"] * rows_sweep / 16384.0
            nq[mode]["cpu_baseline"] = {"value": round(byts / dt / 1e9, 3), "unit": "GB/s", "cores": threads,
                                        "kind": "oracle", "sample": "first %d of 16384 rows" % rows_sweep}
    if "nvfp4_gemm_8192" in extra:
        S = 8192
        aq, asf, ats = oracle.quantize_nvfp4(synth.mx_x(rows_mx, S), oracle.SF_TILED)
        bq, bsf, bts = oracle.quantize_nvfp4(synth.mx_w(S, S), oracle.SF_TILED)
        t0 = time.perf_counter()
        oracle.gemm_nvfp4(aq, asf, ats, bq, bsf, bts, oracle.SF_TILED)
        dt = time.perf_counter() - t0
        extra["nvfp4_gemm_8192"]["cpu_baseline"] = {"value": round(2.0 * rows_mx * S * S / dt / 1e12, 5),
                                                    "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                                    "sample": "first %d of 8192 rows of X (tensor scale from those "
                                                              "rows), all of W, fp64 sums" % rows_mx}


def cpu_baseline_sample(x_host, w_host, target_s: float = 10.0):
    """The oracle as it stands, on a bounded sample of the headline workload:
    quantize the first R rows of X (1x128), quantize W (128x128), and the fp64
    GEMM of those R rows against all of W. Scaled to TFLOP/s of that sample."""
    import oracle

    threads = oracle.default_threads()
    qb, sb = oracle.quantize(w_host, oracle.E4M3, oracle.BLOCK_128x128)
    rows = 8
    while True:
        t0 = time.perf_counter()
        qa, sa = oracle.quantize(x_host[:rows], oracle.E4M3, oracle.TILE_1x128)
        oracle.gemm(qa, sa, oracle.TILE_1x128, qb, sb, oracle.BLOCK_128x128)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or rows >= M:
            break
        rows = min(M, max(rows * 2, int(rows * target_s / max(dt, 1e-3))))
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "first %d of %d rows of X, all of W (%dx%d), fp64 sums; %.1f s" % (rows, M, N, K, dt)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from fp8_block_scaled_04_gb300 import synth
    import oracle

    x_host = synth.prefill_x(M, K)
    w_host = synth.prefill_w(N, K)
    threads = oracle.default_threads()
    qb, sb = oracle.quantize(w_host, oracle.E4M3, oracle.BLOCK_128x128)
    rows = 4

    def one_step():
        qa, sa = oracle.quantize(x_host[:rows], oracle.E4M3, oracle.TILE_1x128)
        oracle.gemm(qa, sa, oracle.TILE_1x128, qb, sb, oracle.BLOCK_128x128)

    # size the per-step sample so the whole run stays within a few minutes
    t0 = time.perf_counter()
    one_step()
    dt = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(M, rows * budget / max(dt, 1e-3))))
    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    sec = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * N * K / sec / 1e12
    sample = "first %d of %d rows of X per step, all of W (%dx%d), fp64 sums" % (rows, M, N, K)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--workload", default="all", choices=["all", "sweep", "decode", "mx", "nvfp4", "next"],
                    help="all: the headline step plus the other workloads; otherwise that workload alone")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baselines")
    ap.add_argument("--stub-step", action="store_true",
                    help="check of the rank plumbing on CPU: a sleep stands in for the step (measures nothing)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args.gpus, sys.argv[1:]))
    if args.stub_step:
        run_stub(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.workload != "all":
        run_workload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
