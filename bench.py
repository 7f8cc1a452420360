#!/usr/bin/env python
"""Benchmark of the layer-streamed NF4 LoRA training step on B300.

Workload (one "step"): forward over 32 Llama-3.1-8B-shaped decoder layers
(q 4096x4096, k/v 1024x4096, o 4096x4096, gate/up 14336x4096, down 4096x14336,
NF4 base, LoRA r=16 alpha=32 on all seven projections) then backward in
reverse, M = 1024 tokens, the frozen base streamed layer by layer from pinned
host RAM through two device buffers.  Synthetic seeded data; no trained
weights.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the plain CPU oracle (the reference of this build) on
the host cores, on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train tokens/s (8B-shape NF4 streamed fwd+bwd); % of PCIe/HBM/TC roofline"
UNIT = "tokens/s"
L, M, D, DKV, F, R, ALPHA = 32, 1024, 4096, 1024, 14336, 16, 32.0
WORKLOAD = "llama-3.1-8b-shaped 32-layer NF4 LoRA stack streamed from pinned host RAM, fwd 0..31 + bwd 31..0"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks, throttle reasons)."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
def oracle_layer_sample(m_sample, seed=3):
    """The oracle on a bounded sample of the workload: ONE full-width NF4 layer,
    m_sample tokens.  Returns (seconds per step of the sample, threads used, closure)."""
    import numpy as np
    import seeded_inputs as si
    from oracle import nf4, stack
    c = si.stack_case(seed, 1, m_sample, D, DKV, F, R)
    lw = c["layers"][0]
    q = {n: nf4.quantize(lw[n]["W"]) for n in si.PROJ_NAMES}   # offline (not timed), like the GPU's blobs

    def step():
        layer = {n: dict(W=nf4.dequantize_bf16(*q[n], *lw[n]["W"].shape), A=lw[n]["A"].astype(np.float64),
                         B=lw[n]["B"].astype(np.float64)) for n in si.PROJ_NAMES}
        stack.stack_step(c["h0"], c["dh_top"], [layer], ALPHA, rnd=True)

    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count() or 1])
    except ImportError:   # numpy's BLAS runs one thread per host core by default
        threads = os.cpu_count() or 1
    return step, threads


def cpu_baseline(m_sample=64):
    step, threads = oracle_layer_sample(m_sample)
    step()  # warm
    t0 = time.perf_counter()
    step()
    dt = time.perf_counter() - t0
    tok_s = m_sample / (L * dt)       # the full stack is L such layers
    return {"value": tok_s, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"one full-width NF4 layer (of {L}), {m_sample} tokens, fwd+bwd incl. dequantisation; "
                      f"{dt:.2f} s; tokens/s scaled by 1/{L} layers"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    m_sample = 64
    step, threads = oracle_layer_sample(m_sample)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = m_sample / (L * dt)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 * L * M / m_sample,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "tokens": M, "layers": L, "rank": R,
                                            "sample": f"1 layer x {m_sample} tokens per step"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step: one full-width NF4 layer, {m_sample} tokens, fwd+bwd; "
                                       f"tokens/s scaled by 1/{L} layers"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import layer_streamed_qlora_linear_b300 as sl
    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", local)
    nl = args.layers
    gen = torch.Generator(device=dev).manual_seed(1234 + rank)
    rnd = lambda shape, std: (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)
    shapes = sl.proj_shapes(D, DKV, F)

    # frozen NF4 base: quantised on the device by the library, kept in pinned host RAM
    host_blobs, A, B = [], [], []
    for l in range(nl):
        blob = sl.build_layer_blob(sl.SL_WEIGHT_NF4, D, DKV, F, [rnd((N, K), 0.02) for N, K in shapes])
        h = torch.empty(blob.numel(), dtype=torch.uint8, pin_memory=True)
        h.copy_(blob)
        host_blobs.append(h)
        del blob
        for N, K in shapes:
            A.append(rnd((R, K), 0.02))
            B.append(rnd((N, R), 0.02))
    dA = [torch.empty(a.shape, dtype=torch.float32, device=dev) for a in A]
    dB = [torch.empty(b.shape, dtype=torch.float32, device=dev) for b in B]
    h0 = torch.randn(M, D, generator=gen, device=dev).to(torch.bfloat16).float()
    dh = torch.randn(M, D, generator=gen, device=dev).to(torch.bfloat16).float()
    hL = torch.empty(M, D, device=dev)
    dh0 = torch.empty(M, D, device=dev)
    stk = sl.Stack(sl.SL_WEIGHT_NF4, D, DKV, F, host_blobs)
    ws = torch.empty(stk.workspace_size(M, R), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        stk.step(sl.SL_MODE_STREAMED, h0, dh, A, B, R, ALPHA, hL, dh0, dA, dB, ws)

    # pinned H2D bandwidth of this machine: 1 GiB, best of 10, CUDA events
    hb = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    db = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    best = 1e9
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        db.copy_(hb, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    h2d_peak = (1 << 30) / (best * 1e-3) / 1e9
    del hb, db

    for _ in range(args.warmup):
        step()
    sl.sl_check_device_errors()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    sl.sl_kernel_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    sl.sl_kernel_timing(False)
    clk = clocks.stop()
    ms_total = e0.elapsed_time(e1)
    h2d_step, kernels_step = stk.last_step_stats()
    timing = {name: sl.sl_kernel_timing_read(i) for i, name in enumerate(sl.GEMM_VARIANTS)}
    sl.sl_check_device_errors()
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / args.steps
    value = world * M * args.steps / (ms_total * 1e-3)

    # end to end through the public API: host inputs in, host result out, every step
    h0_h = h0.cpu().pin_memory()
    dh_h = dh.cpu().pin_memory()
    hL_h = torch.empty(M, D, dtype=torch.float32, pin_memory=True)
    h0_d, dh_d = torch.empty_like(h0), torch.empty_like(dh)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        h0_d.copy_(h0_h, non_blocking=True)
        dh_d.copy_(dh_h, non_blocking=True)
        stk.step(sl.SL_MODE_STREAMED, h0_d, dh_d, A, B, R, ALPHA, hL, dh0, dA, dB, ws)
        hL_h.copy_(hL, non_blocking=True)
    barrier()
    e2e_s = time.perf_counter() - t0
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_s], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e = {"value": world * M * args.steps / e2e_s, "unit": UNIT,
           "h2d_bytes_per_step": int(h0_h.numel() * 4 + dh_h.numel() * 4),
           "d2h_bytes_per_step": int(hL_h.numel() * 4)}

    # dominant kernel: the fused NF4 dequant + LoRA tcgen05 GEMM (forward and dX variants)
    n_f, ms_f, fl_f = timing["nf4_fwd"]
    n_x, ms_x, fl_x = timing["nf4_dx"]
    gemm_ms = ms_f + ms_x
    achieved = (fl_f + fl_x) / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else 0.0
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    roofline = {"bound": "tensor", "kernel": "gemm_tc_kernel<NF4> (fused dequant + LoRA fold; fwd and dX)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside a long step)",
                "traffic": None, "launches": n_f + n_x, "avg_launch_ms": gemm_ms / max(1, n_f + n_x),
                "share_of_step": gemm_ms / ms_total}
    stream_roof = {"bound": "pcie_h2d", "h2d_bytes_per_step": h2d_step,
                   "achieved_gbs": h2d_step / (ms_step * 1e-3) / 1e9, "peak_gbs": h2d_peak,
                   "frac": h2d_step / (ms_step * 1e-3) / 1e9 / h2d_peak,
                   "peak_source": "measured in this run: pinned 1 GiB cudaMemcpyAsync, best of 10"}
    per_variant = {k: {"launches": v[0], "ms": v[1], "tflops": (v[2] / (v[1] * 1e-3) / 1e12) if v[1] else 0.0}
                   for k, v in timing.items() if v[0]}

    # resident run of the same kernels (compute-only context number)
    resident = None
    if not args.no_resident:
        dev_blobs = [hb.to(dev) for hb in host_blobs]
        stk_r = sl.Stack(sl.SL_WEIGHT_NF4, D, DKV, F, host_blobs, dev_blobs)
        stk_r.step(sl.SL_MODE_RESIDENT, h0, dh, A, B, R, ALPHA, hL, dh0, dA, dB, ws)
        barrier()
        e0.record(stream)
        nres = max(2, min(args.steps, 5))
        for _ in range(nres):
            stk_r.step(sl.SL_MODE_RESIDENT, h0, dh, A, B, R, ALPHA, hL, dh0, dA, dB, ws)
        e1.record(stream)
        barrier()
        resident = {"tokens_per_s": M * nres / (e0.elapsed_time(e1) * 1e-3),
                    "ms_per_step": e0.elapsed_time(e1) / nres}
        stk_r.close()
        del dev_blobs

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded device RNG weights, NF4 on device)",
                "config": {"workload": WORKLOAD, "tokens": M, "layers": nl, "D": D, "Dkv": DKV, "F": F, "rank": R,
                           "alpha": ALPHA, "base": "NF4 blocksize 64 fp32 absmax",
                           "parallelism": f"replicas x{world} (no collective on the data path)",
                           "l2": "inputs larger than L2 (3.9 GB streamed base + ~5 GB activations per step)"},
                "roofline": roofline, "stream": stream_roof, "kernels": per_variant,
                "e2e": e2e, "gpu_launches": int(kernels_step * args.steps), "clocks": clk,
                "resident": resident, "preflight": {"host_bytes": stk.host_bytes, "buffer_bytes": stk.buffer_bytes}}
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    stk.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=L, help="layers (default 32; fewer only for quick checks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-resident", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
