#!/usr/bin/env python
"""Benchmark of the layer-streamed NF4 LoRA training path on B300.

Default workload (one "step"): forward over 32 Llama-3.1-8B-shaped decoder
layers (q 4096x4096, k/v 1024x4096, o 4096x4096, gate/up 14336x4096, down
4096x14336, NF4 base, LoRA r=16 alpha=32 on all seven projections) then
backward in reverse, M = 1024 tokens, the frozen base streamed layer by layer
from pinned host RAM through two device buffers.  Synthetic seeded data; no
trained weights.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload stack8b|stack8b_dq|stack8b_attn|sft8b|stack_qwen3b|layer8b|attn8b|ce]

Other workloads (not the headline line): the same 32-layer stack with the
absmax double-quantised to 8 bits (the ~3.6 GB pinned store, 113 MB per
layer, that the pages quote); the same stack as full decoder layers (causal
GQA attention with rotary positions over one 1024-token sequence, weighted
RMS norms); one complete SFT step on those layers (embedding rows, the
streamed stack, final norm, the 128256-entry head's chunked cross-entropy,
backward); one 8B layer's causal GQA attention alone (forward and
backward, 8 sequences of 1024 tokens); the 36-layer Qwen2.5-3B-shaped
stack with a bf16 base streamed at M=2048; one Llama-8B layer's seven NF4
LoRA linears resident at M=2048 (fwd+bwd); the LM-head cross-entropy
(M=2048, D=4096, V=128256).

--impl reference times the plain CPU oracle (the reference of this build) on
the host cores, on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train tokens/s (8B-shape NF4 streamed fwd+bwd); % of PCIe/HBM/TC roofline"
UNIT = "tokens/s"
WORKLOADS = {
    "stack8b": dict(kind="stack", base="nf4", L=32, M=1024, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0,
                    name="llama-3.1-8b-shaped 32-layer NF4 LoRA stack streamed from pinned host RAM, "
                         "fwd 0..31 + bwd 31..0"),
    "stack8b_dq": dict(kind="stack", base="nf4dq", L=32, M=1024, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0,
                       name="llama-3.1-8b-shaped 32-layer NF4 LoRA stack, 8-bit double-quantised absmax, streamed "
                            "from pinned host RAM, fwd 0..31 + bwd 31..0"),
    "stack8b_attn": dict(kind="stack", base="nf4", L=32, M=1024, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0,
                         attn=(1024, 500000.0),
                         name="llama-3.1-8b-shaped 32 full decoder layers (causal GQA attention, rotary positions, "
                              "one 1024-token sequence), NF4 LoRA, streamed from pinned host RAM, fwd + bwd"),
    "sft8b": dict(kind="stack", base="nf4", L=32, M=1024, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0,
                  attn=(1024, 500000.0), sft=dict(V=128256, chunk=8192),
                  name="llama-3.1-8b-shaped complete SFT step: embedding, 32 full decoder layers streamed, final "
                       "norm, 128256-entry head cross-entropy (vocab chunks of 8192), backward"),
    "stack_qwen3b": dict(kind="stack", base="bf16", L=36, M=2048, D=2048, Dkv=256, F=11008, r=16, alpha=32.0,
                         name="qwen2.5-3b-shaped 36-layer bf16-base LoRA stack streamed from pinned host RAM"),
    "layer8b": dict(kind="layer", base="nf4", M=2048, D=4096, Dkv=1024, F=14336, r=16, alpha=32.0,
                    name="one llama-3.1-8b-shaped layer: seven NF4 LoRA linears resident, fwd+bwd"),
    "attn8b": dict(kind="attn", M=8192, S=1024, H=32, Hkv=8, theta=500000.0,
                   name="causal GQA attention of one llama-3.1-8b-shaped layer (32 query heads, 8 kv heads, rotary "
                        "positions), forward + backward, 8 sequences of 1024 tokens"),
    "ce": dict(kind="ce", M=2048, D=4096, V=128256, chunk=8192,
               name="LM-head cross-entropy fwd+bwd, vocab-chunked (llama-3.1-8b head)"),
}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def pick_peak(peaks, clk):
    """The dense bf16 denominator for the clock the timed region actually ran at.

    The burst figure was measured with the SM clock at its maximum; the
    sustained one under the power cap, at a much lower clock.  A kernel timed
    while the median SM clock stayed within 3% of its maximum (power-cap
    samples or not) is held to the burst figure; otherwise to the sustained
    one."""
    burst = peaks["bf16_tflops"]
    sus = peaks.get("bf16_tflops_sustained", burst)
    if not clk:
        return sus, "bf16_tflops_sustained: no clock samples from the timed region"
    cap = " (sw_power_cap seen)" if "sw_power_cap" in clk["reasons"] else ""
    if clk["sm_mhz"] >= 0.97 * clk["sm_max_mhz"]:
        return burst, f"bf16_tflops (burst): median SM clock {clk['sm_mhz']:.0f} of {clk['sm_max_mhz']:.0f} MHz{cap}"
    return sus, f"bf16_tflops_sustained: median SM clock {clk['sm_mhz']:.0f} of {clk['sm_max_mhz']:.0f} MHz{cap}"


def _sources_digest(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# The kernel sources whose DRAM traffic a committed ncu summary records.
GEMM_SOURCES = ["layer_streamed_qlora_linear_b300/csrc/" + f
                for f in ("gemm.cu", "gemm.cuh", "gemm2.cuh", "gemm3.cuh", "ptx.cuh", "common.cuh")]


def profiled_traffic(summary, sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel sources as they are now; (None, why) otherwise.

    The summary carries two lines: `traffic_bytes_per_launch: <float>` and
    `sources_sha256: <hex digest of the sources, concatenated in order>`."""
    path = os.path.join(ROOT, summary)
    try:
        text = open(path).read()
    except OSError:
        return None, f"no summary at {summary}"
    val = dig = None
    for line in text.splitlines():
        line = line.strip().strip("`")
        if line.startswith("traffic_bytes_per_launch:"):
            val = float(line.split(":", 1)[1])
        elif line.startswith("sources_sha256:"):
            dig = line.split(":", 1)[1].strip()
    if val is None or dig is None:
        return None, f"{summary} records no traffic for a known source digest"
    if dig != _sources_digest(sources):
        return None, f"the kernel sources changed since {summary} was captured"
    return val, f"ncu dram__bytes_read.sum + dram__bytes_write.sum per launch ({summary})"


def rank_barrier(world):
    """All replicas meet (no-op for one process)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_of(x, world, device):
    """The largest x over all replicas (the timing rule: the slowest rank's time counts)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds_max):
    """Units all replicas processed per second of the slowest replica (weak scaling)."""
    return world * units_per_rank / seconds_max


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def proj_shapes(D, Dkv, F):
    return [("q", D, D), ("k", Dkv, D), ("v", Dkv, D), ("o", D, D), ("gate", F, D), ("up", F, D), ("down", D, F)]


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks, throttle reasons)."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples (set SL_BENCH_OUT to keep them somewhere else); the JSON line carries the summary
        self.path = os.path.join(os.environ.get("SL_BENCH_OUT", tempfile.gettempdir()), f"sl_clocks_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # the sampler's first line, so that the timed region is covered from its start
        t0 = time.time()
        while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
            time.sleep(0.02)

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
def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count() or 1])
    except ImportError:   # numpy's BLAS runs one thread per host core by default
        return os.cpu_count() or 1


def oracle_sample(w):
    """The oracle on a bounded sample of workload w.

    Returns (step, sample_tokens, scale, description): tokens/s of the full
    workload = sample_tokens / (scale * seconds per sample step)."""
    import numpy as np
    import seeded_inputs as si
    from oracle import ce, lora, nf4, stack
    if w["kind"] in ("stack", "layer"):
        ms = 64
        c = si.stack_case(3, 1, ms, w["D"], w["Dkv"], w["F"], w["r"])
        lw = c["layers"][0]
        nf = w["base"] in ("nf4", "nf4dq")
        q = {n: nf4.quantize(lw[n]["W"]) for n in si.PROJ_NAMES} if nf else None  # offline, not timed
        dq = []
        if w["base"] == "nf4dq":   # each absmax group double-quantised as one array (offline, not timed)
            for names in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
                K, Ns = lw[names[0]]["W"].shape[1], [lw[n]["W"].shape[0] for n in names]
                dq.append((names, Ns, K, *nf4.double_quantize(np.concatenate([q[n][1] for n in names]), sum(Ns), K)))

        def base(n):
            return nf4.dequantize_bf16(*q[n], *lw[n]["W"].shape) if nf else lw[n]["W"].astype(np.float64)

        def layer():
            Ws = {}
            if dq:
                for names, Ns, K, qa, a2 in dq:
                    ap, off = nf4.dq_absmax(qa, a2, sum(Ns), K), 0
                    for n, N in zip(names, Ns):
                        Ws[n] = nf4.dequantize_bf16(q[n][0], ap[off * K // 64:(off + N) * K // 64], N, K)
                        off += N
            else:
                Ws = {n: base(n) for n in si.PROJ_NAMES}
            return {n: dict(W=Ws[n], A=lw[n]["A"].astype(np.float64), B=lw[n]["B"].astype(np.float64))
                    for n in si.PROJ_NAMES}

        if w["kind"] == "stack":
            attn = dict(S=ms, theta=w["attn"][1]) if "attn" in w else None
            what = "full decoder layer (attention over one 64-token sequence)" if attn else "layer"
            sft = w.get("sft")
            if sft:   # and 1/L of the head's vocabulary against the same rows
                Vs = sft["V"] // w["L"]
                cc = si.ce_case(5, ms, w["D"], Vs)
                W64 = cc["W"].astype(np.float64)
                nv = int(np.sum(cc["labels"] != -100))

            def step():
                stack.stack_step(c["h0"], c["dh_top"], [layer()], w["alpha"], rnd=True, attn=attn)
                if sft:
                    ce.ce_rows(cc["H"], W64, cc["labels"], max(nv, 1))
            extra = f" and the cross-entropy of the {ms} rows over {Vs} head rows (1/{w['L']} of the vocabulary)" \
                if sft else ""
            return step, ms, w["L"], (f"one full-width {w['base']} {what} (of {w['L']}), {ms} tokens, fwd+bwd "
                                      f"incl. dequantisation{extra}; tokens/s scaled by 1/{w['L']}")
        shp = proj_shapes(w["D"], w["Dkv"], w["F"])
        ys = {n: si.normal_bf16(77 + i, (ms, N), 1.0) for i, (n, N, K) in enumerate(shp)}
        xs = {n: si.normal_bf16(55 + i, (ms, K), 1.0) for i, (n, N, K) in enumerate(shp)}

        def step():
            P = layer()
            for n in si.PROJ_NAMES:
                lora.lora_linear_fwd(xs[n], P[n]["W"], P[n]["A"], P[n]["B"], w["alpha"])
                lora.lora_linear_bwd(xs[n], ys[n], P[n]["W"], P[n]["A"], P[n]["B"], w["alpha"])
        return step, ms, 1, f"the seven linears of one layer at {ms} tokens, fwd+bwd incl. dequantisation"
    if w["kind"] == "attn":   # one sequence, 4 query heads over 1 kv head: 1/64 of the workload
        from oracle import attention
        S, hs = w["S"], 4
        q = si.normal_bf16(61, (S, hs * 128), 1.0)
        k = si.normal_bf16(62, (S, 128), 1.0)
        v = si.normal_bf16(63, (S, 128), 1.0)
        dO = si.normal_bf16(64, (S, hs * 128), 1.0)
        scale = (w["M"] // S) * (w["H"] // hs)

        def step():
            o, _ = attention.attention_fwd(q, k, v, S)
            attention.attention_bwd(q, k, v, o, dO, S)
        return step, w["M"], scale, (f"one {S}-token sequence, {hs} query heads over 1 kv head, fwd+bwd "
                                     f"(1/{scale} of the workload); tokens/s scaled by 1/{scale}")
    # cross-entropy: 16 rows against the whole vocabulary (loss terms and dH rows)
    rows = 16
    cc = si.ce_case(5, rows, w["D"], w["V"])
    W64 = cc["W"].astype(np.float64)
    nv = int(np.sum(cc["labels"] != -100))

    def step():
        ce.ce_rows(cc["H"], W64, cc["labels"], max(nv, 1))
    return step, rows, 1, f"{rows} rows of the {w['M']}-row batch against the full {w['V']}-entry vocabulary"


def cpu_baseline(w):
    step, ms, scale, desc = oracle_sample(w)
    step()
    t0 = time.perf_counter()
    step()
    dt = time.perf_counter() - t0
    return {"value": ms / (scale * dt), "unit": UNIT, "cores": _threads(), "cpu_model": _cpu_model(), "kind": "oracle",
            "sample": f"{desc}; {dt:.2f} s per sample"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    step, ms, scale, desc = oracle_sample(w)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = ms / (scale * dt)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": w["M"] / v * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w["name"], "tokens": w["M"], "sample": desc},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _threads(), "cpu_model": _cpu_model(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- ours
def pinned_h2d_peak(torch, dev):
    """Pinned host -> device copy bandwidth of this machine: 1 GiB, best of 10, CUDA events."""
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
    return (1 << 30) / (best * 1e-3) / 1e9


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
    w = dict(WORKLOADS[args.workload])
    if args.layers and w["kind"] == "stack":
        w["L"] = args.layers
    M = w["M"]
    gen = torch.Generator(device=dev).manual_seed(1234 + rank)
    rnd = lambda shape, std: (torch.randn(*shape, generator=gen, device=dev) * std).to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    extra = {}
    dominant = ("nf4_fwd", "nf4_dx")
    kname = ("gemm_nf4_pair_persistent_kernel / gemm_nf4_pair_kernel (fused NF4 dequant + LoRA fold, "
             "CTA pairs; fwd and dX)")
    h2d_peak = None

    if w["kind"] == "stack":
        kind = {"nf4": sl.SL_WEIGHT_NF4, "nf4dq": sl.SL_WEIGHT_NF4_DQ, "bf16": sl.SL_WEIGHT_BF16}[w["base"]]
        if kind == sl.SL_WEIGHT_BF16:
            dominant = ("bf16_fwd", "bf16_dx")
            kname = "gemm_bf16_pair_persistent_kernel (bf16 base by TMA on CTA pairs + LoRA fold; fwd and dX)"
        D, Dkv, F, L, r, alpha = w["D"], w["Dkv"], w["F"], w["L"], w["r"], w["alpha"]
        shapes = sl.proj_shapes(D, Dkv, F)
        sa, sb = sl.adapter_shapes(D, Dkv, F, r)
        host_blobs, A, B, dA, dB = [], [], [], [], []
        for l in range(L):
            blob = sl.build_layer_blob(kind, D, Dkv, F, [rnd((N, K), 0.02) for N, K in shapes])
            h = torch.empty(blob.numel(), dtype=torch.uint8, pin_memory=True)
            h.copy_(blob)
            host_blobs.append(h)
            del blob
            # each layer's adapters back to back: q/k/v and gate/up run as projection groups
            la, lb = sl.packed_views(sa, torch.bfloat16, dev), sl.packed_views(sb, torch.bfloat16, dev)
            for t, (n0, n1) in zip(la + lb, sa + sb):
                t.copy_(rnd((n0, n1), 0.02))
            A += la
            B += lb
            dA += sl.packed_views(sa, torch.float32, dev)
            dB += sl.packed_views(sb, torch.float32, dev)
        h0 = torch.randn(M, D, generator=gen, device=dev).to(torch.bfloat16).float()
        dh = torch.randn(M, D, generator=gen, device=dev).to(torch.bfloat16).float()
        hL = torch.empty(M, D, device=dev)
        dh0 = torch.empty(M, D, device=dev)
        mix = dict(mixer=sl.SL_MIX_ATTENTION, seq_len=w["attn"][0], rope_theta=w["attn"][1]) if "attn" in w else {}
        stk = sl.Stack(kind, D, Dkv, F, host_blobs, **mix)
        sft = w.get("sft")
        if sft:
            V, chunk = sft["V"], sft["chunk"]
            emb, head = rnd((V, D), 1.0), rnd((V, D), 0.02)
            nfin = torch.ones(D, device=dev)
            tok = torch.randint(0, V, (M,), generator=gen, device=dev, dtype=torch.int32)
            lab = torch.randint(0, V, (M,), generator=gen, device=dev, dtype=torch.int32)
            lab[torch.randperm(M, generator=gen, device=dev)[: round(0.05 * M)]] = -100
            loss = torch.empty(1, device=dev)
            ws = torch.empty(stk.sft_workspace_size(M, r, V, chunk), dtype=torch.uint8, device=dev)

            def step():
                stk.sft_step(sl.SL_MODE_STREAMED, tok, lab, emb, nfin, head, chunk, A, B, r, alpha, loss, dA, dB, ws)
        else:
            ws = torch.empty(stk.workspace_size(M, r), dtype=torch.uint8, device=dev)

            def step():
                stk.step(sl.SL_MODE_STREAMED, h0, dh, A, B, r, alpha, hL, dh0, dA, dB, ws)

        h0_h, dh_h = h0.cpu().pin_memory(), dh.cpu().pin_memory()
        out_h = torch.empty(M, D, dtype=torch.float32, pin_memory=True)
        h0_d, dh_d = torch.empty_like(h0), torch.empty_like(dh)

        def e2e_step():
            h0_d.copy_(h0_h, non_blocking=True)
            dh_d.copy_(dh_h, non_blocking=True)
            stk.step(sl.SL_MODE_STREAMED, h0_d, dh_d, A, B, r, alpha, hL, dh0, dA, dB, ws)
            out_h.copy_(hL, non_blocking=True)
        e2e_bytes = (h0_h.numel() * 4 + dh_h.numel() * 4, out_h.numel() * 4)
        if sft:   # token ids and labels in, the loss out
            tok_h, lab_h = tok.cpu().pin_memory(), lab.cpu().pin_memory()
            loss_h = torch.empty(1, dtype=torch.float32, pin_memory=True)

            def e2e_step():
                tok.copy_(tok_h, non_blocking=True)
                lab.copy_(lab_h, non_blocking=True)
                step()
                loss_h.copy_(loss, non_blocking=True)
            e2e_bytes = (tok_h.numel() * 4 + lab_h.numel() * 4, 4)
        h2d_peak = pinned_h2d_peak(torch, dev)
        wl_extra = {}
        if "attn" in w:
            wl_extra["attention"] = {"seq_len": w["attn"][0], "rope_theta": w["attn"][1], "heads": D // 128,
                                     "kv_heads": Dkv // 128}
        if sft:
            wl_extra["sft"] = {"V": V, "chunk_V": chunk, "ignore_frac": 0.05}
        config = {**wl_extra, "workload": w["name"], "tokens": M, "layers": L, "D": D, "Dkv": Dkv, "F": F, "rank": r,
                  "alpha": alpha, "base": {sl.SL_WEIGHT_NF4: "NF4 blocksize 64 fp32 absmax",
                                           sl.SL_WEIGHT_NF4_DQ: "NF4 blocksize 64, 8-bit absmax (fp32 offset and "
                                                                "scale per 256 blocks)",
                                           sl.SL_WEIGHT_BF16: "bf16"}[kind],
                  "l2": f"inputs larger than L2 ({stk.host_bytes / 1e9:.1f} GB streamed base + activations)"}
    elif w["kind"] == "layer":
        # One decoder layer's seven projections as a framework runs them: q/k/v
        # read the same input and run as one projection group, gate/up likewise;
        # o and down alone.  NF4 weights of a group back to back, adapters too.
        D, Dkv, F, r, alpha = w["D"], w["Dkv"], w["F"], w["r"], w["alpha"]
        shp = dict(zip(("q", "k", "v", "o", "gate", "up", "down"), [(N, K) for _, N, K in proj_shapes(D, Dkv, F)]))
        units = []
        for names in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
            N_g = [shp[n][0] for n in names]
            K = shp[names[0]][1]
            NN = sum(N_g)
            codes = torch.empty(NN * K // 2, dtype=torch.uint8, device=dev)
            absmax = torch.empty(NN * K // 64, dtype=torch.float32, device=dev)
            row = 0
            for N in N_g:   # quantise each projection into its rows of the group weight
                Wt = rnd((N, K), 0.02)
                sl.sl_nf4_quantize(Wt, codes[row * K // 2:(row + N) * K // 2], absmax[row * K // 64:(row + N) * K // 64])
                row += N
                del Wt
            G = len(N_g)
            units.append(dict(w=sl.Weight.nf4(codes, absmax, NN, K), N_g=N_g, G=G, N=NN, K=K, X=rnd((M, K), 1.0),
                              dY=rnd((M, NN), 1.0), A=rnd((G * r, K), 0.02), B=rnd((NN, r), 0.02),
                              Y=torch.empty(M, NN, dtype=torch.bfloat16, device=dev),
                              T=torch.empty(M, G * r, dtype=torch.float32, device=dev),
                              dX=torch.empty(M, K, dtype=torch.bfloat16, device=dev),
                              dA=torch.empty(G * r, K, device=dev), dB=torch.empty(NN, r, device=dev),
                              ws=torch.empty(max(sl.sl_lora_group_workspace_size(M, G, r),
                                                 sl.sl_lora_linear_workspace_size(M, NN, K, r)),
                                             dtype=torch.uint8, device=dev)))

        def step():
            for u in units:
                if u["G"] > 1:
                    sl.sl_lora_group_fwd(u["w"], u["N_g"], u["X"], u["A"], u["B"], r, alpha, u["Y"], u["T"])
                    sl.sl_lora_group_bwd(u["w"], u["N_g"], u["X"], u["dY"], u["A"], u["B"], r, alpha, u["T"], u["dX"],
                                         u["dA"], u["dB"], False, u["ws"])
                else:
                    sl.sl_lora_linear_fwd(u["w"], u["X"], u["A"], u["B"], r, alpha, u["Y"], u["T"], u["ws"])
                    sl.sl_lora_linear_bwd(u["w"], u["X"], u["dY"], u["A"], u["B"], r, alpha, u["T"], u["dX"], u["dA"],
                                          u["dB"], False, u["ws"])

        hosts = [(u["X"].cpu().pin_memory(), u["dY"].cpu().pin_memory()) for u in units]
        res_h = torch.empty(len(units), 8, dtype=torch.float32, pin_memory=True)

        def e2e_step():
            for u, (xh, yh) in zip(units, hosts):
                u["X"].copy_(xh, non_blocking=True)
                u["dY"].copy_(yh, non_blocking=True)
            step()
            for i, u in enumerate(units):   # a slice of every adapter gradient read back
                res_h[i].copy_(u["dA"][0, :8], non_blocking=True)
        e2e_bytes = (sum(xh.numel() * 2 + yh.numel() * 2 for xh, yh in hosts), res_h.numel() * 4)
        # algorithmic work per projection: base fwd + dX (4 M N K) and the LoRA side
        # products (T, U, fold x2, dA, dB); bytes: weights twice, activations
        pj = [shp[n] for n in ("q", "k", "v", "o", "gate", "up", "down")]
        flops = sum(4.0 * M * N * K + 6.0 * M * r * (N + K) for N, K in pj)
        nbytes = sum(2 * (N * K * 0.5625) + 3 * (M * K * 2) + 3 * (M * N * 2) for N, K in pj)
        extra["step_roofline_inputs"] = {"flops": flops, "bytes": nbytes}
        config = {"workload": w["name"], "tokens": M, "D": D, "Dkv": Dkv, "F": F, "rank": r, "alpha": alpha,
                  "base": "NF4 blocksize 64 fp32 absmax", "grouping": "q/k/v and gate/up as projection groups",
                  "l2": "inputs larger than L2 (~0.8 GB touched per step)"}
    elif w["kind"] == "attn":
        S, H, Hkv = w["S"], w["H"], w["Hkv"]
        dominant = ("attn_fwd", "attn_bwd")
        kname = "attn_fwd_kernel + attn_dq_kernel / attn_dkdv_kernel (tcgen05, causal GQA, rotary gradients)"
        q, k, v = rnd((M, H * 128), 1.0), rnd((M, Hkv * 128), 1.0), rnd((M, Hkv * 128), 1.0)
        dO = rnd((M, H * 128), 1.0)
        o = torch.empty(M, H * 128, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(H, M, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        tab = torch.empty(S, 128, device=dev)
        sl.sl_rope_table(S, w["theta"], tab)
        aws = torch.empty(sl.sl_attention_workspace_size(M, H), dtype=torch.uint8, device=dev)

        def step():
            sl.sl_attention_fwd(q, k, v, S, o, lse)
            sl.sl_attention_bwd(q, k, v, o, dO, lse, S, dq, dk, dv, rope_table=tab, ws=aws)

        hosts = [t.cpu().pin_memory() for t in (q, k, v, dO)]
        dq_h = torch.empty(8, H * 128, dtype=torch.bfloat16, pin_memory=True)

        def e2e_step():
            for t, th in zip((q, k, v, dO), hosts):
                t.copy_(th, non_blocking=True)
            step()
            dq_h.copy_(dq[:8], non_blocking=True)
        e2e_bytes = (sum(th.numel() * 2 for th in hosts), dq_h.numel() * 2)
        pairs = (M // S) * H * S * (S + 1) / 2
        # algorithmic work: 2 products forward, 5 backward (S recomputed once), 2 x 128 FLOPs each per
        # visible pair; bytes: q, k, v, dO read, o written and read, dq, dk, dv written
        extra["step_roofline_inputs"] = {"flops": 7 * 2.0 * 128 * pairs,
                                         "bytes": 2.0 * (3 * M * H * 128 + 3 * M * Hkv * 128 + M * H * 128)}
        config = {"workload": w["name"], "tokens": M, "seq_len": S, "heads": H, "kv_heads": Hkv,
                  "rope_theta": w["theta"], "l2": "inputs larger than L2 (q, o, dO, dq 64 MB each)"}
    else:  # cross-entropy
        D, V, chunk = w["D"], w["V"], w["chunk"]
        dominant = ("ce_logits", "ce_dh")
        kname = ("gemm_bf16_pair_persistent_kernel CE epilogues (logits chunk with exp, rescaled dH accumulation; "
                 "CTA pairs)")
        H = rnd((M, D), 1.0)
        Wh = rnd((V, D), 0.02)
        lab = torch.randint(0, V, (M,), generator=gen, device=dev, dtype=torch.int32)
        lab[torch.randperm(M, generator=gen, device=dev)[: round(0.05 * M)]] = -100
        loss = torch.empty(1, device=dev)
        dH = torch.empty(M, D, device=dev)
        ws = torch.empty(sl.sl_ce_workspace_size(M, D, V, chunk), dtype=torch.uint8, device=dev)

        def step():
            sl.sl_ce_fwd_bwd(H, Wh, lab, loss, dH, ws, chunk_V=chunk)

        Hh, labh = H.cpu().pin_memory(), lab.cpu().pin_memory()
        loss_h = torch.empty(1, dtype=torch.float32, pin_memory=True)

        def e2e_step():
            H.copy_(Hh, non_blocking=True)
            lab.copy_(labh, non_blocking=True)
            step()
            loss_h.copy_(loss, non_blocking=True)
        e2e_bytes = (Hh.numel() * 2 + labh.numel() * 4, 4)
        # algorithmic work: the logits GEMM and the dH GEMM (2 x 2 M V D); head read twice
        extra["step_roofline_inputs"] = {"flops": 2 * 2.0 * M * V * D, "bytes": V * D * 2.0 * 2 + M * D * 6.0}
        extra["extra_bytes_per_logit"] = ws.numel() / (M * V)
        config = {"workload": w["name"], "tokens": M, "D": D, "V": V, "chunk_V": chunk, "ignore_frac": 0.05,
                  "l2": "inputs larger than L2 (1.05 GB head read per GEMM pass)"}

    for _ in range(args.warmup):
        step()
    sl.sl_check_device_errors()

    def barrier():
        torch.cuda.synchronize()
        rank_barrier(world)
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return max_over_ranks_of(x, world, dev)

    # timed region: K steps, CUDA events on the compute stream
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    launches0 = sl.sl_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    launches_timed = sl.sl_launch_count() - launches0
    ms_total = max_over_ranks(e0.elapsed_time(e1))
    ms_step = ms_total / args.steps
    value = whole_job_rate(M * args.steps, world, ms_total * 1e-3)
    h2d_step = kernels_step = None
    if w["kind"] == "stack":
        h2d_step, kernels_step = stk.last_step_stats()

    # the same K steps again with a CUDA event pair around every tensor-core GEMM launch
    sl.sl_kernel_timing(True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms_instr = e0.elapsed_time(e1)
    sl.sl_kernel_timing(False)
    timing = {name: sl.sl_kernel_timing_read(i) for i, name in enumerate(sl.TIMED_VARIANTS)}
    clock = {name: sl.sl_kernel_timing_read_clock(i) for i, name in enumerate(sl.TIMED_VARIANTS) if i <= 5}
    sl.sl_check_device_errors()

    # end to end through the public API: host inputs in, host result out, every step
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    e2e = {"value": whole_job_rate(M * args.steps, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": int(e2e_bytes[0]),
           "d2h_bytes_per_step": int(e2e_bytes[1])}

    n_d = sum(timing[k][0] for k in dominant)
    ms_d = sum(timing[k][1] for k in dominant)
    fl_d = sum(timing[k][2] for k in dominant)
    achieved = fl_d / (ms_d * 1e-3) / 1e12 if ms_d > 0 else 0.0
    # DRAM bytes per launch of the dominant kernel: from the committed ncu summary of the same
    # kernels (one layer's NF4 GEMM launches of the 8B stack at M = 1024), only while the kernel
    # sources are the ones it was captured on; null elsewhere
    traffic, traffic_note = None, None
    if w["kind"] == "stack" and w["base"] == "nf4" and w["D"] == 4096 and w["M"] == 1024:
        traffic, why = profiled_traffic("profiles/ncu_nf4_gemm_dram_traffic_stack4_m1024.md", GEMM_SOURCES)
        traffic_note = {"unit": "bytes per launch", "source": why}
    peak, peak_why = pick_peak(peaks, clk)
    burst = peaks["bf16_tflops"]
    sus = peaks.get("bf16_tflops_sustained", burst)
    # the same launches timed by the kernels themselves on the device clock: an event pair
    # around a launch also counts the delay of its timestamps, which a host-to-device copy
    # in flight (the streamed step) stretches by ~16 us
    n_c = sum(clock.get(k, (0, 0.0))[0] for k in dominant)
    ms_c = sum(clock.get(k, (0, 0.0))[1] for k in dominant)
    achieved_c = fl_d / (ms_c * 1e-3) / 1e12 if ms_c > 0 and n_c == n_d else None
    roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} {peak_why}",
                "frac_burst": achieved / burst, "frac_sustained": achieved / sus,
                "achieved_device_clock": achieved_c,
                "frac_device_clock": achieved_c / peak if achieved_c else None,
                "device_clock_timing": "each launch's span from its first CTA past the dependency wait to its last "
                                       "CTA's completed stores (%globaltimer), summed over the same launches",
                "traffic": traffic, "traffic_note": traffic_note, "launches": n_d,
                "avg_launch_ms": ms_d / max(1, n_d),
                "share_of_step": ms_d / ms_instr,
                "timing": "per-launch CUDA event pairs (libsl, on the launching stream) over a second timed "
                          "region of the same K steps"}
    per_variant = {}
    for k, v in timing.items():
        if not v[0]:
            continue
        rate = v[2] / (v[1] * 1e-3) if v[1] else 0.0
        per_variant[k] = ({"launches": v[0], "ms": v[1], "gbs": rate / 1e9} if k in sl.RANK_R_VARIANTS
                          else {"launches": v[0], "ms": v[1], "tflops": rate / 1e12})
        if k in clock and clock[k][0] == v[0] and clock[k][1] > 0:
            per_variant[k]["ms_device_clock"] = clock[k][1]
            per_variant[k]["tflops_device_clock"] = v[2] / (clock[k][1] * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded device RNG)",
            "config": dict(config, parallelism=f"replicas x{world} (no collective on the data path)"),
            "roofline": roofline, "kernels": per_variant, "e2e": e2e, "clocks": clk,
            "gpu_launches": int(launches_timed)}
    if w["kind"] == "stack":
        line["stream"] = {"bound": "pcie_h2d", "h2d_bytes_per_step": h2d_step,
                          "achieved_gbs": h2d_step / (ms_step * 1e-3) / 1e9, "peak_gbs": h2d_peak,
                          "frac": h2d_step / (ms_step * 1e-3) / 1e9 / h2d_peak,
                          "peak_source": "measured in this run: pinned 1 GiB cudaMemcpyAsync, best of 10"}
        line["preflight"] = {"host_bytes": stk.host_bytes, "buffer_bytes": stk.buffer_bytes}
        if not args.no_resident:
            dev_blobs = [hb.to(dev) for hb in host_blobs]
            stk_r = sl.Stack(kind, D, Dkv, F, host_blobs, dev_blobs, **mix)
            stk_r.step(sl.SL_MODE_RESIDENT, h0, dh, A, B, r, alpha, hL, dh0, dA, dB, ws)
            barrier()
            e0.record(stream)
            nres = max(2, min(args.steps, 5))
            for _ in range(nres):
                stk_r.step(sl.SL_MODE_RESIDENT, h0, dh, A, B, r, alpha, hL, dh0, dA, dB, ws)
            e1.record(stream)
            barrier()
            line["resident"] = {"tokens_per_s": M * nres / (e0.elapsed_time(e1) * 1e-3),
                                "ms_per_step": e0.elapsed_time(e1) / nres}
            # the same resident steps with a CUDA event pair around every tensor-core launch
            sl.sl_kernel_timing(True)
            barrier()
            e0.record(stream)
            for _ in range(nres):
                stk_r.step(sl.SL_MODE_RESIDENT, h0, dh, A, B, r, alpha, hL, dh0, dA, dB, ws)
            e1.record(stream)
            barrier()
            sl.sl_kernel_timing(False)
            rk = {}
            for i, name in enumerate(sl.TIMED_VARIANTS):
                n_, ms_, wk = sl.sl_kernel_timing_read(i)
                if n_:
                    rate = wk / (ms_ * 1e-3) if ms_ else 0.0
                    rk[name] = ({"launches": n_, "ms_per_step": ms_ / nres, "gbs": rate / 1e9}
                                if name in sl.RANK_R_VARIANTS else
                                {"launches": n_, "ms_per_step": ms_ / nres, "tflops": rate / 1e12})
                    if i <= 5:
                        nc_, msc_ = sl.sl_kernel_timing_read_clock(i)
                        if nc_ == n_ and msc_ > 0:
                            rk[name]["tflops_device_clock"] = wk / (msc_ * 1e-3) / 1e12
            line["resident"]["kernels"] = rk
            line["resident"]["ms_per_step_timed"] = e0.elapsed_time(e1) / nres
            # the pages' exactness check at this configuration: one more streamed step on the same
            # inputs into separate outputs (adapters laid out the same way), compared bit for bit
            # with the resident step's hL, dh0 and every dA, dB
            hL_s, dh0_s = torch.empty_like(hL), torch.empty_like(dh0)
            dA_s, dB_s = [], []
            for _ in range(L):
                dA_s += sl.packed_views(sa, torch.float32, dev)
                dB_s += sl.packed_views(sb, torch.float32, dev)
            stk.step(sl.SL_MODE_STREAMED, h0, dh, A, B, r, alpha, hL_s, dh0_s, dA_s, dB_s, ws)
            torch.cuda.synchronize()
            same = lambda x, y: torch.equal(x.view(torch.int32), y.view(torch.int32))
            bad = [n for n, x, y in [("hL", hL_s, hL), ("dh0", dh0_s, dh0)] if not same(x, y)]
            bad += [f"dA[{i}]" for i, (x, y) in enumerate(zip(dA_s, dA)) if not same(x, y)]
            bad += [f"dB[{i}]" for i, (x, y) in enumerate(zip(dB_s, dB)) if not same(x, y)]
            line["streamed_equals_resident"] = not bad
            line["streamed_vs_resident"] = {"compared": f"hL, dh0 and {len(dA) + len(dB)} adapter gradients",
                                            "mismatched": bad[:8]}
            sl.sl_check_device_errors()
            stk_r.close()
            del dev_blobs
    else:
        fl, nb = extra["step_roofline_inputs"]["flops"], extra["step_roofline_inputs"]["bytes"]
        t_roof = max(fl / (peaks["bf16_tflops"] * 1e12), nb / (peaks["hbm_gbs"] * 1e9))
        sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        t_roof_s = max(fl / (sus * 1e12), nb / (peaks["hbm_gbs"] * 1e9))
        pk, pk_why = pick_peak(peaks, clk)
        t_roof_c = max(fl / (pk * 1e12), nb / (peaks["hbm_gbs"] * 1e9))
        line["step_roofline"] = {"frac_at_clock": t_roof_c / (ms_step * 1e-3), "peak_at_clock": f"{peak_src} {pk_why}",
                                 "algorithmic_flops": fl, "algorithmic_bytes": nb,
                                 "roofline_ms": t_roof * 1e3, "frac": t_roof / (ms_step * 1e-3),
                                 "peaks": f"{peak_src} bf16_tflops (burst) and hbm_gbs",
                                 "roofline_ms_sustained": t_roof_s * 1e3,
                                 "frac_sustained": t_roof_s / (ms_step * 1e-3),
                                 "peaks_sustained": f"{peak_src} bf16_tflops_sustained (multi-ms step under the "
                                                    "power cap) and hbm_gbs"}
        if "extra_bytes_per_logit" in extra:
            line["extra_device_bytes_per_logit"] = extra["extra_bytes_per_logit"]
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if w["kind"] == "stack":
        stk.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: 10 for the stacks, 200 for layer8b, 100 for attn8b, 50 for ce)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="stack8b")
    ap.add_argument("--layers", type=int, default=0, help="stack depth override (quick checks only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-resident", action="store_true")
    args = ap.parse_args()
    if args.steps <= 0:
        args.steps = {"layer8b": 200, "ce": 50, "attn8b": 100}.get(args.workload, 10)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
