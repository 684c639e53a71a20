#!/usr/bin/env python3
"""Benchmark of the exact streaming attention forward on GB300.

One step = one call of the forward pass over the whole workload (default:
the packed variable-length causal batch, 16 sequences with seed-7 lengths,
H=16, D=128, BF16).  Prints ONE JSON line with throughput in TFLOP/s
(convention 4*N^2*D per head, halved for causal), ms/step, the roofline of
the kernel, an end-to-end number through the host-buffer C entry point, the
CPU oracle baseline, and per-workload microsecond timings.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the FP64 CPU oracle as reference arm

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of
the workload (the forward pass has no cross-GPU exchange); value = total work
of all ranks / max elapsed time over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16 peak; µs/call (1 GPU)"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# Per-workload timing, by family: the workloads of one family are variants of one problem (a
# layout, a mask, a scaled input), timed in a fresh random order within each sample, as the pages
# time their candidate kernels; families run one after another, so that a small problem's samples
# do not start from caches another, unrelated problem has just swept.
PER_CONFIG_FAMILIES = [["n129_d32_f16_causal"],
                       ["n512_d64_f16_causal", "n512_d64_f16_noncausal", "n512_d64_f16_causal_qx30"],
                       ["b4_h16_n4096_d128_bf16", "b4_h16_n4096_d128_bf16_bnhd"],
                       ["gqa_b2_h32x8_n8192_d128_bf16"], ["varlen16_h16_d128_bf16"], ["chunk2048_cache16384_gqa"],
                       ["window4096_n16384", "global64_window4096_n16384"], ["decode_b8_h32x8_k32768"],
                       ["bwd_b4_h16_n4096_d128_bf16", "bwd_gqa_b2_h32x8_n8192_d128_bf16"]]
PER_CONFIG = [n for fam in PER_CONFIG_FAMILIES for n in fam]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="varlen16_h16_d128_bf16")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload microbenchmarks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    """Ranks from torchrun's environment: NCCL over one GPU per rank, or gloo
    on a host without GPUs (where only the reference arm and the rank
    plumbing run)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


KERNEL_SOURCES = {"attn_fwd_kernel": ("attn_fwd_kernel.cuh", "sm103_ptx.cuh"),
                  "attn_bwd_kernel": ("attn_bwd_kernel.cuh", "sm103_ptx.cuh")}


def kernel_source_digest(kernel: str = "attn_fwd_kernel"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_19_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(w):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu summary, if it was taken on the current kernel source;
    else None."""
    kernel = "attn_bwd_kernel" if w.backward else "attn_fwd_kernel"
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f).get("kernels", {}).get(kernel, {})
    except (OSError, ValueError):
        return None
    if d.get("source_sha256") != kernel_source_digest(kernel):
        return None
    entry = d.get("workloads", {}).get(w.name)
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- GPU side

def device_inputs(w, device):
    """Seeded inputs copied to the device in the workload's storage layout, plus
    preallocated outputs (nothing is allocated inside timed regions)."""
    import torch
    from exact_tiled_attention_19_gb300 import workloads as W
    inp = W.make_inputs(w)
    dev = {}
    for n in ("q", "k", "v"):
        t = inp[n]
        if w.layout == "bnhd":
            dev[n] = t.permute(0, 2, 1, 3).contiguous().to(device).permute(0, 2, 1, 3)
        else:
            dev[n] = t.to(device)
    if w.layout == "varlen":
        T = sum(w.seqlens)
        dev["cu"] = inp["cu_seqlens"].to(device)
        dev["cu_host"] = inp["cu_seqlens"]
        if "cu_seqlens_k" in inp:
            dev["cu_k"] = inp["cu_seqlens_k"].to(device)
        dev["o"] = torch.empty((T, w.Hq, w.D), dtype=w.dtype, device=device)
        dev["lse"] = torch.empty((w.Hq, T), dtype=torch.float32, device=device)
    else:
        dev["o"] = torch.empty((w.B, w.Hq, w.N, w.D), dtype=w.dtype, device=device)
        dev["lse"] = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=device)
    if w.backward:
        from exact_tiled_attention_19_gb300 import binding
        g = torch.Generator().manual_seed(1)
        inp["dout"] = torch.randn(inp["q"].shape, generator=g, dtype=torch.float32).to(w.dtype)
        dev["dout"] = inp["dout"].to(device)
        win = dict(window_left=w.window_left, window_right=w.window_right)
        binding.attention(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale, out=dev["o"],
                          lse=dev["lse"], **win)
        dev["dq"] = torch.empty_like(dev["q"])
        dev["dk"] = torch.empty_like(dev["k"])
        dev["dv"] = torch.empty_like(dev["v"])
        dev["ws"] = torch.empty(max(binding.attn_bwd_workspace_size(w.B, w.Hq, w.N, w.D), 1), dtype=torch.uint8,
                                device=device)
        torch.cuda.synchronize()
    if w.splitkv:
        from exact_tiled_attention_19_gb300 import binding
        rc, n = binding.attn_fwd_splitkv_plan(w.B, w.Hq, w.Hkv, w.N, w.keys)
        assert rc == 0, rc
        dev["splits"] = n
        need = binding.attn_fwd_splitkv_workspace_size(w.B, w.Hq, w.N, w.D, n)
        dev["ws"] = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    return inp, dev


def launches_per_call(w):
    """Kernels one call launches: the split-KV path adds the merge launch,
    the backward pass a launch before (row statistics) and after (dQ)."""
    if w.backward:
        return 3
    return 2 if w.splitkv and w.keys > 0 else 1


def make_call(w, dev, stream):
    from exact_tiled_attention_19_gb300 import binding
    win = dict(window_left=w.window_left, window_right=w.window_right)
    if w.layout == "varlen":
        kw = {}
        if "cu_k" in dev:
            kw = dict(cu_seqlens_k=dev["cu_k"], max_seqlen_k=max(w.seqlens_k))

        def call():
            binding.attention_varlen(dev["q"], dev["k"], dev["v"], dev["cu"], max(w.seqlens), causal=w.causal,
                                     scale=w.scale, out=dev["o"], lse=dev["lse"], stream=stream, **kw, **win)
    elif w.backward:
        def call():
            binding.attention_backward(dev["q"], dev["k"], dev["v"], dev["o"], dev["lse"], dev["dout"],
                                       causal=w.causal, scale=w.scale, dq=dev["dq"], dk=dev["dk"], dv=dev["dv"],
                                       workspace=dev["ws"], stream=stream, **win)
    elif w.num_global > 0:
        def call():
            binding.attention_global(dev["q"], dev["k"], dev["v"], num_global=w.num_global, causal=w.causal,
                                     scale=w.scale, out=dev["o"], lse=dev["lse"], stream=stream, **win)
    elif w.splitkv:
        def call():
            binding.attention_splitkv(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale,
                                      num_splits=dev["splits"], workspace=dev["ws"], out=dev["o"], lse=dev["lse"],
                                      stream=stream, **win)
    else:
        def call():
            binding.attention(dev["q"], dev["k"], dev["v"], causal=w.causal, scale=w.scale, out=dev["o"],
                              lse=dev["lse"], stream=stream, **win)
    return call


def time_steps(call, stream, K, W, world, sampler=None):
    """W untimed calls, then exactly K timed calls bracketed by a barrier and
    a device synchronisation; CUDA events on the launching stream time the
    whole region and every launch."""
    import torch
    for _ in range(W):
        call()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if sampler:
        sampler.start()
        time.sleep(0.3)  # let the sampler take its first readings
    start.record(stream)
    for a, b in evs:
        a.record(stream)
        call()
        b.record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    total_ms = start.elapsed_time(end)
    per_launch_ms = [a.elapsed_time(b) for a, b in evs]
    return total_ms, per_launch_ms, clocks


def time_e2e(w, inp, dev, stream, K, W, world):
    """The same workload through the host-buffer C entry point: each step
    copies Q, K, V (and cu_seqlens) from pinned host memory, runs the kernel
    and copies O and lse back."""
    import torch
    from exact_tiled_attention_19_gb300 import binding
    if not w.square or w.backward or w.splitkv:
        return None  # the host-buffer entry points run the plain forward pass
    pin = {n: inp[n].contiguous().pin_memory() for n in ("q", "k", "v")}
    o_h = torch.empty(dev["o"].shape, dtype=w.dtype).pin_memory()
    l_h = torch.empty(dev["lse"].shape, dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty(pin[n].shape, dtype=w.dtype, device=dev["o"].device) for n in ("q", "k", "v"))
    dtype = 1 if w.dtype == torch.bfloat16 else 0
    h = stream.cuda_stream
    if w.layout == "varlen":
        cu_h = inp["cu_seqlens"].contiguous().pin_memory()
        cu_d = torch.empty_like(dev["cu"])
        T = sum(w.seqlens)

        def call():
            rc = binding.attn_fwd_varlen_host(pin["q"].data_ptr(), pin["k"].data_ptr(), pin["v"].data_ptr(),
                                              o_h.data_ptr(), l_h.data_ptr(), cu_h.data_ptr(), dq.data_ptr(),
                                              dk.data_ptr(), dv.data_ptr(), dev["o"].data_ptr(),
                                              dev["lse"].data_ptr(), cu_d.data_ptr(), len(w.seqlens),
                                              max(w.seqlens), T, w.Hq, w.Hkv, w.D, dtype, int(w.causal), w.scale, h)
            assert rc == 0, rc
        h2d = sum(pin[n].numel() * pin[n].element_size() for n in pin) + cu_h.numel() * 4
    else:
        if w.layout != "bhnd":
            return None  # the host entry point takes contiguous [B,H,N,D] buffers

        def call():
            rc = binding.attn_fwd_host(pin["q"].data_ptr(), pin["k"].data_ptr(), pin["v"].data_ptr(),
                                       o_h.data_ptr(), l_h.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                       dv.data_ptr(), dev["o"].data_ptr(), dev["lse"].data_ptr(), w.B, w.Hq,
                                       w.Hkv, w.N, w.D, dtype, int(w.causal), w.scale, h)
            assert rc == 0, rc
        h2d = sum(pin[n].numel() * pin[n].element_size() for n in pin)
    d2h = o_h.numel() * o_h.element_size() + l_h.numel() * 4
    # Three timed regions of K steps each; the median region is reported.  A
    # region lasts a fraction of a second, and a stall of the host's copy path
    # (tens of milliseconds, seen now and then on these shared hosts) would
    # otherwise decide the figure.
    regions = []
    for rep in range(3):
        total_ms, _, _ = time_steps(call, stream, K, W if rep == 0 else 1, world)
        regions.append(max_over_ranks(total_ms, world) / K)
    # sanity: the host copy of O equals the device result of the resident run
    ok = bool(torch.equal(o_h, dev["o"].cpu()))
    return {"ms_per_step": statistics.median(regions), "ms_per_step_regions": [round(x, 4) for x in regions],
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "matches_device_result": ok}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = sum(i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def oracle_sample(w):
    """A bounded, deterministic slice of the workload for the CPU oracle:
    (description, list of (q_rows, k, v, positions) problems, convention FLOPs).
    Packed batch: the sequence whose length is closest to 10000, every head.
    Batched: batch 0, the first two query heads, every row."""
    from exact_tiled_attention_19_gb300 import workloads as W
    import torch
    g = torch.Generator().manual_seed(0)
    if w.layout == "varlen":
        s = min(range(len(w.seqlens)), key=lambda i: abs(w.seqlens[i] - 10000))
        L = w.seqlens[s]
        inp = W.make_inputs(w)
        t0 = int(inp["cu_seqlens"][s])
        heads = list(range(w.Hq))
        probs = []
        for h in heads:
            hk = h // (w.Hq // w.Hkv)
            probs.append(tuple(inp[n][t0:t0 + L, hh].float().double().numpy()
                               for n, hh in (("q", h), ("k", hk), ("v", hk))))
        desc = f"sequence {s} (L={L}) of the packed batch, all {w.Hq} heads"
        flops = 4.0 * L * L * w.D * len(heads) / (2 if w.causal else 1)
        return desc, probs, flops
    inp = W.make_inputs(w)
    heads = list(range(min(2, w.Hq)))
    probs = []
    dout = torch.randn(inp["q"].shape, generator=g, dtype=torch.float32).to(w.dtype) if w.backward else None
    for h in heads:
        hk = h // (w.Hq // w.Hkv)
        prob = tuple(inp[n][0, hh].float().double().numpy() for n, hh in (("q", h), ("k", hk), ("v", hk)))
        if w.backward:
            prob = prob + (dout[0, h].float().double().numpy(),)
        probs.append(prob)
    desc = f"batch 0, query heads {heads}, all {w.N} rows"
    flops = head_flops(w) * len(heads)
    return desc, probs, flops


def head_flops(w):
    """The metric's FLOPs of one (sequence, query head) of a batched workload
    (every one is the same size)."""
    return w.flops() / (w.B * w.Hq)


def run_oracle_problem(prob, w):
    import oracle
    win = dict(window_left=w.window_left, window_right=w.window_right)
    if w.num_global > 0:
        win["num_global"] = w.num_global
    if w.backward:
        q, k, v, do = (x[None, None] for x in prob)
        return oracle.attention_backward_dense(q, k, v, do, causal=w.causal, scale=w.scale, **win)
    q, k, v = prob
    return oracle.attention_rows(q, k, v, np.arange(q.shape[0]), causal=w.causal, scale=w.scale, **win)


def cpu_baseline(w):
    desc, probs, flops = oracle_sample(w)
    t0 = time.perf_counter()
    for prob in probs:
        run_oracle_problem(prob, w)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": desc + " (NumPy float64; BLAS matmuls multi-threaded, elementwise steps on one core)",
            "seconds": dt, "host_cores": len(os.sched_getaffinity(0)), "cpu_model": provenance_cpu_model()}


def reference_arm(args, w, world, rank):
    """Times the FP64 CPU oracle as it stands: every step is one head of the
    oracle sample (rank 0 only)."""
    if rank != 0:
        return None
    desc, probs, flops = oracle_sample(w)
    step_flops = flops / len(probs)  # one head per step; every head of the sample is the same size
    for i in range(args.warmup):
        run_oracle_problem(probs[i % len(probs)], w)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run_oracle_problem(probs[i % len(probs)], w)
    dt = time.perf_counter() - t0
    value = step_flops * args.steps / dt / 1e12
    sample = f"one head per step of {desc}"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_config(w, n_gpus):
    cfg = {"workload": f"{w.name}: {w.description}", "global_batch": w.total_tokens * n_gpus,
           "seq_len": w.N if w.layout != "varlen" else f"packed, max {max(w.seqlens)}",
           "heads": f"Hq={w.Hq} Hkv={w.Hkv}", "head_dim": w.D, "causal": w.causal,
           "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU",
           "l2": f"inputs larger than L2 ({w.io_bytes() / 1e9:.2f} GB algorithmic bytes per step)"
           if w.io_bytes() > 200e6 else "warm L2 (inputs smaller than L2)"}
    if w.layout != "varlen" and w.keys != w.N:
        cfg["key_len"] = w.keys
    if w.window_left >= 0 or w.window_right >= 0:
        cfg["window"] = {"left": w.window_left, "right": w.window_right}
    if w.num_global > 0:
        cfg["global_tokens"] = w.num_global
    if not w.square:
        cfg["flops"] = "exact eligible (query, key) pairs x 4 x D per head"
    return cfg


# ---------------------------------------------------------------- correctness gate and per-workload timing

def correctness_gate(w, inp, dev, pool=None):
    """Every timed variant first matches the oracle.  Small workloads: every
    element.  Large ones: every (batch or sequence, head) on a stratified row
    sample (the first and last 256 rows of each sequence and both rows at
    every 128-row boundary), the oracle spread over the host cores.  Returns
    (ok, max |dO|, max |dlse|) for the forward pass, (ok, worst error / bound,
    None) for the backward pass."""
    import oracle
    import torch
    from tests.oracle_pool import compare_workload, stratified_rows
    tol = 2e-3 if w.dtype == torch.float16 else 1e-2
    f64 = lambda t: t.float().double().cpu().numpy()
    if w.backward:
        ok, ratio = backward_gate(w, inp, dev, f64)
        return ok, ratio, None
    o, lse = dev["o"], dev["lse"]
    if not bool(torch.isfinite(o).all()) or not bool(torch.isfinite(lse).all()):
        return False, float("inf"), float("inf")
    if w.layout != "varlen" and w.N * w.B * w.Hq <= 4096:
        ro, rl = oracle.attention_dense(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), causal=w.causal, scale=w.scale,
                                        window_left=w.window_left, window_right=w.window_right,
                                        num_global=w.num_global)
        do, dl = float(np.max(np.abs(f64(o) - ro))), float(np.max(np.abs(f64(lse) - rl)))
    else:
        r = compare_workload(w, inp, o.cpu(), lse.cpu(), rows_of=stratified_rows, pool=pool)
        do, dl = r["max_abs_dO"], r["max_abs_dlse"]
    return do <= tol and dl <= 1e-3, do, dl


def backward_gate(w, inp, dev, f64):
    """Sampled rows of (batch 0, KV head 0) of dQ, dK, dV against the oracle,
    each element within u |G| + 8 u M (M the sum of the absolute values of
    its terms, u the input type's half-ulp), as in the GPU parity tests.
    Returns (ok, worst error / bound)."""
    import oracle
    import torch
    u = 2.0 ** -9 if w.dtype == torch.bfloat16 else 2.0 ** -12
    g = w.Hq // w.Hkv
    rows = np.array(sorted({0, 1, 127, 128, w.N // 2, w.N - 1}))
    out = oracle.attention_backward_sampled(f64(inp["q"][0, :g]), f64(inp["k"][0, 0]), f64(inp["v"][0, 0]),
                                            f64(inp["dout"][0, :g]), rows, rows, causal=w.causal, scale=w.scale,
                                            group=g, window_left=w.window_left, window_right=w.window_right,
                                            magnitudes=True)
    gpu = (f64(dev["dq"][0, :g])[:, rows], f64(dev["dk"][0, 0])[rows], f64(dev["dv"][0, 0])[rows])
    worst = 0.0
    for got, ref, mag in zip(gpu, out[:3], out[3:]):
        bound = u * np.abs(ref) + 8 * u * mag + 1e-6 * max(float(mag.max()), 1e-30)
        worst = max(worst, float((np.abs(got - ref) / bound).max()))
    return worst <= 1.0, worst


def per_config_report(stream, device, peaks, pool, gated=None, samples=7, calls=20, warm=5, seed=0):
    """Page-style timing of every workload: a correctness gate first; 5
    warm-up calls; 7 samples of 20 calls each, per call the median (with min,
    max and every raw sample kept), CUDA events and CUDA-graph replay as
    separate experiments.  Within each sample the workloads of one family
    (PER_CONFIG_FAMILIES) run in a fresh random order (seeded, recorded)."""
    from exact_tiled_attention_19_gb300 import workloads as W
    import torch
    gated = gated or {}
    rng = np.random.default_rng(seed)
    out, orders = {}, {}
    for fam in PER_CONFIG_FAMILIES:
        live = {}
        for name in fam:
            w = W.WORKLOADS[name]
            inp, dev = device_inputs(w, device)
            call = make_call(w, dev, stream)
            with torch.cuda.stream(stream):
                call()
            torch.cuda.synchronize()
            ok, err, err_lse = gated[name] if name in gated else correctness_gate(w, inp, dev, pool)
            entry = {"gate": "pass" if ok else "FAIL"}
            if w.backward:
                entry["gate_error_to_bound_ratio"] = err
            else:
                entry["gate_max_abs_dO"] = err
                entry["gate_max_abs_dlse"] = err_lse
            out[name] = entry
            del inp
            if ok:
                live[name] = (w, dev, call)
        graphs, ev, gr = {}, {n: [] for n in live}, {n: [] for n in live}
        with torch.cuda.stream(stream):
            for name, (w, dev, call) in live.items():
                for _ in range(warm):
                    call()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(calls):
                        call()
                g.replay()
                graphs[name] = g
            torch.cuda.synchronize()
            fam_orders = []
            for _ in range(samples):
                order = [str(n) for n in rng.permutation(list(live))]
                fam_orders.append(order)
                for name in order:
                    call = live[name][2]
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(calls):
                        call()
                    b.record(stream)
                    b.synchronize()
                    ev[name].append(a.elapsed_time(b) * 1e3 / calls)
                    a.record(stream)
                    graphs[name].replay()
                    b.record(stream)
                    b.synchronize()
                    gr[name].append(a.elapsed_time(b) * 1e3 / calls)
            orders[" / ".join(fam)] = fam_orders
        for name, (w, dev, call) in live.items():
            e, g = ev[name], gr[name]
            entry = out[name]
            entry.update({"us_event_median": round(statistics.median(e), 3), "us_event_min": round(min(e), 3),
                          "us_event_max": round(max(e), 3), "us_graph_median": round(statistics.median(g), 3),
                          "us_graph_min": round(min(g), 3), "us_graph_max": round(max(g), 3),
                          "us_event_samples": [round(x, 3) for x in e], "us_graph_samples": [round(x, 3) for x in g]})
            us = entry["us_graph_median"]
            tf = w.flops() / (us * 1e-6) / 1e12
            entry["tflops_graph"] = round(tf, 2)
            entry["frac_of_bf16_peak"] = round(tf / peaks["bf16_tflops"], 4)
            entry["achieved_gbs_graph"] = round(w.io_bytes() / (us * 1e-6) / 1e9, 1)
            entry["frac_of_hbm"] = round(entry["achieved_gbs_graph"] / peaks["hbm_gbs"], 4)
            if w.splitkv:
                entry["num_splits"] = dev["splits"]
        del graphs, live
        torch.cuda.empty_cache()
    meta = {"samples": samples, "calls_per_sample": calls, "warmup_calls": warm, "order_seed": seed,
            "families": PER_CONFIG_FAMILIES, "variant_order_per_sample": orders}
    return out, meta


def provenance_cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    cpu_model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    cpu_model = line.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    try:
        lscpu = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in lscpu.splitlines():
            if line.startswith("Model name:"):
                cpu_model = line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return cpu_model


def provenance(device_index):
    """Runtime metadata: source hashes, GPU and CPU names, host cores."""
    import platform
    import torch
    csrc = os.path.join(ROOT, "exact_tiled_attention_19_gb300", "csrc")
    every = hashlib.sha256()
    for name in sorted(os.listdir(csrc)) + ["../../include/etattn.h"]:
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                every.update(name.encode() + b"\0" + f.read())
    return {"source_sha256": {**{k: kernel_source_digest(k) for k in KERNEL_SOURCES},
                              "csrc_and_header": every.hexdigest()},
            "bench_py_sha256": hashlib.sha256(open(os.path.abspath(__file__), "rb").read()).hexdigest(),
            "gpu_name": torch.cuda.get_device_name(device_index), "cuda_runtime": torch.version.cuda,
            "torch": torch.__version__, "cpu_model": provenance_cpu_model(),
            "host_cores": len(os.sched_getaffinity(0)),
            "python": platform.python_version()}


def main():
    args = parse_args()
    from exact_tiled_attention_19_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    world, rank, local = dist_setup()

    if args.impl == "reference":
        line = reference_arm(args, w, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    # The oracle's process pool (correctness gates) is started with "spawn"
    # before any GPU work, on the rank that gates.
    from tests.oracle_pool import spawn_pool
    from contextlib import nullcontext
    with (spawn_pool() if rank == 0 else nullcontext()) as pool:
        return run_ours(args, w, world, rank, local, pool)


def run_ours(args, w, world, rank, local, pool):
    import torch
    from exact_tiled_attention_19_gb300 import binding
    binding.load_library()  # fails loudly if the CUDA library is missing
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)

    inp, dev = device_inputs(w, device)
    call = make_call(w, dev, stream)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    gate = correctness_gate(w, inp, dev, pool) if rank == 0 else (True, 0.0, 0.0)
    if not gate[0]:
        print(json.dumps({"metric": METRIC, "error": f"correctness gate failed (max |dO| or error/bound {gate[1]}, "
                                                     f"max |dlse| {gate[2]})"}))
        return 1

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    with torch.cuda.stream(stream):
        total_ms, per_launch, clocks = time_steps(call, stream, args.steps, max(3, args.warmup), world, sampler)
    total_ms = max_over_ranks(total_ms, world)
    flops = w.flops()
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    launch_ms = statistics.mean(per_launch)
    achieved = flops / (launch_ms * 1e-3) / 1e12
    status = binding.etattn_read_device_status(clear=True, stream=stream.cuda_stream)

    e2e = None
    if not args.no_e2e:
        with torch.cuda.stream(stream):
            r = time_e2e(w, inp, dev, stream, args.steps, max(3, args.warmup), world)
        if r is not None:
            e2e = {"value": flops * world / (r["ms_per_step"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": r["h2d_bytes_per_step"], "d2h_bytes_per_step": r["d2h_bytes_per_step"],
                   "ms_per_step": r["ms_per_step"], "ms_per_step_regions": r["ms_per_step_regions"],
                   "timing": f"median of three timed regions of {args.steps} steps",
                   "host_result_matches_device": r["matches_device_result"]}

    del dev
    torch.cuda.empty_cache()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    per_cfg = per_cfg_meta = None
    if rank == 0 and not args.no_per_config:
        per_cfg, per_cfg_meta = per_config_report(stream, device, peaks, pool, gated={w.name: gate})

    if rank != 0:
        return 0
    if w.memory_bound:
        gbs = w.io_bytes() / (launch_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": measured_traffic(w),
                    "peak_source": "HBM copy, measured (MEASURED_PEAKS.json)" if peak_src == "measured"
                    else "HBM copy, fallback",
                    "algorithmic_bytes_per_launch": w.io_bytes(), "algorithmic_flops_per_launch": flops,
                    "launch_ms_mean": round(launch_ms, 4),
                    "note": "a split-KV call is two launches (slices, merge); the time covers both"
                    if w.splitkv else ""}
    else:
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic": measured_traffic(w),
                    "peak_source": f"bf16 dense burst, {peak_src} (MEASURED_PEAKS.json)"
                    if peak_src == "measured" else "bf16 dense burst, fallback",
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "algorithmic_flops_per_launch": flops, "exact_causal_flops_per_launch": w.flops_exact(),
                    "algorithmic_bytes_per_launch": w.io_bytes(), "launch_ms_mean": round(launch_ms, 4)}
    roofline["launch_ms_samples"] = [round(x, 4) for x in per_launch]
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f16",
        "data": "synthetic (seeded N(0,1) Q/K/V; seed-7 packed lengths)", "config": workload_config(w, world),
        "us_per_call": round(total_ms / args.steps * 1e3, 2),
        "frac_of_bf16_peak": round(value / world / peaks["bf16_tflops"], 4),
        "roofline": roofline,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps * launches_per_call(w), "clocks": clocks,
        "device_status": status,
        "correctness_gate": {"max_abs_dO" if not w.backward else "error_to_bound_ratio": gate[1],
                             "max_abs_dlse": gate[2],
                             "rows": "every element" if (w.layout != "varlen" and w.N * w.B * w.Hq <= 4096)
                             else "every head; first and last 256 rows of each sequence and every 128-row boundary"},
        "provenance": provenance(device.index),
        "per_config": per_cfg, "per_config_timing": per_cfg_meta,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
