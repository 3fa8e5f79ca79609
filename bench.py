"""Benchmark: varlen attention forward TFLOPS and fraction of the GB300 roofline.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                        [--workload NAME] [--no-extra] [--no-cpu-baseline]

One step = one fa_varlen_fwd call over the whole packed batch of the
workload.  The default workload is the largest single-GPU configuration: one
65536-token image, 16 heads, head dim 128, non-causal, returning the LSE
(`long_65536`).  Inputs are resident in HBM before timing; L2 is flushed (a
512 MB write) before every timed step and outside its CUDA-event pair.
Prints one JSON line on rank 0.  Unless --no-extra is given, the line also
carries an "extra" block that times every other workload of the suite (ViT
full and windowed at every head dim, the long sequences, the MLA prefill
cases, sparse-MLA decode, split-KV and packed-GQA cases) with its roofline
fraction; those inputs are drawn on the device (parity is the tests' job).

`--impl reference` times the fp64 CPU oracle (the only reference arm this
method has) on a bounded sample of the same workload and prints the same
line with "impl": "reference".

Multi-GPU: the path has no exchange step, so N > 1 runs N independent
replicas (one per rank, launched by torchrun); the timed region is bracketed
by barriers and the maximum over ranks is taken.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from varlen_flashattention_forward_gb300 import metrics, workloads  # noqa: E402

METRIC = "varlen attention fwd TFLOPS and % of GB300 BF16 tensor peak (decode: % HBM BW)"
L2_FLUSH_BYTES = 512 << 20

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# the dominant kernel, from the ncu captures summarised in profiles/.  A value
# holds only for the kernel source it was measured on (sha256 prefix of the
# listed files); after any change the bench reports null until re-captured.
_CSRC = os.path.join(REPO, "varlen_flashattention_forward_gb300", "csrc")
MEASURED_TRAFFIC = {
    # profiles/varlen_fwd_long_65536_d128.md: one full-size launch
    "long_65536": (1.12e9 + 258.55e6, "5ddaada870faa9d4", ["varlen_fwd_kernel.cuh", "sm103_ptx.cuh"]),
    # profiles/varlen_fwd_vit_full_d80.md
    "vit_full_d80": (134.28e6 + 23.57e6, "5ddaada870faa9d4", ["varlen_fwd_kernel.cuh", "sm103_ptx.cuh"]),
    # profiles/sparse_decode_128tok.md: one full-size (128-token) launch
    "sparse_mla_decode": (312.90e6 + 3.77e6, "555aefb1cc5b44d6",
                          ["sparse_decode_kernel.cuh", "sm103_ptx.cuh", "fa_api.cu"]),
}


def measured_traffic(workload: str):
    import hashlib
    entry = MEASURED_TRAFFIC.get(workload)
    if entry is None:
        return None
    value, digest, files = entry
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(_CSRC, f), "rb") as fh:
            m.update(fh.read())
    return value if m.hexdigest()[:16] == digest else None


def load_peaks():
    path = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p.get("hbm_gbs", 6800.0), "bf16_tflops": p.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", 1700.0),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, sm_max, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                sm_max = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput of `world` replicas that each processed
    `units_per_rank` units, timed by the slowest rank (ms_max): units per second."""
    return units_per_rank * world / (ms_max * 1e-3)


# ------------------------------------------------------------ CPU oracle timing
_HOST_INPUTS = {}


def oracle_sample_rate(w, budget_s: float, seed: int = 0):
    """Times the fp64 oracle on a random sample of (token, head) rows of the
    workload; returns (flops/s, rows, seconds, threads)."""
    import oracle
    if w.name not in _HOST_INPUTS:   # drawn once per workload, reused by every step
        _HOST_INPUTS.clear()
        _HOST_INPUTS[w.name] = w.make_inputs()
    q, k, v, cq, ck = _HOST_INPUTS[w.name]
    rng = np.random.default_rng(seed)
    counts = np.concatenate([metrics.visible_keys_per_row(lq, lk, w.causal, *w.window)
                             for lq, lk in zip(w.lens_q, w.lens_k)])
    n_rows_total = w.total_q * w.num_heads

    def run(n):
        rows = np.sort(rng.choice(n_rows_total, size=n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.varlen_attention(q, k, v, cq, ck, w.softmax_scale, w.causal, *w.window, rows=rows)
        dt = time.perf_counter() - t0
        flops = 2.0 * float(counts[rows // w.num_heads].sum()) * (w.d_qk + w.d_v)
        return flops, dt, n

    flops, dt, n = run(32)
    target = max(32, min(n_rows_total, int(n * budget_s / max(dt, 1e-3))))
    flops, dt, n = run(target)
    return flops / dt, n, dt, oracle.num_threads()


# ------------------------------------------------------------ GPU timing
def time_varlen(w, steps, warmup, device, world, on_device=False, e2e=True, kv_hint=None,
                q_hint=None):
    """CUDA-event times of fa_varlen_fwd on workload w (L2 flushed before each
    step, outside the events), the clocks seen meanwhile, and (e2e) the end
    to end time per step with pinned host inputs copied in and the outputs
    copied back."""
    import varlen_flashattention_forward_gb300 as fa
    if on_device:
        qd, kd, vd, cqd, ckd = w.make_inputs_on(device)
    else:
        q, k, v, cq, ck = w.make_inputs()
        qd, kd, vd, cqd, ckd = (t.to(device) for t in (q, k, v, cq, ck))
    out = torch.empty((w.total_q, w.num_heads, w.d_v), dtype=torch.bfloat16, device=device)
    lse = (torch.empty((w.num_heads, w.total_q), dtype=torch.float32, device=device)
           if w.return_lse else None)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    args = (qd, kd, vd, cqd, ckd, max(w.lens_q) if q_hint is None else q_hint,
            max(w.lens_k) if kv_hint is None else kv_hint, w.softmax_scale, w.causal,
            w.window[0], w.window[1], out, lse)
    for _ in range(warmup):
        fa.fa_varlen_fwd(*args)
    torch.cuda.synchronize(device)
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status word set during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index or 0) as clk:
        for i in range(steps):
            flush.fill_(float(i))                     # evict inputs from L2
            starts[i].record(stream)
            fa.fa_varlen_fwd(*args)
            ends[i].record(stream)
        torch.cuda.synchronize(device)
    barrier(world)
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if not e2e:
        if fa.fa_get_device_status() != fa.FA_OK:
            raise RuntimeError("device status word set during timing")
        return times_ms, clk.summary(), None, 0, 0

    # End to end through the public API with host buffers: pinned host inputs
    # copied in, kernel, outputs (O and, if returned, the LSE) copied back,
    # every step.
    hq, hk, hv, hcq, hck = (t.pin_memory() for t in (q, k, v, cq, ck))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory() if lse is not None else None
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hcq, hck))
    d2h = hout.numel() * hout.element_size() + (
        hlse.numel() * hlse.element_size() if hlse is not None else 0)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(steps, 10))
    for _ in range(2):
        fa.fa_varlen_fwd(*args)
    torch.cuda.synchronize(device)
    e_start.record(stream)
    for _ in range(e2e_steps):
        qd.copy_(hq, non_blocking=True)
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        cqd.copy_(hcq, non_blocking=True)
        ckd.copy_(hck, non_blocking=True)
        fa.fa_varlen_fwd(*args)
        hout.copy_(out, non_blocking=True)
        if hlse is not None:
            hlse.copy_(lse, non_blocking=True)
    e_end.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status word set during timing")
    return times_ms, clk.summary(), e2e_ms, h2d, d2h


def time_decode(d, steps, warmup, device, world, e2e=True):
    """Device time of fa_sparse_mla_decode on the decode workload (inputs drawn
    on the device for speed; parity is covered by the tests), and the end to
    end time with the step's inputs (Q, page table, top-k indices) copied in
    from pinned host memory and the output (O, LSE) copied back.  The latent
    cache is resident state, as in serving, and is not copied."""
    import varlen_flashattention_forward_gb300 as fa
    page_table, topk = d.make_indices()
    g = torch.Generator(device=device).manual_seed(d.seed)
    cache = torch.randn((d.num_pages, 64, 576), generator=g, device=device).bfloat16()
    q = torch.randn((d.num_tokens, d.num_heads, 576), generator=g, device=device).bfloat16()
    pt, ti = page_table.to(device), topk.to(device)
    out = torch.empty((d.num_tokens, d.num_heads, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((d.num_heads, d.num_tokens), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        fa.fa_sparse_mla_decode(q, cache, pt, ti, d.softmax_scale, out, lse)
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    for i in range(steps):
        flush.fill_(float(i))                     # evict the last step's rows from L2
        starts[i].record(stream)
        fa.fa_sparse_mla_decode(q, cache, pt, ti, d.softmax_scale, out, lse)
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    ts = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if not e2e:
        if fa.fa_get_device_status() != fa.FA_OK:
            raise RuntimeError("device status word set during timing")
        del cache
        return ts, None, 0, 0

    hq, hpt, hti = q.cpu().pin_memory(), pt.cpu().pin_memory(), ti.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hpt, hti))
    d2h = sum(t.numel() * t.element_size() for t in (hout, hlse))
    e2e_steps = max(3, min(steps, 10))
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e_start.record(stream)
    for i in range(e2e_steps):
        flush.fill_(float(i))
        q.copy_(hq, non_blocking=True)
        pt.copy_(hpt, non_blocking=True)
        ti.copy_(hti, non_blocking=True)
        fa.fa_sparse_mla_decode(q, cache, pt, ti, d.softmax_scale, out, lse)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
    e_end.record(stream)
    torch.cuda.synchronize(device)
    # The flush of each end-to-end step is taken out again.
    f_start = torch.cuda.Event(enable_timing=True)
    f_end = torch.cuda.Event(enable_timing=True)
    f_start.record(stream)
    for i in range(e2e_steps):
        flush.fill_(float(i))
    f_end.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = (e_start.elapsed_time(e_end) - f_start.elapsed_time(f_end)) / e2e_steps
    if fa.fa_get_device_status() != fa.FA_OK:
        raise RuntimeError("device status word set during timing")
    del cache
    return ts, e2e_ms, h2d, d2h


def decode_launches_per_step(d):
    """Kernel launches of one fa_sparse_mla_decode call of this size, as the
    library's own planner (fa_sparse_mla_decode_plan) gives them: 1, or 2
    when the split cuts tokens between CTAs and a merge kernel combines them."""
    import varlen_flashattention_forward_gb300 as fa
    launches, _ = fa.fa_sparse_mla_decode_plan(d.num_tokens, d.num_heads, d.topk)
    return launches


def varlen_plan(w, q_hint=None, kv_hint=None):
    """[grid, split, heads_per_tile] of the workload's launch (fa_varlen_fwd_plan)."""
    import varlen_flashattention_forward_gb300 as fa
    return list(fa.fa_varlen_fwd_plan(
        len(w.lens_q), w.total_q, w.total_k, w.num_heads, w.num_heads_k, w.d_qk, w.d_v,
        max(w.lens_q) if q_hint is None else q_hint,
        max(w.lens_k) if kv_hint is None else kv_hint, w.causal, *w.window))


def _roofline(flops, byts, ms, peaks):
    """Bound, and the fraction of the roofline time (the slower of compute at
    the bf16 peak and bytes at the HBM copy rate) the measured time reaches."""
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    return ("tensor" if t_tensor >= t_hbm else "hbm"), max(t_tensor, t_hbm) * 1e3 / ms


EXTRA_VARLEN = ["tiny", "vit_full_d64", "vit_full_d72", "vit_full_d80", "vit_full_d128",
                "vit_window_d64", "vit_window_d72", "vit_window_d80", "vit_window_d128",
                "vit_window64_d80", "long_16384", "long_36864", "long_65536", "mla_causal",
                "mla_chunked", "mla_swa"]


def extra_lines(steps, warmup, device, peaks, skip=()):
    """Every other workload of the suite: device time (mean and best of the
    steps), TFLOPS, GB/s and the roofline fraction."""
    res = {}
    for name in EXTRA_VARLEN + [n for n in workloads.EXTRA_ONLY if n not in EXTRA_VARLEN]:
        if name in skip:
            continue
        w = (workloads.VARLEN_BENCH.get(name) or workloads.EXTRA_ONLY[name])()
        try:
            t, _, _, _, _ = time_varlen(w, steps, warmup, device, 1, on_device=True, e2e=False)
        except Exception as exc:  # report and continue with the rest
            res[name] = {"error": str(exc)[:200]}
            continue
        ms = statistics.mean(t)
        flops = metrics.varlen_flops(w)
        byts = metrics.varlen_alg_bytes(w)
        bound, frac = _roofline(flops, byts, ms, peaks)
        res[name] = {"ms": round(ms, 4), "ms_min": round(min(t), 4),
                     "tflops": round(flops / ms / 1e9, 1), "gbs": round(byts / ms / 1e6, 1),
                     "bound": bound, "roofline_frac": round(frac, 4),
                     "grid_split": varlen_plan(w)}
        if name.startswith("splitkv"):
            # The same call with a max_seqlen_k hint of 1, which keeps the
            # launch unsplit (the hint steers only the launch shape).
            try:
                t1, _, _, _, _ = time_varlen(w, steps, warmup, device, 1, on_device=True,
                                             e2e=False, kv_hint=1)
                res[name]["unsplit_ms"] = round(statistics.mean(t1), 4)
                res[name]["split_speedup"] = round(statistics.mean(t1) / ms, 2)
            except Exception as exc:
                res[name]["unsplit_error"] = str(exc)[:200]
        if name.startswith("gqa"):
            # The same call with a max_seqlen_q hint large enough that no
            # heads are packed (the hint steers only the launch shape).
            try:
                t1, _, _, _, _ = time_varlen(w, steps, warmup, device, 1, on_device=True,
                                             e2e=False, q_hint=1 << 20)
                res[name]["unpacked_ms"] = round(statistics.mean(t1), 4)
                res[name]["unpacked_grid_split"] = varlen_plan(w, q_hint=1 << 20)
                res[name]["pack_speedup"] = round(statistics.mean(t1) / ms, 2)
            except Exception as exc:
                res[name]["unpacked_error"] = str(exc)[:200]
        torch.cuda.empty_cache()
    try:
        d = workloads.DecodeWorkload()
        t, _, _, _ = time_decode(d, steps, warmup, device, 1, e2e=False)
        ms = statistics.mean(t)
        byts = metrics.decode_alg_bytes(d)
        res["decode"] = {"ms": round(ms, 4), "ms_min": round(min(t), 4),
                         "gbs": round(byts / ms / 1e6, 1), "bound": "hbm",
                         "hbm_frac": round(byts / ms / 1e6 / peaks["hbm_gbs"], 4),
                         "tflops": round(metrics.decode_flops(d) / ms / 1e9, 1)}
    except Exception as exc:
        res["decode"] = {"error": str(exc)[:200]}
    torch.cuda.empty_cache()
    return res


def decode_oracle_rate(d, budget_s, seed=0):
    """fp64 oracle on a random sample of (token, head) rows of the decode
    workload (small cache: only the sampled tokens' pages are drawn)."""
    import oracle
    pt, ti = d.make_indices()
    q = d.make_q()
    rng = np.random.default_rng(seed)
    # Only the pages the sampled tokens reference are materialised; the
    # others are never read by the oracle.
    def run(n_tok):
        toks = np.sort(rng.choice(d.num_tokens, size=n_tok, replace=False))
        pages = pt[toks].reshape(-1).long()
        g = torch.Generator().manual_seed(seed)
        small = workloads._randn((pages.numel(), d.page_size, 576), g, 1.0)
        remap = torch.arange(pages.numel(), dtype=torch.int32).view(n_tok, -1)
        t0 = time.perf_counter()
        oracle.sparse_mla_decode(q[toks].contiguous(), small, remap, ti[toks].contiguous(),
                                 d.softmax_scale)
        dt = time.perf_counter() - t0
        return n_tok * d.topk * 576 * 2.0, dt, n_tok
    byts, dt, n = run(1)
    n2 = max(1, min(d.num_tokens, int(budget_s / max(dt, 1e-3))))
    byts, dt, n = run(n2)
    return byts / dt, n, dt, oracle.num_threads()


def main_decode(a, world, rank, local, peaks):
    """Sparse-MLA decode line: bound by HBM bandwidth."""
    d = workloads.DecodeWorkload()
    if a.decode_tokens:
        # Smaller case (profiling): same per-token shape, fewer tokens/pages.
        d = workloads.DecodeWorkload(num_tokens=a.decode_tokens,
                                     num_pages=a.decode_tokens * d.pages_per_token)
    byts = metrics.decode_alg_bytes(d)
    config = {"workload": "sparse_mla_decode", "num_tokens": d.num_tokens,
              "num_heads": d.num_heads, "topk": d.topk, "context": d.context,
              "num_pages": d.num_pages, "page_size": d.page_size,
              "l2": "flushed before every timed step (512 MB write)",
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if a.impl == "reference":
        if rank != 0:
            return
        rates = [decode_oracle_rate(d, a.cpu_budget / 4, seed=s)
                 for s in range(a.warmup + a.steps)][a.warmup:]
        val = statistics.mean(r[0] for r in rates) / 1e9
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": byts / (val * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": rates[0][3], "kind": "oracle",
                             "sample": f"{rates[0][1]} tokens per step, fp64 oracle"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import varlen_flashattention_forward_gb300 as fa
    fa.load_library()
    with ClockSampler(local) as clk:
        times, e2e_ms, h2d, d2h = time_decode(d, a.steps, a.warmup, device, world)
    ms = max_over_ranks(statistics.mean(times), world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    gbs = byts / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(whole_job_rate(byts, ms, world) / 1e9, 1), "unit": "GB/s",
        "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "traffic": (measured_traffic("sparse_mla_decode")
                                 if d.num_tokens == 128 else None),
                     "peak_source": peaks["source"] + " HBM copy",
                     "kernel": "sparse_decode_kernel<64>", "alg_bytes_per_launch": byts,
                     "alg_flops_per_launch": metrics.decode_flops(d)},
        "tflops": round(metrics.decode_flops(d) / (ms * 1e-3) / 1e12, 1),
        "e2e": {"value": round(whole_job_rate(byts, e2e_ms, world) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": a.steps * decode_launches_per_step(d), "clocks": clk.summary(),
    }
    if not a.no_cpu_baseline:
        rate, n, dt, threads = decode_oracle_rate(d, a.cpu_budget)
        line["cpu_baseline"] = {"value": rate / 1e9, "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": f"{n} tokens, {dt:.1f} s, fp64"}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_65536",
                    help="a varlen workload name or 'decode'")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the headline workload only (no extra block)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-tokens", type=int, default=0,
                    help="decode workload with this many tokens (default: 128)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)

    world, rank, local = dist_setup()
    peaks = load_peaks()
    if a.workload == "decode":
        return main_decode(a, world, rank, local, peaks)
    w = workloads.VARLEN_BENCH[a.workload]()
    flops = metrics.varlen_flops(w)
    byts = metrics.varlen_alg_bytes(w)
    config = {"workload": w.name, "lens": w.lens_q, "num_heads": w.num_heads,
              "d_qk": w.d_qk, "d_v": w.d_v, "causal": w.causal, "window": list(w.window),
              "return_lse": w.return_lse, "l2": "flushed before every timed step (512 MB write)",
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}

    if a.impl == "reference":
        if rank != 0:
            return
        rates = []
        for s in range(a.warmup + a.steps):
            rate, n, dt, threads = oracle_sample_rate(w, budget_s=a.cpu_budget / 4, seed=s)
            if s >= a.warmup:
                rates.append(rate)
        val = statistics.mean(rates) / 1e12
        ms = flops / (val * 1e12) * 1e3
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n} random (token, head) rows per step, fp64 oracle, "
                                       f"scaled to the workload's flop count"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import varlen_flashattention_forward_gb300 as fa
    fa.load_library()

    times_ms, clocks, e2e_ms, h2d, d2h = time_varlen(w, a.steps, a.warmup, device, world)
    ms = statistics.mean(times_ms)
    ms = max_over_ranks(ms, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    tflops = whole_job_rate(flops, ms, world) / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": measured_traffic(w.name),
                     "peak_source": peaks["source"] + " bf16 burst",
                     "kernel": "varlen_fwd_kernel<%d,%d>" % (w.d_qk, w.d_v),
                     "alg_flops_per_launch": flops, "alg_bytes_per_launch": byts},
        "e2e": {"value": round(whole_job_rate(flops, e2e_ms, world) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": a.steps,
        "clocks": clocks,
        "ms_per_step_min": round(min(times_ms), 5),
        "ms_per_step_median": round(statistics.median(times_ms), 5),
    }
    if not a.no_cpu_baseline:
        rate, n, dt, threads = oracle_sample_rate(w, budget_s=a.cpu_budget)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{n} random (token, head) rows, {dt:.1f} s, fp64"}
    if not a.no_extra and world == 1:
        line["extra"] = extra_lines(max(5, a.steps // 2), 3, device, peaks, skip=(w.name,))
        line["extra_note"] = ("every other workload, inputs drawn on the device, "
                              f"{max(5, a.steps // 2)} timed steps each after 3 warm-up steps, "
                              "L2 flushed before each step; roofline_frac = max(flops / bf16 "
                              "burst peak, alg. bytes / HBM copy peak) / time")
    print(json.dumps(line))


if __name__ == "__main__":
    main()
