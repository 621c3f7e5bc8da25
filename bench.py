#!/usr/bin/env python3
"""Attention-forward bench on GB300.

One step = one causal GQA prefill forward of the Llama-3-8B-shaped workload
(B=1, Hq=32, Hkv=8, T=8192, D=128, bf16 I/O), through libattn.so's C ABI on
inputs already resident in HBM.  The same run also times, under "secondary":
the stream-K decode (B=64, Hq=32, Hkv=8, Tk=4096, D=128) on a dense and on a
paged cache, the decode with eight query heads per KV head (B=32, Hq=64), the GPT-2-small-shaped prefill (B=8, H=12, T=1024, D=64), the
T=4096 non-causal prefill, the T=8192 prefill with a 4096-key sliding window
and with fp16 I/O, and a packed batch of 32 sequences of 128..8192 tokens.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on a bounded sample of the same workload instead; ``--sweep`` prints
the prefill time against T; ``--profile-case`` runs one named workload for ncu.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (causal prefill) & decode KV GB/s, % of GB300 roofline"
PRIMARY = "llama3_8b_prefill_bf16_b1_hq32_hkv8_t8192_d128_causal"
DECODE = "gqa_decode_bf16_b64_hq32_hkv8_tk4096_d128"
GQA8_DECODE = "gqa8_decode_bf16_b32_hq64_hkv8_tk4096_d128"
PAGED_DECODE = "gqa_paged_decode_bf16_b64_hq32_hkv8_tk4096_d128_p16"
GPT2 = "gpt2s_prefill_bf16_b8_h12_t1024_d64_causal"
VARLEN = "llama3_8b_varlen_prefill_bf16_32seq_len128to8192_hq32_hkv8_d128_causal"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

PREFILL_SOURCES = ["transformer_attention_fwd_gb300/csrc/prefill_bf16.cu",
                   "transformer_attention_fwd_gb300/csrc/prefill_common.cuh",
                   "transformer_attention_fwd_gb300/csrc/sm100.cuh"]
PREFILL_D64_SOURCES = ["transformer_attention_fwd_gb300/csrc/prefill_d64.cu",
                       "transformer_attention_fwd_gb300/csrc/prefill_common.cuh",
                       "transformer_attention_fwd_gb300/csrc/sm100.cuh"]
DECODE_SOURCES = ["transformer_attention_fwd_gb300/csrc/decode_bf16.cu",
                  "transformer_attention_fwd_gb300/csrc/sm100.cuh"]
VARLEN_SOURCES = PREFILL_SOURCES + ["transformer_attention_fwd_gb300/csrc/varlen_sched.cu"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true",
                    help="time only the primary workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", default=None, metavar="WORKLOAD",
                    help="only run --warmup + --steps calls of this named workload "
                         "(no L2 flush, clocks, e2e or baselines): the command ncu captures")
    ap.add_argument("--sweep", action="store_true",
                    help="time the prefill over T = 64 .. 4096 (8192) and print one JSON line "
                         "per point (the T^2 curve); not the bench line")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def code_text(text):
    """C++/CUDA source with comments and blank lines removed, so that an edit
    to a comment does not count as a change of the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                  # string literal: keep as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def load_traffic(bench_key, sources):
    """DRAM bytes per launch from a committed ncu summary under profiles/, or
    None if there is none or the kernel source changed since the capture."""
    cur = source_hash(sources)
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".txt", ".md")):
            continue
        text = open(os.path.join(pdir, name), encoding="utf-8").read()
        if f"bench_key: {bench_key}" not in text:
            continue
        m_hash = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if m_hash and m_tr and m_hash.group(1) == cur:
            return float(m_tr.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside and self.samples:  # region shorter than the sampling period
            inside = [min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in inside for n, v in zip(names, p[5:9]) if v == "Active"})
        pw = [num(p[3]) for _, p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside)}


def row_flops(w, rows):
    """Metric FLOPs of a set of query rows: 4 * visible_keys * D each (the
    causal metric halves 4*Tq*Tk*D; per row it is 4*(i + Tk - Tq + 1)*D)."""
    import numpy as np
    i = rows % w.Tq
    vis = np.minimum(i + (w.Tk - w.Tq) + 1, w.Tk) if w.causal else np.full_like(i, w.Tk)
    return float((4.0 * vis * w.D).sum())


def cpu_oracle_rate(w, target_s, seed=0):
    """Time the float64 oracle on random rows of workload w; returns
    (TFLOP/s-equivalent in the metric's units, seconds, rows, flops)."""
    import numpy as np
    import oracle
    from transformer_attention_fwd_gb300.inputs import make_workload
    q, k, v = make_workload(w, seed)
    rng = np.random.default_rng(seed)
    total = w.B * w.Hq * w.Tq
    n = 256
    rows = np.sort(rng.choice(total, size=min(n, total), replace=False))
    t = time.perf_counter()
    oracle.attention_f64(q, k, v, w.causal, rows=rows)
    dt = time.perf_counter() - t
    n = int(min(total, max(n, n * target_s / max(dt, 1e-6))))
    rows = np.sort(rng.choice(total, size=n, replace=False))
    t = time.perf_counter()
    oracle.attention_f64(q, k, v, w.causal, rows=rows)
    dt = time.perf_counter() - t
    fl = row_flops(w, rows)
    return fl / dt / 1e12, dt, n, fl


# ---------------------------------------------------------------------------
# GPU measurement
# ---------------------------------------------------------------------------
def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's x (x itself without a process group): the
    job's time is its slowest rank's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms_per_step):
    """Units per second of the whole job: every rank processes units_per_rank
    per step, and a step takes the slowest rank's time."""
    return units_per_rank * world / (ms_per_step * 1e-3)


# GPU-side spin before each timed call (clock cycles, ~50 us at 2 GHz): the
# host enqueues the start event, the call and the end event while the GPU
# spins, so the events time the kernels and not the Python binding's launch
# overhead (which the end-to-end figure does include).
SPIN_CYCLES = 100_000


def time_steps(fn, steps, warmup, flush=None, spin=True):
    """Warm up, then time `steps` calls with CUDA events on the current stream,
    flushing L2 (outside the event pairs) before each call when asked."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        if spin:
            torch.cuda._sleep(SPIN_CYCLES)
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_ours(args, rank, world):
    import torch
    from transformer_attention_fwd_gb300 import build as b
    b.build()
    from transformer_attention_fwd_gb300 import attn
    from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_workload

    dist = None
    if world > 1:
        import torch.distributed as dist
    dev = torch.cuda.current_device()
    peaks, peak_src = load_peaks()
    w = WORKLOADS[PRIMARY]
    q, k, v = make_workload(w, seed=0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        flush_buf.zero_()

    def step():
        attn.attn_fwd(qd, kd, vd, causal=True, out=od, lse=lsed)

    step()
    assert attn.device_status() == attn.ATTN_OK, attn.last_error()
    _, _, kernels_per_step = attn.last_launch_info()

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    times = time_steps(step, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    st = attn.device_status()
    assert st == attn.ATTN_OK, attn.last_error()

    total_ms = max_over_ranks(sum(times), dist, "cuda")
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(w.flops, world, ms_per_step) / 1e12
    kernel_tflops = w.flops / (ms_per_step * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    traffic = load_traffic("prefill_llama3_t8192_causal", PREFILL_SOURCES)

    # End to end: pinned host inputs -> attn_fwd_host -> pinned host outputs.
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.empty(od.shape, dtype=od.dtype, pin_memory=True)
    lh = torch.empty(lsed.shape, dtype=lsed.dtype, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        # One C-ABI call on host buffers: copies in, compute, copies out,
        # pipelined over chunks of (b, hkv) pairs inside the library.
        attn.attn_fwd_host(qh, kh, vh, causal=True, out=oh, lse=lh)

    e2e_times = time_steps(e2e_step, e2e_steps, 2, spin=False)
    e2e_ms = sum(e2e_times) / e2e_steps
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v))
    d2h = od.numel() * od.element_size() + lsed.numel() * 4

    secondary = {}
    if not args.no_secondary:
        secondary = run_secondary(args, attn, peaks, flush)

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": PRIMARY, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq,
                   "Tk": w.Tk, "D": w.D, "causal": True, "flops_per_step": w.flops,
                   "inputs": "N(0,1) seed 0 rounded to bf16", "l2": "flushed before every step "
                   "(256 MiB write, outside the timed events)",
                   "timing": "CUDA events around each call on the launching stream; a GPU-side "
                   "spin precedes each call so that the host's launch overhead stays outside "
                   "the events (the e2e figure includes it)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(kernel_tflops, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(kernel_tflops / peak, 4),
                     "traffic": traffic, "peak_source": f"bf16_tflops burst ({peak_src})"},
        "e2e": {"value": round(w.flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clocks,
        "secondary": secondary,
    }
    return result


def run_secondary(args, attn, peaks, flush):
    import torch
    from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload
    out = {}
    steps = max(5, min(args.steps, 100))
    # Decode: K+V = 1 GiB >> L2, no flush needed.
    w = WORKLOADS[DECODE]
    q, k, v = (x.cuda() for x in make_workload(w, 0))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    fn = lambda: attn.attn_fwd(q, k, v, causal=False, out=o, lse=lse)  # noqa: E731
    fn()
    _, splits, kernels = attn.last_launch_info()
    times = time_steps(fn, steps, 5)
    ms = sum(times) / steps
    gbs = w.io_bytes() / (ms * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out["decode"] = {
        "workload": DECODE, "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 5),
        "algorithmic_bytes": w.io_bytes(),
        "mode": "stream-K, one key slice per SM" if splits == 0 else f"{splits} splits",
        "kernels_per_step": kernels,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4),
                     "traffic": load_traffic("decode_b64_tk4096", DECODE_SOURCES),
                     "note": "step time includes the stream kernel and the fragment combine kernel"},
    }
    del q, k, v, o, lse
    # Eight query heads per KV head: automatic mode runs the tensor-core
    # prefill kernel over the query-head groups.
    w = WORKLOADS[GQA8_DECODE]
    q, k, v = (x.cuda() for x in make_workload(w, 0))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    fn = lambda: attn.attn_fwd(q, k, v, causal=False, out=o, lse=lse)  # noqa: E731
    fn()
    _, items, kernels = attn.last_launch_info()
    times = time_steps(fn, steps, 5)
    ms = sum(times) / steps
    gbs = w.io_bytes() / (ms * 1e-3) / 1e9
    out["gqa8_decode"] = {
        "workload": GQA8_DECODE, "value": round(gbs, 1), "unit": "GB/s",
        "ms_per_step": round(ms, 5), "algorithmic_bytes": w.io_bytes(),
        "mode": f"tensor-core prefill kernel over the query-head groups, {items} work items",
        "kernels_per_step": kernels,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4),
                     "traffic": load_traffic("gqa8_decode_b32_tk4096", PREFILL_SOURCES),
                     "note": "K+V (537 MB) exceed L2; no flush needed"},
    }
    del q, k, v, o, lse
    # The same decode against a paged cache (16-token blocks in a random order).
    from transformer_attention_fwd_gb300.inputs import PAGED_WORKLOADS, make_paged_workload
    pw = PAGED_WORKLOADS[PAGED_DECODE]
    q, kv, bt, sl = (x.cuda() for x in make_paged_workload(pw, 0))
    o = torch.empty_like(q)
    lse = torch.empty((pw.B, pw.Hq), dtype=torch.float32, device="cuda")
    fn = lambda: attn.attn_fwd_decode_paged(q, kv, bt, sl, out=o, lse=lse)  # noqa: E731
    fn()
    _, _, kernels = attn.last_launch_info()
    times = time_steps(fn, steps, 5)
    ms = sum(times) / steps
    gbs = pw.io_bytes() / (ms * 1e-3) / 1e9
    out["paged_decode"] = {
        "workload": PAGED_DECODE, "value": round(gbs, 1), "unit": "GB/s",
        "ms_per_step": round(ms, 5), "algorithmic_bytes": pw.io_bytes(),
        "kernels_per_step": kernels,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4),
                     "traffic": load_traffic("paged_decode_b64_tk4096_p16", DECODE_SOURCES),
                     "note": "step time includes the stream kernel (which also sums the request "
                             "lengths) and the fragment combine kernel"},
    }
    del q, kv, bt, sl, o, lse
    # GPT-2-small-shaped causal prefill, D = 64.
    w = WORKLOADS[GPT2]
    q, k, v = (x.cuda() for x in make_workload(w, 0))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    fn = lambda: attn.attn_fwd(q, k, v, causal=True, out=o, lse=lse)  # noqa: E731
    times = time_steps(fn, steps, 5, flush)
    ms = sum(times) / steps
    tf = w.flops / (ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    out["gpt2s_prefill"] = {
        "workload": GPT2, "value": round(tf, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "traffic": load_traffic("prefill_gpt2s_d64", PREFILL_D64_SOURCES)},
    }
    # Non-causal T=4096 variant of the primary workload.
    w = WORKLOADS["llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_noncausal"]
    q, k, v = (x.cuda() for x in make_workload(w, 0))
    o = torch.empty_like(q)
    fn = lambda: attn.attn_fwd(q, k, v, causal=False, out=o, want_lse=False)  # noqa: E731
    times = time_steps(fn, steps, 5, flush)
    ms = sum(times) / steps
    tf = w.flops / (ms * 1e-3) / 1e12
    out["llama3_noncausal_t4096"] = {
        "workload": w.name, "value": round(tf, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "traffic": load_traffic("prefill_llama3_t4096_noncausal", PREFILL_SOURCES)},
    }
    # Sliding window of 4096 keys on the primary workload's shapes.
    w = WORKLOADS[PRIMARY]
    q, k, v = (x.cuda() for x in make_workload(w, 0))
    o = torch.empty_like(q)
    W = 4096
    fn = lambda: attn.attn_fwd_window(q, k, v, W, out=o, want_lse=False)  # noqa: E731
    times = time_steps(fn, steps, 5, flush)
    ms = sum(times) / steps
    pairs = W * (W + 1) // 2 + (w.Tq - W) * W  # visible (query, key) pairs of one head
    tf = 4.0 * pairs * w.D * w.B * w.Hq / (ms * 1e-3) / 1e12
    out["llama3_window4096_t8192"] = {
        "workload": f"{PRIMARY}_window{W}", "value": round(tf, 3), "unit": "TFLOP/s",
        "ms_per_step": round(ms, 5), "flops_per_step": 4.0 * pairs * w.D * w.B * w.Hq,
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "traffic": load_traffic("prefill_llama3_t8192_window4096", PREFILL_SOURCES)},
    }
    del q, k, v, o
    # The primary workload with fp16 I/O.
    q, k, v = (x.cuda() for x in make_qkv(w.B, w.Hq, w.Hkv, w.Tq, w.Tk, w.D, "f16", 0))
    o = torch.empty_like(q)
    fn = lambda: attn.attn_fwd(q, k, v, causal=True, out=o, want_lse=False)  # noqa: E731
    times = time_steps(fn, steps, 5, flush)
    ms = sum(times) / steps
    tf = w.flops / (ms * 1e-3) / 1e12
    out["llama3_f16_t8192"] = {
        "workload": PRIMARY.replace("bf16", "f16"), "value": round(tf, 3), "unit": "TFLOP/s",
        "ms_per_step": round(ms, 5),
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "traffic": load_traffic("prefill_llama3_t8192_f16", PREFILL_SOURCES),
                     "note": "fp16 and bf16 share the measured dense peak"},
    }
    del q, k, v, o
    # Packed variable-length prefill: 32 sequences of 128..8192 tokens.
    from transformer_attention_fwd_gb300.inputs import VARLEN_WORKLOADS, make_varlen_workload
    vw = VARLEN_WORKLOADS[VARLEN]
    q, k, v, cq, ck = (x.cuda() for x in make_varlen_workload(vw, 0))
    o = torch.empty_like(q)
    lse = torch.empty((vw.Hq, q.shape[0]), dtype=torch.float32, device="cuda")
    fn = lambda: attn.attn_fwd_varlen(q, k, v, cq, ck, vw.causal, out=o, lse=lse)  # noqa: E731
    fn()
    _, _, kernels = attn.last_launch_info()
    times = time_steps(fn, steps, 5, flush)
    ms = sum(times) / steps
    tf = vw.flops() / (ms * 1e-3) / 1e12
    out["llama3_varlen_mix"] = {
        "workload": VARLEN, "value": round(tf, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
        "flops_per_step": vw.flops(), "tokens": int(q.shape[0]), "kernels_per_step": kernels,
        "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                     "traffic": load_traffic("prefill_varlen_mix", VARLEN_SOURCES),
                     "note": "step time includes the two scheduling kernels"},
    }
    del q, k, v, cq, ck, o, lse
    assert attn.device_status() == attn.ATTN_OK, attn.last_error()
    # Prefill time against T (L2 flushed before each call).
    out["t_sweep"] = {
        "note": "bf16 prefill, L2 flushed before every call; growth = t(T) / t(T/2), "
                "which tends to 4 once the T^2 work dominates the fixed per-call cost",
        "steps_per_point": 20,
        "points": sweep_points(attn, 20, 3, flush)}
    return out


def run_reference(args):
    """The float64 oracle on the host cores, on bounded samples of the primary
    workload: each step computes a fixed random sample of query rows."""
    import numpy as np
    import oracle
    from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_workload
    w = WORKLOADS[PRIMARY]
    q, k, v = make_workload(w, 0)
    cores = oracle.default_threads()
    budget_s = 150.0
    per_step = max(0.05, min(1.0, budget_s / max(1, args.steps + args.warmup)))
    _, dt, n, _ = cpu_oracle_rate(w, per_step)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(w.B * w.Hq * w.Tq, size=n, replace=False))
    fl = row_flops(w, rows)
    for _ in range(args.warmup):
        oracle.attention_f64(q, k, v, True, rows=rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_f64(q, k, v, True, rows=rows)
    total = time.perf_counter() - t
    ms = total / args.steps * 1e3
    value = fl / (ms * 1e-3) / 1e12
    sample = f"{n} random query rows of {PRIMARY} per step ({fl / 1e9:.2f} GFLOP)"
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": PRIMARY, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq,
                   "Tk": w.Tk, "D": w.D, "causal": True},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_profile_case(args):
    import torch
    from transformer_attention_fwd_gb300 import build as b
    b.build()
    from transformer_attention_fwd_gb300 import attn
    from transformer_attention_fwd_gb300.inputs import (PAGED_WORKLOADS, WORKLOADS, make_paged_workload,
                                                        make_qkv, make_workload)
    from transformer_attention_fwd_gb300.inputs import VARLEN_WORKLOADS, make_varlen_workload
    if args.profile_case in VARLEN_WORKLOADS:
        vw = VARLEN_WORKLOADS[args.profile_case]
        q, k, v, cq, ck = (x.cuda() for x in make_varlen_workload(vw, 0))
        fn = lambda: attn.attn_fwd_varlen(q, k, v, cq, ck, vw.causal)  # noqa: E731
        times = time_steps(fn, args.steps, args.warmup)
        if attn.device_status() != attn.ATTN_OK:
            raise RuntimeError(attn.last_error())
        ms = sum(times) / len(times)
        print(json.dumps({"profile_case": vw.name, "ms_per_step": round(ms, 5),
                          "tflops": round(vw.flops() / (ms * 1e-3) / 1e12, 3)}), flush=True)
        return 0
    if args.profile_case in PAGED_WORKLOADS:
        pw = PAGED_WORKLOADS[args.profile_case]
        q, kv, bt, sl = (x.cuda() for x in make_paged_workload(pw, 0))
        fn = lambda: attn.attn_fwd_decode_paged(q, kv, bt, sl)  # noqa: E731
        times = time_steps(fn, args.steps, args.warmup)
        if attn.device_status() != attn.ATTN_OK:
            raise RuntimeError(attn.last_error())
        ms = sum(times) / len(times)
        print(json.dumps({"profile_case": pw.name, "ms_per_step": round(ms, 5),
                          "gbs": round(pw.io_bytes() / (ms * 1e-3) / 1e9, 1)}), flush=True)
        return 0
    # The primary workload's sliding-window and fp16 lines.
    name, window, dtype = args.profile_case, 0, None
    if name == PRIMARY + "_window4096":
        name, window = PRIMARY, 4096
    elif name == PRIMARY.replace("bf16", "f16"):
        name, dtype = PRIMARY, "f16"
    w = WORKLOADS[name]
    if dtype is None:
        q, k, v = (x.cuda() for x in make_workload(w, 0))
    else:
        q, k, v = (x.cuda() for x in make_qkv(w.B, w.Hq, w.Hkv, w.Tq, w.Tk, w.D, dtype, 0))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    if window:
        fn = lambda: attn.attn_fwd_window(q, k, v, window, out=o, lse=lse)  # noqa: E731
    else:
        fn = lambda: attn.attn_fwd(q, k, v, causal=w.causal, out=o, lse=lse)  # noqa: E731
    times = time_steps(fn, args.steps, args.warmup)
    st = attn.device_status()
    if st != attn.ATTN_OK:
        raise RuntimeError(attn.last_error())
    ms = sum(times) / len(times)
    print(json.dumps({"profile_case": w.name, "ms_per_step": round(ms, 5),
                      "tflops": round(w.flops / (ms * 1e-3) / 1e12, 3),
                      "gbs": round(w.io_bytes() / (ms * 1e-3) / 1e9, 1)}), flush=True)
    return 0


SWEEP_SHAPES = [
    # (name, B, Hq, Hkv, D, causal, largest T)
    ("mha_b1_h4_d64", 1, 4, 4, 64, False, 4096),
    ("llama3_8b_b1_hq32_hkv8_d128_causal", 1, 32, 8, 128, True, 8192),
]


def sweep_points(attn, steps, warmup, flush):
    """Prefill time against sequence length, T = 64, 128, .., doubling, for
    each SWEEP_SHAPES entry ("第 11 章 · Attention 入门" §11 exercises: the
    T sweep).  The growth column is t(T) / t(T/2), which tends to 4 once the
    T^2 work dominates the launch and pipeline-fill latency."""
    import torch
    from transformer_attention_fwd_gb300.inputs import make_qkv
    points = []
    for name, B, Hq, Hkv, D, causal, tmax in SWEEP_SHAPES:
        prev = None
        T = 64
        while T <= tmax:
            q, k, v = (x.cuda() for x in make_qkv(B, Hq, Hkv, T, T, D, "bf16", 0))
            o = torch.empty_like(q)
            fn = lambda: attn.attn_fwd(q, k, v, causal=causal, out=o, want_lse=False)  # noqa: E731
            times = time_steps(fn, steps, warmup, flush)
            ms = sum(times) / steps
            flops = 4.0 * B * Hq * T * T * D * (0.5 if causal else 1.0)
            points.append({"sweep": name, "T": T, "ms_per_step": round(ms, 5),
                           "tflops": round(flops / (ms * 1e-3) / 1e12, 3),
                           "growth": None if prev is None else round(ms / prev, 3)})
            prev = ms
            T *= 2
            del q, k, v, o
    if attn.device_status() != attn.ATTN_OK:
        raise RuntimeError(attn.last_error())
    return points


def run_sweep(args):
    """--sweep: the T sweep alone, one JSON line per point."""
    import torch
    from transformer_attention_fwd_gb300 import build as b
    b.build()
    from transformer_attention_fwd_gb300 import attn
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush = lambda: flush_buf.fill_(1)  # noqa: E731
    for pt in sweep_points(attn, max(5, min(args.steps, 200)), max(3, args.warmup), flush):
        print(json.dumps(pt), flush=True)
    return 0


def main():
    args = parse_args()
    if args.profile_case:
        return run_profile_case(args)
    if args.sweep:
        return run_sweep(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    result = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            from transformer_attention_fwd_gb300.inputs import WORKLOADS
            import oracle
            w = WORKLOADS[PRIMARY]
            rate, dt, n, fl = cpu_oracle_rate(w, 10.0)
            result["cpu_baseline"] = {
                "value": round(rate, 6), "unit": "TFLOP/s", "cores": oracle.default_threads(),
                "kind": "oracle",
                "sample": f"{n} random query rows of {PRIMARY} ({fl / 1e9:.1f} GFLOP, "
                          f"{dt:.1f} s wall)"}
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
