"""Benchmark of the fused exact-attention forward on GB300.

Default workload: bf16 forward, B=1, H=16, N=16384, d=128, causal -- the
d=128, N=16k point of the 16384-token sweep (hidden 2048), the largest bf16
single-GPU configuration at the head dimension and length where the
throughput target is set -- FLOPs counted as 4 B H N^2 d / 2.  One step = one
fused forward over the batch (load, QK^T, online softmax, correction, PV and
epilogue all inside one kernel launch).  The same line carries, as extra
objects: the non-causal variant of that point ("noncausal"), the B=2, H=32,
N=4096 causal shape ("c2"), the FP8 path (prep of Q, K, V with block scales +
Hadamard rotation, then the FP8 forward) on its workload (B=2, H=16, N=8192,
d=128, non-causal, outlier inputs; "fp8"), and the backward on the pages'
Fig. 6 point (B=1, H=16, N=16384, d=128, non-causal; FLOPs 2.5 x the
forward's; "bwd").  The "e2e" object is the same metric with host buffers,
through the library's host-buffer entries (attn_fwd_host, attn_fwd_fp8_host,
attn_bwd_host): the copies in and out are inside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c3_d128_n16k|c2|c4|c5|gqa|bwd|bwd_c2|bwd_d64|sparse|fp8_d256|
                                fp8_d256_causal|c3:N:d:causal|fp8:N:d:causal|bwd:N:causal[:d]]
                    [--quick]

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own
device (weak scaling, no collective on the data path); `value` is the work of
all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, fp8) on 1 GB300 and % of dense tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}

DEFAULT_WORKLOAD = "c3_d128_n16k"

WORKLOADS = {
    "c3_d128_n16k": dict(name="bf16 fwd B=1 H=16 N=16384 d=128 causal (16384 tokens, hidden 2048)", B=1, H=16,
                         N=16384, d=128, causal=True, window=0, dtype="bf16"),
    "c3_d128_n16k_noncausal": dict(name="bf16 fwd B=1 H=16 N=16384 d=128 non-causal (16384 tokens, hidden 2048)",
                                   B=1, H=16, N=16384, d=128, causal=False, window=0, dtype="bf16"),
    "c2": dict(name="bf16 fwd B=2 H=32 N=4096 d=128 causal", B=2, H=32, N=4096, d=128, causal=True, window=0,
               dtype="bf16"),
    "c4": dict(name="fp8 e4m3 fwd B=2 H=16 N=8192 d=128 non-causal, outliers, block scales + Hadamard",
               B=2, H=16, N=8192, d=128, causal=False, window=0, dtype="fp8"),
    "c5": dict(name="bf16 fwd B=1 H=8 N=32768 d=128 causal, 4096-token sliding window", B=1, H=8, N=32768,
               d=128, causal=True, window=4096, dtype="bf16"),
    "gqa": dict(name="bf16 fwd grouped-query B=2 H=32 H_kv=8 N=8192 d=128 causal", B=2, H=32, Hkv=8, N=8192,
                d=128, causal=True, window=0, dtype="bf16"),
    # The backward's headline point on the pages (Fig. 6: d=128, 16k tokens,
    # hidden 2048, non-causal N=16k) and the forward's headline shape.
    "bwd": dict(name="bf16 bwd B=1 H=16 N=16384 d=128 non-causal", B=1, H=16, N=16384, d=128, causal=False,
                window=0, dtype="bf16", direction="bwd"),
    "bwd_c2": dict(name="bf16 bwd B=2 H=32 N=4096 d=128 causal", B=2, H=32, N=4096, d=128, causal=True, window=0,
                   dtype="bf16", direction="bwd"),
    "bwd_d64": dict(name="bf16 bwd B=1 H=32 N=16384 d=64 non-causal", B=1, H=32, N=16384, d=64, causal=False,
                    window=0, dtype="bf16", direction="bwd"),
    # The pages' FP8 figure: d = 256, 16k tokens with hidden 2048 (8 heads), N = 16k.
    "fp8_d256": dict(name="fp8 e4m3 fwd B=1 H=8 N=16384 d=256 non-causal, outliers, block scales + Hadamard", B=1, H=8,
                     N=16384, d=256, causal=False, window=0, dtype="fp8"),
    "fp8_d256_causal": dict(name="fp8 e4m3 fwd B=1 H=8 N=16384 d=256 causal, outliers, block scales + Hadamard", B=1, H=8,
                            N=16384, d=256, causal=True, window=0, dtype="fp8"),
    # Block-sparse forward: a band of +-8 key blocks around the diagonal plus
    # every 8th key block (128 x 128 blocks; about 24 % of them visible).
    "sparse": dict(name="bf16 fwd block-sparse B=1 H=16 N=16384 d=128 non-causal, band +-8 blocks + every 8th block",
                   B=1, H=16, N=16384, d=128, causal=False, window=0, dtype="bf16", sparse="band8_stride8"),
}


def block_mask(w: dict) -> np.ndarray:
    """The workload's block mask (B, H, T, T), uint8."""
    T = (w["N"] + 127) // 128
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    if w.get("sparse") != "band8_stride8":
        raise SystemExit(f"unknown block pattern {w.get('sparse')}")
    m = ((np.abs(i - j) <= 8) | (j % 8 == 0)).astype(np.uint8)
    return np.ascontiguousarray(np.broadcast_to(m, (w["B"], w["H"], T, T)))


def visible_pairs(w: dict, rows=None) -> int:
    """Exact number of (query, key) pairs that take part, over all heads
    (block mask, causal and window), for all query rows or the given ones."""
    N = w["N"]
    rows = np.arange(N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    lo = np.maximum(0, rows - w["window"] + 1) if w["window"] > 0 else np.zeros(len(rows), dtype=np.int64)
    hi = rows if w["causal"] else np.full(len(rows), N - 1)
    if not w.get("sparse"):
        return int(np.sum(hi - lo + 1)) * w["B"] * w["H"]
    m = block_mask(w)[0, 0].astype(bool)          # the pattern is the same for every head
    keys = np.arange(N)
    total = 0
    for r, a, b in zip(rows, lo, hi):
        kb = m[r // 128][keys[a:b + 1] // 128]
        total += int(np.count_nonzero(kb))
    return total * w["B"] * w["H"]


def workload(spec: str) -> dict:
    if spec in WORKLOADS:
        return dict(WORKLOADS[spec])
    if spec.startswith("c3:"):
        _, n, d, c = spec.split(":")
        n, d, c = int(n), int(d), c in ("1", "true", "causal")
        return dict(name=f"bf16 fwd sweep point N={n} d={d} {'causal' if c else 'non-causal'} (16384 tokens, "
                         f"hidden 2048)", B=16384 // n, H=2048 // d, N=n, d=d, causal=c, window=0, dtype="bf16")
    if spec.startswith("fp8:"):
        _, n, d, c = spec.split(":")
        n, d, c = int(n), int(d), c in ("1", "true", "causal")
        return dict(name=f"fp8 e4m3 fwd sweep point N={n} d={d} {'causal' if c else 'non-causal'} (16384 tokens, "
                         f"hidden 2048), outliers, block scales + Hadamard", B=16384 // n, H=2048 // d, N=n, d=d,
                    causal=c, window=0, dtype="fp8")
    if spec.startswith("bwd:"):
        parts = spec.split(":")
        n, c = int(parts[1]), parts[2] in ("1", "true", "causal")
        d = int(parts[3]) if len(parts) > 3 else 128
        return dict(name=f"bf16 bwd sweep point N={n} d={d} {'causal' if c else 'non-causal'} (16384 tokens, "
                         f"hidden 2048)", B=16384 // n, H=2048 // d, N=n, d=d, causal=c, window=0, dtype="bf16",
                    direction="bwd")
    raise SystemExit(f"unknown workload {spec}")


def attended_pairs(N: int, causal: bool, window: int) -> int:
    """Exact count of visible (query, key) pairs of one head."""
    i = np.arange(N, dtype=np.int64)
    hi = i if causal else np.full(N, N - 1)
    lo = np.maximum(0, i - window + 1) if window > 0 else np.zeros(N, dtype=np.int64)
    return int(np.sum(hi - lo + 1))


def flops_per_step(w: dict) -> float:
    """Forward: 4 B H N^2 d, halved when causal; with a window, 4 d x the
    attended pairs.  Backward: 2.5 x the forward (five matrix products
    against two, the pages' convention)."""
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    mult = 2.5 if w.get("direction") == "bwd" else 1.0
    if w.get("sparse"):
        return mult * 4.0 * d * visible_pairs(w)
    if w["window"] > 0:
        return mult * 4.0 * B * H * d * attended_pairs(N, w["causal"], w["window"])
    return mult * 4.0 * B * H * N * N * d / (2.0 if w["causal"] else 1.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def cublaslt_fp8_peak():
    """The e4m3 GEMM throughput measured on this GPU type by `--fp8-peak`
    (stored beside the ncu summaries), for context beside the nominal-ratio
    denominator; None when absent."""
    try:
        with open(os.path.join(ROOT, "profiles", "fp8_gemm_peak.json")) as f:
            return json.load(f).get("fp8_tflops")
    except (OSError, ValueError):
        return None


# The sources each timed kernel is compiled from: a recorded DRAM traffic
# figure is used only while these files are unchanged.
KERNEL_SOURCES = {
    "attn_fwd": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_fwd_kernel.cuh", "attn_launch.cuh", "fwd_bf16_d128.cu"),
    "attn_fwd_fp8": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_fwd_kernel.cuh", "attn_launch.cuh", "fwd_fp8_d128.cu"),
    "attn_fwd_fp8_d256": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_fwd_kernel.cuh", "attn_fwd_la_kernel.cuh",
                          "attn_launch.cuh", "fwd_fp8_d256.cu"),
    "attn_fwd_fp8_d64": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_fwd_kernel.cuh", "attn_launch.cuh",
                         "fwd_fp8_d64.cu"),
    "fp8_prep": ("fp8_prep.cu", "fp8_prep.cuh", "fp8_prep_tc.cu", "sm103_ptx.cuh"),
    "attn_bwd": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_bwd_kernel.cuh", "attn_bwd.cu", "attn_bwd.cuh"),
    "attn_fwd_sparse": ("sm103_ptx.cuh", "sm103_bulk.cuh", "attn_fwd_kernel.cuh", "attn_launch.cuh",
                        "fwd_sparse_d128.cu"),
}


def kernel_source_hash(kernel: str = "attn_fwd") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_71_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(f"{kernel}/{workload_key}")
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            rows.append(parts)
        if not rows and self.lines:   # uuid formats differ: take the first GPU listed
            first = self.lines[0].split(",")[0].strip()
            rows = [[p.strip() for p in ln.split(",")] for ln in self.lines if ln.split(",")[0].strip() == first]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_inputs(w, device, seed=0):
    """Seeded synthetic inputs on the device (bf16 bit patterns from synth)."""
    import torch

    from exact_attention_71_gb300 import synth
    outliers = w["dtype"] == "fp8"
    B, N, H, d = w["B"], w["N"], w["H"], w["d"]
    Hkv = w.get("Hkv", H)
    arrs = (synth.tensor_bf16((B, N, H, d), seed, synth.STREAM_Q, outliers),
            synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_K, outliers),
            synth.tensor_bf16((B, N, Hkv, d), seed, synth.STREAM_V, outliers))
    if w.get("direction") == "bwd":
        arrs = arrs + (synth.tensor_bf16((B, N, H, d), seed, STREAM_DOUT),)
    return [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device) for a in arrs], arrs


STREAM_DOUT = 4    # synth stream of the upstream gradient dO


def time_loop(fn, steps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def time_loop_two_streams(fn, steps, streams):
    """time_loop for work spread over two streams: the start event is on the
    first, the second waits for it; the end event is recorded on the first
    after it has waited for everything queued on the second."""
    import torch
    a, b = streams
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(a)
    b.wait_event(e0)
    for _ in range(steps):
        fn()
    eb = torch.cuda.Event()
    eb.record(b)
    a.wait_event(eb)
    e1.record(a)
    e1.synchronize()
    return e0.elapsed_time(e1)


def _oracle_inputs(w, arrs=None):
    from exact_attention_71_gb300 import synth
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    if arrs is None:
        Hkv = w.get("Hkv", H)
        o_ = w["dtype"] == "fp8"
        arrs = (synth.tensor_bf16((B, N, H, d), 0, synth.STREAM_Q, o_),
                synth.tensor_bf16((B, N, Hkv, d), 0, synth.STREAM_K, o_),
                synth.tensor_bf16((B, N, Hkv, d), 0, synth.STREAM_V, o_))
        if w.get("direction") == "bwd":
            arrs = arrs + (synth.tensor_bf16((B, N, H, d), 0, STREAM_DOUT),)
    return arrs


def _oracle_run(w, arrs, size, cores):
    """One bounded sample of the workload on the fp64 oracle: `size` seeded
    query rows of every head (forward), or the first `size` query heads in
    full (backward, whose key gradients need every query row).  Returns
    (seconds, flops, description)."""
    import oracle

    from exact_attention_71_gb300 import synth
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    t0 = time.perf_counter()
    if w.get("direction") == "bwd":
        q, k, v, do = arrs
        group = H // k.shape[2]
        nh = max(group, size // group * group)
        sl, skv = slice(0, nh), slice(0, nh // group)
        oracle.attention_bwd(q[:, :, sl], k[:, :, skv], v[:, :, skv], do[:, :, sl], causal=w["causal"],
                             window=w["window"], nthreads=cores)
        t = time.perf_counter() - t0
        flops = flops_per_step(dict(w, H=nh))
        return t, flops, f"{nh} of {H} query heads in full x {B} batch ({flops / 1e9:.2f} GFLOP, fp64, {cores} threads)"
    q, k, v = arrs[:3]
    rows = synth.sample_rows(N, size, seed=17)
    bm = block_mask(w) if w.get("sparse") else None
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=w["causal"], window=w["window"], rows=rows, nthreads=cores, block_mask=bm)
    t = time.perf_counter() - t0
    flops = 4.0 * d * visible_pairs(w, rows)
    return t, flops, f"{len(rows)} seeded query rows per head x all {B * H} heads ({flops / 1e9:.2f} GFLOP, fp64, {cores} threads)"


def _oracle_size(w, arrs, target_s, cores):
    """Grows the sample until one run takes at least target_s / 2."""
    size = 1 if w.get("direction") == "bwd" else 2
    limit = w["H"] if w.get("direction") == "bwd" else w["N"]
    while True:
        t, flops, desc = _oracle_run(w, arrs, size, cores)
        if t >= target_s / 2 or size >= limit:
            return size, t, flops, desc
        size = min(limit, int(size * max(1.5, min(8.0, 0.6 * target_s / max(t, 1e-3)))) + 1)


def cpu_baseline(w, budget_s=12.0, arrs=None):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of
    the same workload; throughput in the same unit (TFLOPS of attention
    arithmetic)."""
    arrs = _oracle_inputs(w, arrs)
    cores = os.cpu_count() or 1
    _, t, flops, desc = _oracle_size(w, arrs, budget_s, cores)
    out = {"value": flops / t / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
           "sample": desc + f", {t:.1f} s"}
    # The same oracle on one core, on a smaller sample (a per-core figure).
    _, t1, flops1, desc1 = _oracle_size(w, arrs, budget_s / 4, 1)
    out["one_core"] = {"value": flops1 / t1 / 1e12, "unit": "TFLOPS", "sample": desc1 + f", {t1:.1f} s"}
    return out


def run_reference(args, w, key):
    """The oracle arm: W untimed and K timed steps, each the same bounded
    sample of the workload (sized once so that the whole run stays within
    about two minutes of CPU time); value = the median step's throughput."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    arrs = _oracle_inputs(w)
    per_step = min(args.ref_budget, max(0.05, 120.0 / (args.steps + args.warmup)))
    size, _, _, _ = _oracle_size(w, arrs, per_step, cores)
    for _ in range(args.warmup):
        _oracle_run(w, arrs, size, cores)
    per = []
    desc = ""
    for _ in range(max(1, args.steps)):
        t, flops, desc = _oracle_run(w, arrs, size, cores)
        per.append(flops / t / 1e12)
    val = float(np.median(per))
    cb = {"value": val, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
          "sample": desc + f"; median of {len(per)} timed steps"}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "N": w["N"],
                                             "d": w["d"], "causal": w["causal"], "window": w["window"]},
            "cpu_baseline": cb, "e2e": {"value": val, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0},
            "vs_baseline": None}
    print(json.dumps(line), flush=True)


def measure_spec_peak():
    """Spec dense tensor peak pinned by this repository's own tcgen05
    microbenchmark (mma_peak.cu beside this file): SMs x measured dense FLOP per
    clock per SM x the maximum SM clock."""
    src = os.path.join(ROOT, "mma_peak.cu")
    exe = os.path.join(ROOT, "_build", "mma_peak")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", ROOT, "-o", exe, src],
                   check=True)
    res = json.loads(subprocess.run([exe], check=True, capture_output=True, text=True).stdout.strip())
    mhz = res["max_sm_mhz"]
    res["bf16_tflops_spec"] = round(res["sms"] * res["bf16_flop_per_clk_per_sm"] * mhz * 1e6 / 1e12, 1)
    res["e4m3_tflops_spec"] = round(res["sms"] * res["e4m3_flop_per_clk_per_sm"] * mhz * 1e6 / 1e12, 1)
    res["how"] = ("one CTA per SM issuing 4096 back-to-back 128x256 tcgen05 MMAs (both operands in shared "
                  "memory); FLOP/clk/SM from the slowest SM's clock64 time; spec = SMs x that x max SM clock")
    print(json.dumps(res), flush=True)


def spec_peak():
    try:
        with open(os.path.join(ROOT, "profiles", "spec_dense_peak.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def measure_fp8_peak():
    """Dense e4m3 GEMM throughput of cuBLASLt (torch._scaled_mm, 8192^3,
    bf16 output), measured like the bf16 peak: best of 10 (burst) and back to
    back for 4 s (sustained)."""
    import torch
    n = 8192
    a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()
    one = torch.ones((), device="cuda")

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flops = 2.0 * n ** 3
    with ClockSampler(None) as clk:
        t0 = time.perf_counter()
        cnt = 0
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        while time.perf_counter() - t0 < 4.0:
            for _ in range(20):
                mm()
            cnt += 20
            torch.cuda.synchronize()
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
    out = {"fp8_tflops": round(flops / (best / 1e3) / 1e12, 1),
           "fp8_tflops_sustained": round(flops * cnt / (ms / 1e3) / 1e12, 1),
           "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3 (2 N^3): best of 10 (burst) and back to back "
                  "for 4 s (sustained), CUDA events", "clocks": clk.summary(),
           "gpu": torch.cuda.get_device_name(0), "torch": torch.__version__}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--quick", action="store_true", help="skip e2e, FP8 and CPU baseline (profiling runs)")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--fp8-peak", action="store_true", help="measure the cuBLASLt e4m3 GEMM peak and exit")
    ap.add_argument("--spec-peak", action="store_true", help="measure the tcgen05 spec dense peak and exit")
    ap.add_argument("--sweep", choices=["bf16", "fp8", "bwd"],
                    help="time every point of the 16384-token sweep (one JSON line each) and exit")
    args = ap.parse_args()
    if args.fp8_peak:
        measure_fp8_peak()
        return
    if args.spec_peak:
        measure_spec_peak()
        return
    if args.sweep:
        run_sweep(args.sweep, args.warmup)
        return
    w = workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w, args.workload)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist

    from exact_attention_71_gb300 import api

    ws, rank, local = dist_setup()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    # Multi-rank: the global batch is B x world; each rank owns a contiguous
    # shard of it (no data exchange between ranks).
    from exact_attention_71_gb300.shard import batch_shard
    b_start, b_stop = batch_shard(w["B"] * ws, ws, rank)
    global_batch = w["B"] * ws
    w = dict(w, B=b_stop - b_start)
    # Two resident input sets (> L2 each) used alternately, so no step finds
    # the previous step's inputs in the 129 MB L2.
    bwd = w.get("direction") == "bwd"
    sets = []
    arrs0 = None
    for s in range(2):
        tensors, arrs = make_inputs(w, device, seed=s + 2 * b_start)
        if s == 0:
            arrs0 = arrs
        q, k, v = tensors[:3]
        if w["dtype"] == "fp8":
            q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, sign_seed=1234)
            sets.append((q8, k8, v8, qs, ks, vs))
        elif w.get("sparse"):
            sets.append((q, k, v, torch.from_numpy(block_mask(w)).to(device)))
        elif bwd:
            # The backward consumes the forward's O and LSE, computed once here.
            o_s, lse_s = api.attn_fwd(q, k, v, causal=w["causal"], window=w["window"])
            sets.append((tensors[3], q, k, v, o_s, lse_s))
        else:
            sets.append((q, k, v))
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    if bwd:
        grads = (torch.empty_like(sets[0][1]), torch.empty_like(sets[0][2]), torch.empty_like(sets[0][3]))
        work = torch.empty(api.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)
    step_idx = [0]

    def step():
        s = sets[step_idx[0] & 1]
        step_idx[0] += 1
        if w["dtype"] == "fp8":
            api.attn_fwd_fp8(*s, causal=w["causal"], window=w["window"], out=o, lse=lse, stream=stream)
        elif bwd:
            api.attn_bwd(*s, causal=w["causal"], window=w["window"], dq=grads[0], dk=grads[1], dv=grads[2],
                         workspace=work, stream=stream)
        elif w.get("sparse"):
            api.attn_fwd_sparse(*s, causal=w["causal"], window=w["window"], out=o, lse=lse, stream=stream)
        else:
            api.attn_fwd(*s, causal=w["causal"], window=w["window"], out=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass
    with ClockSampler(uuid if rank == 0 else None) as clk:
        barrier()
        ms = time_loop(step, args.steps, stream)
        barrier()
    t_local = torch.tensor([ms], dtype=torch.float64, device=device)
    if ws > 1:
        dist.all_reduce(t_local, op=dist.ReduceOp.MAX)
    ms_total = float(t_local.item())
    rc, site = api.device_status(stream)
    if rc != 0:
        raise SystemExit(f"device status {rc} (site {site:#x})")

    flops = flops_per_step(w)
    ms_step = ms_total / args.steps
    value = ws * flops * args.steps / (ms_total / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    achieved = flops / (ms_step / 1e3) / 1e12
    kernel = ("attn_fwd_fp8" + {128: "", 256: "_d256", 64: "_d64"}[w["d"]]) if w["dtype"] == "fp8" else (
        "attn_bwd" if bwd else ("attn_fwd_sparse" if w.get("sparse") else "attn_fwd"))
    if w["dtype"] == "fp8":
        fp8_peak = peaks.get("fp8_tflops") or 2.0 * peaks["bf16_tflops"]
        peak, peak_note = fp8_peak, f"{peak_src} bf16 burst x 2 (nominal fp8:bf16 ratio)"
    else:
        peak, peak_note = peaks["bf16_tflops"], f"{peak_src} bf16 burst (cuBLAS)"
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": recorded_traffic(kernel, args.workload),
            "peak_source": peak_note,
            "frac_of_sustained": round(achieved / (peaks.get("bf16_tflops_sustained", peak) *
                                                   (2.0 if w["dtype"] == "fp8" else 1.0)), 4)}
    sp = spec_peak()
    if sp:
        roof["frac_of_spec_dense"] = round(achieved / sp["e4m3_tflops_spec" if w["dtype"] == "fp8" else
                                                       "bf16_tflops_spec"], 4)
    if w["dtype"] == "fp8" and cublaslt_fp8_peak():
        roof["frac_of_cublaslt_fp8_gemm"] = round(achieved / cublaslt_fp8_peak(), 4)
    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w["dtype"] == "bf16" else "e4m3", "data": "synthetic",
            "config": {"workload": w["name"], "B": B, "H": H, "H_kv": w.get("Hkv", H), "N": N, "d": d,
                       "causal": w["causal"],
                       "window": w["window"], "flops_per_step": flops,
                       "flop_convention": ("4 d x visible (query, key) pairs after the block mask" if w.get("sparse")
                                           else "4 B H N^2 d, halved for causal; window: 4 d x attended pairs")
                                          + ("; backward 2.5 x" if bwd else ""),
                       "l2": "inputs larger than L2 (two resident input sets, alternated per step)",
                       "global_batch": global_batch,
                       "parallelism": f"batch shards x{ws}, no collective on the data path"},
            "roofline": roof, "gpu_launches": args.steps * (3 if bwd else 1),
            "clocks": clk.summary() if rank == 0 else None}
    if bwd:
        line["roofline"]["note"] = ("achieved counts the whole backward step: the fused kernel plus the two "
                                    "memory-bound launches around it (D / accumulator zeroing, dQ conversion)")

    if not args.quick:
        # Every rank runs the end-to-end leg on its own shard at the same
        # time (a barrier right before the timed loop); the job's figure is
        # all ranks' work over the slowest rank's time.
        e2e = e2e_measure(api, w, device, stream, arrs0, flops, steps=min(args.steps, 100),
                          sync=(lambda: dist.barrier()) if ws > 1 else None)
        if ws > 1:
            t_e2e = torch.tensor([e2e["ms_per_step"]], dtype=torch.float64, device=device)
            dist.all_reduce(t_e2e, op=dist.ReduceOp.MAX)
            e2e = job_e2e(e2e, float(t_e2e.item()), ws, flops)
        if rank == 0:
            line["e2e"] = e2e
    if not args.quick and rank == 0:
        if args.workload == DEFAULT_WORKLOAD:
            line["noncausal"] = fwd_secondary(api, device, stream, "c3_d128_n16k_noncausal",
                                              steps=min(args.steps, 200))
            line["c2"] = fwd_secondary(api, device, stream, "c2", steps=min(args.steps, 200))
            line["fp8"] = fp8_secondary(api, device, stream, steps=min(args.steps, 200))
            line["bwd"] = bwd_secondary(api, device, stream, steps=min(args.steps, 50))
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.ref_budget, arrs=arrs0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def job_e2e(rank_e2e: dict, ms_slowest: float, ws: int, flops_per_rank: float) -> dict:
    """The whole job's end-to-end figure from one rank's: every rank moved
    the same bytes and did the same work in its step, and the job's step
    takes the slowest rank's time."""
    out = dict(rank_e2e)
    out["ms_per_step"] = round(ms_slowest, 4)
    out["value"] = round(ws * flops_per_rank / (ms_slowest / 1e3) / 1e12, 2)
    out["h2d_bytes_per_step"] = rank_e2e["h2d_bytes_per_step"] * ws
    out["d2h_bytes_per_step"] = rank_e2e["d2h_bytes_per_step"] * ws
    out["ranks"] = ws
    return out


def e2e_measure(api, w, device, stream, arrs, flops, steps, sync=None):
    """Same metric through the public API with HOST buffers: pinned host
    Q, K, V copied to the device, the forward, O and LSE copied back, all
    inside the timed region."""
    import torch
    if w.get("direction") == "bwd":
        return e2e_measure_bwd(api, w, device, stream, arrs, flops, steps, sync)
    hmask = torch.from_numpy(block_mask(w)).pin_memory() if w.get("sparse") else None
    dmask = torch.empty_like(hmask, device=device) if hmask is not None else None
    hq, hk, hv = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in arrs)
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    dq, dk, dv = (torch.empty_like(t, device=device) for t in (hq, hk, hv))
    do = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=device)
    dl = torch.empty((B, H, N), dtype=torch.float32, device=device)
    ho = torch.empty((B, N, H, d), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    fp8 = w["dtype"] == "fp8"
    launches = 4 if fp8 else 1
    host_path = hmask is None
    if host_path:
        # The library's host-buffer entries: chunks of sequences staged
        # through two device slots, copies overlapping the compute (and the
        # previous step's copies).  FP8: prep of Q, K, V + forward per chunk.
        wsb = (api.fwd_fp8_host_workspace_bytes if fp8 else api.fwd_host_workspace_bytes)(B, H, H, N, d)
        ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        seqs_per_chunk = -(-B // min(B, 4))
        launches = -(-B // seqs_per_chunk) * (4 if fp8 else 1)

    # Host path: consecutive steps alternate between two streams (two requests
    # in flight), so one step's input copies can start while the previous
    # step's outputs are still coming back; each step's own copies and
    # forward stay ordered on its stream.
    streams = [stream, torch.cuda.Stream(device=device)]
    host_out = [(ho, hl), (torch.empty_like(ho).pin_memory(), torch.empty_like(hl).pin_memory())]
    turn = [0]

    def step():
        if host_path:
            s_ = streams[turn[0] & 1]
            o_, l_ = host_out[turn[0] & 1]
            turn[0] += 1
            if fp8:
                api.attn_fwd_fp8_host(hq, hk, hv, api.MODE_BLOCK_HADAMARD, 1234, causal=w["causal"],
                                      window=w["window"], out=o_, lse=l_, workspace=ws, stream=s_)
            else:
                api.attn_fwd_host(hq, hk, hv, causal=w["causal"], window=w["window"], out=o_, lse=l_, workspace=ws,
                                  stream=s_)
            return
        with torch.cuda.stream(stream):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            if fp8:
                q8, k8, v8, qs, ks, vs = api.fp8_prepare_qkv(dq, dk, dv, api.MODE_BLOCK_HADAMARD, 1234,
                                                             stream=stream)
                api.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=w["causal"], window=w["window"], out=do,
                                 lse=dl, stream=stream)
            elif hmask is not None:
                dmask.copy_(hmask, non_blocking=True)
                api.attn_fwd_sparse(dq, dk, dv, dmask, causal=w["causal"], window=w["window"], out=do, lse=dl,
                                    stream=stream)
            else:
                api.attn_fwd(dq, dk, dv, causal=w["causal"], window=w["window"], out=do, lse=dl, stream=stream)
            ho.copy_(do, non_blocking=True)
            hl.copy_(dl, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    if sync:
        sync()
    if host_path:
        ms = time_loop_two_streams(step, steps, streams) / steps
    else:
        ms = time_loop(step, steps, stream) / steps
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 + (hmask.numel() if hmask is not None else 0)
    d2h = ho.numel() * 2 + hl.numel() * 4
    out = {"value": round(flops / (ms / 1e3) / 1e12, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "kernel_launches_per_step": launches}
    if host_path:
        out["api"] = (("attn_fwd_fp8_host" if fp8 else "attn_fwd_host") +
                      " (pinned host buffers; per-sequence chunks, copies overlapped with the compute; two streams)")
    return out


def fwd_secondary(api, device, stream, key, steps):
    """A further bf16 forward workload, timed like the main line (two
    resident input sets larger than L2, alternated per step)."""
    import torch
    w = dict(WORKLOADS[key])
    sets = [make_inputs(w, device, seed=s)[0] for s in range(2)]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    idx = [0]

    def fn():
        q, k, v = sets[idx[0] & 1]
        idx[0] += 1
        api.attn_fwd(q, k, v, causal=w["causal"], window=w["window"], out=o, lse=lse, stream=stream)

    for _ in range(5):
        fn()
    torch.cuda.synchronize(device)
    ms = time_loop(fn, steps, stream) / steps
    flops = flops_per_step(w)
    peaks, src = load_peaks()
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": w["name"], "flops_per_step": flops, "ms": round(ms, 5), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4), "steps": steps,
            "traffic": recorded_traffic("attn_fwd", key)}


def bwd_secondary(api, device, stream, steps):
    """The backward on its headline point (the pages' Fig. 6: d=128,
    non-causal, N=16k, 16 heads), timed like the main line."""
    import torch
    w = dict(WORKLOADS["bwd"])
    tensors, _ = make_inputs(w, device, seed=0)
    do, (q, k, v) = tensors[3], tensors[:3]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    o, lse = api.attn_fwd(q, k, v, causal=False)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    work = torch.empty(api.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)

    def fn():
        api.attn_bwd(do, q, k, v, o, lse, causal=False, dq=dq, dk=dk, dv=dv, workspace=work, stream=stream)

    for _ in range(3):
        fn()
    torch.cuda.synchronize(device)
    ms = time_loop(fn, steps, stream) / steps
    flops = flops_per_step(w)
    peaks, src = load_peaks()
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": w["name"], "flops_per_step": flops, "ms": round(ms, 4), "tflops": round(tf, 1),
            "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4), "launches_per_step": 3,
            "flop_convention": "2.5 x the forward's 4 B H N^2 d (five products against two)"}


def e2e_measure_bwd(api, w, device, stream, arrs, flops, steps, sync=None):
    """Backward end to end with HOST buffers: pinned Q, K, V, dO and the
    forward's O, LSE copied in, the backward, dQ, dK, dV copied back, all
    inside the timed region (through attn_bwd_host)."""
    import torch
    host = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in arrs]
    hq, hk, hv, hdo = host
    dq_, dk_, dv_, ddo = (torch.empty_like(t, device=device) for t in host)
    o_dev, lse_dev = api.attn_fwd(dq_.copy_(hq), dk_.copy_(hk), dv_.copy_(hv), causal=w["causal"], window=w["window"])
    ho, hl = o_dev.cpu().pin_memory(), lse_dev.cpu().pin_memory()
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    Hkv = hk.shape[2]
    # The library's host-buffer backward: chunks of sequences staged through
    # two device slots; consecutive steps alternate between two streams so
    # that one step's copies overlap the previous step's backward.
    ws = torch.empty(api.bwd_host_workspace_bytes(B, H, Hkv, N, d), dtype=torch.uint8, device=device)
    outs = [tuple(torch.empty_like(t).pin_memory() for t in (hq, hk, hv)) for _ in range(2)]
    streams = [stream, torch.cuda.Stream(device=device)]
    turn = [0]

    def step():
        i = turn[0] & 1
        turn[0] += 1
        gq, gk, gv = outs[i]
        api.attn_bwd_host(hdo, hq, hk, hv, ho, hl, causal=w["causal"], window=w["window"], dq=gq, dk=gk, dv=gv,
                          workspace=ws, stream=streams[i])

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    if sync:
        sync()
    ms = time_loop_two_streams(step, steps, streams) / steps
    hgq, hgk, hgv = outs[0]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, ho, hl))
    d2h = sum(t.numel() * t.element_size() for t in (hgq, hgk, hgv))
    seqs_per_chunk = -(-B // min(B, 4))
    return {"value": round(flops / (ms / 1e3) / 1e12, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "kernel_launches_per_step": 3 * -(-B // seqs_per_chunk),
            "api": "attn_bwd_host (pinned host buffers; per-sequence chunks, copies overlapped with the compute; "
                   "two streams)"}


def fp8_secondary(api, device, stream, steps):
    """FP8 path on its workload: prep (3 tensors) + FP8 forward, and the
    forward alone."""
    import torch
    w = dict(WORKLOADS["c4"])
    (q, k, v), _ = make_inputs(w, device, seed=0)
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    prepped = api.fp8_prepare_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 1234, stream=stream)

    def fwd_only():
        api.attn_fwd_fp8(*prepped, causal=False, out=o, lse=lse, stream=stream)

    def with_prep():
        pp = api.fp8_prepare_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 1234, stream=stream)
        api.attn_fwd_fp8(*pp, causal=False, out=o, lse=lse, stream=stream)

    flops = flops_per_step(w)
    out = {"workload": w["name"], "flops_per_step": flops}
    for name, fn in (("fwd", fwd_only), ("prep_plus_fwd", with_prep)):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(device)
        ms = time_loop(fn, steps, stream) / steps
        out[name] = {"ms": round(ms, 5), "tflops": round(flops / (ms / 1e3) / 1e12, 1)}
    peaks, src = load_peaks()
    fp8_peak = peaks.get("fp8_tflops") or 2.0 * peaks["bf16_tflops"]
    out["frac_of_fp8_peak"] = round(out["fwd"]["tflops"] / fp8_peak, 4)
    out["fp8_peak"] = fp8_peak
    out["fp8_peak_source"] = f"{src} bf16 burst x 2 (nominal fp8:bf16 ratio)"
    if cublaslt_fp8_peak():
        out["frac_of_cublaslt_fp8_gemm"] = round(out["fwd"]["tflops"] / cublaslt_fp8_peak(), 4)
        out["cublaslt_fp8_gemm_tflops"] = cublaslt_fp8_peak()
    return out


def run_sweep(kind: str, warmup: int):
    """Every point of the 16384-token sweep (hidden 2048: B = 16384 / N,
    H = 2048 / d) for one path, in one process: per point, inputs of
    B x N x H x d (each tensor 64 MB, larger than L2 together), W untimed
    launches, then about half a second of launches timed with CUDA events on
    the launching stream, the SM clock sampled meanwhile."""
    import torch

    from exact_attention_71_gb300 import api
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    uuid = None
    try:
        uuid = subprocess.run(["nvidia-smi", "--query-gpu=uuid", "--format=csv,noheader", "-i", "0"],
                              capture_output=True, text=True, timeout=30).stdout.strip() or None
    except Exception:
        pass
    peaks, src = load_peaks()
    dims = (64, 128) if kind == "bwd" else (64, 128, 256)
    for d in dims:
        for causal in (False, True):
            for n in (512, 1024, 2048, 4096, 8192, 16384):
                prefix = {"bf16": "c3", "fp8": "fp8", "bwd": "bwd"}[kind]
                key = f"{prefix}:{n}:{d}:{int(causal)}" if kind != "bwd" else f"bwd:{n}:{int(causal)}:{d}"
                w = workload(key)
                tensors, _ = make_inputs(w, device, seed=0)
                q, k, v = tensors[:3]
                B, H, N = w["B"], w["H"], w["N"]
                o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=device)
                lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
                if kind == "bf16":
                    def fn():
                        api.attn_fwd(q, k, v, causal=causal, out=o, lse=lse, stream=stream)
                elif kind == "fp8":
                    pp = api.fp8_prepare_qkv(q, k, v, api.MODE_BLOCK_HADAMARD, 1234, stream=stream)

                    def fn():
                        api.attn_fwd_fp8(*pp, causal=causal, out=o, lse=lse, stream=stream)
                else:
                    do = tensors[3]
                    api.attn_fwd(q, k, v, causal=causal, out=o, lse=lse, stream=stream)
                    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                    work = torch.empty(api.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=device)

                    def fn():
                        api.attn_bwd(do, q, k, v, o, lse, causal=causal, dq=dq, dk=dk, dv=dv, workspace=work,
                                     stream=stream)
                for _ in range(warmup):
                    fn()
                torch.cuda.synchronize(device)
                probe = time_loop(fn, 3, stream) / 3
                steps = max(10, min(2000, int(500.0 / max(probe, 1e-3))))
                with ClockSampler(uuid) as cs:
                    ms = time_loop(fn, steps, stream) / steps
                st = api.device_status()
                if st[0] != 0:
                    raise SystemExit(f"device status {st} at {key}")
                flops = flops_per_step(w)
                tf = flops / (ms / 1e3) / 1e12
                peak = peaks["bf16_tflops"] * (2.0 if kind == "fp8" else 1.0)
                sp = spec_peak()
                sp_tf = (sp or {}).get("e4m3_tflops_spec" if kind == "fp8" else "bf16_tflops_spec")
                print(json.dumps({"sweep": kind, "workload": key, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                                  "ms": round(ms, 5), "tflops": round(tf, 1), "frac_of_measured_peak": round(tf / peak, 4),
                                  "frac_of_spec_dense": round(tf / sp_tf, 4) if sp_tf else None, "steps": steps,
                                  "clocks": cs.summary()}), flush=True)
                del tensors, q, k, v, o, lse
                torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
