#!/usr/bin/env python
"""Benchmark of one attention step (forward + backward) on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
fa_fwd (O, L) then fa_bwd (D, dK, dV, dQ) through the C ABI.  The default
workload is the GQA long-sequence shape: B=2, Hq=32, Hkv=8, N=8192, d=128,
bf16, causal.  Throughput counts FLOPs as 4*B*H*N^2*d for the forward
(halved under the causal mask) plus 2.5x that for the backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own copy of
the workload (its shard of an N-times larger batch: the (batch, kv-head)
units are independent, so there is no collective on the data path) and
`value` is the total over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_io_aware_20_gb300.inputs import WORKLOADS, Workload, make_inputs  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s (4·B·H·N²·d) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "gqa8k"
L2_BYTES = 129 * 2**20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Sources each timed kernel is built from: a recorded DRAM-traffic figure is
# used only while these files are unchanged.
_COMMON_SOURCES = ["exact_io_aware_20_gb300/csrc/fa_api.cu",
                   "exact_io_aware_20_gb300/csrc/fa_internal.h",
                   "exact_io_aware_20_gb300/csrc/block_list.cuh",
                   "exact_io_aware_20_gb300/csrc/sm103_ptx.cuh"]
KERNEL_SOURCES = {
    "fwd": ["exact_io_aware_20_gb300/csrc/fa_fwd_kernel.cuh",
            "exact_io_aware_20_gb300/csrc/fa_fwd.cu"] + _COMMON_SOURCES,
    "bwd_main": ["exact_io_aware_20_gb300/csrc/fa_bwd_fused_kernel.cuh",
                 "exact_io_aware_20_gb300/csrc/fa_bwd_fused.cu",
                 "exact_io_aware_20_gb300/csrc/fa_bwd_kernel.cuh"] + _COMMON_SOURCES,
    "bwd_dq": ["exact_io_aware_20_gb300/csrc/fa_bwd_dq_kernel.cuh",
               "exact_io_aware_20_gb300/csrc/fa_bwd_dq.cu"] + _COMMON_SOURCES,
}


# Small shapes for profiler captures (--mode case): one kernel of each kind
# on a few hundred MB, larger than L2.  name -> (workload, deterministic backward)
PROFILE_CASES = {
    "gqa8k_b1": (WORKLOADS["gqa8k"].with_(B=1), False),
    "gpt_layer_b2": (WORKLOADS["gpt_layer"].with_(B=2), False),
    "gpt_layer_causal_b2": (WORKLOADS["gpt_layer_causal"].with_(B=2), False),
    "d64": (Workload("d64", 1, 16, 16, 4096, 64, "bf16", False, 7), False),
    "head256_b1": (WORKLOADS["head256"].with_(B=1), False),
    "head256_b1_det": (WORKLOADS["head256"].with_(B=1), True),
}


def run_case(args):
    """One forward and two backward calls of a small shape: the launches a
    profiler capture selects from (-k <kernel> -s <launches to skip> -c 1)."""
    torch.cuda.set_device(0)
    from exact_io_aware_20_gb300 import binding
    binding.load()
    w, det = PROFILE_CASES[args.case]
    q, k, v, do = make_inputs(w, "cuda")
    o, lse = binding.forward(q, k, v, w.causal, w.scale)
    for _ in range(2):
        binding.backward(q, k, v, o, lse, do, w.causal, w.scale, deterministic=det)
    binding.device_status()
    print(json.dumps({"case": args.case, "shape": f"B={w.B} Hq={w.H} Hkv={w.Hkv} N={w.N} d={w.d} "
                                                 f"{w.dtype} causal={int(w.causal)}",
                      "deterministic": det}), flush=True)
    return 0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the forward / backward timings of the other workloads")
    ap.add_argument("--mode", choices=["train", "decode", "blocksparse", "case"], default="train",
                    help="train: fwd+bwd step (the headline); decode: short-query forward; "
                         "blocksparse: fwd+bwd step under a random block mask; case: one "
                         "forward and two backward calls of a --case, for profiler captures")
    ap.add_argument("--case", default="gqa8k_b1", choices=sorted(PROFILE_CASES),
                    help="case: the shape to run (see PROFILE_CASES)")
    ap.add_argument("--density", type=float, default=0.25,
                    help="blocksparse: fraction of 128x128 blocks kept")
    ap.add_argument("--decode-nq", type=int, default=1)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller profiling captures)")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """The source without its comments and with whitespace collapsed, so that
    a comment edit does not invalidate a measurement of unchanged code (the
    sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.txt, if taken on this exact source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    if kind not in KERNEL_SOURCES:
        return None
    src = kernel_source_hash(kind)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kind and \
                parts[1] == workload and parts[2] == src:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for row in csv.reader(io.StringIO(out)):
            if len(row) >= 9:
                self.rows.append([c.strip() for c in row])
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1])]
        mx = [num(r[2]) for r in self.rows if num(r[2])]
        power = [num(r[3]) for r in self.rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() in ("active", "0x1", "1")})
        top = max(mx) if mx else None
        loaded = [s for s in sm if top and s > 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": top,
                "power_w_max": max(power) if power else None, "samples": len(self.rows),
                "reasons": reasons}


class NvmlPoller:
    """SM clock, power and clock-event reasons read through NVML every few
    milliseconds (the timed region of the default run lasts well under a
    second, too short for nvidia-smi's 100 ms sampling).  Read-only queries;
    None when the NVML library is not present."""
    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.002):
        import ctypes
        self.ct = ctypes
        self.period = period_s
        self.samples = []
        self.lib = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) != 0:
                return
            self.lib, self.h, self.max_mhz = lib, h, float(mx.value)
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception:
            self.lib = None

    def _sample(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, ct.c_int(1), ct.byref(clk)) != 0:
            return
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.reasons_fn(self.h, ct.byref(rs))
        self.samples.append((float(clk.value), pw.value / 1000.0, int(rs.value)))

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        if self.lib is not None:
            def loop():
                while not self._stop.is_set():
                    self._sample()
                    time.sleep(self.period)
            self._t = threading.Thread(target=loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self.lib is not None:
            self._t.join(timeout=2)
        return False

    def summary(self):
        if self.lib is None or not self.samples:
            return None
        sm = [s[0] for s in self.samples]
        loaded = [s for s in sm if s > 0.5 * self.max_mhz] or sm
        reasons = sorted({name for s in self.samples for bit, name in self.REASONS.items()
                          if s[2] & bit})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(loaded), "power_w_max": max(s[1] for s in self.samples),
                "samples": len(self.samples), "reasons": reasons, "source": "nvml, 2 ms"}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(w: Workload, target_pairs: float):
    """A bounded sample of the workload for the CPU oracle: whole (batch,
    kv-head) groups in order, the last one cut to its final rows (the rows
    with the most keys under the mask).  Returns ([(b, kh, r0, r1)], pairs)
    with r0..r1 flattened rows g*N + i of the group, and the number of
    unmasked query-key pairs it covers."""
    G = w.H // w.Hkv

    def row_pairs(r):
        i = r % w.N
        return (i + 1) if w.causal else w.N

    segments, pairs = [], 0
    for u in range(w.B * w.Hkv):
        b, kh = divmod(u, w.Hkv)
        r1 = G * w.N
        r0 = r1
        while r0 > 0 and pairs < target_pairs:
            r0 -= 1
            pairs += row_pairs(r0)
        segments.append((b, kh, r0, r1))
        if pairs >= target_pairs:
            break
    return segments, pairs


def run_oracle_sample(w: Workload, q, k, v, do, segments):
    import oracle
    G = w.H // w.Hkv
    t0 = time.perf_counter()
    for (b, kh, r0, r1) in segments:
        sl = slice(kh * G, (kh + 1) * G)
        oracle.backward_rows(q[b, sl], k[b, kh], v[b, kh], do[b, sl], r0, r1, w.causal, w.scale)
    return time.perf_counter() - t0


def describe(segments, pairs, w):
    G = w.H // w.Hkv
    parts = [f"(b{b},kvh{kh}) rows {r0}..{r1 - 1} of {G * w.N}" for b, kh, r0, r1 in segments]
    return (f"fp64 C oracle forward+backward over {len(segments)} (batch, kv-head) group(s) of "
            f"the {w.name} shape: " + "; ".join(parts) + f" ({pairs} unmasked query-key pairs)")


def cpu_baseline(w: Workload, target_seconds: float):
    """The oracle as it stands, on this host's cores, over a bounded sample."""
    import oracle
    q, k, v, do = make_inputs(w)
    threads = oracle.num_threads()
    # calibrate on a small slab, then size the sample for ~target_seconds
    seg, pairs = oracle_sample(w, 4e6)
    dt = run_oracle_sample(w, q, k, v, do, seg)
    seg, pairs = oracle_sample(w, pairs / max(dt, 1e-6) * target_seconds)
    dt = run_oracle_sample(w, q, k, v, do, seg)
    flops = pairs * 4.0 * w.d * 3.5      # metric FLOPs of these pairs: fwd + 2.5x bwd
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "seconds": round(dt, 3), "cpu": cpu_model(),
            "sample": describe(seg, pairs, w) + f", {threads} threads"}


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm
    implementer / part codes), with the number of logical CPUs."""
    fields = {}
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if ":" in line:
                    key, val = (s.strip() for s in line.split(":", 1))
                    fields.setdefault(key, val)
    except OSError:
        return "unknown"
    name = fields.get("model name") or " ".join(
        f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields) or "unknown"
    return f"{name}, {os.cpu_count()} logical CPUs"


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    q, k, v, do = make_inputs(w)
    import oracle
    threads = oracle.num_threads()
    seg, pairs = oracle_sample(w, 16e6)
    flops = pairs * 4.0 * w.d * 3.5
    for _ in range(args.warmup):
        run_oracle_sample(w, q, k, v, do, seg)
    times = []
    for _ in range(args.steps):
        times.append(run_oracle_sample(w, q, k, v, do, seg))
    total = sum(times)
    value = flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} Hq={w.H} Hkv={w.Hkv} N={w.N} d={w.d} "
                               f"{w.dtype} causal={int(w.causal)}",
                   "sample_per_step": describe(seg, pairs, w)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(), "sample": "per step: " + describe(seg, pairs, w)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- decode regime
def decode_result(steps: int, warmup: int, nq: int = 1) -> dict:
    """Short-query forward over a long key cache (decoding after a prefix):
    memory-bound, so the metric is GB/s of Q, K, V read and O, L written
    against the measured copy bandwidth.  Times fa_fwd_splitkv (key axis
    split over CTAs, partials merged) and fa_fwd_qk (one pass)."""
    from exact_io_aware_20_gb300 import binding
    binding.load()
    B, H, Hkv, Nq, Nk, d = 8, 32, 8, nq, 8192, 128
    w = Workload("decode", B, H, Hkv, Nq, d, "bf16", True, 1006)
    q, k, v, _ = make_inputs(w, "cuda", Nk=Nk)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, device="cuda")
    need = int(binding.load().fa_fwd_splitkv_workspace_size(B, H, Hkv, Nq, Nk, d, 0))
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    nbytes = (q.numel() + k.numel() + v.numel() + o.numel()) * 2 + lse.numel() * 4
    peaks, src = load_peaks()
    res = {}
    for name, fn in (("splitkv", lambda: binding.forward_splitkv(q, k, v, True, w.scale, 0, o, lse, ws)),
                     ("one_pass", lambda: binding.forward(q, k, v, True, w.scale, o, lse))):
        for _ in range(max(warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        res[name] = {"ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "frac_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    binding.device_status()
    return {
        "metric": "decode attention forward GB/s (Q,K,V read + O,L written)", "unit": "GB/s",
        "value": res["splitkv"]["GB/s"], "higher_is_better": True, "steps": steps,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode: B={B} Hq={H} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} bf16, "
                               f"causal (bottom-right), inputs larger than L2 ({nbytes >> 20} MiB)"},
        "peak": {"hbm_gbs": peaks["hbm_gbs"], "source": src},
        "splitkv": res["splitkv"], "one_pass": res["one_pass"],
        "splits_auto": need and int(need // (B * H * Nq * (d + 1) * 4)) or 1}


def run_decode(args):
    torch.cuda.set_device(0)
    print(json.dumps(decode_result(args.steps, args.warmup, args.decode_nq)), flush=True)
    return 0


# ---------------------------------------------------------------- block-sparse
def kept_pairs(mask: torch.Tensor, N: int, causal: bool) -> int:
    """(query, key) pairs a shared block mask [1, N/128, N/128] keeps per head
    (N a multiple of 128), with the causal diagonal blocks half kept."""
    nb = N // 128
    keep = mask[0].bool().cpu()
    if not causal:
        return int(keep.sum()) * 128 * 128
    below = int((keep & torch.ones(nb, nb, dtype=torch.bool).tril(-1)).sum())
    diag = int((keep & torch.eye(nb, dtype=torch.bool)).sum())
    return below * 128 * 128 + diag * (128 * 129 // 2)


def blocksparse_result(workload: str, density: float, steps: int, warmup: int) -> dict:
    """fa_fwd_blocksparse + fa_bwd_blocksparse on a workload's shapes under a
    seeded random block mask (one pattern for all heads): TFLOP/s counted on
    the kept (query, key) pairs only, and the time against the dense step."""
    from exact_io_aware_20_gb300 import binding
    from exact_io_aware_20_gb300.inputs import make_block_mask
    binding.load()
    w = WORKLOADS[workload]
    q, k, v, do = make_inputs(w, "cuda")
    mask = make_block_mask(1, w.N, w.N, density, w.seed, "cuda")
    pairs = kept_pairs(mask, w.N, w.causal) * w.B * w.H
    flops = 4.0 * w.d * pairs * 3.5          # forward 4d, backward 2.5x that, per kept pair
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d), dtype=torch.uint8,
                     device="cuda")

    def sparse_step():
        binding.forward_blocksparse(q, k, v, mask, w.causal, w.scale, o, lse)
        binding.backward_blocksparse(q, k, v, o, lse, do, mask, w.causal, w.scale, dq, dk, dv, ws)

    def dense_step():
        binding.forward(q, k, v, w.causal, w.scale, o, lse)
        binding.backward(q, k, v, o, lse, do, w.causal, w.scale, dq, dk, dv, ws)

    res = {}
    for name, fn in (("sparse", sparse_step), ("dense", dense_step)):
        for _ in range(max(warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / steps
    binding.device_status()
    peaks, src = load_peaks()
    value = flops / (res["sparse"] * 1e-3) / 1e12
    dense_pairs = w.B * w.H * (w.N * (w.N + 1) // 2 if w.causal else w.N * w.N)
    del q, k, v, do, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return {
        "metric": "block-sparse attention fwd+bwd TFLOP/s (kept pairs)", "unit": "TFLOP/s",
        "value": round(value, 1), "higher_is_better": True, "steps": steps,
        "warmup": warmup, "ms_per_step": round(res["sparse"], 4), "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{w.name} (B={w.B} Hq={w.H} Hkv={w.Hkv} N={w.N} d={w.d}, "
                               f"causal={w.causal}) under a random 128x128 block mask, "
                               f"density {density}, shared by all heads; inputs larger "
                               f"than L2"},
        "kept_fraction": round(pairs / dense_pairs, 4),
        "dense_ms_per_step": round(res["dense"], 4),
        "speedup_vs_dense": round(res["dense"] / res["sparse"], 3),
        "frac_of_burst": round(value / peaks["bf16_tflops"], 4), "peak_source": src}


def run_blocksparse(args):
    torch.cuda.set_device(0)
    print(json.dumps(blocksparse_result(args.workload, args.density, args.steps, args.warmup)),
          flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "decode":
        return run_decode(args)
    if args.mode == "blocksparse":
        return run_blocksparse(args)
    if args.mode == "case":
        return run_case(args)
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from exact_io_aware_20_gb300 import binding
    binding.load()

    base = WORKLOADS[args.workload]
    if args.batch:
        base = base.with_(B=args.batch)
    w = base.with_(seed=base.seed + 7919 * rank)
    q_h, k_h, v_h, do_h = make_inputs(w)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o, lse = binding.forward(q, k, v, w.causal, w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.forward(q, k, v, w.causal, w.scale, out=o, lse=lse, stream=stream)
        binding.backward(q, k, v, o, lse, do, w.causal, w.scale, dq=dq, dk=dk, dv=dv,
                         workspace=ws, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    binding.device_status()

    # ------------------------------------------------ device-timed region
    def timed_region():
        binding.timing_enable(4 * args.steps + 8)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clocks, NvmlPoller(local) as nvml:
            barrier()
            torch.cuda.synchronize()
            step_evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
            ev0.record(stream)
            for i in range(args.steps):
                step()
                step_evs[i].record(stream)
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
        binding.device_status()
        # each step's own time (the line's value is over the whole region)
        step_ms = [ev0.elapsed_time(step_evs[0])] + \
            [step_evs[i - 1].elapsed_time(step_evs[i]) for i in range(1, args.steps)]
        kernel_times = binding.timing_read()
        binding.timing_enable(0)
        return ev0.elapsed_time(ev1), step_ms, kernel_times, clocks, nvml

    def throttled(clocks, nvml) -> list:
        """Clock-event reasons that void a measurement (a power cap does not)."""
        seen = set((nvml.summary() or {}).get("reasons", [])) | set(clocks.summary().get("reasons", []))
        bad = sorted(seen & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"})
        if world > 1:    # every rank takes the same decision
            import torch.distributed as dist
            t = torch.tensor([1.0 if bad else 0.0], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            if t.item() > 0 and not bad:
                bad = ["on another rank"]
        return bad

    ms_total, step_ms, kernel_times, clocks, nvml = timed_region()
    remeasured = throttled(clocks, nvml)
    if remeasured:
        # a slowdown during the region: measure once more and report that one
        ms_total, step_ms, kernel_times, clocks, nvml = timed_region()
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / args.steps
    flops_step = w.flops_fwd() + w.flops_bwd()
    value = world * flops_step / (ms_step * 1e-3) / 1e12

    # ------------------------------------------------ end to end through the public API
    pin = lambda t: t.pin_memory()  # noqa: E731
    q_p, k_p, v_p, do_p = (pin(t) for t in (q_h, k_h, v_h, do_h))
    outs_p = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in (q_p, k_p, v_p, do_p))
    d2h = sum(t.numel() * t.element_size() for t in outs_p)

    def e2e_step():
        for dst, src in ((q, q_p), (k, k_p), (v, v_p), (do, do_p)):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(outs_p, (o, lse, dq, dk, dv)):
            dst.copy_(src, non_blocking=True)

    def timed_e2e(body):
        body(1)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        body(args.e2e_steps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = e0.elapsed_time(e1) / args.e2e_steps
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    def serial(n, start=None):
        for _ in range(n):
            e2e_step()

    # Pipelined: two device copies of the inputs and outputs; step i's inputs
    # go up on one copy stream while step i - 1 computes, its outputs come
    # back on another while step i + 1 computes.  Every step still copies all
    # of its inputs in and all of its outputs out inside the timed region.
    sets = [(q, k, v, do, o, lse, dq, dk, dv, ws)]
    sets.append(tuple(torch.empty_like(t) for t in sets[0]))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def pipelined(n, start=None):
        comp_done, out_done = [None, None], [None, None]
        if start is not None:
            s_in.wait_event(start)
            s_out.wait_event(start)
        for i in range(n):
            j = i % 2
            qq, kk, vv, dd, oo, ll, gq, gk, gv, wk = sets[j]
            if comp_done[j] is not None:      # step i - 2 has read this set's inputs
                s_in.wait_event(comp_done[j])
            with torch.cuda.stream(s_in):
                for dst, src in ((qq, q_p), (kk, k_p), (vv, v_p), (dd, do_p)):
                    dst.copy_(src, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
            stream.wait_event(in_done)
            if out_done[j] is not None:       # step i - 2's outputs have left this set
                stream.wait_event(out_done[j])
            binding.forward(qq, kk, vv, w.causal, w.scale, out=oo, lse=ll, stream=stream)
            binding.backward(qq, kk, vv, oo, ll, dd, w.causal, w.scale, dq=gq, dk=gk, dv=gv,
                             workspace=wk, stream=stream)
            comp_done[j] = torch.cuda.Event()
            comp_done[j].record(stream)
            s_out.wait_event(comp_done[j])
            with torch.cuda.stream(s_out):
                for dst, src in zip(outs_p, (oo, ll, gq, gk, gv)):
                    dst.copy_(src, non_blocking=True)
            out_done[j] = torch.cuda.Event()
            out_done[j].record(s_out)
        for ev in out_done:
            if ev is not None:
                stream.wait_event(ev)

    ms_e2e_serial = timed_e2e(serial)
    ms_e2e = timed_e2e(pipelined)
    binding.device_status()

    if rank != 0:
        return 0

    # ------------------------------------------------ roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    clk = nvml.summary() or clocks.summary()
    if nvml.summary() is not None:
        clk["nvidia_smi"] = clocks.summary()
    dom = max(kernel_times, key=lambda kk: kernel_times[kk][0])
    dom_ms, dom_n = kernel_times[dom]
    per_launch_ms = dom_ms / max(dom_n, 1)
    if dom in ("fwd", "bwd_main", "bwd_dq"):
        # products per kernel, each w.flops_fwd() / 2: forward 2; backward 5,
        # or 4 in the main kernel and 3 in the query-outer dQ kernel when dQ
        # is computed there (S and dP formed again)
        dq_outer = kernel_times.get("bwd_dq", (0.0, 0))[1] > 0
        fl = {"fwd": 2.0, "bwd_main": 4.0 if dq_outer else 5.0, "bwd_dq": 3.0}[dom] * \
            w.flops_fwd() / 2

        achieved = fl / (per_launch_ms * 1e-3) / 1e12
        peak, why = choose_tensor_peak(peaks, peak_src, clk, ms_total * 1e-3)
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": why,
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    else:
        rows = w.B * w.H * w.N
        by = rows * w.d * 2 * 2 + rows * 4 + rows * w.d * 4 if dom == "bwd_pre" else \
            rows * w.d * (4 + 2)
        achieved = by / (per_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} copy bandwidth"}
    roof["traffic"] = recorded_traffic(dom, w.name)
    roof["ms_per_launch"] = round(per_launch_ms, 4)

    kernels = {}
    for kind, (ms, n) in kernel_times.items():
        if n:
            kernels[kind] = {"ms_per_launch": round(ms / n, 4), "launches": n,
                             "share": round(ms / sum(x[0] for x in kernel_times.values()), 4)}
    fwd_ms = kernel_times["fwd"][0] / max(kernel_times["fwd"][1], 1)
    bwd_ms = sum(kernel_times[kk][0] for kk in ("bwd_pre", "bwd_main", "bwd_convert", "bwd_dq")
                 if kk in kernel_times) / max(kernel_times["bwd_main"][1], 1)
    gpu_launches = sum(n for _, n in kernel_times.values())

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "ms_per_step_median": round(statistics.median(step_ms), 4),
        "ms_per_step_min": round(min(step_ms), 4),
        "config": {"workload": f"{w.name}: B={w.B} Hq={w.H} Hkv={w.Hkv} N={w.N} d={w.d} "
                               f"{w.dtype} causal={int(w.causal)}, N(0,1) inputs, seed {w.seed}",
                   "step": "fa_fwd + fa_bwd (O, L, dQ, dK, dV)",
                   "l2": f"inputs larger than L2: {round(step_bytes(w) / 2**20)} MiB touched per "
                         f"step vs {L2_BYTES // 2**20} MiB L2",
                   "parallelism": f"{world} rank(s), one workload copy each, no collective"},
        "pct_of_peak": {
            "step": round(value / world / peaks["bf16_tflops"], 4),
            "fwd": round(w.flops_fwd() / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "bwd": round(w.flops_bwd() / (bwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "denominator": f"{peak_src} bf16 burst {peaks['bf16_tflops']} TFLOP/s"},
        "fwd_tflops": round(w.flops_fwd() / (fwd_ms * 1e-3) / 1e12, 1),
        "bwd_tflops": round(w.flops_bwd() / (bwd_ms * 1e-3) / 1e12, 1),
        "kernels": kernels,
        "exp_rate": exp_rate(w, fwd_ms, kernel_times, binding.measure_ex2_rate(stream)),
        "roofline": roof,
        "dq_reduce": dq_reduce(w, kernel_times, stream),
        "e2e": {"value": round(world * flops_step / (ms_e2e * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "path": "pinned host Q,K,V,dO -> device, fa_fwd + fa_bwd, O,L,dQ,dK,dV -> "
                        "pinned host; two device buffer sets, inputs and outputs copied on their "
                        "own streams overlapping the neighbouring steps' compute",
                "serial_ms_per_step": round(ms_e2e_serial, 4),
                "serial_value": round(world * flops_step / (ms_e2e_serial * 1e-3) / 1e12, 2)},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        **({"remeasured_after": remeasured} if remeasured else {}),
        "timed_region_s": round(ms_total * 1e-3, 4),
    }
    if world == 1 and not args.no_per_config:
        line["bwd_deterministic"] = time_deterministic_bwd(w, q, k, v, o, lse, do, dq, dk, dv, ws,
                                                           stream, peaks)
        line["per_config"] = per_config(dev, peaks, peak_src)
        # the measurement plan's other regimes, in compact form: decode
        # (split-KV over an 8192-key cache) and block-sparse (the gqa8k
        # shapes under random block masks)
        dec = decode_result(20, 3)
        line["decode"] = {"GB/s": dec["value"], "frac_hbm": dec["splitkv"]["frac_hbm"],
                          "ms": dec["splitkv"]["ms"], "one_pass_GB/s": dec["one_pass"]["GB/s"],
                          "splits": dec["splits_auto"], "workload": dec["config"]["workload"]}
        line["blocksparse"] = {}
        for dens in (0.1, 0.25):
            bs = blocksparse_result("gqa8k", dens, 5, 3)
            line["blocksparse"][str(dens)] = {
                "tflops_kept_pairs": bs["value"], "ms_per_step": bs["ms_per_step"],
                "speedup_vs_dense": bs["speedup_vs_dense"], "kept_fraction": bs["kept_fraction"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(base, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def choose_tensor_peak(peaks, peak_src, clk, region_s):
    """The dense bf16 peak a kernel timed in this run is held against: the
    burst figure (a GEMM timed alone at full clock) unless the timed region
    lasted several seconds and the SM clock under load fell below its maximum,
    which is the regime of the sustained figure (a GEMM loop of seconds under
    the power cap)."""
    sm, mx = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz")
    at_max = sm is not None and mx and sm >= 0.97 * mx
    if region_s >= 3.0 and sm is not None and not at_max:
        return peaks["bf16_tflops_sustained"], (
            f"{peak_src} bf16 sustained: timed region {region_s:.2f} s, median SM clock "
            f"{sm:.0f} of {mx:.0f} MHz")
    clock = f"median SM clock {sm:.0f} of {mx:.0f} MHz" if sm is not None else "clock not sampled"
    return peaks["bf16_tflops"], (
        f"{peak_src} bf16 burst: timed region {region_s:.3f} s, {clock}")


def time_deterministic_bwd(w, q, k, v, o, lse, do, dq, dk, dv, ws, stream, peaks, iters=10):
    """fa_bwd_deterministic on the same workload (query-outer dQ kernel, no
    atomics): the reproducible alternative to the default backward."""
    from exact_io_aware_20_gb300 import binding

    def bwd():
        binding.backward(q, k, v, o, lse, do, w.causal, w.scale, dq=dq, dk=dk, dv=dv,
                         workspace=ws, stream=stream, deterministic=True)
    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        bwd()
    e1.record(stream)
    torch.cuda.synchronize()
    binding.device_status()
    ms = e0.elapsed_time(e1) / iters
    tf = w.flops_bwd() / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tflops": round(tf, 1),
            "frac_of_burst": round(tf / peaks["bf16_tflops"], 4)}


# Forward and backward timings of the other workloads of the measurement plan.
PER_CONFIG = ["tiny", "gpt_layer", "gpt_layer_causal", "long_seq", "head256"]


def fwd_bytes(w: Workload) -> int:
    """Algorithmic bytes of the forward: Q, K, V read, O and L written."""
    q = w.B * w.H * w.N * w.d * 2
    kv = w.B * w.Hkv * w.N * w.d * 2
    return 2 * q + 2 * kv + w.B * w.H * w.N * 4


def bwd_bytes(w: Workload) -> int:
    """Algorithmic bytes of the backward: Q, K, V, O, dO, L read, dQ, dK, dV written."""
    q = w.B * w.H * w.N * w.d * 2
    kv = w.B * w.Hkv * w.N * w.d * 2
    return 4 * q + 4 * kv + w.B * w.H * w.N * 4


def per_config(dev, peaks, peak_src, iters: int = 10):
    """Forward and backward of each workload timed separately with CUDA
    events on the launch stream (inputs larger than L2, except the tiny one,
    whose calls are replayed from CUDA graphs with a write of twice the L2
    size before each timed call)."""
    from exact_io_aware_20_gb300 import binding
    out = {}
    stream = torch.cuda.Stream(device=dev)     # graphs are captured off the default stream
    for name in PER_CONFIG:
        w = WORKLOADS[name]
        q, k, v, do = (t.to(dev) for t in make_inputs(w))
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.N, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d),
                         dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()    # the copies above ran on the default stream

        def fwd():
            binding.forward(q, k, v, w.causal, w.scale, out=o, lse=lse, stream=stream)

        def bwd():
            binding.backward(q, k, v, o, lse, do, w.causal, w.scale, dq=dq, dk=dk, dv=dv,
                             workspace=ws, stream=stream)

        res = {}
        if name == "tiny":
            flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
            for part, fn in (("fwd", fwd), ("bwd", bwd)):
                for _ in range(3):
                    fn()
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                times = []
                for _ in range(4 * iters):
                    with torch.cuda.stream(stream):
                        flush.fill_(1)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    with torch.cuda.stream(stream):
                        g.replay()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    times.append(e0.elapsed_time(e1))
                res[part] = statistics.median(times)
                # eager calls back to back through the Python binding (host
                # argument checks, cached tensor maps, launches): their
                # average spacing on the GPU timeline
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(200):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
                res[part + "_eager"] = e0.elapsed_time(e1) / 200
            del flush
        else:
            for part, fn in (("fwd", fwd), ("bwd", bwd)):
                for _ in range(3):
                    fn()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(iters):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
                res[part] = e0.elapsed_time(e1) / iters
        binding.device_status()
        entry = {"shape": f"B={w.B} Hq={w.H} Hkv={w.Hkv} N={w.N} d={w.d} {w.dtype} "
                          f"causal={int(w.causal)}"}
        for part, flops, nbytes in (("fwd", w.flops_fwd(), fwd_bytes(w)),
                                    ("bwd", w.flops_bwd(), bwd_bytes(w))):
            ms = res[part]
            tf = flops / (ms * 1e-3) / 1e12
            entry[part] = {"ms": round(ms, 5), "tflops": round(tf, 2),
                           "frac_of_burst": round(tf / peaks["bf16_tflops"], 4),
                           "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
            if name == "tiny":
                entry[part]["us"] = round(ms * 1e3, 2)
                entry[part]["eager_us"] = round(res[part + "_eager"] * 1e3, 2)
        out[name] = entry
        del q, k, v, do, o, lse, dq, dk, dv, ws
        torch.cuda.empty_cache()
    out["notes"] = (f"frac_of_burst against the {peak_src} bf16 burst peak "
                    f"{peaks['bf16_tflops']} TFLOP/s; gbs = algorithmic bytes (inputs read and "
                    f"outputs written once) / time; backward = preprocess + main + dQ kernels")
    return out


def exp_rate(w: Workload, fwd_ms: float, kernel_times, peak_per_s: float) -> dict:
    """Exponentials per second: one per unmasked score in the forward kernel;
    in the backward the kernels that form P (the main kernel, and at d = 128
    with the query-outer dQ kernel that one too, which forms it again),
    against the ex2 rate measured on this GPU in the same run
    (fa_measure_ex2_rate)."""
    scores = w.B * w.H * w.N * w.N / (2 if w.causal else 1)
    out = {"peak_per_s": round(peak_per_s, 1),
           "peak_source": "measured: fa_measure_ex2_rate (independent ex2.approx chains on every SM)",
           "fwd_per_s": round(scores / (fwd_ms * 1e-3), 1)}
    out["fwd_frac"] = round(out["fwd_per_s"] / peak_per_s, 4)
    for kind in ("bwd_main", "bwd_dq"):
        ms, n = kernel_times.get(kind, (0.0, 0))
        if n:
            out[kind + "_per_s"] = round(scores / (ms / n * 1e-3), 1)
            out[kind + "_frac"] = round(out[kind + "_per_s"] / peak_per_s, 4)
    return out


def dq_reduce_bytes(w: Workload) -> int:
    """Bytes the d = 128 main kernel adds into the fp32 dQ accumulator: one
    128-row x d tile per (key tile, query tile, head) step it walks (under the
    mask only the query tiles at or below each key tile's diagonal)."""
    n_t = (w.N + 127) // 128
    steps = sum(n_t - (jt if w.causal else 0) for jt in range(n_t)) * w.H * w.B
    return steps * 128 * w.d * 4


def dq_reduce(w: Workload, kernel_times, stream):
    """The resource that bounds the d = 128 backward main kernel: the SMs'
    outflow of fp32 reduce-adds (each step's 64 KB dQ tile), as bytes per
    second over the kernel's time against the rate measured on this GPU in
    the same run (fa_measure_reduce_rate, 128 MiB of targets like the
    accumulator)."""
    from exact_io_aware_20_gb300 import binding
    ms, n = kernel_times.get("bwd_main", (0.0, 0))
    if w.d != 128 or not n:
        return None
    scratch = torch.empty(128 << 20, dtype=torch.uint8, device="cuda")
    peak = binding.measure_reduce_rate(scratch, stream)
    del scratch
    by = dq_reduce_bytes(w)
    achieved = by / (ms / n * 1e-3)
    return {"kernel": "bwd_main", "bytes_per_launch": by, "achieved_tbs": round(achieved / 1e12, 3),
            "peak_tbs": round(peak / 1e12, 3), "frac": round(achieved / peak, 4),
            "peak_source": "measured: fa_measure_reduce_rate (16 KB bulk reduce-adds, one CTA per SM)"}


def step_bytes(w: Workload) -> int:
    q = w.B * w.H * w.N * w.d * 2
    kv = w.B * w.Hkv * w.N * w.d * 2
    rows = w.B * w.H * w.N
    # fwd: Q,K,V in, O,L out; bwd: Q,K,V,O,dO,L in, dQ,dK,dV out, D and dQ accumulator
    return (q + 2 * kv + q + rows * 4) + (3 * q + 2 * kv + rows * 4 + q + 2 * kv + rows * 4
                                          + 2 * rows * w.d * 4)


if __name__ == "__main__":
    sys.exit(main())
