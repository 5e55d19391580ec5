#!/usr/bin/env python
"""Benchmark: exact attention forward + backward on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch: fa_fwd (forward
kernel) then fa_bwd (D preprocess, block-sparse column lists, dK/dV/dQ
kernel, dQ convert), by default on the block-sparse long-sequence workload
B=1 H=8 N=65536 d=64 with a 512x512 mask of 128x128 blocks (a diagonal band
of width 3 plus uniformly random blocks, 5% nonzero), bf16 storage, fp32
accumulation: the largest of the five configurations and one inside the
N >= 4K, d = 64 regime.  Inputs are synthetic (seeded normals, see
workloads.py); --workload selects the others.

Timing: W warm-up steps, then exactly K steps, each bracketed by CUDA events
on the launching stream; L2 is flushed (a 256 MiB buffer is rewritten)
between steps, outside the events.  A barrier and a device synchronise
bracket the timed loop; the per-rank time is the sum of the step events and
the job time is the maximum over ranks.  value = counted FLOPs of all ranks
/ job time.  FLOPs: 4*N*L*d per (b, h) forward (L = key bound, x0.5 causal,
x nonzero-block fraction), 2.5x that backward.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs an independent replica (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "sparse64k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20
# forward, D preprocess, dK/dV/dQ, dQ convert; plus the column-list kernel
# when a block mask is given
KERNELS_PER_STEP = 4


# ---------------------------------------------------------------- helpers


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "fa_bwd_main_kernel": ("fa_bwd.cu", "fa_sm103.cuh", "fa_kernels.cuh"),
    "fa_fwd_kernel": ("fa_fwd.cu", "fa_fwd_common.cuh", "fa_sm103.cuh", "fa_kernels.cuh"),
    "fa_bwd_d128_kernel": ("fa_bwd_d128.cu", "fa_sm103.cuh", "fa_kernels.cuh"),
    "fa_fwd_d128_kernel": ("fa_fwd_d128.cu", "fa_fwd_common.cuh", "fa_sm103.cuh",
                           "fa_kernels.cuh"),
}


def _code_text(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to one
    space: what the compiler sees, so that editing a comment does not mark a
    capture stale.  String and character literals are kept as written."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _sources_hash(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "exact_io_aware_25_gb300", "csrc", n)) as f:
            h.update(_code_text(f.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when no
    capture matches this kernel and workload or the kernel's sources changed
    since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get(f"{kernel}:{workload}")
    except (OSError, ValueError):
        return None
    if not entry or kernel not in KERNEL_SOURCES:
        return None
    if entry.get("sources") != _sources_hash(KERNEL_SOURCES[kernel]):
        return None
    return entry.get("bytes")


def step_stats(ms):
    """Per-step spread of CUDA-event times (ms): mean, min, median, p90, max."""
    xs = sorted(ms)
    n = len(xs)
    pick = lambda f: xs[min(n - 1, max(0, int(math.ceil(f * n)) - 1))]
    return {"mean": statistics.mean(xs), "min": xs[0], "p50": statistics.median(xs),
            "p90": pick(0.9), "max": xs[-1], "n": n}


def counted_flops(spec, kv_len, block_mask=None):
    """Forward FLOPs 4*N*L*d per (b, h) with L the key bound of batch b
    (N*N for no padding, halved under causal, times the nonzero-block
    fraction under a block mask), backward 2.5x forward."""
    N, d, H = spec.N, spec.d, spec.H
    lens = [min(int(x), N) for x in kv_len] if kv_len is not None else [N] * spec.B
    fwd = sum(4.0 * N * L * d * H for L in lens)
    nominal = 4.0 * N * N * d * H * spec.B
    if spec.causal:
        fwd *= 0.5
        nominal *= 0.5
    if block_mask is not None:
        frac = float((block_mask != 0).sum()) / block_mask.size
        fwd *= frac
        nominal *= frac
    return {"fwd": fwd, "bwd": 2.5 * fwd, "step": 3.5 * fwd, "nominal_step": 3.5 * nominal}


class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (ctypes) while the
    timed region runs; falls back to `nvidia-smi -lms` if NVML is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._h = None
        self._proc = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            idx = cuda_index
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [p for p in vis.split(",") if p.strip()]
            if parts and all(p.strip().isdigit() for p in parts) and cuda_index < len(parts):
                idx = int(parts[cuda_index])
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
        except OSError:
            self._nvml = None
        self._index = cuda_index

    def _poll_nvml(self):
        nv, h = self._nvml, self._h
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if get_r(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self._thread.start()
        else:
            import subprocess
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown")
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self._index), f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            names = ["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6 or not f[0].isdigit():
                    continue
                self.samples.append(int(f[0]))
                self.max_mhz = int(f[1]) if f[1].isdigit() else self.max_mhz
                for name, val in zip(names, f[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# ---------------------------------------------------------------- distributed


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank scalar (timing only; no data-path exchange)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- oracle timing


def time_oracle(w, budget_s: float, max_units=None, dropout=0.0, seed=0):
    """Times the fp64 oracle (forward + backward) on whole (b, h) heads of the
    workload until budget_s has elapsed; returns (flops counted, seconds,
    heads, threads)."""
    import numpy as np
    import oracle
    import workloads as W
    spec = w.spec
    threads = os.cpu_count() or 1
    p8 = oracle.drop_p8(dropout) if dropout > 0 else 0
    q, k, v, do = (w.f64(n) for n in ("q", "k", "v", "do"))
    done_flops, elapsed, heads = 0.0, 0.0, 0
    order = [(b, h) for b in range(spec.B) for h in range(spec.H)]
    for (b, h) in order:
        if elapsed >= budget_s or (max_units is not None and heads >= max_units):
            break
        sl = (slice(b, b + 1), slice(h, h + 1))
        kv = None if w.kv_len is None else w.kv_len[b:b + 1]
        qs, ks, vs, ds = (x[sl] for x in (q, k, v, do))
        t0 = time.perf_counter()
        # (the single head keeps its own index 0 for the keep mask: timing only)
        oracle.forward(qs, ks, vs, spec.scale, causal=spec.causal, kv_len=kv,
                       block_mask=w.block_mask, nthreads=threads, p8=p8, seed=seed)
        oracle.backward(qs, ks, vs, ds, spec.scale, causal=spec.causal, kv_len=kv,
                        block_mask=w.block_mask, nthreads=threads, p8=p8, seed=seed)
        elapsed += time.perf_counter() - t0
        one = W.Spec(**{**spec.__dict__, "B": 1, "H": 1})
        done_flops += counted_flops(one, kv, w.block_mask)["step"]
        heads += 1
    del np
    return done_flops, elapsed, heads, threads


# ---------------------------------------------------------------- arms


def allowed_keys(spec, kv_len, block_mask, b, i):
    """Number of keys query row i of batch b attends to (for FLOP counting)."""
    N = spec.N
    L = N if kv_len is None else max(0, min(int(kv_len[b]), N))
    lim = min(L, i + 1) if spec.causal else L
    if block_mask is None:
        return lim
    row = block_mask[i // 128]
    full_tiles = lim // 128
    n = 128 * int(np.count_nonzero(row[:full_tiles]))
    if lim % 128 and row[full_tiles]:
        n += lim % 128
    return n


def time_oracle_rows(w, rows, dropout=0.0, seed=0):
    """Times the oracle's forward and the dQ side of its backward on the given
    global query rows (bh * N + i); returns (flops counted, seconds, threads).
    Counted per row: 4*L*d forward plus 6*L*d backward (S, dP and dQ, the
    part of the 10*L*d backward convention that belongs to the row's dQ);
    the key-side dK / dV work is not part of this sample."""
    import oracle
    spec = w.spec
    threads = os.cpu_count() or 1
    p8 = oracle.drop_p8(dropout) if dropout > 0 else 0
    q, k, v, do = (w.f64(n) for n in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    oracle.forward(q, k, v, spec.scale, causal=spec.causal, kv_len=w.kv_len,
                   block_mask=w.block_mask, rows=rows, nthreads=threads, p8=p8, seed=seed)
    oracle.backward(q, k, v, do, spec.scale, causal=spec.causal, kv_len=w.kv_len,
                    block_mask=w.block_mask, q_rows=rows, k_rows=np.zeros(0, np.int64),
                    nthreads=threads, p8=p8, seed=seed)
    t = time.perf_counter() - t0
    flops = 0.0
    for g in rows:
        bh, i = divmod(int(g), spec.N)
        flops += 10.0 * allowed_keys(spec, w.kv_len, w.block_mask, bh // spec.H, i) * spec.d
    return flops, t, threads


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only).  Each
    step is a bounded sample of the workload: whole (b, h) heads (forward +
    backward) when one head fits the per-step budget, else seeded query rows
    spread over the heads (forward + the dQ side of the backward)."""
    if rank != 0:
        return 0
    import workloads as W
    w = W.make(args.workload) if args.head_dim == 64 else W.make(args.workload, d=args.head_dim)
    spec = w.spec
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    rng = np.random.default_rng(4242)
    total_rows = spec.B * spec.H * spec.N
    # per-row cost from a small probe, to decide between whole heads and rows
    probe = np.sort(rng.choice(total_rows, size=min(total_rows, 64), replace=False))
    f_p, t_p, threads = time_oracle_rows(w, probe, dropout=args.dropout, seed=args.seed)
    head_est = t_p / len(probe) * spec.N * 1.4
    if head_est <= per_step_budget:
        # one whole head, timed (max_units bounds it; the budget must not stop it first)
        f1, t1, _, threads = time_oracle(w, float("inf"), max_units=1, dropout=args.dropout,
                                         seed=args.seed)
        heads_per_step = max(1, min(spec.B * spec.H, int(per_step_budget / max(t1, 1e-6))))
        run = lambda: time_oracle(w, float("inf"), max_units=heads_per_step,
                                  dropout=args.dropout, seed=args.seed)[:2]
        sample = (f"{heads_per_step} of {spec.B * spec.H} (b, h) heads per step "
                  f"(forward + backward, full rows)")
    else:
        # blocks of 64 consecutive query rows (half a tile: rows that share
        # their allowed key tiles), drawn uniformly over all heads
        blk = 64
        n_blocks = total_rows // blk
        per_blk = max(t_p / len(probe), 1e-9) * blk
        nb = max(1, min(n_blocks, int(per_step_budget / per_blk)))
        steps_rows = [(np.sort(rng.choice(n_blocks, size=nb, replace=False))[:, None] * blk
                       + np.arange(blk)[None, :]).ravel() for _ in range(args.steps)]
        it = iter(steps_rows)
        run = lambda: time_oracle_rows(w, next(it), dropout=args.dropout, seed=args.seed)[:2]
        sample = (f"{nb * blk} of {total_rows} query rows per step ({nb} blocks of {blk} "
                  f"consecutive rows drawn uniformly over the (b, h) heads, seed 4242): forward "
                  f"+ the dQ side of the backward, counted at 10*L*d per row (one whole head, "
                  f"forward + backward, takes about {head_est:.0f} s here)")
    for _ in range(args.warmup):
        time_oracle_rows(w, probe, dropout=args.dropout, seed=args.seed)
    tot_f, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t = run()
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC if spec.d == 64 else METRIC.replace("(bf16,", f"(bf16, d={spec.d},"),
        "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.dropout, args.seed),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


WORKLOAD_NAMES = {
    "tiny": "tiny exact-attention check, fwd+bwd",
    "bert": "BERT-large-shaped encoder attention, fwd+bwd",
    "gpt2": "GPT-2-small-shaped causal decoder attention, fwd+bwd",
    "gpt2_4k": "long-context GPT-2-shaped causal attention with peaky keys, fwd+bwd",
    "sparse64k": "block-sparse long-sequence attention (s=0.05), fwd+bwd",
}


def workload_config(w, dropout=0.0, seed=0):
    s = w.spec
    cfg = {"workload": WORKLOAD_NAMES.get(s.name, s.name),
           "B": s.B, "H": s.H, "N": s.N, "d": s.d, "causal": s.causal, "scale": s.scale,
           "kv_len": None, "block_mask": None,
           "flops": "algorithmic: 4*N*L*d per head fwd (L = key bound; x0.5 causal; x nonzero "
                    "block fraction), x3.5 fwd+bwd",
           "l2": "flushed between timed steps (256 MiB write outside the events)",
           "parallelism": "replicas"}
    if w.kv_len is not None:
        cfg["kv_len"] = "uniform [256, 512] per sequence (seed 2), keys past it masked"
    if w.block_mask is not None:
        cfg["block_mask"] = (f"{w.block_mask.shape[0]}x{w.block_mask.shape[1]} of 128x128 blocks, "
                             f"{int(w.block_mask.sum())} nonzero")
    if dropout > 0:
        cfg["dropout"] = {"p": dropout, "seed": seed,
                          "mask": "counter-based hash per 2x2 block, regenerated in both passes"}
    return cfg


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import exact_io_aware_25_gb300 as fa
    import workloads as W

    fa.lib()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = W.make(args.workload) if args.head_dim == 64 else W.make(args.workload, d=args.head_dim)
    s = w.spec
    B, H, N, d = s.B, s.H, s.N, s.d
    fl = counted_flops(s, w.kv_len, w.block_mask)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)

    q, k, v, do = dev(w.q), dev(w.k), dev(w.v), dev(w.do)
    kv_len = torch.from_numpy(w.kv_len).to(device) if w.kv_len is not None else None
    mask = (torch.from_numpy(w.block_mask).to(device) if w.block_mask is not None else None)
    o = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    stream = torch.cuda.current_stream(device)
    # Auxiliary memory, measured: everything allocated beyond the inputs
    # (Q, K, V, dO, masks) and the outputs O, dQ, dK, dV from here until one
    # forward + backward has finished -- the lse the forward leaves for the
    # backward and the backward's workspace -- as the allocator's peak, and
    # the device's free memory before and after (the library itself
    # allocates nothing).
    torch.cuda.synchronize(device)
    base_alloc = torch.cuda.memory_allocated(device)
    torch.cuda.reset_peak_memory_stats(device)
    free0 = torch.cuda.mem_get_info(device)[0]
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)

    p_drop, seed = args.dropout, args.seed

    def fwd_call():
        if p_drop > 0:
            fa.fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, s.scale, s.causal, kv_len, mask,
                              p_drop, seed, stream)
        else:
            fa.fa_fwd(q, k, v, o, lse, B, H, N, d, s.scale, s.causal, kv_len, mask, stream)

    def bwd_call():
        if p_drop > 0:
            fa.fa_bwd_dropout(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, s.scale, s.causal,
                              kv_len, mask, p_drop, seed, ws, ws_bytes, stream)
        else:
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, s.scale, s.causal, kv_len,
                      mask, ws, ws_bytes, stream)

    def step():
        fwd_call()
        bwd_call()

    step()
    torch.cuda.synchronize(device)
    fa.fa_check(stream)
    aux_peak = torch.cuda.max_memory_allocated(device) - base_alloc
    aux_free_delta = free0 - torch.cuda.mem_get_info(device)[0]
    materialised = 2 * B * H * N * N * 2
    aux = {"measured_peak_bytes": int(aux_peak),
           "lse_bytes": int(lse.numel() * 4), "workspace_bytes": int(ws_bytes),
           "device_free_delta_bytes": int(aux_free_delta),
           "materialised_s_p_bf16_bytes": int(materialised),
           "ratio_materialised_over_measured": materialised / max(1, aux_peak),
           "how": "torch allocator peak above the inputs and outputs over one fa_fwd + fa_bwd "
                  "(lse + backward workspace); device free-memory delta over the same span "
                  "(allocator rounding included); baseline = S and P in bf16 for every (b, h)"}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    fa.fa_check(stream)

    K = args.steps
    ev_step0, ev_step1, ev_k0, ev_k1, ev_fwd1, bm0, bm1 = (
        [torch.cuda.Event(enable_timing=True) for _ in range(K)] for _ in range(7))
    for e in bm0 + bm1:  # torch creates the CUDA event on first record
        e.record(stream)
    sampler = ClockSampler(local)
    barrier(world, device)
    torch.cuda.synchronize(device)
    # no collector pause while the host enqueues the timed steps (a pause longer
    # than the queue the host has built up would show as GPU idle time)
    gc.collect()
    gc.disable()
    sampler.start()
    wall0 = time.perf_counter()
    # the timed steps: events only at each step's two ends (an event between two
    # kernels would end the overlap of the second one's launch with the first)
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev_step0[i].record(stream)
        fwd_call()
        bwd_call()
        ev_step1[i].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    # the kernel-timing pass, inside the same clock sampling: K more steps with
    # events at the forward's end and around the backward's main kernel
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev_k0[i].record(stream)
        fwd_call()
        ev_fwd1[i].record(stream)
        fa.fa_set_bwd_main_events(bm0[i], bm1[i])
        bwd_call()
        ev_k1[i].record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    gc.enable()
    fa.fa_set_bwd_main_events(None, None)
    barrier(world, device)
    fa.fa_check(stream)

    step_ms = [ev_step0[i].elapsed_time(ev_step1[i]) for i in range(K)]
    inst_ms = [ev_k0[i].elapsed_time(ev_k1[i]) for i in range(K)]
    fwd_ms = [ev_k0[i].elapsed_time(ev_fwd1[i]) for i in range(K)]
    bwd_main_ms = [bm0[i].elapsed_time(bm1[i]) for i in range(K)]
    spread = {"step": step_stats(step_ms), "fwd": step_stats(fwd_ms),
              "bwd_main": step_stats(bwd_main_ms), "step_with_kernel_events": step_stats(inst_ms)}
    t_rank = sum(step_ms) / 1e3
    t_job = max_over_ranks(t_rank, world, device)
    value = fl["step"] * K * world / t_job / 1e12

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    fwd_avg = statistics.mean(fwd_ms) / 1e3
    bwd_avg = statistics.mean(bwd_main_ms) / 1e3
    bwd_dominant = bwd_avg >= fwd_avg
    if d == 64:
        dominant = "fa_bwd_main_kernel" if bwd_dominant else "fa_fwd_kernel"
    else:
        dominant = "fa_bwd_d128_kernel" if bwd_dominant else "fa_fwd_d128_kernel"
    dom_flops = fl["bwd"] if bwd_dominant else fl["fwd"]
    dom_t = bwd_avg if bwd_dominant else fwd_avg
    achieved = dom_flops / dom_t / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": load_traffic(dominant, args.workload) if p_drop == 0 else None,
                "kernel": dominant, "peak_source": f"bf16_tflops (burst) of {peak_src}",
                "algorithmic_flops_per_launch": dom_flops,
                "avg_launch_ms": dom_t * 1e3}

    # ---- end to end through the public API: pinned host in, host out
    e2e_steps = max(3, min(args.e2e_steps, K))
    hq, hk, hv, hdo = (torch.from_numpy(x.view(np.int16)).pin_memory() for x in (w.q, w.k, w.v, w.do))
    hkv = torch.from_numpy(w.kv_len).pin_memory() if w.kv_len is not None else None
    hmask = torch.from_numpy(w.block_mask).pin_memory() if w.block_mask is not None else None
    ho, hdq, hdk, hdv = (torch.empty(q.shape, dtype=torch.int16).pin_memory() for _ in range(4))
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    dq_i, dk_i, dv_i, do_i = (t.view(torch.int16) for t in (dq, dk, dv, do))
    qi, ki, vi, oi = (t.view(torch.int16) for t in (q, k, v, o))
    arena_bytes = fa.fa_host_arena_size(B, H, N, d)
    arena = torch.empty(arena_bytes, dtype=torch.uint8, device=device) if p_drop == 0 else None

    def e2e_host_api():
        # one call: the library copies each head group in, runs it and copies
        # its results out, overlapping the three across groups
        fa.fa_fwd_bwd_host(hq, hk, hv, hdo, ho, hlse, hdq, hdk, hdv, B, H, N, d, s.scale,
                           s.causal, hkv, hmask, 0, arena, arena_bytes, stream)

    def e2e_serial():
        # the device entry points between plain copies on one stream
        qi.copy_(hq, non_blocking=True)
        ki.copy_(hk, non_blocking=True)
        vi.copy_(hv, non_blocking=True)
        do_i.copy_(hdo, non_blocking=True)
        if hkv is not None:
            kv_len.copy_(hkv, non_blocking=True)
        step()
        ho.copy_(oi, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
        hdq.copy_(dq_i, non_blocking=True)
        hdk.copy_(dk_i, non_blocking=True)
        hdv.copy_(dv_i, non_blocking=True)

    def time_e2e(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(device)
        gc.collect()
        gc.disable()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        barrier(world, device)
        for i in range(e2e_steps):
            flush.fill_(i & 0xFF)
            e0[i].record(stream)
            fn()
            e1[i].record(stream)
        torch.cuda.synchronize(device)
        gc.enable()
        fa.fa_check(stream)
        return max_over_ranks(sum(e0[i].elapsed_time(e1[i]) for i in range(e2e_steps)) / 1e3,
                              world, device)

    t_bytes = q.numel() * 2
    h2d = 4 * t_bytes + (hkv.numel() * 4 if hkv is not None else 0)
    d2h = 4 * t_bytes + hlse.numel() * 4
    t_serial = time_e2e(e2e_serial)
    serial = {"value": fl["step"] * e2e_steps * world / t_serial / 1e12,
              "ms_per_step": 1e3 * t_serial / e2e_steps,
              "api": "fa_fwd / fa_bwd on device buffers between plain copies on one stream"}
    if p_drop == 0:
        e2e_t = time_e2e(e2e_host_api)
        h2d += hmask.numel() if hmask is not None else 0   # the host call copies the mask too
        e2e = {"value": fl["step"] * e2e_steps * world / e2e_t / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": 1e3 * e2e_t / e2e_steps,
               "api": "fa_fwd_bwd_host: pinned host buffers, copies of each head group "
                      "overlapped with the kernels of the previous one",
               "serial_copies": serial}
    else:
        # the host-buffer entry points have no dropout
        e2e = {"value": serial["value"], "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": serial["ms_per_step"], "api": serial["api"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t, heads, threads = time_oracle(w, args.cpu_budget, dropout=p_drop, seed=seed)
        est = t * fl["step"] / f   # the same rate over the whole workload
        cpu = {"value": f / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{heads} of {B * H} (b, h) heads, forward + backward, full rows; "
                         f"{t:.1f} s of fp64 C oracle work",
               "seconds": t,
               "extrapolated_full_workload_s": est,
               "extrapolation": f"the sampled heads' time scaled by counted FLOPs to all "
                                f"{B * H} heads (labelled estimate, not measured)"}

    if rank == 0:
        line = {
            "metric": METRIC if d == 64 else METRIC.replace("(bf16,", f"(bf16, d={d},"),
            "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_job / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, p_drop, seed),
            "pct_of_peak": value / peak,
            "fwd": {"tflops": fl["fwd"] / fwd_avg / 1e12, "ms": fwd_avg * 1e3},
            "bwd_main": {"tflops": fl["bwd"] / bwd_avg / 1e12, "ms": bwd_avg * 1e3},
            "nominal_tflops": fl["nominal_step"] * K * world / t_job / 1e12,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (KERNELS_PER_STEP + (w.block_mask is not None)) * K,
            "clocks": sampler.summary(),
            "step_ms_stats": spread,
            "timing": "value: the K timed steps, CUDA events only at each step's two ends; "
                      "fwd, bwd_main and roofline: a second pass of K steps inside the same "
                      "clock sampling with events at the forward's end and around the "
                      "backward's main kernel (an event between two kernels ends the overlap "
                      "of the second one's launch with the first)",
            "wall_s_timed_region": wall,
            "aux_memory": aux,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- forward only (any head dim)

def run_fwd_only(args, rank, world, local):
    """Times fa_fwd alone (--fwd-only) on a workload, at its head dimension
    or the one --head-dim gives.  Same timing rules as the fwd+bwd line; the
    metric is forward TFLOP/s."""
    import numpy as np
    import torch

    import exact_io_aware_25_gb300 as fa
    import workloads as W

    fa.lib()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = W.make(args.workload, d=args.head_dim)
    s = w.spec
    B, H, N, d = s.B, s.H, s.N, s.d
    fl = counted_flops(s, w.kv_len, w.block_mask)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)

    q, k, v = dev(w.q), dev(w.k), dev(w.v)
    kv_len = torch.from_numpy(w.kv_len).to(device) if w.kv_len is not None else None
    mask = (torch.from_numpy(w.block_mask).to(device) if w.block_mask is not None else None)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        fa.fa_fwd(q, k, v, o, lse, B, H, N, d, s.scale, s.causal, kv_len, mask, stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    fa.fa_check(stream)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(local)
    barrier(world, device)
    torch.cuda.synchronize(device)
    # no collector pause while the host enqueues the timed steps (a pause longer
    # than the queue the host has built up would show as GPU idle time)
    gc.collect()
    gc.disable()
    sampler.start()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    gc.enable()
    barrier(world, device)
    fa.fa_check(stream)
    t_job = max_over_ranks(sum(ev0[i].elapsed_time(ev1[i]) for i in range(K)) / 1e3, world,
                           device)
    value = fl["fwd"] * K * world / t_job / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    kernel = "fa_fwd_d128_kernel" if d == 128 else "fa_fwd_kernel"
    roofline = {"bound": "tensor", "achieved": value / world, "peak": peak, "unit": UNIT,
                "frac": value / world / peak, "traffic": None, "kernel": kernel,
                "peak_source": f"bf16_tflops (burst) of {peak_src}",
                "algorithmic_flops_per_launch": fl["fwd"], "avg_launch_ms": 1e3 * t_job / K}

    e2e_steps = max(3, min(args.e2e_steps, K))
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).pin_memory() for x in (w.q, w.k, w.v))
    hkv = torch.from_numpy(w.kv_len).pin_memory() if w.kv_len is not None else None
    hmask = torch.from_numpy(w.block_mask).pin_memory() if w.block_mask is not None else None
    ho = torch.empty(q.shape, dtype=torch.int16).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    arena_bytes = fa.fa_host_arena_size(B, H, N, d)
    arena = torch.empty(arena_bytes, dtype=torch.uint8, device=device)

    def e2e_step():
        fa.fa_fwd_host(hq, hk, hv, ho, hlse, B, H, N, d, s.scale, s.causal, hkv, hmask, 0, arena,
                       arena_bytes, stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(device)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.fill_(i & 0xFF)
        e0[i].record(stream)
        e2e_step()
        e1[i].record(stream)
    torch.cuda.synchronize(device)
    fa.fa_check(stream)
    e2e_t = max_over_ranks(sum(e0[i].elapsed_time(e1[i]) for i in range(e2e_steps)) / 1e3,
                           world, device)
    t_bytes = q.numel() * 2
    h2d = 3 * t_bytes + (hkv.numel() * 4 if hkv is not None else 0) + (
        hmask.numel() if hmask is not None else 0)
    e2e = {"value": fl["fwd"] * e2e_steps * world / e2e_t / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": t_bytes + hlse.numel() * 4,
           "steps": e2e_steps, "ms_per_step": 1e3 * e2e_t / e2e_steps,
           "api": "fa_fwd_host: pinned host buffers, copies of each head group overlapped "
                  "with the kernels of the previous one"}
    if rank == 0:
        cfg = workload_config(w)
        cfg["workload"] = cfg["workload"].replace("fwd+bwd", f"forward only, d={d}")
        line = {
            "metric": f"attention fwd TFLOP/s (bf16, d={d}, 1\u00d7GB300) and % of dense BF16 peak",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_job / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "pct_of_peak": value / world / peak, "roofline": roofline, "cpu_baseline": None,
            "e2e": e2e, "gpu_launches": K, "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- split-KV decode

DECODE = {"B": 16, "H": 16, "Nq": 1, "Nk": 32768, "d": 64, "scale": 0.125, "seed": 6}


def decode_inputs():
    """Decode-shaped inputs: one query per (b, h) against a 32K-key cache;
    Q, K, V iid N(0, 1) in fp32 (numpy PCG64, draw order Q, K, V), rounded
    to bf16 (RNE)."""
    import numpy as np
    import workloads as W
    c = DECODE
    rng = np.random.default_rng(c["seed"])
    q = W.f32_to_bf16_bits(rng.standard_normal((c["B"], c["H"], c["Nq"], c["d"]), dtype=np.float32))
    k = W.f32_to_bf16_bits(rng.standard_normal((c["B"], c["H"], c["Nk"], c["d"]), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((c["B"], c["H"], c["Nk"], c["d"]), dtype=np.float32))
    return q, k, v


def run_decode(args, rank, world, local):
    """Split-KV forward on the decode workload: TFLOP/s of 4*Nq*Nk*d per head
    and the K/V read bandwidth against the measured HBM copy peak."""
    import numpy as np
    import torch

    import exact_io_aware_25_gb300 as fa
    import workloads as W

    fa.lib()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    c = DECODE
    B, H, Nq, Nk, d, scale = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["scale"]
    hq, hk, hv = decode_inputs()

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)

    q, k, v = dev(hq), dev(hk), dev(hv)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
    nbytes = fa.fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        fa.fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, None, 0, ws, nbytes, stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        step()
    fa.fa_check(stream)
    K = args.steps
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(local)
    barrier(world, device)
    torch.cuda.synchronize(device)
    # no collector pause while the host enqueues the timed steps (a pause longer
    # than the queue the host has built up would show as GPU idle time)
    gc.collect()
    gc.disable()
    sampler.start()
    for i in range(K):
        flush.fill_(i & 0xFF)
        e0[i].record(stream)
        step()
        e1[i].record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    gc.enable()
    fa.fa_check(stream)
    t_rank = sum(e0[i].elapsed_time(e1[i]) for i in range(K)) / 1e3
    t_job = max_over_ranks(t_rank, world, device)
    flops = 4.0 * Nq * Nk * d * B * H
    kv_bytes = 2.0 * B * H * Nk * d * 2
    value = flops * K * world / t_job / 1e12
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = kv_bytes * K / t_rank / 1e9

    # end to end: pinned host Q, K, V in, O and lse out, every step
    e2e_steps = max(3, min(args.e2e_steps, 5))
    pq, pk, pv = (torch.from_numpy(x.view(np.int16)).pin_memory() for x in (hq, hk, hv))
    po = torch.empty(q.shape, dtype=torch.int16).pin_memory()
    pl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    qi, ki, vi, oi = (t.view(torch.int16) for t in (q, k, v, o))
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        a0[i].record(stream)
        qi.copy_(pq, non_blocking=True)
        ki.copy_(pk, non_blocking=True)
        vi.copy_(pv, non_blocking=True)
        step()
        po.copy_(oi, non_blocking=True)
        pl.copy_(lse, non_blocking=True)
        a1[i].record(stream)
    torch.cuda.synchronize(device)
    e2e_t = max_over_ranks(sum(a0[i].elapsed_time(a1[i]) for i in range(e2e_steps)) / 1e3,
                           world, device)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = os.cpu_count() or 1
        heads, t_cpu = 0, 0.0
        for b in range(B):
            for h in range(H):
                if t_cpu >= args.cpu_budget:
                    break
                t0 = time.perf_counter()
                oracle.forward_qk(W.bf16_bits_to_f64(hq[b:b + 1, h:h + 1]),
                                  W.bf16_bits_to_f64(hk[b:b + 1, h:h + 1]),
                                  W.bf16_bits_to_f64(hv[b:b + 1, h:h + 1]), scale,
                                  nthreads=threads)
                t_cpu += time.perf_counter() - t0
                heads += 1
        cpu = {"value": 4.0 * Nq * Nk * d * heads / t_cpu / 1e12, "unit": UNIT, "cores": threads,
               "kind": "oracle", "sample": f"{heads} of {B * H} (b, h) heads, forward",
               "seconds": t_cpu}

    if rank == 0:
        line = {
            "metric": "split-KV decode forward TFLOP/s (bf16, 1\u00d7GB300)",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_job / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode: one query per head against a 32K-key cache",
                       "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "scale": scale,
                       "splits": "auto (about two CTAs per SM)",
                       "l2": "flushed between timed steps; K and V (2.1 GB) exceed L2 anyway",
                       "parallelism": "replicas"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "traffic": None,
                         "kernel": "fa_fwd_kernel (split mode) + fa_fwd_merge_kernel",
                         "peak_source": f"hbm_gbs of {peak_src}",
                         "algorithmic_bytes_per_launch": kv_bytes},
            "cpu_baseline": cpu,
            "e2e": {"value": flops * e2e_steps * world / e2e_t / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": (pq.numel() + pk.numel() + pv.numel()) * 2,
                    "d2h_bytes_per_step": po.numel() * 2 + pl.numel() * 4,
                    "steps": e2e_steps, "ms_per_step": 1e3 * e2e_t / e2e_steps},
            "gpu_launches": 2 * K,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name from workloads.py (the reported line uses sparse64k), or "
                         "'decode' for the split-KV forward on a decode-shaped problem")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="drop probability of the fused dropout (0 = plain attention)")
    ap.add_argument("--seed", type=int, default=1234, help="dropout seed")
    ap.add_argument("--head-dim", type=int, default=64, choices=[64, 128],
                    help="head dimension of the workload (the reported line uses 64)")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward alone")
    args = ap.parse_args(argv)
    rank, world, local = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        if args.workload == "decode":
            return run_decode(args, rank, world, local)
        if args.fwd_only:
            return run_fwd_only(args, rank, world, local)
        return run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
