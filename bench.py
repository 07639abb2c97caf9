#!/usr/bin/env python3
"""Benchmark of the SSD forward pass (tokens/s and roofline fraction).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one whole forward pass -- chunk_cumsum, fwd_pass_state and
compute_out -- over one batch of the workload's synthetic inputs, resident in
HBM.  Each timed step is bracketed by CUDA events on the launching stream and
preceded by an untimed 256 MiB write that flushes L2.  For N > 1 (torchrun,
one process per GPU) every rank runs an independent replica on its own batch
(the (batch, head) slices are independent; there is no exchange step), the
timed region is bracketed by a barrier and a device synchronize, and the job
time is the maximum over ranks.

Besides the headline value the JSON line carries:
  roofline      the dominant kernel's algorithmic HBM bytes per launch over its
                CUDA-event duration, against the measured copy bandwidth;
  e2e           the same metric through the public API with pinned host
                buffers, host<->device copies inside the timed region
                (ssd_fwd_host: the copies of one batch slice overlap the
                computation of another);
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the workload;
  clocks        SM clocks and throttle reasons sampled during the timed region.
``--impl reference`` times the oracle alone (rank 0 only) on the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_sequence_chunk_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "mamba2_layer_bf16"
METRIC = "SSD fwd tokens/s on 1 GB300 and % of roofline (HBM GB/s / tensor-pipe)"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(synth.WORKLOADS) + list(synth.CONTEXT_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--decode", action="store_true",
                    help="time ssd_step (one token per stream) on the decode configuration "
                         "instead of the forward pass")
    ap.add_argument("--gdn", action="store_true",
                    help="time the Gated DeltaNet chunk kernels (chunk_fwd_h + chunk_fwd_o) "
                         "instead of the forward pass")
    ap.add_argument("--profile", type=int, default=0, metavar="ITERS",
                    help="run ITERS untimed forward passes of the workload and exit (the "
                         "command the profiles/ ncu captures run)")
    ap.add_argument("--conv1d", action="store_true",
                    help="time the depthwise causal conv1d on the Mamba-2 block's xBC shape "
                         "instead of the forward pass")
    return ap.parse_args()


# Decode configuration for --decode: the Mamba-2-layer head shape with 64 streams,
# one token per stream and step (state 168 MB: larger than L2).
DECODE = dict(batch=64, nheads=80, headdim=64, dstate=128, ngroups=1, dtype="bf16")
DECODE_METRIC = "SSD decode tokens/s on 1 GB300 (ssd_step, one token per stream) and % of HBM roofline"


# --- algorithmic byte model (per launch; the method's minimum traffic) -----------

def byte_model(w: synth.Workload) -> dict:
    """Bytes each kernel must move if it reads its operands once and writes its
    results once (the three-kernel method; no per-token states, no Q x Q matrix)."""
    b, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk
    s = 2 if w.dtype == "bf16" else 4
    nc = -(-L // Q)
    Lp = nc * Q
    x = b * L * H * P * s
    bc = b * L * G * N * s
    dt = b * L * H * 4
    gcs = b * H * Lp * 4
    hid = b * H * nc * P * N * s
    st = b * H * P * N * 4
    init = st if w.init_std > 0 else 0
    D = H * 4 if w.with_D else 0
    return {
        "chunk_cumsum": dt + H * 4 + 2 * gcs,                    # dt, A -> Gcs, dtT
        "fwd_pass_state": x + bc + 2 * gcs + init + hid + st,    # x, B, Gcs, dtT, init -> hiddens, final
        "compute_out": x + 2 * bc + 2 * gcs + hid + D + x,       # x, B, C, Gcs, dtT, hiddens, D -> y
    }


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's figure (the job's time is set by its last rank); a
    no-op on one rank.  The ranks are independent replicas, so this reduction of
    the timings is the only collective in the benchmark."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own replica of the workload
    (weak scaling), so the job does world x tokens per step in the slowest rank's time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def launches_per_step(w: synth.Workload, sms: int) -> int:
    """Kernels one ssd_fwd enqueues (same rules as the library's launchers):
    three for bf16 (chunk_cumsum, fwd_pass_state, compute_out), five when
    fwd_pass_state takes its two-pass form for long chains (local pass, scan,
    apply pass) on either of its kernels; four for fp32 (chunk products and scan
    for step 2)."""
    if w.dtype != "bf16":
        return 4
    hpg = w.nheads // w.ngroups
    nc = -(-w.seqlen // w.chunk)
    paired = w.dstate <= 128 and w.headdim <= 64 and w.nheads % 2 == 0 and hpg % 2 == 0
    if paired:
        rows = w.batch * w.nheads                 # the scan's grid rows
        W = w.batch * w.nheads // 2 * nc
        G = min(W, sms, 1024 // 4)
    else:
        rows = w.batch * w.nheads * -(-w.dstate // 128) * -(-w.headdim // 64)
        W = rows * nc
        G = min(W, 2 * sms, 1024 // 2)            # two CTAs per SM
    two = nc >= 64 and G > 0 and -(-W // G) <= nc // 2 and rows <= 65535
    return 5 if two else 3


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dram_traffic_record():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by kernel,
    with the source digest they were taken at."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    rec = {}
    if os.path.exists(p):
        for line in open(p):
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#"):
                rec[(parts[0], parts[1])] = (float(parts[2]), parts[3])
    return rec


# The source files whose kernels serve each step (every dtype and shape path).
KERNEL_SOURCES = {"chunk_cumsum": ["chunk_cumsum.cu"],
                  "fwd_pass_state": ["fwd_pass_state_tc.cu", "tf32_path.cu", "simt_path.cu"],
                  "compute_out": ["compute_out_tc.cu", "tf32_path.cu", "simt_path.cu"],
                  "ssd_step": ["ssd_step.cu"], "causal_conv1d": ["causal_conv1d.cu"],
                  "gdn": ["gdn_chunk.cu", "tf32_path.cu"]}


def source_digest(kernel: str) -> str:
    """Digest of one step's kernel sources and the shared headers: a recorded
    DRAM-traffic figure is valid only while this digest is unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "state_space_sequence_chunk_gb300", "csrc")
    names = KERNEL_SOURCES[kernel] + sorted(n for n in os.listdir(csrc) if n.endswith(".cuh"))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu record, or None when there is
    none or the kernel's source has changed since it was taken."""
    rec = dram_traffic_record().get((kernel, workload))
    if rec is not None and rec[1] == source_digest(kernel):
        return rec[0]
    return None


# --- clocks ----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --- CPU oracle baseline ---------------------------------------------------------

def cpu_baseline(w: synth.Workload, inp: dict, target_s: float) -> dict:
    """The fp64 oracle, single-threaded, on whole-sequence (batch, head) slices
    of the workload; projected to the full workload's tokens/s."""
    import oracle
    lib = oracle.load()
    H, G = w.nheads, w.ngroups
    pairs = [(b, h) for b in range(w.batch) for h in range(H)]
    rng = np.random.default_rng(0)
    order = rng.permutation(len(pairs))

    def run(bh):
        b, h = bh
        g = h // (H // G)
        oracle.recurrence(
            inp["x"][b:b + 1, :, h:h + 1], inp["dt"][b:b + 1, :, h:h + 1], inp["A"][h:h + 1],
            inp["B"][b:b + 1, :, g:g + 1], inp["C"][b:b + 1, :, g:g + 1],
            None if inp["D"] is None else inp["D"][h:h + 1],
            None if inp["init_state"] is None else inp["init_state"][b:b + 1, h:h + 1], lib=lib)

    done, t_total = 0, 0.0
    while done < len(pairs) and t_total < target_s:
        t0 = time.perf_counter()
        run(pairs[order[done]])
        t_total += time.perf_counter() - t0
        done += 1
    per_slice = t_total / done
    full_s = per_slice * len(pairs)
    return {"value": w.tokens / full_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of {len(pairs)} (batch, head) slices, full {w.seqlen}-token "
                      f"sequences, fp64, single thread; {t_total:.1f} s measured, "
                      f"projected {full_s:.1f} s for the whole workload",
            "all_cores": all_cores_oracle(w, run, pairs, order, target_s / 2)}


def all_cores_oracle(w: synth.Workload, run, pairs, order, target_s: float) -> dict:
    """The same oracle on every host core: one thread per core takes whole
    (batch, head) slices from a shared counter until about target_s has passed
    (the C oracle runs without the interpreter lock, so the threads run in
    parallel); projected to the full workload's tokens/s."""
    import threading
    n = os.cpu_count() or 1
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t_end = time.perf_counter() + target_s

    def worker():
        while True:
            with lock:
                if state["next"] >= len(pairs) or time.perf_counter() > t_end:
                    return
                i = state["next"]
                state["next"] += 1
            run(pairs[order[i]])
            with lock:
                state["done"] += 1

    t0 = time.perf_counter()
    threads = [threading.Thread(target=worker) for _ in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    wall = time.perf_counter() - t0
    done = max(state["done"], 1)
    full_s = wall * len(pairs) / done
    return {"value": w.tokens / full_s, "unit": "tokens/s", "cores": n,
            "sample": f"{done} of {len(pairs)} (batch, head) slices on {n} threads in "
                      f"{wall:.1f} s, projected {full_s:.1f} s for the whole workload"}


def reference_arm(args, w: synth.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = synth.make_inputs(w)
    import oracle
    lib = oracle.load()
    H, G = w.nheads, w.ngroups
    pairs = [(b, h) for b in range(w.batch) for h in range(H)]

    def step(i):
        b, h = pairs[i % len(pairs)]
        g = h // (H // G)
        # bounded sample of the workload: one (batch, head) slice, first 512 tokens
        T = min(w.seqlen, 512)
        oracle.recurrence(
            inp["x"][b:b + 1, :T, h:h + 1], inp["dt"][b:b + 1, :T, h:h + 1], inp["A"][h:h + 1],
            inp["B"][b:b + 1, :T, g:g + 1], inp["C"][b:b + 1, :T, g:g + 1],
            None if inp["D"] is None else inp["D"][h:h + 1],
            None if inp["init_state"] is None else inp["init_state"][b:b + 1, h:h + 1], lib=lib)
        return T

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    toks = 0
    for i in range(args.steps):
        toks += step(args.warmup + i)
    el = time.perf_counter() - t0
    # one slice-token is 1/H of a workload token (a token carries H heads)
    value = toks / el / H
    T = min(w.seqlen, 512)
    sample = (f"each step: one (batch, head) slice x {T} tokens of the workload "
              f"({T / H:.2f} workload tokens), fp64 oracle, single thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            # measured: wall time of one step as run (one bounded slice sample)
            "ms_per_step": el / args.steps * 1e3,
            # projection, not measured: the same rate over one whole workload step
            "projected_ms_per_workload_step": w.tokens / value * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w: synth.Workload) -> dict:
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
            "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk,
            "io_dtype": w.dtype, "state_dtype": "f32",
            "l2": "flushed before every timed step (256 MiB write)"}


# --- GPU arm ---------------------------------------------------------------------

# conv1d configuration for --conv1d: the Mamba-2 layer's xBC channels
# (H*P + 2*G*N = 5120 + 256), batch 4, 4096 tokens, width 4, bf16 (x 176 MB).
CONV = dict(batch=4, dim=80 * 64 + 2 * 128, seqlen=4096, width=4)
CONV_METRIC = "causal conv1d tokens/s on 1 GB300 (Mamba-2 xBC channels) and % of HBM roofline"


def conv1d_main(args):
    """ssd_causal_conv1d timed like the forward pass (W untimed runs, K timed runs,
    L2 flushed before each, CUDA events)."""
    import torch
    import state_space_sequence_chunk_gb300 as ssd
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    b, d, L, W = CONV["batch"], CONV["dim"], CONV["seqlen"], CONV["width"]
    rng = np.random.default_rng(20261202 + 11)
    x_np = rng.standard_normal((b, d, L)).astype(np.float32)
    w_np = (rng.standard_normal((d, W)) / 2).astype(np.float32)
    b_np = rng.standard_normal(d).astype(np.float32)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = torch.from_numpy(x_np).to(dev).to(torch.bfloat16)
    w = torch.from_numpy(w_np).to(dev)
    bias = torch.from_numpy(b_np).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    run = lambda: ssd.causal_conv1d(x, w, bias)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for s0, s1 in evs:
        flush.fill_(1)
        s0.record(stream)
        run()
        s1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b2) for a, b2 in evs)
    x_h = x.cpu().pin_memory()
    out_h = torch.empty_like(x_h).pin_memory()
    x_d = torch.empty_like(x)

    def e2e():
        x_d.copy_(x_h, non_blocking=True)
        out_h.copy_(ssd.causal_conv1d(x_d, w, bias), non_blocking=True)

    for _ in range(3):
        e2e()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(20)]
    for s0, s1 in eev:
        flush.fill_(1)
        s0.record(stream)
        e2e()
        s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b2) for a, b2 in eev)
    clocks = sampler.stop()
    algo = 2 * b * d * L * 2 + d * W * 4 + d * 4
    peak, peak_kind = measured_peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    line = {
        "metric": CONV_METRIC, "value": b * L / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "causal_conv1d_xbc_bf16", "batch": b, "dim": d, "seqlen": L,
                   "width": W, "l2": "flushed before every step"},
        "roofline": {"bound": "hbm", "kernel": "causal_conv1d", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic("causal_conv1d", "causal_conv1d_xbc_bf16"),
                     "algorithmic_bytes": algo},
        "e2e": {"value": b * L / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.numel() * 2, "d2h_bytes_per_step": out_h.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        nrows = 0
        t_cpu = 0.0
        xb = x.float().cpu().numpy()
        while t_cpu < min(args.cpu_seconds, 5.0) and nrows < d:
            t0 = time.perf_counter()
            oracle.causal_conv1d(xb[:1, nrows:nrows + 64], w_np[nrows:nrows + 64], b_np[nrows:nrows + 64])
            t_cpu += time.perf_counter() - t0
            nrows += 64
        full = t_cpu / min(nrows, d) * d * b
        line["cpu_baseline"] = {"value": b * L / full, "unit": "tokens/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{min(nrows, d)} of {b * d} channel rows, fp64, single "
                                          f"thread; {t_cpu:.2f} s measured, projected {full:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


# Gated DeltaNet configuration for --gdn: 4 sequences of 4096 tokens, 16 heads,
# K = V = 128, chunk 64, fp32 (the gallery's kernels use C = 64 and K/V 64-128).
GDN = dict(B=4, T=4096, H=16, K=128, V=128, chunk=64)
GDN_METRIC = "Gated DeltaNet chunk_fwd_h + chunk_fwd_o tokens/s on 1 GB300 and % of roofline (HBM GB/s / tensor-pipe)"
# Nominal dense tensor rates of GB300 (TF32 1.1, bf16 2.25 PFLOP/s): the TF32 peak
# is the measured bf16 GEMM rate scaled by their ratio.
TF32_PER_BF16 = 1.1 / 2.25


def gdn_bytes(B: int, T: int, H: int, K: int, V: int, C: int) -> int:
    """Algorithmic bytes of one Gated DeltaNet step (fp32, each operand read once
    and each result written once): chunk_fwd_h reads k, w [B,T,H,K], u [B,T,H,V],
    g [B,T,H] and h0 [B,H,K,V] and writes h [B,H,NT,K,V], v_new [B,T,H,V] and the
    final state; chunk_fwd_o reads q, k, v_new, h and g and writes o [B,T,H,V]."""
    NT = -(-T // C)
    return 4 * (B * T * H * (4 * K + 4 * V + 2) + B * H * K * V * (2 + 2 * NT))


def tf32_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]) * TF32_PER_BF16, \
                "measured bf16 GEMM rate x nominal TF32/bf16 ratio (1.1/2.25)"
    return 1900.0 * TF32_PER_BF16, "fallback bf16 rate x nominal TF32/bf16 ratio"


def gdn_main(args):
    import torch
    import state_space_sequence_chunk_gb300 as ssd
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    B, T, H, K, V, C = (GDN[k] for k in ("B", "T", "H", "K", "V", "chunk"))
    rng = np.random.default_rng(20261202 + 13)
    f32 = lambda a: a.astype(np.float32)
    q = f32(rng.standard_normal((B, T, H, K)) / np.sqrt(K))
    k = f32(rng.standard_normal((B, T, H, K)) / np.sqrt(K))
    w = f32(rng.standard_normal((B, T, H, K)) / np.sqrt(K) * 0.5)
    u = f32(rng.standard_normal((B, T, H, V)))
    gamma = -np.abs(rng.normal(0.05, 0.03, (B, T, H)))
    g = np.zeros_like(gamma)
    for t in range(T):
        g[:, t] = gamma[:, t] + (g[:, t - 1] if t % C else 0.0)
    g = f32(g)
    h0 = f32(rng.standard_normal((B, H, K, V)) * 0.1)
    dev = lambda a: torch.from_numpy(a).cuda()
    tq, tk, tw, tu, tg, th0 = map(dev, (q, k, w, u, g, h0))

    def step():
        h, v_new, fin = ssd.gdn_chunk_fwd_h(tk, tw, tu, tg, th0, chunk=C)
        return ssd.gdn_chunk_fwd_o(tq, tk, v_new, h, tg, chunk=C)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for s0, s1 in evs:
        flush.fill_(1)
        s0.record(stream)
        step()
        s1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b2) for a, b2 in evs)
    host = {n: torch.from_numpy(a).pin_memory() for n, a in (("q", q), ("k", k), ("w", w), ("u", u), ("g", g))}
    dev_in = {n: torch.empty_like(t, device="cuda") for n, t in host.items()}
    o_h = torch.empty((B, T, H, V), dtype=torch.float32).pin_memory()

    def e2e():
        for n, t in host.items():
            dev_in[n].copy_(t, non_blocking=True)
        h, v_new, _ = ssd.gdn_chunk_fwd_h(dev_in["k"], dev_in["w"], dev_in["u"], dev_in["g"], th0, chunk=C)
        o_h.copy_(ssd.gdn_chunk_fwd_o(dev_in["q"], dev_in["k"], v_new, h, dev_in["g"], chunk=C),
                  non_blocking=True)

    for _ in range(2):
        e2e()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for s0, s1 in eev:
        flush.fill_(1)
        s0.record(stream)
        e2e()
        s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b2) for a, b2 in eev)
    # per-kernel breakdown (same launches, L2 flushed before each)
    h1, vn1, _ = ssd.gdn_chunk_fwd_h(tk, tw, tu, tg, th0, chunk=C)
    per = {"gdn_fwd_h": [], "gdn_fwd_o": []}
    for _ in range(5):
        for name, fn in (("gdn_fwd_h", lambda: ssd.gdn_chunk_fwd_h(tk, tw, tu, tg, th0, chunk=C)),
                         ("gdn_fwd_o", lambda: ssd.gdn_chunk_fwd_o(tq, tk, vn1, h1, tg, chunk=C))):
            flush.fill_(1)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            fn()
            a1.record(stream)
            per[name].append((a0, a1))
    torch.cuda.synchronize()
    kms = {n: statistics.mean(a.elapsed_time(b2) for a, b2 in v) for n, v in per.items()}
    clocks = sampler.stop()
    NT = -(-T // C)
    macs = B * H * NT * (2 * C * K * V + C * K * V + C * (C + 1) // 2 * (K + V))
    achieved = 2 * macs / (ms * 1e-3) / 1e12
    peak_tf, peak_kind_tf = tf32_peak()
    step_bytes = gdn_bytes(B, T, H, K, V, C)
    hbm, hbm_kind = measured_peaks()
    bw = step_bytes / (ms * 1e-3) / 1e9
    hbm_bound = step_bytes / (hbm * 1e9) >= 2 * macs / (peak_tf * 1e12)
    line = {
        "metric": GDN_METRIC, "value": B * T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "gdn_chunk_f32", "B": B, "T": T, "H": H, "K": K, "V": V, "chunk": C,
                   "l2": "flushed before every step"},
        # the binding bound is the slower of the bytes at HBM bandwidth and the
        # FLOPs at the TF32 tensor rate; the other is reported beside it
        "roofline": dict(
            ({"bound": "hbm", "kernel": "gdn_fwd_h + gdn_fwd_o", "achieved": bw, "peak": hbm,
              "peak_kind": hbm_kind, "unit": "GB/s", "frac": bw / hbm}
             if hbm_bound else
             {"bound": "tensor", "kernel": "gdn_fwd_h + gdn_fwd_o", "achieved": achieved,
              "peak": peak_tf, "peak_kind": peak_kind_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf}),
            # DRAM bytes of both launches of one step
            traffic=recorded_traffic("gdn", "gdn_chunk_f32"),
            algorithmic_bytes=step_bytes, algorithmic_flops=2 * macs,
            tensor={"achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": achieved / peak_tf, "peak_kind": peak_kind_tf}),
        "e2e": {"value": B * T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": sum(t.numel() * 4 for t in host.values()),
                "d2h_bytes_per_step": o_h.numel() * 4},
        "kernels_ms": kms,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        Ts = 256   # a bounded sample: one head of one sequence, 256 tokens
        t0 = time.perf_counter()
        hs, vns, _ = oracle.gdn_fwd_h(k[:1, :Ts, :1], w[:1, :Ts, :1], u[:1, :Ts, :1], g[:1, :Ts, :1],
                                      h0[:1, :1], chunk=C)
        oracle.gdn_fwd_o(q[:1, :Ts, :1], k[:1, :Ts, :1], vns, hs, g[:1, :Ts, :1], chunk=C)
        t_cpu = time.perf_counter() - t0
        full = t_cpu * (B * H) * (T / Ts)
        line["cpu_baseline"] = {"value": B * T / full, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"1 of {B * H} (sequence, head) pairs, {Ts} of {T} tokens, "
                                          f"fp64, single thread; {t_cpu:.2f} s, projected {full:.0f} s"}
    print(json.dumps(line), flush=True)
    return 0


def decode_main(args):
    """ssd_step timed like the forward pass: W untimed steps, K timed steps with an
    L2 flush before each, CUDA events on the launching stream.  The state stays in
    HBM between steps (as in a decode loop); x, dt, B, C of one token per stream
    are the step's inputs."""
    import torch
    import state_space_sequence_chunk_gb300 as ssd
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = synth.Workload("decode_step_bf16", DECODE["batch"], 1, DECODE["nheads"], DECODE["headdim"],
                       DECODE["dstate"], DECODE["ngroups"], 64, DECODE["dtype"], init_std=0.1,
                       seed=20261202 + 9)
    inp = synth.make_inputs(w)
    dev = torch.device("cuda", torch.cuda.current_device())
    up = lambda a, dt=None: None if a is None else (torch.from_numpy(a).to(dev) if dt is None
                                                    else torch.from_numpy(a).to(dev).to(dt))
    x, B, C = (up(inp[k], torch.bfloat16) for k in ("x", "B", "C"))
    dt, A, D = up(inp["dt"]), up(inp["A"]), up(inp["D"])
    state = up(inp["init_state"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    step = lambda: ssd.ssd_step(x, dt, A, B, C, D, state)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for s0, s1 in evs:
        flush.fill_(1)
        s0.record(stream)
        step()
        s1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # end to end: the token's inputs from pinned host memory, y back to the host
    host = {k: torch.from_numpy(inp[k]).to(torch.bfloat16 if k in ("x", "B", "C") else torch.float32)
            .pin_memory() for k in ("x", "dt", "B", "C")}
    y_h = torch.empty(tuple(x.shape), dtype=torch.bfloat16).pin_memory()
    dev_in = {k: torch.empty_like(v, device=dev) for k, v in host.items()}

    def e2e():
        for k, v in host.items():
            dev_in[k].copy_(v, non_blocking=True)
        y = ssd.ssd_step(dev_in["x"], dev_in["dt"], A, dev_in["B"], dev_in["C"], D, state)
        y_h.copy_(y, non_blocking=True)

    for _ in range(3):
        e2e()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(20)]
    for s0, s1 in eev:
        flush.fill_(1)
        s0.record(stream)
        e2e()
        s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in eev)
    clocks = sampler.stop()
    b, H, P, N, G = w.batch, w.nheads, w.headdim, w.dstate, w.ngroups
    algo = 2 * b * H * P * N * 4 + 2 * b * H * P * 2 + b * H * 4 + 2 * b * G * N * 2 + 2 * H * 4
    peak, peak_kind = measured_peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    line = {
        "metric": DECODE_METRIC, "value": b / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "streams": b, "tokens_per_step": 1, "nheads": H,
                   "headdim": P, "dstate": N, "ngroups": G, "l2": "flushed before every step"},
        "roofline": {"bound": "hbm", "kernel": "ssd_step", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic("ssd_step", w.name), "algorithmic_bytes": algo},
        "e2e": {"value": b / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": y_h.numel() * y_h.element_size()},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["init_state"], lib=oracle.load())
        t_cpu = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": b / t_cpu, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"the whole step ({b} streams x {H} heads, one token), "
                                          f"fp64, single thread; {t_cpu:.3f} s"}
    print(json.dumps(line), flush=True)
    return 0


def profile_main(args, w: synth.Workload) -> int:
    """``--profile ITERS``: ITERS untimed ssd_fwd calls on the workload, then a
    device synchronise and a check of the kernels' error bits -- a short,
    fixed launch sequence for ncu captures (no L2 flush, no timing)."""
    import torch
    import state_space_sequence_chunk_gb300 as ssd
    inp = synth.make_inputs(w)
    dev = torch.device("cuda")
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = {k: (None if v is None else torch.from_numpy(v).to(dev)) for k, v in inp.items()}
    for k in ("x", "B", "C"):
        t[k] = t[k].to(tdt)
    dims = ssd.dims_for(t["x"], t["B"], w.chunk)
    ws = torch.empty(ssd.ssd_fwd_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    y = torch.empty_like(t["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    for _ in range(args.profile):
        ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                    chunk_size=w.chunk, workspace=ws, out=y, final_out=fin)
    torch.cuda.synchronize()
    errs = ssd.ssd_take_device_errors()
    if errs:
        print(f"device error bits {errs:#x}", file=sys.stderr)
        return 1
    print(f"{w.name}: {args.profile} forward passes ok")
    return 0


def copy_roofline(h2d_bytes: int, d2h_bytes: int, dev, reps: int = 5) -> dict:
    """Pinned host<->device copy rates on this machine, and the time the step's own
    copies take alone (h2d_bytes in on one stream while d2h_bytes go out on
    another, as ssd_fwd_host overlaps them): the floor under the e2e figure."""
    import torch
    hin = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    hout = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    din = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dout = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            el = time.perf_counter() - t0
            best = el if best is None else min(best, el)
        return best

    def h2d():
        with torch.cuda.stream(s_in):
            din.copy_(hin, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            hout.copy_(dout, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": h2d_bytes / t_in / 1e9, "d2h_gbs": d2h_bytes / t_out / 1e9,
            "copies_alone_ms": t_both * 1e3,
            "how": "pinned buffers of the step's input and output bytes; both directions at "
                   f"once on two streams; best of {reps}, wall clock around a device sync"}


def main():
    args = parse()
    if args.decode:
        return decode_main(args)
    if args.conv1d:
        return conv1d_main(args)
    if args.gdn:
        return gdn_main(args)
    w = synth.workload(args.workload)
    if args.impl == "reference":
        return reference_arm(args, w)
    if args.profile:
        return profile_main(args, w)

    import ctypes
    import torch
    import torch.distributed as dist

    import state_space_sequence_chunk_gb300 as ssd

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())

    lib = ssd.load_library()
    inp = synth.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def up(a, dtype=None):
        if a is None:
            return None
        t = torch.from_numpy(a).to(dev)
        return t.to(dtype) if dtype is not None else t

    x, B, C = up(inp["x"], tdt), up(inp["B"], tdt), up(inp["C"], tdt)
    dt, A, D, init = up(inp["dt"]), up(inp["A"]), up(inp["D"]), up(inp["init_state"])
    y = torch.empty_like(x)
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    dims = ssd.dims_for(x, B, w.chunk)
    ws_bytes = ssd.ssd_fwd_workspace_bytes(dims)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        ssd.ssd_fwd(x, dt, A, B, C, D, init, chunk_size=w.chunk, workspace=ws, out=y,
                    final_out=fin)

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        fwd()
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)

    # headline: K whole steps, each timed with events, L2 flushed in between
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sync_all()
    for s0, s1 in evs:
        flush.fill_(1)
        s0.record(stream)
        fwd()
        s1.record(stream)
    sync_all()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, w.tokens, ms_per_step)

    # per-kernel breakdown through the three step entry points (same launches)
    gb, hb = ssd.ssd_intermediate_bytes(dims)
    gcs = ws[:gb].view(torch.float32)
    off = (gb + 255) // 256 * 256
    dtT = ws[off:off + gb].view(torch.float32)
    hid = ws[2 * off:2 * off + hb]
    scr = ws[2 * off + (hb + 255) // 256 * 256:]   # fwd_pass_state scratch (the rest)
    P = ctypes.c_void_p
    ptr = lambda t: None if t is None else P(t.data_ptr())
    st = P(stream.cuda_stream)
    kern = {"chunk_cumsum": lambda: lib.ssd_chunk_cumsum(ctypes.byref(dims), ptr(dt), ptr(A),
                                                         ptr(gcs), ptr(dtT), st),
            "fwd_pass_state": lambda: lib.ssd_fwd_pass_state(ctypes.byref(dims), ptr(x), ptr(B),
                                                             ptr(gcs), ptr(dtT), ptr(init),
                                                             ptr(hid), ptr(fin), ptr(scr),
                                                             ctypes.c_size_t(scr.numel()), st),
            "compute_out": lambda: lib.ssd_compute_out(ctypes.byref(dims), ptr(x), ptr(B),
                                                       ptr(C), ptr(gcs), ptr(dtT), ptr(hid),
                                                       ptr(D), ptr(y), st)}
    per = {k: [] for k in kern}
    nrep = max(10, min(args.steps, 50))
    for _ in range(nrep):
        for k, f in kern.items():
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = f()
            e1.record(stream)
            if rc != 0:
                raise RuntimeError(f"{k} returned {rc}")
            per[k].append((e0, e1))
    torch.cuda.synchronize()
    kms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in per.items()}

    # e2e through the public API with pinned host buffers
    host = {k: (None if v is None else torch.from_numpy(v).to(tdt if k in ("x", "B", "C") else
                                                          torch.float32).pin_memory())
            for k, v in inp.items()}
    y_h = torch.empty(y.shape, dtype=tdt).pin_memory()
    f_h = torch.empty(fin.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = y_h.numel() * y_h.element_size() + f_h.numel() * f_h.element_size()
    # ssd_fwd_host: batch slices whose copies overlap the other slices' compute
    nslices = max(1, min(w.batch, 4))
    staging = torch.empty(max(ssd.ssd_fwd_host_staging_bytes(
        ssd.dims_for(host["x"], host["B"], w.chunk), nslices), 256), dtype=torch.uint8, device=dev)

    def e2e_step():
        ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["B"], host["C"], host["D"],
                         host["init_state"], chunk_size=w.chunk, nslices=nslices,
                         staging=staging, out=y_h, final_out=f_h)

    for _ in range(3):
        e2e_step()
    e2e_n = max(5, min(args.steps, 20))
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(e2e_n)]
    sync_all()
    for s0, s1 in eev:
        flush.fill_(1)
        s0.record(stream)
        e2e_step()
        s1.record(stream)
    sync_all()
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in eev), world, dev)
    clocks = sampler.stop()
    copies = copy_roofline(h2d, d2h, dev)
    copies["frac"] = copies["copies_alone_ms"] / e2e_ms

    if rank == 0:
        model = byte_model(w)
        dom = max(kms, key=kms.get)
        peak, peak_kind = measured_peaks()
        achieved = model[dom] / (kms[dom] * 1e-3) / 1e9
        traffic = recorded_traffic(dom, w.name)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_of(w),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "algorithmic_bytes": model[dom]},
            "kernels_ms": kms,
            "method_roofline_frac": sum(model.values()) / (ms_per_step * 1e-3) / 1e9 / peak,
            "e2e": {"value": job_throughput(world, w.tokens, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": f"ssd_fwd_host, {nslices} batch slices",
                    # the copies alone over the e2e step time: how close e2e is to
                    # the host link's own limit
                    "copy_roofline": copies},
            "gpu_launches": launches_per_step(w, torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
