#!/usr/bin/env python3
"""Benchmark of the gated delta-rule hot path on GB300.

One JSON line on stdout (rank 0).  The headline workload is the KDA
long-context chunked prefill (B=1, H=32, T=131072, dk=dv=128, C=64, bf16
q/k/v, float32 state, per-channel decay): ``value`` is tokens/s (B*T tokens,
all heads) with inputs already resident in HBM.  ``roofline`` holds the
dominant kernel against the bytes it must move itself, the whole call
against the path's algorithmic bytes (``roofline.call``), every kernel of
the call (``roofline.kernels``: time, own bytes, fraction of the measured
HBM peak, and, where an ncu capture of the current source is committed
under profiles/, its DRAM traffic and tensor-pipe utilisation) and the
call's DRAM traffic over its algorithmic bytes.  The same run measures:
``configs``, the DeltaNet (4 x 8 x 2048, d = 64) and Gated DeltaNet
(8 x 16 x 8192, d = 128) prefill workloads with the same rooflines;
``decode``, the KDA decode step (256 sequences x 32 heads, d=128, float32
state updated in place, 1000 steps over a cycled pool of 16 token sets),
state GB/s; ``e2e``, the headline prefill through kda_chunk_fwd_host from
page-locked host memory (median of >= 10 steps) with the measured host-link
rate; ``variants`` and ``attn_res``; ``cpu_baseline``, the float64 oracle on
the host cores (and on one core).

Timing: W warm-up calls, then K timed calls bracketed by a barrier and
``torch.cuda.synchronize()`` on both sides, CUDA events on the launching
stream, max over ranks.  The headline's inputs (6.4 GB per prefill call) and
the decode state (0.54 GB) are larger than the 129 MB L2, so no flush is
needed between their calls; the DeltaNet workload (34 MB) is timed call by
call with an L2 flush in between.  ``--sections`` limits the run to some
sections (profiler captures).

``--impl reference`` times the float64 CPU oracle instead (the reference arm:
this method has no reference implementation, so the oracle, as it stands, is
the comparison program), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

SECTIONS = ("variants", "e2e", "configs", "decode", "attn_res")
METRIC = "KDA chunked prefill tokens/s (H=32,d=128); decode-step state GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------- workload accounting

def prefill_algorithmic_bytes(w):
    """Bytes a prefill call must move at least: q, k, v and o once each in
    their storage type, beta and log_alpha once, h0 / hT once each."""
    es = 2 if w.dtype == "bf16" else 4
    per_token_head = es * (2 * w.dk + w.dv) + 4 + es * w.dv
    per_token_head += {"none": 0, "scalar": 4, "channel": 4 * w.dk}[w.alpha]
    state = 4 * w.dk * w.dv * (2 if w.h0_sd > 0 else 1)
    return w.B * w.H * (w.T * per_token_head + state)


def prefill_kernel_bytes(w, kernels):
    """The share of the path's algorithmic bytes each kernel of a prefill call
    must move itself: the tensor path's prep reads the inputs (q, k, v, beta,
    log_alpha), its scan writes o and hT and reads h0; a single kernel (the
    CUDA-core path) moves all of them.  The per-chunk records the prep hands
    to the scan are not algorithmic bytes: they are the design's own traffic."""
    es = 2 if w.dtype == "bf16" else 4
    la = {"none": 0, "scalar": 4, "channel": 4 * w.dk}[w.alpha]
    th = w.B * w.H * w.T
    inputs = th * (es * (2 * w.dk + w.dv) + 4 + la)
    outputs = th * es * w.dv + w.B * w.H * 4 * w.dk * w.dv * (2 if w.h0_sd > 0 else 1)
    if len(kernels) == 1:
        return {kernels[0]: inputs + outputs}
    return {k: (inputs if "prep" in k else outputs) for k in kernels}


def prefill_algorithmic_flops(w):
    """Triangle-exploited flop count per call: 6 d^2 + 5 C d + C^2/3 per
    token-head (state products W S, Q S, K^T u at 2 dk dv each; A, W, U, M,
    M u at about C d each with the triangles skipped; the C x C solve)."""
    d = w.dk
    return w.B * w.H * w.T * (6 * d * d + 5 * w.C * d + w.C * w.C / 3.0)


def decode_algorithmic_bytes(w):
    es = 2 if w.dtype == "bf16" else 4
    la = {"none": 0, "scalar": 4, "channel": 4 * w.dk}[w.alpha]
    per_state = 2 * 4 * w.dk * w.dv + es * (2 * w.dk + w.dv) + la + 4 + es * w.dv
    return w.N * w.H * per_state


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_delta_rule_wise_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_profile(kernel, src_hash, workload="kda_prefill_bf16"):
    """The committed ncu figures of `kernel` on `workload` (DRAM bytes per
    launch, tensor-pipe utilisation), if they were taken on the current
    kernel source; else {}."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel if workload == "kda_prefill_bf16" else f"{kernel}@{workload}")
    if not e or e.get("source_hash") != src_hash:
        return {}
    return e


def recorded_traffic(kernel, src_hash, workload="kda_prefill_bf16"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    return recorded_profile(kernel, src_hash, workload).get("bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            # raw samples: KDA_CLOCKS_DIR if set, else the system temp directory
            # (the JSON line carries their summary)
            out_dir = os.environ.get("KDA_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"kda_clocks_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 0.25 * max(x["power"] for x in rows)] or rows
        reasons = sorted({name for r in rows for name, key in
                          (("hw_slowdown", "hw"), ("hw_thermal_slowdown", "hwt"),
                           ("sw_thermal_slowdown", "swt"), ("sw_power_cap", "swp"))
                          if r[key].lower() == "active"})
        return {"sm_mhz": float(np.median([r["sm"] for r in busy])),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------- distributed

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    import torch
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local, dist


def barrier(dist, torch_mod=None):
    if torch_mod is not None and torch_mod.cuda.is_available():
        torch_mod.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    if torch_mod is not None and torch_mod.cuda.is_available():
        torch_mod.cuda.synchronize()


def max_over_ranks(x, dist, device=None):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing

def oracle_prefill_rate(w, heads, T_sample, threads):
    """Tokens/s of the float64 oracle on ``heads`` x the first T_sample tokens
    of workload ``w``, one thread per head; scaled to whole tokens (all H
    heads per token)."""
    import oracle
    oracle.build()
    x = W.prefill_inputs(w.with_(T=T_sample), heads=heads)
    la = x["log_alpha"]
    t0 = time.perf_counter()
    oracle.recurrent_heads(x["q"][:, None], x["k"][:, None], x["v"][:, None], x["beta"][:, None],
                           None if la is None else la[:, None],
                           None if x["h0"] is None else x["h0"][:, None], threads=threads)
    dt = time.perf_counter() - t0
    token_heads = len(heads) * T_sample
    return token_heads / dt / w.H, dt, token_heads


# Arm CPU part numbers (implementer 0x41) of the cores these boxes use.
_ARM_PARTS = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
              "0xd8e": "Arm Neoverse-N3", "0xd84": "Arm Neoverse-V3"}


def cpu_info():
    """The host CPU's model name: lscpu's, else /proc/cpuinfo's model name,
    else the Arm part number translated."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    part = None
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":", 1)[0].strip().lower()
            if key == "model name":
                return line.split(":", 1)[1].strip()
            if key == "cpu part" and part is None:
                part = line.split(":", 1)[1].strip()
    except OSError:
        pass
    if part:
        return _ARM_PARTS.get(part.lower(), f"Arm CPU part {part}")
    return platform.processor() or platform.machine()


def cpu_baseline(w, threads, tokens_all, tokens_one):
    """The oracle on the host cores: `threads` heads x `tokens_all` tokens, one
    thread per head, and one head x `tokens_one` tokens on a single thread."""
    heads = [(0, h) for h in range(threads)]
    rate, dt, n = oracle_prefill_rate(w, heads, tokens_all, threads)
    rate1, dt1, n1 = oracle_prefill_rate(w, [(0, 0)], tokens_one, 1)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{threads} of {w.H} heads x first {tokens_all} tokens ({n} token-heads) "
                      f"in {dt:.1f}s, float64, one thread per head; tokens/s = "
                      f"token-heads/s / H",
            "one_core": {"value": rate1, "unit": "tokens/s",
                         "token_heads_per_s": rate1 * w.H,
                         "sample": f"1 head x first {tokens_one} tokens ({n1} token-heads) in "
                                   f"{dt1:.1f}s on one thread"},
            "cpu": cpu_info(), "host_cpus": os.cpu_count()}


def run_reference(args, rank, world, dist):
    """The reference arm: the float64 oracle on host cores, rank 0 only."""
    if rank != 0:
        return 0
    w = W.KDA_PREFILL_BF16
    threads = max(1, min(os.cpu_count() or 1, w.H))
    heads = [(0, h) for h in range(threads)]
    T_s = args.ref_tokens
    rates, times = [], []
    for i in range(args.warmup + args.steps):
        r, dt, n = oracle_prefill_rate(w, heads, T_s, threads)
        if i >= args.warmup:
            rates.append(r)
            times.append(dt)
    value = float(np.median(rates))
    sample = (f"{threads} of {w.H} heads x first {T_s} of {w.T} tokens per step "
              f"({threads * T_s} token-heads), float64, one thread per head; tokens/s = "
              f"token-heads/s / H")
    rate1, dt1, n1 = oracle_prefill_rate(w, [(0, 0)], max(1024, T_s // 4), 1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * float(np.median(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk=dv={w.dk} C={w.C} "
                                   f"bf16 inputs, per-channel decay (oracle on a sample)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample, "cpu": cpu_info(),
                             "host_cpus": os.cpu_count(),
                             "one_core": {"value": rate1, "unit": "tokens/s",
                                          "sample": f"1 head x {n1} tokens on one thread"}},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def fill_prefill_host(w, torch):
    """Pinned host tensors holding the workload in its storage types."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    B, H, T = w.B, w.H, w.T
    h = dict(q=torch.empty((B, H, T, w.dk), dtype=dt, pin_memory=True),
             k=torch.empty((B, H, T, w.dk), dtype=dt, pin_memory=True),
             v=torch.empty((B, H, T, w.dv), dtype=dt, pin_memory=True),
             beta=torch.empty((B, H, T), dtype=torch.float32, pin_memory=True))
    if w.alpha == "channel":
        h["log_alpha"] = torch.empty((B, H, T, w.dk), dtype=torch.float32, pin_memory=True)
    elif w.alpha == "scalar":
        h["log_alpha"] = torch.empty((B, H, T), dtype=torch.float32, pin_memory=True)
    else:
        h["log_alpha"] = None
    h["h0"] = (torch.empty((B, H, w.dk, w.dv), dtype=torch.float32, pin_memory=True)
               if w.h0_sd > 0 else None)

    def sink(b, hh, d):
        for key, t in h.items():
            if t is not None:
                t[b, hh].copy_(torch.from_numpy(d[key]).to(t.dtype))

    W.prefill_inputs(w, sink=sink)
    return h


def prefill_roofline(kda, w, per_kernel, ms_call, peaks, peak_src):
    """Roofline of a prefill call: the dominant kernel against the bytes it
    must move itself (the object's top level), the whole call against the
    path's algorithmic bytes, every kernel on its own bytes with its ncu DRAM
    traffic and tensor-pipe utilisation where a capture of the current
    source is committed, and the call's DRAM traffic over its algorithmic
    bytes."""
    alg = prefill_algorithmic_bytes(w)
    own = prefill_kernel_bytes(w, list(per_kernel))
    kernels = {}
    traffic_total = 0
    for kname, kms in per_kernel.items():
        prof = recorded_profile(kname, kernel_source_hash(kda.kernel_sources(kname)), w.name)
        ach = own[kname] / (kms * 1e-3) / 1e9
        kernels[kname] = {"ms": kms, "own_bytes": own[kname], "achieved": ach,
                          "frac": ach / peaks["hbm_gbs"],
                          "traffic": prof.get("bytes_per_launch"),
                          "tensor_pipe_pct": prof.get("tensor_pipe_pct")}
        traffic_total = (None if traffic_total is None or prof.get("bytes_per_launch") is None
                         else traffic_total + prof["bytes_per_launch"])
    kname = max(per_kernel, key=per_kernel.get)
    k = kernels[kname]
    call_ach = alg / (ms_call * 1e-3) / 1e9
    return {"kernel": kname, "bound": "hbm", "unit": "GB/s", "achieved": k["achieved"],
            "peak": peaks["hbm_gbs"], "frac": k["frac"], "traffic": k["traffic"],
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "algorithmic_bytes_per_launch": own[kname],
            "achieved_is": f"{kname}'s own algorithmic bytes / its mean launch time",
            "call": {"achieved": call_ach, "frac": call_ach / peaks["hbm_gbs"],
                     "ms": ms_call, "algorithmic_bytes": alg,
                     "dram_traffic": traffic_total,
                     "traffic_over_algorithmic": (traffic_total / alg if traffic_total else None)},
            "kernels": kernels}


def time_prefill_config(kda, torch, w, dev, stream, steps, warmup, peaks, peak_src):
    """tokens/s and rooflines of one synthetic prefill workload (inputs in HBM).
    Each call is timed on its own with CUDA events around each kernel; a
    workload whose bytes do not exceed twice the L2 gets an L2 flush (a
    512 MB write) between calls, outside the timed events."""
    host = fill_prefill_host(w, torch)
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    del host
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=dt, device=dev)
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    ws = kda.workspace_for(d["q"], d["v"], w.C, d["log_alpha"])
    meta = (w.B, w.H, w.T, w.dk, w.dv, w.C, kda.KDA_BF16 if w.dtype == "bf16" else kda.KDA_F32,
            {"none": kda.KDA_ALPHA_NONE, "scalar": kda.KDA_ALPHA_SCALAR,
             "channel": kda.KDA_ALPHA_CHANNEL}[w.alpha])
    n_launch = kda.kda_chunk_fwd_launches(*meta)
    knames = kda.kda_chunk_fwd_kernel_names(*meta)
    alg = prefill_algorithmic_bytes(w)
    flush = alg < 2 * 126 * 2 ** 20
    scratch = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if flush else None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)]
          for _ in range(steps)]
    for row in ev:           # create the CUDA events (torch creates them on first record)
        for e in row:
            e.record(stream)

    def call(events=None):
        kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], o, hT,
                             w.C, ws, stream, kda.KDA_PATH_AUTO, events)

    for _ in range(warmup):
        call()
    for i in range(steps):
        if flush:
            scratch.fill_(i & 255)
        call(ev[i])
    kda.kda_chunk_fwd_status(ws, stream)
    ms = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps)]
    per_kernel = {n: float(np.median([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]))
                  for j, n in enumerate(knames)}
    ms_call = float(np.median(ms))
    tokens = w.B * w.T
    out = {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk=dv={w.dk} C={w.C} {w.dtype} "
                       f"q/k/v, fp32 state, decay {w.alpha}, h0 {'N(0,%g)' % w.h0_sd if w.h0_sd else '0'}",
           "value": tokens / (ms_call * 1e-3), "unit": "tokens/s", "ms_per_call": ms_call,
           "ms_per_call_all": [round(x, 4) for x in ms], "steps": steps,
           "l2": ("flushed between calls (512 MB write)" if flush
                  else f"inputs larger than L2 ({alg / 1e9:.2f} GB per call); no flush"),
           "kernels": knames,
           "roofline": prefill_roofline(kda, w, per_kernel, ms_call, peaks, peak_src)}
    del d, o, hT, ws, scratch
    torch.cuda.empty_cache()
    return out


def host_link_gbs(torch, dev, stream, nbytes=1 << 30, reps=3):
    """Host -> device copy rate from page-locked memory (one cudaMemcpyAsync of
    `nbytes`, best of `reps`), the ceiling of the end-to-end number."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = float("inf")
    with torch.cuda.stream(stream):
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
    del src, dst
    return nbytes / (best * 1e-3) / 1e9


def run_e2e(kda, torch, w, host, o, hT, dev, stream, args, dist, world, tokens):
    """The prefill end to end through kda_chunk_fwd_host: inputs copied in from
    page-locked host memory and outputs copied back inside the timed region."""
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    o_host = torch.empty_like(o, device="cpu").pin_memory()
    hT_host = torch.empty_like(hT, device="cpu").pin_memory()
    d2h = o_host.numel() * o_host.element_size() + hT_host.numel() * hT_host.element_size()

    # kda_chunk_fwd_host: segments of the sequence (every head, a sixteenth
    # of T each), each segment's copy-in, prefill and copy-out overlapped with its
    # neighbours', the state carried from segment to segment
    hbuf = kda.host_buffer_for(host["q"], host["v"], w.C, host["log_alpha"], device=dev)

    def e2e_step():
        kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["beta"], host["log_alpha"],
                               host["h0"], o_host, hT_host, w.C, hbuf, 0, stream)

    for _ in range(min(2, args.warmup)):
        e2e_step()
    e2e_steps = max(10, args.steps)
    barrier(dist, torch)
    # an event after every step as well: the host link is shared with other
    # tenants of the machine, and the per-step times show a slow stretch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    evs[0].record(stream)
    for i in range(e2e_steps):
        e2e_step()
        evs[i + 1].record(stream)
    barrier(dist, torch)
    e2e_step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(e2e_steps)]
    # median step: the host link is shared with the machine's other tenants,
    # and a single slow step would move a mean
    e2e_ms = max_over_ranks(float(np.median(e2e_step_ms)), dist, dev)
    link = host_link_gbs(torch, dev, stream)
    e2e = {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "ms_per_step_is": f"median of {e2e_steps} steps",
           "ms_per_step_mean": float(np.mean(e2e_step_ms)),
           "step_ms": [round(x, 3) for x in e2e_step_ms],
           "h2d_gbs": link, "h2d_floor_ms": h2d / (link * 1e9) * 1e3,
           "h2d_gbs_is": "one 1 GiB cudaMemcpyAsync from page-locked memory, best of 3",
           "api": "kda_chunk_fwd_host from pinned host memory, 16 segments of T (all heads), "
                  "copy-in / prefill / copy-out of neighbouring segments overlapped",
           "steps": e2e_steps}
    del o_host, hT_host, hbuf
    return e2e


def run_attn_res(kda, torch, dev, stream, args, dist, world, peaks, peak_src):
    """AttnRes depth mixing: 9 stacked blocks (8 AttnRes blocks and the
    partial one) of 4096 tokens x 7168, bf16; HBM-bound."""
    ar_nb, ar_rows, ar_D = 9, 4096, 7168
    g = torch.Generator(device=dev).manual_seed(5)
    Var = torch.randn((ar_nb, ar_rows, ar_D), device=dev, generator=g).to(torch.bfloat16)
    war = torch.randn(ar_D, device=dev, generator=g) / ar_D ** 0.5
    har = torch.empty((ar_rows, ar_D), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        kda.kda_attn_res(Var, war, har, 1e-6, stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ar_steps = max(args.steps, 10)
    barrier(dist, torch)
    a.record(stream)
    for _ in range(ar_steps):
        kda.kda_attn_res(Var, war, har, 1e-6, stream)
    b.record(stream)
    barrier(dist, torch)
    ar_ms = max_over_ranks(a.elapsed_time(b) / ar_steps, dist, dev)
    ar_bytes = (ar_nb + 1) * ar_rows * ar_D * 2 + ar_D * 4
    attn_res = {"workload": f"n_blocks={ar_nb} rows={ar_rows} D={ar_D} bf16 (synthetic; the pages "
                            f"give the block count, not the model width)",
                "value": world * ar_bytes / (ar_ms * 1e-3) / 1e9, "unit": "GB/s",
                "us_per_call": ar_ms * 1e3, "steps": ar_steps,
                "roofline": {"kernel": "attn_res_kernel", "bound": "hbm", "unit": "GB/s",
                             "achieved": ar_bytes / (ar_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                             "frac": ar_bytes / (ar_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                             "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                             "traffic": recorded_traffic(
                                 "attn_res_kernel",
                                 kernel_source_hash(kda.kernel_sources("attn_res_kernel"))),
                             "algorithmic_bytes_per_launch": ar_bytes}}
    del Var, war, har
    return attn_res


def run_ours(args, rank, world, local, dist):
    import torch

    import gated_delta_rule_wise_gb300 as kda

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library()
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    sections = set(SECTIONS if args.sections == "all" else args.sections.split(","))
    w = W.KDA_PREFILL_BF16
    if args.seq_len:  # shorter sequences for profiler captures; not the headline
        w = w.with_(T=args.seq_len)
    wd = W.KDA_DECODE_BF16

    # ---- inputs
    t0 = time.perf_counter()
    host = fill_prefill_host(w, torch)
    log(f"[bench] generated {w.name} inputs in {time.perf_counter() - t0:.1f}s")
    d = {k: (None if v is None else v.to(dev, non_blocking=False)) for k, v in host.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=torch.bfloat16, device=dev)
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    ws = kda.workspace_for(d["q"], d["v"], w.C, d["log_alpha"])
    meta = (w.B, w.H, w.T, w.dk, w.dv, w.C, kda.KDA_BF16, kda.KDA_ALPHA_CHANNEL)
    launches_per_call = kda.kda_chunk_fwd_launches(*meta)
    knames = kda.kda_chunk_fwd_kernel_names(*meta)

    def prefill(events=None):
        kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], o, hT,
                             w.C, ws, stream, kda.KDA_PATH_AUTO, events)

    # per-step events: one before each kernel launch of the call, one after the last
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(launches_per_call + 1)]
          for _ in range(args.steps)]
    for row in ev:           # create the CUDA events (torch creates them on first record)
        for e in row:
            e.record(stream)
    for _ in range(args.warmup):
        prefill()
    kda.kda_chunk_fwd_status(ws, stream)

    with ClockSampler(local) as clk:
        barrier(dist, torch)
        for i in range(args.steps):
            prefill(ev[i])
        barrier(dist, torch)
    kda.kda_chunk_fwd_status(ws, stream)
    step_ms = [ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps)]
    per_kernel = {n: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1])
                                    for i in range(args.steps)]))
                  for j, n in enumerate(knames)}
    ms_step = max_over_ranks(float(np.mean(step_ms)), dist, dev)
    tokens = w.B * w.T
    value = world * tokens / (ms_step * 1e-3)
    clocks = clk.summary()

    # ---- rooflines: the whole call, and each kernel on the bytes it must move
    # itself, all timed inside the timed region
    alg_bytes = prefill_algorithmic_bytes(w)
    alg_flops = prefill_algorithmic_flops(w)
    roof = prefill_roofline(kda, w, per_kernel, ms_step, peaks, peak_src)
    roof["algorithmic_flops_per_launch"] = alg_flops
    roof["tensor_tflops_per_call"] = alg_flops / (ms_step * 1e-3) / 1e12

    # ---- the other update rule and the fused input maps, same workload
    def time_variant(rule, maps):
        beta_arg = None if rule != kda.KDA_RULE_DELTA else d["beta"]
        state = rule != kda.KDA_RULE_LINEAR_NORM   # the normalised rule keeps (S, z) internal

        def call():
            kda.kda_chunk_fwd_rule(d["q"], d["k"], d["v"], beta_arg, d["log_alpha"],
                                   d["h0"] if state else None, o, hT if state else None, w.C, ws,
                                   rule, maps, stream)

        for _ in range(args.warmup):
            call()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist, torch)
        a.record(stream)
        for _ in range(args.steps):
            call()
        b.record(stream)
        barrier(dist, torch)
        kda.kda_chunk_fwd_status(ws, stream)
        ms = max_over_ranks(a.elapsed_time(b) / args.steps, dist, dev)
        return {"value": world * tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
                "steps": args.steps}

    def time_path(path):  # the headline call through another path of kda_chunk_fwd_ex
        def call():
            kda.kda_chunk_fwd_ex(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["h0"], o, hT,
                                 w.C, ws, stream, path)

        for _ in range(args.warmup):
            call()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist, torch)
        a.record(stream)
        for _ in range(args.steps):
            call()
        b.record(stream)
        barrier(dist, torch)
        kda.kda_chunk_fwd_status(ws, stream)
        ms = max_over_ranks(a.elapsed_time(b) / args.steps, dist, dev)
        return {"value": world * tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
                "steps": args.steps}

    variants = {} if "variants" not in sections else {
        "linear_attention": dict(
            time_variant(kda.KDA_RULE_LINEAR, 0),
            rule="S = Diag(a) S + k v^T, o = S^T q (kda_chunk_fwd_rule, KDA_RULE_LINEAR)"),
        "fused_input_maps": dict(
            time_variant(kda.KDA_RULE_DELTA, kda.KDA_MAP_QK_SILU_NORM | kda.KDA_MAP_BETA_SIGMOID),
            maps="q, k <- normalize(silu(.)), beta <- sigmoid(.) inside the prep kernel"),
        "normalised_linear_attention": dict(
            time_variant(kda.KDA_RULE_LINEAR_NORM, kda.KDA_MAP_QK_ELU1),
            rule="q, k <- elu(.) + 1; S = Diag(a) S + k v^T, z = a z + k, o = S^T q / q.z "
                 "(kda_chunk_fwd_rule, KDA_RULE_LINEAR_NORM, KDA_MAP_QK_ELU1)"),
        "pipelined_call": dict(
            time_path(kda.KDA_PATH_TENSOR_PIPELINED),
            path="the headline call in 16 sequence segments, each segment's prep beside the "
                 "previous segment's one-CTA-per-head scan (KDA_PATH_TENSOR_PIPELINED); "
                 "the headline value uses the two-launch call"),
    }

    # ---- end to end through the public API with host buffers
    e2e = None
    if "e2e" in sections:
        e2e = run_e2e(kda, torch, w, host, o, hT, dev, stream, args, dist, world, tokens)
    del d, host, o, hT, ws
    torch.cuda.empty_cache()

    # ---- the other synthetic prefill workloads, each with its own roofline
    configs = {}
    if "configs" in sections and (not args.seq_len or args.sections != "all"):
        for wc in (W.DELTANET_BF16, W.GDN_BF16):
            t0 = time.perf_counter()
            configs[wc.name] = time_prefill_config(kda, torch, wc, dev, stream,
                                                   args.steps, args.warmup, peaks, peak_src)
            log(f"[bench] {wc.name}: {configs[wc.name]['ms_per_call']:.3f} ms per call "
                f"({time.perf_counter() - t0:.1f}s with input generation)")

    # ---- decode
    dec = None
    if args.decode_steps > 0 and "decode" in sections:
        S = torch.from_numpy(W.decode_state(wd)).to(dev)
        pool = []
        for i in range(wd.pool):
            tk = W.decode_tokens(wd, i)
            pool.append({k: (None if v is None else torch.from_numpy(v).to(dev).to(
                torch.bfloat16 if k in ("q", "k", "v") else torch.float32))
                for k, v in tk.items()})
        od = torch.empty((wd.N, wd.H, wd.dv), dtype=torch.bfloat16, device=dev)

        def dstep(i):
            p = pool[i % wd.pool]
            kda.kda_decode_step(p["q"], p["k"], p["v"], p["beta"], p["log_alpha"], S, od, stream)

        for i in range(max(3, args.warmup)):
            dstep(i)
        with ClockSampler(local) as dclk:
            barrier(dist, torch)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(args.decode_steps):
                dstep(i)
            b.record(stream)
            barrier(dist, torch)
        dms = max_over_ranks(a.elapsed_time(b) / args.decode_steps, dist, dev)
        dbytes = decode_algorithmic_bytes(wd)
        dsrc = kernel_source_hash(kda.kernel_sources("decode_step_kernel"))
        dec = {"workload": f"{wd.name}: N={wd.N} H={wd.H} dk=dv={wd.dk} fp32 state "
                           f"({4 * wd.N * wd.H * wd.dk * wd.dv / 1e6:.0f} MB) in place, bf16 q/k/v, "
                           f"per-channel decay, {args.decode_steps} steps over {wd.pool} token sets",
               "value": world * dbytes / (dms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": dms, "tokens_per_s": world * wd.N / (dms * 1e-3),
               "gpu_launches": args.decode_steps,
               "roofline": {"kernel": "decode_step_kernel", "bound": "hbm", "unit": "GB/s",
                            "achieved": dbytes / (dms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                            "frac": dbytes / (dms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                            "traffic": recorded_traffic("decode_step_kernel", dsrc),
                            "algorithmic_bytes_per_launch": dbytes},
               "clocks": dclk.summary()}
        del S, pool, od
        torch.cuda.empty_cache()

    attn_res = run_attn_res(kda, torch, dev, stream, args, dist, world, peaks, peak_src) \
        if "attn_res" in sections else None

    # ---- CPU baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = max(1, min(os.cpu_count() or 1, w.H))
        cpu = cpu_baseline(w, threads, args.cpu_tokens, args.cpu_tokens // 4)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk=dv={w.dk} "
                                       f"C={w.C}, bf16 q/k/v, fp32 state, per-channel decay "
                                       f"log_alpha~N({w.la_mu},{w.la_sd}), h0=0, seed {w.seed}",
                           "per_gpu_tokens": tokens,
                           "l2": f"inputs larger than L2 ({alg_bytes / 1e9:.1f} GB per call); "
                                 f"no flush",
                           "parallelism": f"replicas x{world}"},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "configs": configs,
                "gpu_launches": launches_per_call * args.steps,
                "clocks": clocks, "decode": dec, "variants": variants, "attn_res": attn_res}
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--cpu-tokens", type=int, default=131072,
                    help="tokens per head in the CPU-baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=16384,
                    help="tokens per head in each reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sections", default="all",
                    help="comma list of the sections to run besides the headline prefill "
                         f"(of {','.join(SECTIONS)}; default all): profiler captures of one "
                         "section")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="prefill T other than the workload's 131072 (profiler captures "
                         "of a smaller case; the line then names that T and is not the "
                         "headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local, dist = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world, dist)
        return run_ours(args, rank, world, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
