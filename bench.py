#!/usr/bin/env python
"""Benchmark: decode attention over an asymmetrically quantized KV cache on GB300.

One step = one pass of the whole hot path on one batch:
  kvq_quantize_append (one new token per sequence; windows that fill are
  quantized into the pages) then kvq_decode_attention (split-K kernel +
  combine) for one query per (sequence, query head).

Default workload (--config 5): 64 sequences with ragged contexts drawn
log-uniform in [1024, 65536) tokens (seeded), 32 query / 8 KV heads, head_dim
128, 16-token pages in a random physical order, INT8 symmetric per-channel keys
(64-token groups) stored pre-RoPE (theta 500000, rotated after dequantization),
INT4 asymmetric per-token values, a 64-token bf16 residual window.
--config 3 (Llama-3.1-8B-shaped, 2-bit KIVI-style, 32K) and --config 4
(Llama-3.1-70B-shaped, FP8 E4M3, or E5M2 with --fp8 e5m2, 128K) time the
decode call alone.  --config 1 (one fp32 head of 4096 tokens, INT8 keys per
channel or, with --k-axis tensor, per tensor) and --config 2 (one fp32 kv-head
of 512 tokens read by 64 query heads, INT4 asymmetric keys per channel or, with
--k-axis token, per token) are latency-bound: their inputs fit in L2, so L2 is
flushed (a 256 MiB write) before every decode call, outside its events, and
the time is the sum of the calls' own event times.  Defaults: 20 warm-up and 200 timed steps; every decode call
is also bracketed by events, and roofline.us_per_launch (mean) and
us_per_launch_median come from those.

value = algorithmic bytes per step (packed codes + scale/min metadata + window
+ q + out, plus the append's reads and writes) / device time per step, in
GB/s; the inputs of configs 3-5 (>0.5 GB) are larger than L2, so no flush is
needed between their steps.
--impl reference times the CPU oracle (float64 numpy) on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
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

import kvq_inputs as W  # noqa: E402

METRIC = "quantized-KV decode attention: KV bytes GB/s (% of HBM peak), µs/step"
INT2, INT4, INT8, FP8, FP8_E5M2 = 2, 4, 8, 9, 10
FP8_MAX = {FP8: 448.0, FP8_E5M2: 57344.0}  # calibration qmax of each FP8 format
LATENCY_CONFIGS = (1, 2)  # inputs that fit in L2: flushed before every call
REF_MAX_TOKENS = 8192  # the reference arm's streams: prefixes of at most this many tokens
FLUSH_BYTES = 256 << 20
FP8_FORMATS = {"e4m3": FP8, "e5m2": FP8_E5M2}
SYM, ASYM = 0, 1
TEN, TOK, CH = 0, 1, 2
F32, BF16 = 0, 1

# kernels this library launches per call (append: fold + window/lengths;
# attention: split-K + combine)
LAUNCHES_APPEND = 2
LAUNCHES_ATTENTION = 2

# DRAM bytes (read + write) of one full-size split-kernel launch, from one ncu
# capture of a smaller case of the same kernel scaled by algorithmic bytes
# (profiles/split_rope_i8i4_paged_ragged_b16.md, split_fp8_70b_layer_b2.md,
# split_int2_8b_layer_b8.md); to be re-captured whenever that kernel changes.
SPLIT_TRAFFIC = {5: 1827.6e6, 4: 2192.4e6, 3: 558.1e6}
SPLIT_KERNEL = {5: "split_rope_i8i4_kernel", 4: "split_fp8_kernel", 3: "split_int2_kernel",
                1: "split_generic_kernel", 2: "split_generic_kernel"}
K_AXES = {"tensor": 0, "token": 1, "channel": 2}


def static_qmax(fmt) -> float:
    """Calibration qmax of a per-tensor format: the FP8 maximum, or 2^(b-1)-1."""
    return FP8_MAX[fmt] if fmt in FP8_MAX else float((1 << (fmt - 1)) - 1)


def workload_spec(cid: int, batch: int = 0, fp8: str = "e4m3", meta: str = "f32", k_axis: str = "channel") -> dict:
    spec = _workload_spec(cid, batch, fp8, k_axis)
    spec["meta"] = meta  # stored scales / minima: "f32" or "f16" (binary16, scale up / minimum down)
    spec["flush"] = cid in LATENCY_CONFIGS
    if meta == "f16":
        spec["name"] += ", fp16 scales/minima"
    return spec


def _workload_spec(cid: int, batch: int = 0, fp8: str = "e4m3", k_axis: str = "channel") -> dict:
    w = W.WORKLOADS[cid]
    if batch:  # the first `batch` sequences of the workload (smaller captures for ncu)
        import dataclasses
        w = dataclasses.replace(w, batch=min(batch, w.batch))
    if cid == 1:
        if k_axis == "tensor":  # INT8 per-tensor K and V, static scales absmax/127
            return dict(w=w, k=(INT8, SYM, TEN, 0), v=(INT8, SYM, TEN, 0), R=0, P=256, rope=0, theta=1e4,
                        append=False, name="single fp32 head, 4096 tokens, Hq1/Hkv1/D128, INT8 per-tensor K and V "
                                           "(static absmax/127 scales)")
        if k_axis != "channel":
            raise SystemExit("--config 1 takes --k-axis channel or tensor")
        return dict(w=w, k=(INT8, SYM, CH, 4096), v=(INT8, SYM, TOK, 0), R=4096, P=4096, rope=0, theta=1e4,
                    append=False, name="single fp32 head, 4096 tokens, Hq1/Hkv1/D128, INT8 K per-channel (one "
                                       "4096-token group) + INT8 V per-token")
    if cid == 2:
        if k_axis == "token":
            return dict(w=w, k=(INT4, ASYM, TOK, 0), v=(INT4, ASYM, TOK, 0), R=0, P=512, rope=0, theta=1e4,
                        append=False, name="single fp32 kv-head, 512 tokens, 64 query heads, D128, INT4 asym K "
                                           "per-token + V per-token")
        if k_axis != "channel":
            raise SystemExit("--config 2 takes --k-axis channel or token")
        return dict(w=w, k=(INT4, ASYM, CH, 512), v=(INT4, ASYM, TOK, 0), R=512, P=512, rope=0, theta=1e4,
                    append=False, name="single fp32 kv-head, 512 tokens, 64 query heads, D128, INT4 asym K "
                                       "per-channel (one 512-token group) + V per-token")
    if cid == 5:
        return dict(w=w, k=(INT8, SYM, CH, 64), v=(INT4, ASYM, TOK, 128), R=64, P=16, rope=1, theta=500000.0,
                    append=True, name="paged ragged 1K-64K (sum T ~1.0M), Hq32/Hkv8/D128, INT8 per-channel "
                                      "pre-RoPE K (G64, theta 5e5) + INT4 asym per-token V, 64-token bf16 window, "
                                      "16-token pages; append + decode per step")
    if cid == 3:
        return dict(w=w, k=(INT2, ASYM, CH, 32), v=(INT2, ASYM, TOK, 32), R=128, P=256, rope=0, theta=1e4,
                    append=False, name="Llama-3.1-8B decode layer, B16, 32768 quantized + 127 window tokens, "
                                       "Hq32/Hkv8/D128, KIVI 2-bit K per-channel (G32) + V per-token (g32)")
    if cid == 4:
        f = FP8_FORMATS[fp8]
        return dict(w=w, k=(f, SYM, TEN, 0), v=(f, SYM, TEN, 0), R=0, P=256, rope=0, theta=1e4, append=False,
                    name=f"Llama-3.1-70B decode layer, B8, 131072 tokens, Hq64/Hkv8/D128, FP8 {fp8.upper()} K/V "
                         f"with per-head absmax/{FP8_MAX[f]:g} scales")
    raise SystemExit(f"unknown --config {cid}")


# ------------------------------------------------------------------ byte accounting

def _is_fp8(fmt):
    return fmt in FP8_MAX


def _bits(fmt):
    return 8 if _is_fp8(fmt) else fmt


def quantized_bytes(spec, n: int) -> int:
    """Packed codes plus scale/min metadata of n quantized tokens of one kv-head."""
    D = spec["w"].head_dim
    kf, kmode, kaxis, kg = spec["k"]
    vf, vmode, vaxis, vg = spec["v"]
    nmk = 2 if kmode == ASYM and not _is_fp8(kf) else 1
    nmv = 2 if vmode == ASYM and not _is_fp8(vf) else 1
    mb = 2 if spec.get("meta") == "f16" else 4  # bytes per stored scale / minimum
    total = n * D * (_bits(kf) + _bits(vf)) // 8
    if kaxis == CH:
        total += (n // kg) * D * mb * nmk
    elif kaxis == TOK:
        total += n * (D // (kg or D)) * mb * nmk
    if vaxis == TOK:
        total += n * (D // (vg or D)) * mb * nmv
    return total


def head_bytes(spec, T: int) -> int:
    """Bytes one (sequence, kv-head) contributes to a decode call: its quantized
    tokens plus its window tokens (K and V, source dtype)."""
    w = spec["w"]
    src = 2 if w.src_dtype == "bf16" else 4
    R = spec["R"]
    nq = T if R == 0 else R * (T // R)
    return quantized_bytes(spec, nq) + (T - nq) * w.head_dim * 2 * src


def attention_bytes(spec, lens) -> int:
    """Algorithmic bytes one decode-attention call must move."""
    w = spec["w"]
    src = 2 if w.src_dtype == "bf16" else 4
    total = sum(w.num_kv_heads * head_bytes(spec, T) for T in lens)
    return total + len(lens) * w.num_q_heads * w.head_dim * (src + 4)  # q in, fp32 out


def append_bytes(spec, lens_before) -> int:
    """Algorithmic bytes of appending one token to every sequence: read the new
    K and V rows; write them to the window, or, when the window fills, read its
    R-1 older tokens and write the R tokens' codes and metadata."""
    w = spec["w"]
    H, D = w.num_kv_heads, w.head_dim
    src = 2 if w.src_dtype == "bf16" else 4
    R = spec["R"]
    total = 0
    for T in lens_before:
        total += 2 * H * D * src
        if R == 0:
            total += H * quantized_bytes(spec, 1)
        elif (T + 1) % R == 0:
            total += 2 * (R - 1) * H * D * src + H * quantized_bytes(spec, R)
        else:
            total += 2 * H * D * src
    return total


# ------------------------------------------------------------------ CPU oracle leg

_ORACLE_STATES = {}  # per worker process: quantized streams already built, by job


def _oracle_state(cid, b, h, T, fp8, meta, k_axis):
    """The oracle's quantized stream of one (sequence, kv-head), its queries and
    static scales (built once per worker process and kept)."""
    key = (cid, b, h, T, fp8, meta, k_axis)
    if key not in _ORACLE_STATES:
        from oracle import kvq_oracle as O
        spec = workload_spec(cid, 0, fp8, meta, k_axis)
        w = spec["w"]
        cfg = O.Config(w.num_q_heads, w.num_kv_heads, w.head_dim, O.QSpec(*spec["k"]), O.QSpec(*spec["v"]),
                       spec["R"], spec["P"], spec["rope"], spec["theta"],
                       O.BF16 if w.src_dtype == "bf16" else O.F32, meta_dtype=O.F16 if meta == "f16" else O.F32)
        K = W.kv_block(w, b, h, W.KIND_K, 0, T)
        V = W.kv_block(w, b, h, W.KIND_V, 0, T)
        ks = O.calibrate_absmax(K, static_qmax(spec["k"][0])) if spec["k"][2] == TEN else 0.0
        vs = O.calibrate_absmax(V, static_qmax(spec["v"][0])) if spec["v"][2] == TEN else 0.0
        st = O.quantize_stream(cfg, K, V, ks, vs)
        q = W.queries(w, 0)[b % w.batch, h * cfg.n_rep:(h + 1) * cfg.n_rep].astype(np.float64)
        _ORACLE_STATES[key] = (O, cfg, st, q, ks, vs)
    return _ORACLE_STATES[key]


def _oracle_decode(job, steps):
    """Run the oracle's decode (dequantize + RoPE + attention) `steps` times on
    one sampled (sequence, kv-head) stream; seconds taken."""
    cid, b, h, T, _, fp8, meta, k_axis = job
    O, cfg, st, q, ks, vs = _oracle_state(cid, b, h, T, fp8, meta, k_axis)
    t0 = time.perf_counter()
    for _ in range(steps):
        O.decode_head(cfg, st, q, ks, vs)
    return time.perf_counter() - t0


def _oracle_proc(jobs, inbox, outbox):
    """One worker process of OraclePool: build the quantized streams of its jobs,
    report ready, then for every request run each job's decode and report the
    seconds; one BLAS thread (set by the parent's environment)."""
    for j in jobs:
        _oracle_state(*[j[k] for k in (0, 1, 2, 3, 5, 6, 7)])
    outbox.put(0.0)
    while True:
        steps = inbox.get()
        if steps is None:
            return
        outbox.put(sum(_oracle_decode(j, j[4] if steps < 0 else steps) for j in jobs))


def oracle_jobs(cid, n_streams, steps, fp8, meta, k_axis, max_tokens=0):
    """A seeded sample of the workload's (sequence, kv-head) streams as oracle
    jobs; streams longer than max_tokens (if set) are cut to that prefix."""
    spec = workload_spec(cid, 0, fp8, meta, k_axis)
    w = spec["w"]
    lens = W.lengths(w)
    g = np.random.default_rng(1234)
    picks = [(int(g.integers(0, w.batch)), int(g.integers(0, w.num_kv_heads))) for _ in range(n_streams)]
    cap = 16384 if cid == 4 else 0  # 131072-token streams: a prefix keeps the sample bounded
    if max_tokens:
        cap = min(cap, max_tokens) if cap else max_tokens
    return [(cid, b, h, min(int(lens[b]), cap) if cap else int(lens[b]), steps, fp8, meta, k_axis)
            for b, h in picks]


def oracle_job_bytes(jobs):
    """Bytes the sampled streams contribute to decode calls: each stream's KV
    bytes plus its query heads' q and out, per timed step."""
    total = 0
    for (cid, b, h, T, steps, fp8, meta, k_axis) in jobs:
        spec = workload_spec(cid, 0, fp8, meta, k_axis)
        w = spec["w"]
        src = 2 if w.src_dtype == "bf16" else 4
        total += (head_bytes(spec, T) + (w.num_q_heads // w.num_kv_heads) * w.head_dim * (src + 4)) * steps
    return total


class OraclePool:
    """Spawned oracle worker processes, one BLAS thread each, with a fixed share
    of the jobs (job i goes to process i mod procs).  Each process builds its
    quantized streams once at start-up (untimed); a pass then starts every
    process at once and ends when the last one finishes, so the pass's wall time
    holds decode work only."""

    ENV = ["OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"]

    def __init__(self, procs, jobs):
        import multiprocessing as mp
        try:
            cores = len(os.sched_getaffinity(0))
        except AttributeError:
            cores = os.cpu_count() or 1
        self.procs = max(1, min(cores, procs, len(jobs)))
        self.old = {k: os.environ.get(k) for k in self.ENV}
        for k in self.ENV:
            os.environ[k] = "1"
        ctx = mp.get_context("spawn")
        self.outbox = ctx.Queue()
        self.inboxes = [ctx.Queue() for _ in range(self.procs)]
        self.ps = [ctx.Process(target=_oracle_proc, args=(jobs[i::self.procs], self.inboxes[i], self.outbox),
                               daemon=True) for i in range(self.procs)]
        for p in self.ps:
            p.start()
        for _ in self.ps:  # every stream built
            self.outbox.get()

    def run(self, steps=-1):
        """(summed decode seconds, wall seconds) of one pass: every job's decode
        `steps` times (-1: each job's own step count)."""
        t0 = time.perf_counter()
        for q in self.inboxes:
            q.put(steps)
        busy = sum(self.outbox.get() for _ in self.ps)
        return busy, time.perf_counter() - t0

    def close(self):
        for q in self.inboxes:
            q.put(None)
        for p in self.ps:
            p.join(timeout=60)
        for k, val in self.old.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val


def cpu_oracle_throughput(cid: int, n_streams: int, steps: int = 1, fp8: str = "e4m3", meta: str = "f32",
                          k_axis: str = "channel", append: bool = False):
    """Oracle GB/s on a bounded sample of the workload's streams: bytes of the
    timed decodes over the wall time of the pass, in a spawned process pool (one
    BLAS thread per process, one process per available core), and the same
    sample on one core.  Building the quantized streams happens in an untimed
    first pass."""
    jobs = oracle_jobs(cid, n_streams, steps, fp8, meta, k_axis)
    nbytes = oracle_job_bytes(jobs)
    pool = OraclePool(len(jobs), jobs)
    try:
        busy, wall = pool.run()
    finally:
        pool.close()
    one = OraclePool(1, jobs)
    try:
        one_jobs = [j[:4] + (1,) + j[5:] for j in jobs]  # one step per stream on one core
        _, wall1 = one.run(1)
    finally:
        one.close()
    return dict(value=nbytes / wall / 1e9, unit="GB/s", cores=pool.procs, kind="oracle",
                value_1core=oracle_job_bytes(one_jobs) / wall1 / 1e9,
                sample=f"{len(jobs)} (sequence, kv-head) streams of the workload ("
                       f"{sum(j[3] for j in jobs)} tokens), decode = dequantize + RoPE + attention in float64, "
                       f"{steps} step(s) each; value = bytes / wall time of the pass over {pool.procs} spawned "
                       f"processes x 1 BLAS thread ({busy:.1f} s CPU, {wall:.1f} s wall); value_1core = one "
                       f"step per stream in one process ({wall1:.1f} s wall)"
                       + ("; the append of each step is not timed on the CPU" if append else ""))


# ------------------------------------------------------------------ ranks

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    identity for one rank.  `device`: where the process group's tensors live
    (the GPU for NCCL, the CPU for gloo)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: float, world: int, elapsed_ms: float) -> float:
    """Whole-job GB/s: every replica moves the same bytes in the slowest rank's time."""
    return bytes_per_rank * world / (elapsed_ms / 1e3) / 1e9


# ------------------------------------------------------------------ GPU leg

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def hold_device(ms: float = 20.0):
    """Keep the GPU busy for about `ms` before a timed region, so the host queues
    the region's launches while it waits and no step waits on the host (a host
    hiccup at the start of the loop would otherwise show up as device time)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(ms * 1e-3 * 2.0e9))


def build_cache(spec, device, extra_tokens, gen_seed=1):
    """Fill a cache with the workload's prefill through kvq_quantize_append.
    bf16 workloads are drawn on the device with a seeded torch generator
    (N(0,1), K outlier channels from kvq_inputs.outliers); the small fp32
    workloads take the host streams of kvq_inputs.kv_block.  Static per-tensor
    scales (FP8, per-tensor INT) come from kvq_calibrate_absmax."""
    import torch
    import asymmetric_quantized_kv_gb300 as K
    w = spec["w"]
    Bn, H, D, Hq = w.batch, w.num_kv_heads, w.head_dim, w.num_q_heads
    lens = [int(x) for x in W.lengths(W.WORKLOADS[w.cid])][:w.batch]
    P = spec["P"]
    src_f32 = w.src_dtype == "f32"
    cfg = K.make_config(Hq, H, D, spec["k"], spec["v"], spec["R"], P, spec["rope"], spec["theta"],
                        F32 if src_f32 else BF16, 2 if spec.get("meta") == "f16" else 0)
    need = [(T + extra_tokens + P - 1) // P for T in lens]
    maxp = max(need)
    n_pages = sum(need)
    perm = W.page_permutation(n_pages, 5)
    bt = np.zeros((Bn, maxp), np.int32)
    o = 0
    for b in range(Bn):
        bt[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    cache = K.PagedKVCache(cfg, Bn, maxp, n_pages, bt, device=device)
    if src_f32:  # small workloads: every stream at once, [B, T, Hkv, D] fp32
        T = max(lens)
        kk = torch.from_numpy(np.stack([np.stack([W.kv_block(w, b, h, W.KIND_K, 0, T) for h in range(H)], 1)
                                        for b in range(Bn)])).to(device)
        vv = torch.from_numpy(np.stack([np.stack([W.kv_block(w, b, h, W.KIND_V, 0, T) for h in range(H)], 1)
                                        for b in range(Bn)])).to(device)
        for kind, src, dst in ((0, kk, cache.k_scale), (1, vv, cache.v_scale)):
            f = spec["k" if kind == 0 else "v"]
            if f[2] == TEN:
                K.kvq_calibrate_absmax(cfg, src.reshape(-1, H, D).contiguous(), Bn * T, static_qmax(f[0]), dst)
        cache.append(kk, vv, torch.tensor(lens, dtype=torch.int32, device=device))
        torch.cuda.synchronize(device)
        return cfg, cache, lens
    scale = W.torch_outlier_scale(w, device)
    g = torch.Generator(device=device)
    g.manual_seed(gen_seed)
    chunk = 4096 if Bn * H * D * 4096 * 2 < (1 << 31) else 1024
    if _is_fp8(spec["k"][0]):  # calibrate on the whole source, then append it (same draws)
        state = g.get_state()
        kmax = torch.zeros(H, device=device)
        vmax = torch.zeros(H, device=device)
        done = 0
        while done < max(lens):
            n = min(chunk, max(lens) - done)
            kk, vv = W.torch_kv_chunk(w, g, Bn, n, scale, device)
            kk = kk.transpose(0, 1).reshape(-1, H, D)
            vv = vv.transpose(0, 1).reshape(-1, H, D)
            tmp = torch.empty(H, device=device)
            K.kvq_calibrate_absmax(cfg, kk.contiguous(), kk.shape[0], FP8_MAX[spec["k"][0]], tmp)
            kmax = torch.maximum(kmax, tmp)
            K.kvq_calibrate_absmax(cfg, vv.contiguous(), vv.shape[0], FP8_MAX[spec["v"][0]], tmp)
            vmax = torch.maximum(vmax, tmp)
            done += n
        cache.k_scale.copy_(kmax)
        cache.v_scale.copy_(vmax)
        g.set_state(state)
    done = 0
    while done < max(lens):
        n = min(chunk, max(lens) - done)
        per = torch.tensor([max(0, min(n, T - done)) for T in lens], dtype=torch.int32, device=device)
        kk, vv = W.torch_kv_chunk(w, g, Bn, n, scale, device)
        cache.append(kk, vv, per)
        done += n
    torch.cuda.synchronize(device)
    return cfg, cache, lens


def run_gpu(args, spec, rank, world):
    import torch
    import torch.distributed as dist
    import asymmetric_quantized_kv_gb300 as K
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = spec["w"]
    Bn, H, D, Hq = w.batch, w.num_kv_heads, w.head_dim, w.num_q_heads
    steps, warm = args.steps, args.warmup
    total_steps = warm + steps + (warm + steps if args.e2e else 0)
    cfg, cache, lens = build_cache(spec, device, total_steps + 1)
    g = torch.Generator(device=device)
    g.manual_seed(77 + rank)
    sdt = torch.float32 if w.src_dtype == "f32" else torch.bfloat16
    q_all = torch.randn(total_steps, Bn, Hq, D, generator=g, device=device).to(sdt)
    k_all = torch.randn(total_steps, Bn, 1, H, D, generator=g, device=device).to(sdt)
    v_all = torch.randn(total_steps, Bn, 1, H, D, generator=g, device=device).to(sdt)
    # inputs that fit in L2: a write larger than L2 before every timed call
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device) if spec["flush"] else None
    out = torch.empty(Bn, Hq, D, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    do_append = spec["append"]

    def step(i):
        if do_append:
            K.kvq_quantize_append(cfg, cache.c, k_all[i], v_all[i], 1, None, stream)
        K.kvq_decode_attention(cfg, cache.c, q_all[i], out, 0.0, cache.workspace, stream)

    cur = list(lens)
    for i in range(warm):
        step(i)
        if do_append:
            cur = [T + 1 for T in cur]
    torch.cuda.synchronize(device)
    # bytes of the timed steps, from the known lengths
    step_bytes = []
    att_bytes = []
    for i in range(steps):
        ab = append_bytes(spec, cur) if do_append else 0
        if do_append:
            cur = [T + 1 for T in cur]
        tb = attention_bytes(spec, cur)
        att_bytes.append(tb)
        step_bytes.append(ab + tb)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    att_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    hold_device()
    ev0.record(stream)
    for i in range(steps):
        j = warm + i
        if flush is not None:
            flush.fill_(i & 255)
        if do_append:
            K.kvq_quantize_append(cfg, cache.c, k_all[j], v_all[j], 1, None, stream)
        att_ev[i][0].record(stream)
        K.kvq_decode_attention(cfg, cache.c, q_all[j], out, 0.0, cache.workspace, stream)
        att_ev[i][1].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(device)
    att_ms = [a.elapsed_time(b) for a, b in att_ev]
    # with flushes in the loop, the step time is the calls' own event times
    elapsed_ms = ev0.elapsed_time(ev1) if flush is None else sum(att_ms)
    clock_info = clocks.stop()
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    status = int(cache.status.item())
    # end to end through the public API: pinned host inputs in, result out, every step
    e2e = None
    if args.e2e:
        hq = q_all[warm + steps:].cpu().pin_memory()
        hk = k_all[warm + steps:].cpu().pin_memory()
        hv = v_all[warm + steps:].cpu().pin_memory()
        host_out = torch.empty((warm + steps,) + tuple(out.shape), dtype=torch.float32).pin_memory()
        dq = torch.empty_like(q_all[0])
        dk = torch.empty_like(k_all[0])
        dv = torch.empty_like(v_all[0])
        e2e_bytes = 0
        cur2 = list(cur)
        def e2e_step(i):
            dq.copy_(hq[i], non_blocking=True)
            if do_append:
                dk.copy_(hk[i], non_blocking=True)
                dv.copy_(hv[i], non_blocking=True)
                K.kvq_quantize_append(cfg, cache.c, dk, dv, 1, None, stream)
            K.kvq_decode_attention(cfg, cache.c, dq, out, 0.0, cache.workspace, stream)
            host_out[i].copy_(out, non_blocking=True)
        for i in range(warm):
            e2e_step(i)
            if do_append:
                cur2 = [T + 1 for T in cur2]
        torch.cuda.synchronize(device)
        for i in range(steps):
            ab = append_bytes(spec, cur2) if do_append else 0
            if do_append:
                cur2 = [T + 1 for T in cur2]
            e2e_bytes += ab + attention_bytes(spec, cur2)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)
        if flush is None:
            # the timed steps run as a serving loop would: one CUDA graph of all of them, captured
            # from the public API calls, in which a copy stream brings step i+1's inputs into the
            # other buffer set and reads step i-1's output back while step i's kernels run.  Every
            # step's copies stay inside the timed region, which ends when the last output is on the
            # host; the graph only removes the host's per-call launch cost.
            cap = torch.cuda.Stream(device)
            cs = torch.cuda.Stream(device)
            dqs = [dq, torch.empty_like(dq)]
            dks = [dk, torch.empty_like(dk)]
            dvs = [dv, torch.empty_like(dv)]
            outs = [out, torch.empty_like(out)]
            in_ready = [torch.cuda.Event() for _ in range(steps)]
            done = [torch.cuda.Event() for _ in range(steps)]
            out_read = [torch.cuda.Event() for _ in range(steps)]

            def h2d(i):  # inputs of timed step i into buffer set i % 2, once step i-2 has used it
                j = i & 1
                with torch.cuda.stream(cs):
                    if i >= 2:
                        cs.wait_event(done[i - 2])
                    dqs[j].copy_(hq[warm + i], non_blocking=True)
                    if do_append:
                        dks[j].copy_(hk[warm + i], non_blocking=True)
                        dvs[j].copy_(hv[warm + i], non_blocking=True)
                    in_ready[i].record(cs)

            graph = torch.cuda.CUDAGraph()
            torch.cuda.synchronize(device)
            with torch.cuda.graph(graph, stream=cap):
                cs.wait_stream(cap)
                h2d(0)
                for i in range(steps):
                    j = i & 1
                    if i + 1 < steps:
                        h2d(i + 1)
                    cap.wait_event(in_ready[i])
                    if i >= 2:
                        cap.wait_event(out_read[i - 2])  # output buffer j is free again
                    if do_append:
                        K.kvq_quantize_append(cfg, cache.c, dks[j], dvs[j], 1, None, cap)
                    K.kvq_decode_attention(cfg, cache.c, dqs[j], outs[j], 0.0, cache.workspace, cap)
                    done[i].record(cap)
                    with torch.cuda.stream(cs):
                        cs.wait_event(done[i])
                        host_out[warm + i].copy_(outs[j], non_blocking=True)
                        out_read[i].record(cs)
                cap.wait_stream(cs)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            hold_device()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize(device)
            e_ms = e0.elapsed_time(e1)
        else:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(steps)]
            for i in range(steps):
                flush.fill_(i & 255)
                pairs[i][0].record(stream)
                e2e_step(warm + i)
                pairs[i][1].record(stream)
            torch.cuda.synchronize(device)
            e_ms = sum(a.elapsed_time(b) for a, b in pairs)
        e_ms = max_over_ranks(e_ms, world, device)
        h2d = dq.numel() * dq.element_size() + (2 * dk.numel() * dk.element_size() if do_append else 0)
        e2e = {"value": job_throughput(e2e_bytes, world, e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": out.numel() * out.element_size(), "ms_per_step": e_ms / steps,
               "mode": ("one CUDA graph of the timed steps' API calls; a copy stream overlaps step i+1's input "
                        "copies and step i-1's output read with step i's kernels" if flush is None else
                        "one step at a time after the L2 flush: input copies, kernels, output read in order")}
    return dict(elapsed_ms=elapsed_ms, step_bytes=step_bytes, att_bytes=att_bytes, att_ms=att_ms,
                clocks=clock_info, status=status, e2e=e2e, lens=cur)


def kcycles(us, clocks):
    """Thousands of SM cycles at the median SM clock sampled during the timed
    region (time x clock: comparable across runs whose clocks differ)."""
    if not clocks or not clocks.get("sm_mhz"):
        return None
    return us * clocks["sm_mhz"] / 1e3


def layer_line(args, cid, peak, peak_kind):
    """Decode-only measurement of another headline layer in the same process
    (the 2-bit 8B layer, the FP8 70B layer): its own cache, events around every
    decode call over the same number of steps, its roofline against the same
    HBM peak."""
    import argparse as _ap
    import torch
    spec = workload_spec(cid)
    sub = _ap.Namespace(**vars(args))
    sub.e2e = False
    r = run_gpu(sub, spec, 0, 1)
    torch.cuda.empty_cache()
    att_ms = statistics.mean(r["att_ms"])
    att_bytes = statistics.mean(r["att_bytes"])
    achieved = att_bytes / (att_ms / 1e3) / 1e9
    return {"workload": spec["name"], "batch": spec["w"].batch, "sum_tokens": int(sum(r["lens"])),
            "us_per_call": att_ms * 1e3, "us_per_call_median": statistics.median(r["att_ms"]) * 1e3,
            "bytes_per_call": att_bytes, "value": achieved, "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": SPLIT_TRAFFIC.get(cid),
                         "kernel": f"kvq_decode_attention: {SPLIT_KERNEL[cid]} + combine (timed together)",
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s"},
            "gpu_launches": args.steps * LAUNCHES_ATTENTION, "clocks": r["clocks"], "device_status": r["status"],
            "kcycles_per_call": kcycles(att_ms * 1e3, r["clocks"])}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-layers", dest="layers", action="store_false",
                    help="skip the 2-bit and FP8 layers that a default (--config 5, one GPU) run adds to its line")
    ap.add_argument("--cpu-streams", type=int, default=16)
    ap.add_argument("--cpu-steps", type=int, default=8)
    ap.add_argument("--batch", type=int, default=0, help="use only the first N sequences (profiling)")
    ap.add_argument("--fp8", default="e4m3", choices=sorted(FP8_FORMATS), help="FP8 format of --config 4")
    ap.add_argument("--meta", default="f32", choices=["f32", "f16"], help="stored scales / minima (configs 3, 5)")
    ap.add_argument("--k-axis", default="channel", choices=sorted(K_AXES),
                    help="key axis of --config 1 (channel or tensor) and --config 2 (channel or token)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.k_axis != "channel" and args.config not in LATENCY_CONFIGS:
        raise SystemExit("--k-axis applies to --config 1 and 2")
    spec = workload_spec(args.config, args.batch, args.fp8, args.meta, args.k_axis)
    w = spec["w"]

    if args.impl == "reference":
        if rank != 0:
            return
        # one pool for the whole run; the warm-up passes build each worker's
        # quantized streams, every timed pass times the decode alone
        jobs = oracle_jobs(args.config, args.cpu_streams, 1, args.fp8, args.meta, args.k_axis,
                           max_tokens=REF_MAX_TOKENS)
        nbytes = oracle_job_bytes(jobs)
        pool = OraclePool(len(jobs), jobs)
        per_step, busy_all, wall_all = [], 0.0, 0.0
        try:
            for _ in range(args.warmup):
                pool.run()
            for _ in range(args.steps):
                busy, wall = pool.run()
                busy_all += busy
                wall_all += wall
                per_step.append(nbytes / wall / 1e9)
        finally:
            pool.close()
        val = statistics.median(per_step)
        detail = dict(value=val, unit="GB/s", cores=pool.procs, kind="oracle",
                      sample=f"{len(jobs)} (sequence, kv-head) streams of the workload (prefixes of at most "
                             f"{REF_MAX_TOKENS} tokens, {sum(j[3] for j in jobs)} tokens) per step, decode = "
                             f"dequantize + RoPE + attention in float64, bytes / wall time of each pass, median "
                             f"over {args.steps} steps after {args.warmup} warm-up passes; {pool.procs} spawned "
                             f"processes x 1 BLAS thread; {busy_all:.1f} s CPU, {wall_all:.1f} s wall")
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": spec["name"]}, "cpu_baseline": detail,
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_throughput(args.config, n_streams=args.cpu_streams, steps=args.cpu_steps, fp8=args.fp8,
                                    meta=args.meta, k_axis=args.k_axis, append=spec["append"])

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_gpu(args, spec, rank, world)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    steps = args.steps
    ms_per_step = r["elapsed_ms"] / steps
    value = job_throughput(sum(r["step_bytes"]), world, r["elapsed_ms"])
    peak, peak_kind = load_peaks()
    att_ms = statistics.mean(r["att_ms"])
    att_bytes = statistics.mean(r["att_bytes"])
    achieved = att_bytes / (att_ms / 1e3) / 1e9
    launches = steps * ((LAUNCHES_APPEND if spec["append"] else 0) + LAUNCHES_ATTENTION)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "us_per_step": ms_per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": spec["name"], "batch": w.batch, "sum_tokens": int(sum(r["lens"])),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": ("flushed before every decode call (a 256 MiB write outside the call's events); "
                          "inputs %.2f MB per call" % (att_bytes / 1e6)) if spec["flush"] else
                         "inputs (%.2f GB per step) larger than the 129 MB L2; no flush" % (att_bytes / 1e9)},
        "pct_of_hbm_peak": 100.0 * value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": SPLIT_TRAFFIC.get(args.config)
                     if not args.batch and args.fp8 == "e4m3" and args.meta == "f32" else None,
                     "kernel": f"kvq_decode_attention: {SPLIT_KERNEL[args.config]} + combine (timed together)",
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "us_per_launch": att_ms * 1e3,
                     "us_per_launch_median": statistics.median(r["att_ms"]) * 1e3,
                     "bytes_per_launch": att_bytes},
        "cpu_baseline": cpu,
        "e2e": r["e2e"],
        "gpu_launches": launches,
        "clocks": r["clocks"],
        "kcycles_per_decode": kcycles(att_ms * 1e3, r["clocks"]),
        "device_status": r["status"],
    }
    if world == 1 and args.config == 5 and args.layers and not args.batch and args.meta == "f32":
        # the other two headline layers, decode alone, each against the HBM roofline
        line["layers"] = {str(cid): layer_line(args, cid, peak, peak_kind) for cid in (3, 4)}
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
