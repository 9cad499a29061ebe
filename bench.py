#!/usr/bin/env python
"""Benchmark of the TurboQuant compressed-KV decode step on GB300.

A step is the whole hot path for one batch: tq_paged_append of one new token
per sequence (K and V encode into the paged pools), then decode attention
over the compressed cache (query prep, split-K pass, merge + inverse WHT).
Default workload: 16 sequences x 32 query heads / 8 KV heads, d=128, context
4096 (4095 cached + 1 appended), 16-token blocks scattered by a random
permutation, bf16 inputs with lognormal per-channel K scales.

Printed (rank 0, one JSON line): GB/s over the algorithmic bytes of a step
(compressed cache read by decode + block ids + query/output + append traffic),
the split-K kernel's live CUDA-event time against the measured HBM peak, the
end-to-end rate through host buffers, and the fp64 CPU oracle timed on this
machine's cores on a bounded sample.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl tq|reference]
With --impl reference the same metric is measured for the fp64 CPU oracle.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn compressed-KV GB/s & % of GB300 HBM peak; encode Mtok/s vs CPU oracle"
WORKLOAD = "llama8b_decode"
L2_BYTES = 129 * 1024 * 1024
# the d = 128 pass and the headers it is built from: the committed traffic figure is used only
# while their combined hash matches the one the counters were taken on
DECODE_SRC = [os.path.join(ROOT, "turboquant_compressed_kv_gb300", "csrc", f)
              for f in ("tq_decode_warp.cu", "tq_split.cuh", "tq_prep.cuh", "tq_internal.cuh")]
PROFILE_JSON = os.path.join(ROOT, "profiles", "decode_warp_llama8b_decode_traffic.txt")


def decode_src_hash():
    h = hashlib.sha256()
    for f in DECODE_SRC:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--main-only", action="store_true",
                    help="skip the ragged / long-context decode and the prefill encode measurements")
    ap.add_argument("--workload", default=None,
                    help="run only this side workload (ragged, long256, verify_q2, hybrid32k, prefill_encode, "
                         "prefill_encode256, prefill_dequant, gq_compare) and print its JSON object; for profiling")
    ap.add_argument("--oracle-single-thread", choices=["decode", "encode"], default=None,
                    help=argparse.SUPPRESS)   # child run of the oracle on one thread (cpu_baseline)
    return ap.parse_args()


# ---------------------------------------------------------------- bytes

def step_bytes(w) -> dict:
    """Algorithmic bytes of one step: what the method must move."""
    d, Hkv = w.head_dim, w.n_kv_heads
    krec, vrec = (8 * d + 64) / 16, (6 * d + 32) / 16      # bytes per token per kv head
    tokens = sum(w.ctx_lens)
    cache = tokens * Hkv * (krec + vrec)
    blocks = sum(math.ceil(L / 16) for L in w.ctx_lens) * 4
    in_bytes = 2 if w.dtype == "bf16" else 4
    q = w.batch * w.n_q_heads * d * in_bytes
    out = w.batch * w.n_q_heads * d * 4
    app = w.batch * Hkv * (2 * d * in_bytes + krec + vrec) if w.append else 0
    return dict(cache=cache, blocks=blocks, q=q, out=out, append=app,
                partial=cache + blocks, step=cache + blocks + q + out + app)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, ln in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- oracle (CPU) arm

def oracle_sample_setup(w, nseq):
    """Cache of the first nseq sequences written by the oracle (setup, untimed)."""
    import numpy as np

    import oracle
    from turboquant_compressed_kv_gb300 import synth
    d = w.head_dim
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    bt, nblk = synth.block_tables(w)
    bt = bt[:nseq]
    used = np.unique(bt)
    remap = {int(b): i for i, b in enumerate(used)}
    bt_s = np.vectorize(remap.get)(bt).astype(np.int32)
    kp = np.zeros((len(used), w.n_kv_heads, 8 * d + 64), np.uint8)
    vp = np.zeros((len(used), w.n_kv_heads, 6 * d + 32), np.uint8)
    for b in range(nseq):
        L = w.prefill_lens[b]
        K, V = synth.kv_tokens(w, b, 0, L)
        sl = synth.slots_for(bt_s, b, 0, L)
        oracle.encode(True, D, S, K, sl, kp)
        oracle.encode(False, D, S, V, sl, vp)
    q = synth.queries(w)[:nseq]
    kn = np.empty((nseq, w.n_kv_heads, d), np.float32)
    vn = np.empty_like(kn)
    for b in range(nseq):
        k1, v1 = synth.kv_tokens(w, b, w.prefill_lens[b], 1)
        kn[b], vn[b] = k1[0], v1[0]
    return dict(D=D, S=S, bt=bt_s, kp=kp, vp=vp, q=q, kn=kn, vn=vn, nseq=nseq)


def oracle_step(w, st):
    import numpy as np

    import oracle
    from turboquant_compressed_kv_gb300 import synth
    n = st["nseq"]
    slots = np.array([synth.slots_for(st["bt"], b, w.prefill_lens[b], 1)[0] for b in range(n)], np.int64)
    if w.append:
        oracle.encode(True, st["D"], st["S"], st["kn"], slots, st["kp"])
        oracle.encode(False, st["D"], st["S"], st["vn"], slots, st["vp"])
    ctx = np.array(w.ctx_lens[:n], np.int32)
    return oracle.decode(st["D"], st["S"], st["q"], w.n_kv_heads, st["kp"], st["vp"], st["bt"], ctx)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_oracle(w, steps, warmup, nseq):
    """Times the oracle (as it stands) on the first nseq sequences; returns (GB/s, seconds/step)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(cores()))
    from turboquant_compressed_kv_gb300 import synth
    import dataclasses
    ws = dataclasses.replace(w, batch=nseq, ctx_lens=w.ctx_lens[:nseq], prefill_lens=w.prefill_lens[:nseq])
    st = oracle_sample_setup(w, nseq)
    for _ in range(warmup):
        oracle_step(w, st)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(w, st)
    dt = (time.perf_counter() - t0) / steps
    return step_bytes(ws)["step"] / dt / 1e9, dt, ws


def run_cpu_encode(w, ntok=4096):
    """Times the oracle's K and V encode (as it stands, OpenMP over vectors) on the first ntok tokens of
    sequence 0, all kv heads; returns (tokens/s, seconds, sample description)."""
    os.environ.setdefault("OMP_NUM_THREADS", str(cores()))
    import numpy as np

    import oracle
    from turboquant_compressed_kv_gb300 import synth
    d, H = w.head_dim, w.n_kv_heads
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    K, V = synth.kv_tokens(w, 0, 0, ntok)
    nblk = (ntok + 15) // 16
    kp = np.zeros((nblk, H, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nblk, H, oracle.record_bytes(False, d)), np.uint8)
    slots = np.arange(ntok, dtype=np.int64)
    oracle.encode(True, D, S, K[:64], slots[:64], kp)     # warm-up (library load)
    t0 = time.perf_counter()
    oracle.encode(True, D, S, K, slots, kp)
    oracle.encode(False, D, S, V, slots, vp)
    dt = time.perf_counter() - t0
    return ntok / dt, dt, f"{ntok} tokens x {H} kv heads of sequence 0 (K and V), one timed pass"


def bench_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from turboquant_compressed_kv_gb300 import synth
    w = synth.workload(WORKLOAD)
    nseq = 1
    gbs, dt, ws = run_cpu_oracle(w, args.steps, args.warmup, nseq)
    n = int(os.environ.get("OMP_NUM_THREADS", cores()))
    sample = (f"{nseq} of {w.batch} sequences per step: append 1 token x {w.n_kv_heads} kv heads (K+V), "
              f"decode {w.n_q_heads} query heads over {w.ctx_lens[0]} tokens")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "fp64 CPU oracle, per-step sample"),
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def max_over_ranks(values, world, device):
    """Element-wise maximum of a list of floats over all ranks (the job takes as long as its slowest
    rank); the identity at world == 1."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_gbs(world, bytes_per_step, seconds_per_step):
    """Whole-job throughput: every rank processes its own batch (replicas), in the slowest rank's time."""
    return world * bytes_per_step / seconds_per_step / 1e9


def workload_config(w, l2_note):
    return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "ctx": w.ctx_lens[0], "block_size": 16, "kv_dtype_in": w.dtype,
            "k_scales": w.k_scale, "parallelism": "replicas (one independent batch per GPU)", "l2": l2_note}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profile_traffic(bytes_per_launch):
    """dram bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    try:
        with open(PROFILE_JSON) as f:
            prof = json.load(f)
        if prof.get("source_sha256_16") != decode_src_hash():
            return None
        return float(prof["dram_bytes_per_launch_full"])
    except Exception:
        return None


def run_ahead(dev, n_iters, body, batch=100, lead_ms=30.0):
    """body(i) for i < n_iters, in batches that each start behind a short spin kernel on the current
    stream, so that the interpreter has queued the whole batch before the GPU reaches it.  Event pairs
    inside body then time device work only: in a plain loop whose calls take the interpreter longer
    to issue than the GPU takes to run them, an event pair around one call also spans the time the
    GPU sat waiting for that call to be queued."""
    import torch
    cycles = int(lead_ms * 1e-3 * 2.2e9)
    for b0 in range(0, n_iters, batch):
        torch.cuda._sleep(cycles)
        for i in range(b0, min(n_iters, b0 + batch)):
            body(i)
        torch.cuda.synchronize(dev)


def timed_batches(dev, n_iters, body, batch=100, lead_ms=30.0):
    """Mean device milliseconds of body(i) over n_iters calls, timed per batch of calls queued behind a
    short spin kernel (one event pair per batch, after the spin), for calls whose issue takes the
    interpreter about as long as the GPU takes to run them."""
    import torch
    cycles = int(lead_ms * 1e-3 * 2.2e9)
    total, done = 0.0, 0
    for b0 in range(0, n_iters, batch):
        n = min(batch, n_iters - b0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(cycles)
        e0.record()
        for i in range(b0, b0 + n):
            body(i)
        e1.record()
        torch.cuda.synchronize(dev)
        total += e0.elapsed_time(e1)
        done += n
    return total / done


def extra_decode(name, steps, warmup, dev):
    """Decode pass (query prep + split-K) on another decode workload; inputs drawn on the device."""
    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache, to_device
    w = synth.workload(name)
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    nb = step_bytes(w)
    cache = PagedCache.create(w, dev)
    cache.prefill_device()
    per_cache = cache.k_pool.numel() + cache.v_pool.numel()
    nrep = max(2, math.ceil(3 * L2_BYTES / per_cache))
    pools = [(cache.k_pool, cache.v_pool)] + [(cache.k_pool.clone(), cache.v_pool.clone())
                                              for _ in range(nrep - 1)]
    q = to_device(synth.queries(w), w.dtype, dev)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=dev)
    max_ctx = max(w.ctx_lens)
    ws = torch.empty(tq.decode_workspace_bytes(d, B, Hq, max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        """One decode call (tq_decode_attn: query prep, then the pass and its merge)."""
        kp, vp = pools[i % nrep]
        tq.decode_attn(cache.params, d, q, Hkv, kp, vp, cache.block_table, ctx, max_ctx, out=out, workspace=ws,
                       status=status)

    def stage_step(i, ev):
        """The same work through the stage calls, with events around the pass (and its merge)."""
        kp, vp = pools[i % nrep]
        tq.decode_qprep(cache.params, d, q, Hkv, ctx, max_ctx, ws)
        ev[0].record(stream)
        tq.decode_splitk(cache.params, d, B, Hq, Hkv, kp, vp, cache.block_table, ctx, max_ctx, out, ws,
                         status=status)
        ev[1].record(stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    run_ahead(dev, steps, lambda i: stage_step(i, kev[i]))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in {name}")
    ms = e0.elapsed_time(e1) / steps
    kms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    peak, _ = measured_peak()
    res = {"config": workload_config(w, f"{nrep} cache copies cycled ({nrep * per_cache / 2**20:.0f} MiB > L2)"),
           "value": round(nb["step"] / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms, 6),
           "steps": steps, "warmup": warmup, "launches_per_step": 3,
           "roofline": {"bound": "hbm", "kernel": "tq_decode_splitk", "kernel_ms": round(kms, 6),
                        "achieved": round(nb["partial"] / (kms * 1e-3) / 1e9, 3), "peak": peak, "unit": "GB/s",
                        "frac": round(nb["partial"] / (kms * 1e-3) / 1e9 / peak, 4),
                        "bytes_per_launch": nb["partial"]}}
    del pools, cache
    torch.cuda.empty_cache()
    return res


def extra_verify(steps, warmup, dev, q_len=2):
    """Speculative verify on the llama8b_decode shape: every sequence appends q_len draft tokens and
    verifies them with q_len causal queries in one tq_decode_step_mq (one read of the cache)."""
    import dataclasses

    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache
    w0 = synth.workload("llama8b_decode")
    w = dataclasses.replace(w0, prefill_lens=[L - q_len for L in w0.ctx_lens])
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    cache = PagedCache.create(w, dev)
    cache.prefill_device()
    per_cache = cache.k_pool.numel() + cache.v_pool.numel()
    nrep = max(2, math.ceil(3 * L2_BYTES / per_cache))
    pools = [(cache.k_pool, cache.v_pool)] + [(cache.k_pool.clone(), cache.v_pool.clone())
                                              for _ in range(nrep - 1)]
    g = torch.Generator(device=dev).manual_seed(1234)
    k_new = torch.randn((B, q_len, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn((B, q_len, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn((B, q_len, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    pre = torch.tensor(w.prefill_lens, dtype=torch.int32, device=dev)
    max_ctx = max(w.ctx_lens)
    ws = torch.empty(tq.decode_workspace_bytes_mq(d, B, q_len, Hq, max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty((B, q_len, Hq, d), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        kp, vp = pools[i % nrep]
        tq.decode_step_mq(cache.params, d, k_new, v_new, q, Hkv, kp, vp, cache.block_table, pre, max_ctx, out=out,
                          workspace=ws, status=status)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    ms = timed_batches(dev, steps, step)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the verify step")
    nb = step_bytes(w0)
    krec, vrec = (8 * d + 64) / 16, (6 * d + 32) / 16
    step_b = nb["partial"] + q_len * (nb["q"] + nb["out"]) + q_len * B * Hkv * (2 * d * 2 + krec + vrec)
    res = {"config": {"workload": "llama8b_verify", "batch": B, "q_len": q_len, "n_q_heads": Hq, "n_kv_heads": Hkv,
                      "head_dim": d, "ctx": max_ctx, "drafts_appended_per_step": q_len,
                      "l2": f"{nrep} cache copies cycled ({nrep * per_cache / 2**20:.0f} MiB > L2)"},
           "value": round(step_b / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
           "queries_per_s": round(B * q_len * Hq / (ms * 1e-3), 1), "ms_per_step": round(ms, 6),
           "steps": steps, "warmup": warmup, "launches_per_step": 3,
           "timing": "batches of 100 steps queued behind a spin kernel, one event pair per batch"}
    del pools, cache
    torch.cuda.empty_cache()
    return res


def extra_dequant(steps, warmup, dev):
    """Bulk dequantisation of the prefill workload's cache (8 x 32768 tokens x 8 kv heads, d=128)
    back to dense bf16 K and V: the input of a chunked prefill over a compressed prefix."""
    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache
    w = synth.workload("prefill")
    d, Hkv = w.head_dim, w.n_kv_heads
    cache = PagedCache.create(w, dev)
    cache.prefill_device()
    ids = torch.cat([cache.block_table[b, :w.prefill_lens[b] // 16] for b in range(w.batch)]).contiguous()
    n = ids.numel()
    ko = torch.empty((n * 16, Hkv, d), dtype=torch.bfloat16, device=dev)
    vo = torch.empty_like(ko)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tq.dequant_k(cache.params, d, cache.k_pool, ids, out=ko, status=status)
        if ev is not None:
            ev[1].record(stream)
        tq.dequant_v(cache.params, d, cache.v_pool, ids, out=vo, status=status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the dequantisation")
    ms = statistics.mean(a.elapsed_time(c) for a, _, c in evs)
    kms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    vms = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    ntok = n * 16
    krec, vrec = (8 * d + 64) / 16, (6 * d + 32) / 16
    kbytes = ntok * Hkv * (krec + d * 2) + n * 4
    vbytes = ntok * Hkv * (vrec + d * 2) + n * 4
    peak, _ = measured_peak()
    res = {"config": {"workload": "prefill_dequant", "sequences": w.batch, "tokens_per_sequence": w.prefill_lens[0],
                      "n_kv_heads": Hkv, "head_dim": d, "out_dtype": "bf16",
                      "l2": f"records {(cache.k_pool.numel() + cache.v_pool.numel()) / 2**20:.0f} MiB in, "
                            f"{2 * ko.numel() * 2 / 2**20:.0f} MiB out (> L2)"},
           "value": round(ntok / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s",
           "gbs": round((kbytes + vbytes) / (ms * 1e-3) / 1e9, 3), "ms_per_step": round(ms, 6),
           "steps": steps, "warmup": warmup, "launches_per_step": 2,
           "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s",
                        "k": {"kernel_ms": round(kms, 6), "achieved": round(kbytes / (kms * 1e-3) / 1e9, 3),
                              "frac": round(kbytes / (kms * 1e-3) / 1e9 / peak, 4), "bytes_per_launch": kbytes},
                        "v": {"kernel_ms": round(vms, 6), "achieved": round(vbytes / (vms * 1e-3) / 1e9, 3),
                              "frac": round(vbytes / (vms * 1e-3) / 1e9 / peak, 4), "bytes_per_launch": vbytes}}}
    del ko, vo, cache
    torch.cuda.empty_cache()
    return res


def extra_hybrid(steps, warmup, dev, history=30720, window=2048):
    """Hybrid-cache decode on the llama8b_decode head shape at 32K context: 30720 compressed tokens plus
    a 2048-token bf16 window of the most recent ones, one softmax over both (tq_decode_attn_hybrid)."""
    import dataclasses

    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache, to_device
    w0 = synth.workload("llama8b_decode")
    w = dataclasses.replace(w0, ctx_lens=[history] * w0.batch, prefill_lens=[history] * w0.batch, append=False)
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    cache = PagedCache.create(w, dev)
    cache.prefill_device()
    per_cache = cache.k_pool.numel() + cache.v_pool.numel() + 2 * B * window * Hkv * d * 2
    nrep = max(2, math.ceil(3 * L2_BYTES / per_cache))
    g = torch.Generator(device=dev).manual_seed(4321)
    sets = []
    for r in range(nrep):
        kp, vp = (cache.k_pool, cache.v_pool) if r == 0 else (cache.k_pool.clone(), cache.v_pool.clone())
        wk = torch.randn((B, window, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
        wv = torch.randn((B, window, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
        sets.append((kp, vp, wk, wv))
    q = to_device(synth.queries(w), w.dtype, dev)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=dev)
    wl = torch.full((B,), window, dtype=torch.int32, device=dev)
    ws = torch.empty(int(tq.load_library().tq_decode_workspace_bytes_hybrid(d, B, Hq, history, window)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        kp, vp, wk, wv = sets[i % nrep]
        tq.decode_attn_hybrid(cache.params, d, q, Hkv, kp, vp, cache.block_table, ctx, history, wk, wv, wl, out=out,
                              workspace=ws, status=status)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the hybrid decode")
    ms = e0.elapsed_time(e1) / steps
    # the window upkeep (tq_hybrid_append): every call finds the windows full, moves each sequence's
    # oldest window token into the compressed history and writes a new token.  The history restarts
    # 256 tokens short of the table's end so that every moved token has a block.
    usteps = min(steps, 200)
    kn = torch.randn((B, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
    vn = torch.randn((B, Hkv, d), generator=g, device=dev).to(torch.bfloat16)
    uctx = torch.full((B,), history - 256, dtype=torch.int32, device=dev)
    uwl = torch.full((B,), window, dtype=torch.int32, device=dev)
    scratch = torch.empty(int(tq.load_library().tq_hybrid_append_scratch_bytes(d, B, Hkv, tq.DTYPE_BF16)),
                          dtype=torch.uint8, device=dev)
    kp0, vp0, wk0, wv0 = sets[0]
    for _ in range(min(warmup, 10)):
        tq.hybrid_append(cache.params, d, kn, vn, wk0, wv0, uwl, cache.block_table, uctx, kp0, vp0, scratch=scratch,
                         status=status)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(usteps):
        tq.hybrid_append(cache.params, d, kn, vn, wk0, wv0, uwl, cache.block_table, uctx, kp0, vp0, scratch=scratch,
                         status=status)
    u1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the hybrid upkeep")
    ums_loop = u0.elapsed_time(u1) / usteps
    # The same calls replayed from a CUDA graph: the device time of the upkeep without the
    # per-call Python and launch overhead of the loop above (a call's kernels take less time than
    # the interpreter needs to issue it).  Each replay restores the lengths first.
    ncap = 50
    uctx0 = torch.full((B,), history - 256, dtype=torch.int32, device=dev)
    uwl0 = torch.full((B,), window, dtype=torch.int32, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        uctx.copy_(uctx0)
        uwl.copy_(uwl0)
        for _ in range(ncap):
            tq.hybrid_append(cache.params, d, kn, vn, wk0, wv0, uwl, cache.block_table, uctx, kp0, vp0,
                             scratch=scratch, status=status)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    nrp = max(1, usteps // ncap)
    u0.record(stream)
    for _ in range(nrp):
        graph.replay()
    u1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the hybrid upkeep (graph)")
    ums = u0.elapsed_time(u1) / (nrp * ncap)
    nb = step_bytes(w)
    win_b = 2 * B * window * Hkv * d * 2
    step_b = nb["partial"] + win_b + nb["q"] + nb["out"]
    res = {"config": {"workload": "llama8b_hybrid32k", "batch": B, "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": d,
                      "compressed_tokens": history, "window_tokens": window, "window_dtype": "bf16",
                      "l2": f"{nrep} copies of cache and window cycled ({nrep * per_cache / 2**20:.0f} MiB > L2)"},
           "value": round(step_b / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms, 6),
           "bytes_per_step": {"compressed": nb["partial"], "window": win_b},
           "steps": steps, "warmup": warmup, "launches_per_step": 5,
           "upkeep": {"call": "tq_hybrid_append", "us_per_call": round(ums * 1e3, 3),
                      "timing": f"{nrp} replays of a CUDA graph of {ncap} calls (the device time per call)",
                      "us_per_call_python_loop": round(ums_loop * 1e3, 3), "calls": usteps,
                      "launches_per_call": 2,
                      "per_call": f"{B * Hkv} K and {B * Hkv} V vectors leave the windows and are encoded; "
                                  f"{B} new tokens written"}}
    del sets, cache
    torch.cuda.empty_cache()
    return res


def extra_encode(steps, warmup, dev, cpu=False, name="prefill"):
    """Bulk encode of a prefill workload into paged storage: "prefill" (8 x 32768 tokens x 8 kv heads,
    d=128, bf16) or "prefill256" (4 x 32768 tokens x 8 kv heads, d=256, bf16, lognormal K scales); with
    cpu, the oracle's encode rate on the host cores beside it."""
    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache
    w = synth.workload(name)
    d, Hkv = w.head_dim, w.n_kv_heads
    cache = PagedCache.create(w, dev)
    ntok = sum(w.prefill_lens)
    Ks, Vs, slots = [], [], []
    for b in range(w.batch):
        K, V = synth.kv_tokens_device(w, b, 0, w.prefill_lens[b], dev)
        Ks.append(K)
        Vs.append(V)
        slots.append(torch.from_numpy(synth.slots_for(cache.block_table_np, b, 0, w.prefill_lens[b])))
    K = torch.cat(Ks)
    V = torch.cat(Vs)
    del Ks, Vs
    sl = torch.cat(slots).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tq.encode_k(cache.params, d, K, sl, cache.k_pool, status=status)
        if ev is not None:
            ev[1].record(stream)
        tq.encode_v(cache.params, d, V, sl, cache.v_pool, status=status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the encode")
    ms = statistics.mean(a.elapsed_time(c) for a, _, c in evs)
    kms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    vms = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    in_b = 2 if w.dtype == "bf16" else 4
    krec, vrec = (8 * d + 64) / 16, (6 * d + 32) / 16
    kbytes = ntok * Hkv * (d * in_b + krec)
    vbytes = ntok * Hkv * (d * in_b + vrec)
    peak, _ = measured_peak()
    res = {"config": {"workload": w.name, "sequences": w.batch, "tokens_per_sequence": w.prefill_lens[0],
                      "n_kv_heads": Hkv, "head_dim": d, "kv_dtype_in": w.dtype, "k_scales": w.k_scale,
                      "l2": f"inputs {(K.numel() + V.numel()) * in_b / 2**20:.0f} MiB > L2, no flush needed"},
           "value": round(ntok / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s",
           "gbs": round((kbytes + vbytes) / (ms * 1e-3) / 1e9, 3), "ms_per_step": round(ms, 6),
           "steps": steps, "warmup": warmup, "launches_per_step": 2,
           "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s",
                        "k": {"kernel_ms": round(kms, 6), "achieved": round(kbytes / (kms * 1e-3) / 1e9, 3),
                              "frac": round(kbytes / (kms * 1e-3) / 1e9 / peak, 4), "bytes_per_launch": kbytes},
                        "v": {"kernel_ms": round(vms, 6), "achieved": round(vbytes / (vms * 1e-3) / 1e9, 3),
                              "frac": round(vbytes / (vms * 1e-3) / 1e9 / peak, 4), "bytes_per_launch": vbytes}}}
    del K, V, cache
    torch.cuda.empty_cache()
    if cpu:
        tps, dt, sample = run_cpu_encode(w)
        res["cpu_baseline"] = {"value": round(tps / 1e6, 6), "unit": "Mtok/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
                               "kind": "oracle", "sample": sample, "seconds": round(dt, 3),
                               "single_thread": oracle_single_thread("encode")}
    return res


def extra_gq(steps, warmup, dev, group=64):
    """Fidelity comparator on the llama8b_decode shape (every sequence at 4096 tokens): the same
    bf16 K / V encoded by TurboQuant and by 4- and 8-bit group quantisation; for each, the decode
    attention's cosine similarity to dense fp32 attention over the uncompressed K / V (information,
    per (sequence, query head)), and the group-quantised decode's time over its own cache bytes."""
    import torch

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache, to_device
    w = synth.workload("llama8b_decode")
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    G, L = Hq // Hkv, max(w.ctx_lens)
    cache = PagedCache.create(w, dev)
    nblk = cache.num_blocks
    gk = {bits: tq.gq_empty_pool(nblk, Hkv, d, bits, group, dev) for bits in (4, 8)}
    gv = {bits: tq.gq_empty_pool(nblk, Hkv, d, bits, group, dev) for bits in (4, 8)}
    Kd = torch.empty((B, L, Hkv, d), dtype=torch.bfloat16, device=dev)
    Vd = torch.empty_like(Kd)
    for b in range(B):
        K, V = synth.kv_tokens_device(w, b, 0, L, dev)
        Kd[b], Vd[b] = K, V
        slots = torch.from_numpy(synth.slots_for(cache.block_table_np, b, 0, L)).to(dev)
        tq.encode_k(cache.params, d, K, slots, cache.k_pool)
        tq.encode_v(cache.params, d, V, slots, cache.v_pool)
        for bits in (4, 8):
            tq.gq_encode(d, bits, group, K, slots, gk[bits])
            tq.gq_encode(d, bits, group, V, slots, gv[bits])
    q = to_device(synth.queries(w), w.dtype, dev)
    ctx = torch.full((B,), L, dtype=torch.int32, device=dev)
    qf = q.float().view(B, Hkv, G, d)
    p = torch.softmax(torch.einsum("bhgd,blhd->bhgl", qf, Kd.float()) / math.sqrt(d), -1)
    ref = torch.einsum("bhgl,blhd->bhgd", p, Vd.float()).reshape(B, Hq, d).double()
    del p, Kd, Vd

    def fidelity(o):
        c = torch.nn.functional.cosine_similarity(o.double(), ref, dim=-1)
        return {"cos_mean": round(float(c.mean()), 6), "cos_min": round(float(c.min()), 6)}

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = tq.decode_attn(cache.params, d, q, Hkv, cache.k_pool, cache.v_pool, cache.block_table, ctx, L,
                         status=status)
    kb, vb = tq.k_record_bytes(d), tq.v_record_bytes(d)
    res = {"config": {"workload": "gq_compare", "batch": B, "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": d,
                      "ctx": L, "group": group, "reference": "dense fp32 attention over the bf16 K / V",
                      "k_scales": w.k_scale},
           "turboquant": {"bits_per_dim": round((kb + vb) * 8 / (2 * 16 * d), 4), **fidelity(out)}}
    # the same comparison with plain N(0,1) keys (no channel scales), information only
    wn = dataclasses.replace(w, k_scale="none")
    Kn = torch.empty((B, L, Hkv, d), dtype=torch.bfloat16, device=dev)
    Vn = torch.empty_like(Kn)
    kpn, vpn = torch.zeros_like(cache.k_pool), torch.zeros_like(cache.v_pool)
    gkn = {bits: tq.gq_empty_pool(nblk, Hkv, d, bits, group, dev) for bits in (4, 8)}
    gvn = {bits: tq.gq_empty_pool(nblk, Hkv, d, bits, group, dev) for bits in (4, 8)}
    for b in range(B):
        K, V = synth.kv_tokens_device(wn, b, 0, L, dev)
        Kn[b], Vn[b] = K, V
        slots = torch.from_numpy(synth.slots_for(cache.block_table_np, b, 0, L)).to(dev)
        tq.encode_k(cache.params, d, K, slots, kpn)
        tq.encode_v(cache.params, d, V, slots, vpn)
        for bits in (4, 8):
            tq.gq_encode(d, bits, group, K, slots, gkn[bits])
            tq.gq_encode(d, bits, group, V, slots, gvn[bits])
    pn = torch.softmax(torch.einsum("bhgd,blhd->bhgl", qf, Kn.float()) / math.sqrt(d), -1)
    refn = torch.einsum("bhgl,blhd->bhgd", pn, Vn.float()).reshape(B, Hq, d).double()
    del pn, Kn, Vn

    def fid_n(o):
        c = torch.nn.functional.cosine_similarity(o.double(), refn, dim=-1)
        return {"cos_mean": round(float(c.mean()), 6), "cos_min": round(float(c.min()), 6)}

    on = tq.decode_attn(cache.params, d, q, Hkv, kpn, vpn, cache.block_table, ctx, L, status=status)
    res["fidelity_n01_keys"] = {"turboquant": fid_n(on)}
    for bits in (4, 8):
        og = tq.gq_decode_attn(d, bits, group, q, Hkv, gkn[bits], gvn[bits], cache.block_table, ctx, L,
                               status=status)
        res["fidelity_n01_keys"][f"gq{bits}"] = fid_n(og)
    del kpn, vpn, gkn, gvn, refn
    bt = cache.block_table
    del cache
    stream = torch.cuda.current_stream()
    peak, _ = measured_peak()
    for bits in (4, 8):
        per_cache = gk[bits].numel() + gv[bits].numel()
        nrep = max(2, math.ceil(3 * L2_BYTES / per_cache))
        pools = [(gk[bits], gv[bits])] + [(gk[bits].clone(), gv[bits].clone()) for _ in range(nrep - 1)]
        ws = torch.empty(tq.gq_decode_workspace_bytes(d, B, Hq, Hkv, L), dtype=torch.uint8, device=dev)
        o = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)

        def step(i):
            kp, vp = pools[i % nrep]
            tq.gq_decode_attn(d, bits, group, q, Hkv, kp, vp, bt, ctx, L, out=o, workspace=ws, status=status)

        for i in range(warmup):
            step(i)
        torch.cuda.synchronize(dev)
        fid = fidelity(o)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        nbytes = B * L * Hkv * 2 * tq.gq_record_bytes(d, bits, group) / 16
        res[f"gq{bits}"] = {"bits_per_dim": tq.gq_record_bytes(d, bits, group) * 8 / (16 * d), **fid,
                            "ms_per_step": round(ms, 6), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 3),
                            "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "launches_per_step": 2,
                            "l2": f"{nrep} cache copies cycled ({nrep * per_cache / 2**20:.0f} MiB > L2)"}
        del pools, ws
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in gq_compare")
    torch.cuda.empty_cache()
    return res


def bench_tq(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import turboquant_compressed_kv_gb300 as tq
    from turboquant_compressed_kv_gb300 import synth
    from turboquant_compressed_kv_gb300.cache import PagedCache, to_device

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tq.load_library()

    w = synth.workload(WORKLOAD)
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    nb = step_bytes(w)
    cache = PagedCache.create(w, dev)
    cache.prefill()
    # Cycle through enough identical cache copies that a step's reads miss L2.
    per_cache = cache.k_pool.numel() + cache.v_pool.numel()
    nrep = max(2, math.ceil(3 * L2_BYTES / per_cache))
    pools = [(cache.k_pool, cache.v_pool)] + [(cache.k_pool.clone(), cache.v_pool.clone())
                                              for _ in range(nrep - 1)]
    K1, V1 = cache.append_inputs()
    q_np = synth.queries(w)
    k_new = to_device(K1, w.dtype, dev)
    v_new = to_device(V1, w.dtype, dev)
    q = to_device(q_np, w.dtype, dev)
    pre = torch.tensor(w.prefill_lens, dtype=torch.int32, device=dev)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=dev)
    max_ctx = max(w.ctx_lens)
    ws = torch.empty(tq.decode_workspace_bytes(d, B, Hq, max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    launches_per_step = 3          # tq_decode_step: append + query prep in one launch, the split-K pass, its merge

    def step(i):
        kp, vp = pools[i % nrep]
        tq.decode_step(cache.params, d, k_new, v_new, q, Hkv, kp, vp, cache.block_table, pre, max_ctx, out=out,
                       workspace=ws, status=status)

    def stage_step(i, ev):
        """The same work through the stage calls, with events around each: the append, the query prep
        and the split-K kernel."""
        kp, vp = pools[i % nrep]
        ev[2].record(stream)
        tq.paged_append(cache.params, d, k_new, v_new, cache.block_table, pre, kp, vp, status=status)
        ev[3].record(stream)
        tq.decode_qprep(cache.params, d, q, Hkv, ctx, max_ctx, ws)
        ev[0].record(stream)
        tq.decode_splitk(cache.params, d, B, Hq, Hkv, kp, vp, cache.block_table, ctx, max_ctx, out, ws,
                         status=status)
        ev[1].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        step(i)
    barrier()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    # device-time loop: K steps between one event pair
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    barrier()
    t_wall1 = time.time()
    total_ms = e0.elapsed_time(e1)
    # the dominant kernel: the split-K pass, timed by events on the launching stream over K steps
    kev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    run_ahead(dev, args.steps, lambda i: stage_step(i, kev[i]))
    barrier()
    kern_ms = [e[0].elapsed_time(e[1]) for e in kev]
    append_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in kev)
    qprep_ms = statistics.mean(e[3].elapsed_time(e[0]) for e in kev)
    # keep the GPU busy a little longer so the sampler sees the loaded clocks
    t_c0 = time.time()
    while time.time() - t_c0 < 1.0:
        for i in range(50):
            step(i)
        torch.cuda.synchronize(dev)
    t_c1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.15, t_c1)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the bench")

    # end-to-end through the public API with pinned host buffers.  The step's inputs (q, new K, new V)
    # sit in one pinned buffer and go over in one copy; the output comes back in one copy.  As a
    # serving loop would, uploads and downloads run on their own streams with double buffers, so
    # that step i's download and step i+1's upload overlap the kernels (every step makes both).
    assert q.dtype == k_new.dtype == v_new.dtype
    nq, nk = q.numel(), k_new.numel()
    hin = torch.empty(nq + 2 * nk, dtype=q.dtype).pin_memory()
    hin[:nq].copy_(torch.from_numpy(np.ascontiguousarray(q_np)).reshape(-1).to(q.dtype))
    hin[nq:nq + nk].copy_(torch.from_numpy(np.ascontiguousarray(K1)).reshape(-1).to(q.dtype))
    hin[nq + nk:].copy_(torch.from_numpy(np.ascontiguousarray(V1)).reshape(-1).to(q.dtype))
    hout = [torch.empty((B, Hq, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    din = [torch.empty(hin.shape, dtype=hin.dtype, device=dev) for _ in range(2)]
    views = [(x[:nq].view(q.shape), x[nq:nq + nk].view(k_new.shape), x[nq + nk:].view(v_new.shape)) for x in din]
    dout = [torch.empty((B, Hq, d), dtype=torch.float32, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        kp, vp = pools[i % nrep]
        b = i & 1
        with torch.cuda.stream(up):        # upload, once step i-2 has read this buffer
            up.wait_event(ev_done[b])
            din[b].copy_(hin, non_blocking=True)
            ev_up[b].record(up)
        stream.wait_event(ev_up[b])
        stream.wait_event(ev_down[b])      # step i-2's output has gone back
        dq, dk, dv = views[b]
        tq.decode_step(cache.params, d, dk, dv, dq, Hkv, kp, vp, cache.block_table, pre, max_ctx, out=dout[b],
                       workspace=ws)
        ev_done[b].record(stream)
        with torch.cuda.stream(down):      # download of this step's output
            down.wait_event(ev_done[b])
            hout[b].copy_(dout[b], non_blocking=True)
            ev_down[b].record(down)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_s = (time.perf_counter() - t0) / args.steps
    h2d = hin.numel() * hin.element_size()
    d2h = hout[0].numel() * 4

    total_ms, e2e_s = max_over_ranks([total_ms, e2e_s], world, dev)
    ms_step = total_ms / args.steps
    value = job_gbs(world, nb["step"], ms_step * 1e-3)
    e2e_value = job_gbs(world, nb["step"], e2e_s)

    kern_avg_ms = statistics.mean(kern_ms)
    achieved = nb["partial"] / (kern_avg_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = profile_traffic(nb["partial"])

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16/f32", "data": "synthetic",
        "arithmetic": ("mixed: mma.sync f16 x f16 with fp32 accumulation; codebook operands are f16 table values "
                       "alpha c[j], the query (qbar/alpha, QJL-scaled u) and the softmax weights enter as f16 hi+lo "
                       "pairs (one f16 above 4 heads); norms fp16 as stored; softmax, value sums, merge and the "
                       "inverse rotation in fp32"),
        "config": workload_config(w, f"{nrep} cache copies cycled ({nrep * per_cache / 2**20:.0f} MiB > L2), "
                                     "no flush needed"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 3), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "decode split-K pass with merge (tq_decode_splitk)", "peak_source": peak_kind,
                     "kernel_ms": round(kern_avg_ms, 6), "bytes_per_launch": nb["partial"]},
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "stages_ms": {"append": round(append_ms, 6), "qprep": round(qprep_ms, 6), "splitk": round(kern_avg_ms, 6),
                      "note": "each stage through its own entry point, timed by events on the stream; the step "
                              "fuses the append with the query prep and overlaps the pass's launch"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                   "samples": clocks["samples"]},
        "bytes_per_step": nb,
    }
    if not args.main_only:
        ksteps = max(3, min(args.steps, 200))
        line["workloads"] = {"ragged": extra_decode("ragged", ksteps, max(3, args.warmup), dev),
                             "long256": extra_decode("long256", ksteps, max(3, args.warmup), dev),
                             "verify_q2": extra_verify(ksteps, max(3, args.warmup), dev),
                             "hybrid32k": extra_hybrid(ksteps, max(3, args.warmup), dev),
                             "prefill_encode": extra_encode(max(3, min(args.steps, 50)), max(3, args.warmup), dev,
                                                            cpu=rank == 0 and world == 1 and not args.no_cpu_baseline),
                             "prefill_encode256": extra_encode(max(3, min(args.steps, 50)), max(3, args.warmup),
                                                               dev, name="prefill256"),
                             "prefill_dequant": extra_dequant(max(3, min(args.steps, 50)), max(3, args.warmup), dev),
                             "gq_compare": extra_gq(max(3, min(args.steps, 100)), max(3, args.warmup), dev)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, dt, _ = run_cpu_oracle(w, 3, 1, 2)
        line["cpu_baseline"] = {"value": round(gbs, 6), "unit": "GB/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
                                "kind": "oracle",
                                "sample": "2 of 16 sequences, full step (append + decode of 32 heads over 4096 "
                                          "tokens), 3 timed repetitions",
                                "single_thread": oracle_single_thread("decode")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def side_workload(args):
    import torch

    import turboquant_compressed_kv_gb300 as tq
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    tq.load_library()
    steps, warmup = max(1, args.steps), max(1, args.warmup)
    runs = {"ragged": lambda: extra_decode("ragged", steps, warmup, dev),
            "long256": lambda: extra_decode("long256", steps, warmup, dev),
            "verify_q2": lambda: extra_verify(steps, warmup, dev),
            "hybrid32k": lambda: extra_hybrid(steps, warmup, dev),
            "prefill_encode": lambda: extra_encode(steps, warmup, dev),
            "prefill_encode256": lambda: extra_encode(steps, warmup, dev, name="prefill256"),
            "prefill_dequant": lambda: extra_dequant(steps, warmup, dev),
            "gq_compare": lambda: extra_gq(steps, warmup, dev)}
    if args.workload not in runs:
        raise SystemExit(f"unknown workload {args.workload}; one of {sorted(runs)}")
    print(json.dumps({"workload": args.workload, **runs[args.workload]()}), flush=True)
    return 0


def oracle_single_thread(kind):
    """The oracle on one host thread, in a child process started with OMP_NUM_THREADS=1 (the thread
    count is fixed when the oracle's OpenMP runtime loads); None if the child fails."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread", kind], env=env,
                           capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def oracle_single_thread_child(kind):
    from turboquant_compressed_kv_gb300 import synth
    if kind == "decode":
        gbs, dt, _ = run_cpu_oracle(synth.workload(WORKLOAD), 1, 0, 1)
        res = {"value": round(gbs, 6), "unit": "GB/s", "cores": 1,
               "sample": "1 of 16 sequences, full step (append + decode of 32 heads over 4096 tokens), one timed pass",
               "seconds": round(dt, 3)}
    else:
        tps, dt, sample = run_cpu_encode(synth.workload("prefill"), ntok=512)
        res = {"value": round(tps / 1e6, 6), "unit": "Mtok/s", "cores": 1, "sample": sample, "seconds": round(dt, 3)}
    print(json.dumps(res), flush=True)
    return 0


def main():
    args = parse()
    if args.oracle_single_thread:
        return oracle_single_thread_child(args.oracle_single_thread)
    if args.impl == "reference":
        return bench_reference(args)
    if args.workload:
        return side_workload(args)
    return bench_tq(args)


if __name__ == "__main__":
    sys.exit(main())
