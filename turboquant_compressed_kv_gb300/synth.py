"""Seeded synthetic workloads shaped like the pages' KV-cache use.

This module only draws random numbers and lays out block tables; it holds
none of the compression or attention arithmetic.  Tests feed the same draws
to the CUDA library and to the fp64 oracle; the benchmark uses them to fill
device memory.

Random streams (numpy PCG64):
  * rotation sign diagonal D:   default_rng(1), D = 1 - 2*integers(0, 2, d)
  * QJL Gaussian matrix S[d,d]: default_rng(2), standard_normal, rounded to binary16 (held as fp32)
  * data: default_rng([seed, stream, index]) so that any one sequence (or
    prefill chunk) can be regenerated alone, without drawing the others.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK = 16

# ---------------------------------------------------------------- shared random matrices


def rotation_signs(d: int, seed: int = 1) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (1 - 2 * rng.integers(0, 2, d)).astype(np.int8)


def qjl_matrix(d: int, seed: int = 2) -> np.ndarray:
    """N(0,1) draws rounded to binary16 (the precision the library holds S at), as fp32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((d, d)).astype(np.float32).astype(np.float16).astype(np.float32)


# ---------------------------------------------------------------- workloads


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_lens: list          # cached tokens per sequence attended by decode
    dtype: str              # "f32" or "bf16" inputs
    k_scale: str            # "outlier20", "lognormal", "outlier10x2pct" or "none"
    prefill_lens: list      # tokens written before the timed step (decode configs)
    append: bool            # one token per sequence is appended inside the step
    contiguous: bool        # identity block table (config 1)
    pool_spare: float       # extra physical blocks, as a fraction
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def workload(name: str) -> Workload:
    """The five workloads of the pages' use case (sizes written out)."""
    if name == "tiny":        # 1 seq, 1 head, d=128, 256 tokens, fp32, channels 3,77 x20
        return Workload(name, 1, 1, 1, 128, [256], "f32", "outlier20", [256], False, True, 0.0)
    if name == "llama8b_decode":   # B16, Hq32, Hkv8, d128, ctx 4096 (4095 + 1 appended)
        return Workload(name, 16, 32, 8, 128, [4096] * 16, "bf16", "lognormal", [4095] * 16,
                        True, False, 0.0)
    if name == "ragged":      # B64, Hq32, Hkv4, d128, ctx ~ U[512, 32768]
        rng = np.random.default_rng([0, 3])
        lens = rng.integers(512, 32768 + 1, 64).tolist()
        return Workload(name, 64, 32, 4, 128, lens, "bf16", "outlier20", lens, False, False, 0.10)
    if name == "prefill":     # 8 x 32768 tokens x Hkv8 x d128, encode only
        return Workload(name, 8, 8, 8, 128, [32768] * 8, "bf16", "outlier10x2pct", [32768] * 8,
                        False, False, 0.0)
    if name == "prefill256":  # 4 x 32768 tokens x Hkv8 x d256, encode only (shaped like long256)
        return Workload(name, 4, 8, 8, 256, [32768] * 4, "bf16", "lognormal", [32768] * 4,
                        False, False, 0.0)
    if name == "long256":     # B4, Hq16, Hkv8, d256, ctx 131072
        return Workload(name, 4, 16, 8, 256, [131072] * 4, "bf16", "lognormal", [131072] * 4,
                        False, False, 0.0)
    raise KeyError(name)


WORKLOADS = ["tiny", "llama8b_decode", "ragged", "prefill", "long256", "prefill256"]


def scaled_down(w: Workload, batch: int, max_ctx: int, seed_shift: int = 0) -> Workload:
    """A smaller instance with the same structure (for parity tests)."""
    lens = [min(int(x), max_ctx) for x in w.ctx_lens[:batch]]
    pre = [min(int(x), max_ctx - (1 if w.append else 0)) for x in w.prefill_lens[:batch]]
    return dataclasses.replace(w, batch=batch, ctx_lens=lens, prefill_lens=pre,
                               name=w.name + f"_b{batch}_c{max_ctx}", seed=w.seed + seed_shift)


def k_channel_scale(w: Workload) -> np.ndarray:
    """[Hkv][d] per-channel multipliers applied to K before rounding."""
    d, H = w.head_dim, w.n_kv_heads
    s = np.ones((H, d), np.float32)
    if w.k_scale == "outlier20":
        s[:, 3] = 20.0
        s[:, 77 % d] = 20.0
    elif w.k_scale == "lognormal":
        rng = np.random.default_rng([w.seed, 11])
        s = rng.lognormal(0.0, 1.0, (H, d)).astype(np.float32)
    elif w.k_scale == "outlier10x2pct":
        rng = np.random.default_rng([w.seed, 12])
        nch = int(round(0.02 * d))
        ch = rng.choice(d, nch, replace=False)
        s[:, ch] = 10.0
    return s


def round_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the storage dtype (bf16 RNE) and return them as fp32."""
    if dtype == "f32":
        return a.astype(np.float32)
    u = a.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def kv_tokens(w: Workload, b: int, start: int, count: int):
    """K and V values of tokens [start, start+count) of sequence b: [count][Hkv][d] fp32
    (already rounded to the input dtype).  Drawn in 256-token chunks so that any
    range regenerates identically."""
    d, H = w.head_dim, w.n_kv_heads
    scale = k_channel_scale(w)
    K = np.empty((count, H, d), np.float32)
    V = np.empty((count, H, d), np.float32)
    CH = 256
    c0 = start // CH
    c1 = (start + count + CH - 1) // CH
    for c in range(c0, c1):
        rng = np.random.default_rng([w.seed, 21, b, c])
        kk = rng.standard_normal((CH, H, d), dtype=np.float32) * scale[None]
        vv = rng.standard_normal((CH, H, d), dtype=np.float32)
        lo = max(start, c * CH)
        hi = min(start + count, (c + 1) * CH)
        K[lo - start:hi - start] = kk[lo - c * CH:hi - c * CH]
        V[lo - start:hi - start] = vv[lo - c * CH:hi - c * CH]
    return round_dtype(K, w.dtype), round_dtype(V, w.dtype)


def queries(w: Workload, step: int = 0) -> np.ndarray:
    rng = np.random.default_rng([w.seed, 31, step])
    q = rng.standard_normal((w.batch, w.n_q_heads, w.head_dim), dtype=np.float32)
    return round_dtype(q, w.dtype)


def block_tables(w: Workload):
    """Returns (block_table[B][max_blocks] int32, num_blocks).

    Each sequence gets ceil(ctx/16) blocks; physical ids are a seeded random
    permutation of the pool (plus spare blocks), so consecutive logical
    blocks are scattered."""
    need = [max(1, math.ceil(L / BLOCK)) for L in w.ctx_lens]
    max_blocks = max(need)
    total = sum(need)
    num_blocks = total + int(math.ceil(total * w.pool_spare))
    if w.contiguous:
        perm = np.arange(num_blocks)
    else:
        perm = np.random.default_rng([w.seed, 41]).permutation(num_blocks)
    bt = np.zeros((w.batch, max_blocks), np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, num_blocks


def slots_for(bt: np.ndarray, b: int, start: int, count: int) -> np.ndarray:
    j = np.arange(start, start + count)
    return (bt[b, j // BLOCK].astype(np.int64) * BLOCK + (j % BLOCK)).astype(np.int64)


def kv_tokens_device(w: Workload, b: int, start: int, count: int, device):
    """K and V of tokens [start, start+count) of sequence b drawn on the device:
    the same distributions as kv_tokens (N(0,1), K times k_channel_scale,
    rounded to the input dtype), from torch's seeded CUDA generator instead of
    numpy's, so that the large throughput workloads need no host-side draws.
    Returns two tensors [count][Hkv][d] in the input dtype (bf16 or fp32).
    The values differ from kv_tokens'; tests use kv_tokens."""
    import torch
    d, H = w.head_dim, w.n_kv_heads
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 1_000_003 + b) * 1_000_003 + start) & 0x7FFFFFFFFFFFFFFF)
    scale = torch.from_numpy(k_channel_scale(w)).to(device)
    K = torch.randn((count, H, d), generator=g, device=device, dtype=torch.float32) * scale
    V = torch.randn((count, H, d), generator=g, device=device, dtype=torch.float32)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return K.to(dt), V.to(dt)
