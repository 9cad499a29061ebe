"""Oracle of the group-quantised KV comparator (numpy).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline may use it, and it
never imports the CUDA library.

Source: SwiftLM README, "Per-Request API Parameters" -- ``kv_bits`` (4 or 8)
turns on MLX-native standard group quantization of the KV cache from token 0,
``kv_group_size`` (default 64) is its group, and the comparison table puts its
saving at "~2-4x vs FP16"; lilting.ch, "TurboQuant V2+V3ハイブリッド実装": the V2
route is linear (affine) quantization.  The pages print no formula; the reading
taken is plain min-max affine quantization per group:

  scale = fp16((max - min) / (2^bits - 1)),   bias = fp16(min),
  code  = clamp(rint((x - bias) / scale), 0, 2^bits - 1)   (0 when scale == 0),
  x~    = scale * code + bias.

The code is an integer decided by floating point, so it is taken in fp32 with
round-to-nearest-even at every step, the precision the kernel uses.  Decoding
and attention are fp64.

Record of one (block, kv head), 16 slots (this library's layout):
  codes  [16][d * bits / 8]   4-bit: coordinate 2j in the low nibble of byte j
  params [16][d / group][2]   fp16 scale, fp16 bias (little-endian)
"""
from __future__ import annotations

import numpy as np

BLOCK = 16


def record_bytes(d: int, bits: int, group: int) -> int:
    return BLOCK * (d * bits // 8 + 4 * (d // group))


def encode(x, bits: int, group: int):
    """x [..., d] -> (codes uint8 [..., d], scale fp16 bits uint16 [..., d/group], bias uint16)."""
    x = np.asarray(x, np.float32)
    d = x.shape[-1]
    xg = x.reshape(x.shape[:-1] + (d // group, group))
    top = np.float32(2 ** bits - 1)
    lo = xg.min(-1)
    hi = xg.max(-1)
    scale = ((hi - lo) / top).astype(np.float16)          # fp32 subtract, fp32 divide, fp16 round
    bias = lo.astype(np.float16)
    sf = scale.astype(np.float32)[..., None]
    zf = bias.astype(np.float32)[..., None]
    pos = sf > 0
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = np.where(pos, (xg - zf) / np.where(pos, sf, np.float32(1)), np.float32(0))
    codes = np.fmin(np.fmax(np.rint(q), np.float32(0)), top).astype(np.uint8)
    return codes.reshape(x.shape), scale.view(np.uint16), bias.view(np.uint16)


def decode_values(codes, scale16, bias16, group: int) -> np.ndarray:
    """x~ = scale * code + bias in fp64, shape of codes."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    s = np.asarray(scale16, np.uint16).view(np.float16).astype(np.float64)
    z = np.asarray(bias16, np.uint16).view(np.float16).astype(np.float64)
    cg = codes.reshape(codes.shape[:-1] + (d // group, group)).astype(np.float64)
    return (cg * s[..., None] + z[..., None]).reshape(codes.shape)


def pack(codes, scale16, bias16, slots, pool: np.ndarray, H: int, bits: int, group: int) -> None:
    """Write (codes [N][H][d], scale16 / bias16 [N][H][d/group]) into slot slots[n] of pool
    (uint8, num_blocks * H * record_bytes, modified in place).  Negative slots are skipped."""
    codes = np.asarray(codes, np.uint8)
    N, _, d = codes.shape
    ng = d // group
    cb = d * bits // 8
    rec = record_bytes(d, bits, group)
    flat = pool.reshape(-1)
    for n in range(N):
        slot = int(slots[n])
        if slot < 0:
            continue
        blk, off = divmod(slot, BLOCK)
        for h in range(H):
            base = (blk * H + h) * rec
            c = codes[n, h].astype(np.uint8)
            if bits == 8:
                row = c
            else:
                row = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
            flat[base + off * cb: base + (off + 1) * cb] = row
            for g in range(ng):
                p = base + BLOCK * cb + (off * ng + g) * 4
                flat[p: p + 2] = np.array([scale16[n, h, g]], np.uint16).view(np.uint8)
                flat[p + 2: p + 4] = np.array([bias16[n, h, g]], np.uint16).view(np.uint8)


def unpack(pool: np.ndarray, d: int, H: int, bits: int, group: int, slots):
    """Inverse of pack for the given slots: (codes [N][H][d], scale16, bias16 [N][H][d/group])."""
    ng = d // group
    cb = d * bits // 8
    rec = record_bytes(d, bits, group)
    flat = np.asarray(pool, np.uint8).reshape(-1)
    N = len(slots)
    codes = np.zeros((N, H, d), np.uint8)
    s16 = np.zeros((N, H, ng), np.uint16)
    z16 = np.zeros((N, H, ng), np.uint16)
    for n, slot in enumerate(slots):
        blk, off = divmod(int(slot), BLOCK)
        for h in range(H):
            base = (blk * H + h) * rec
            row = flat[base + off * cb: base + (off + 1) * cb]
            if bits == 8:
                codes[n, h] = row
            else:
                codes[n, h, 0::2] = row & 15
                codes[n, h, 1::2] = row >> 4
            prm = flat[base + BLOCK * cb + off * ng * 4: base + BLOCK * cb + (off + 1) * ng * 4].copy().view(np.uint16)
            s16[n, h] = prm[0::2]
            z16[n, h] = prm[1::2]
    return codes, s16, z16


def attention(q, K, V) -> np.ndarray:
    """Textbook attention of one query row over rows K, V (fp64): softmax(K q / sqrt d) V."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    if len(K) == 0:
        return np.zeros(q.shape[-1])
    s = K @ q / np.sqrt(q.shape[-1])
    p = np.exp(s - s.max())
    return (p[:, None] * V).sum(0) / p.sum()


def decode(q, Hkv: int, kpool, vpool, block_table, ctx_lens, bits: int, group: int) -> np.ndarray:
    """Decode attention over the group-quantised paged pools: query head h of sequence b
    attends its ctx_lens[b] tokens (token j in block block_table[b][j // 16], slot j % 16)
    of kv head h // (Hq / Hkv) through the decoded keys and values.  out [B][Hq][d] fp64."""
    q = np.asarray(q, np.float64)
    B, Hq, d = q.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, d), np.float64)
    bt = np.asarray(block_table)
    for b in range(B):
        L = max(0, int(ctx_lens[b]))
        if L == 0:
            continue
        j = np.arange(L)
        slots = bt[b, j // BLOCK].astype(np.int64) * BLOCK + j % BLOCK
        K = decode_values(*unpack(kpool, d, Hkv, bits, group, slots), group)
        V = decode_values(*unpack(vpool, d, Hkv, bits, group, slots), group)
        for h in range(Hq):
            out[b, h] = attention(q[b, h], K[:, h // G], V[:, h // G])
    return out
