"""fp64 CPU oracle for TurboQuant KV encode and compressed-cache decode attention.

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``tq_oracle.c`` (plain C,
fp64); this module compiles it with gcc on first use and wraps it with
ctypes/numpy.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import it; the CUDA library never
does, and this module never imports the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 16


def build(force: bool = False) -> str:
    """Compile tq_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=gnu11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
        return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def _declare(L):
    L.tqo_fp16_rne.restype = ctypes.c_uint16
    L.tqo_fp16_rne.argtypes = [ctypes.c_double]
    L.tqo_fp16_value.restype = ctypes.c_double
    L.tqo_fp16_value.argtypes = [ctypes.c_uint16]
    L.tqo_lloyd_max8.restype = _I
    L.tqo_lloyd_max8.argtypes = [_P, _P, _P]
    L.tqo_hadamard_entry.restype = _I
    L.tqo_hadamard_entry.argtypes = [_I, _I]
    L.tqo_rotate.restype = None
    L.tqo_rotate.argtypes = [_I, _P, _P, _P]
    L.tqo_rotate_t.restype = None
    L.tqo_rotate_t.argtypes = [_I, _P, _P, _P]
    L.tqo_encode_vector.restype = None
    L.tqo_encode_vector.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    L.tqo_k_record_bytes.restype = ctypes.c_size_t
    L.tqo_k_record_bytes.argtypes = [_I]
    L.tqo_v_record_bytes.restype = ctypes.c_size_t
    L.tqo_v_record_bytes.argtypes = [_I]
    L.tqo_k_bitpos.restype = None
    L.tqo_k_bitpos.argtypes = [_I, _I, _I, _I, _P, _P]
    L.tqo_v_bitpos.restype = None
    L.tqo_v_bitpos.argtypes = [_I, _I, _I, _I, _P, _P]
    L.tqo_pack_k.restype = None
    L.tqo_pack_k.argtypes = [_I, _P, _I, _P, _P, ctypes.c_uint16, ctypes.c_uint16]
    L.tqo_unpack_k.restype = None
    L.tqo_unpack_k.argtypes = [_I, _P, _I, _P, _P, _P, _P]
    L.tqo_pack_v.restype = None
    L.tqo_pack_v.argtypes = [_I, _P, _I, _P, ctypes.c_uint16]
    L.tqo_unpack_v.restype = None
    L.tqo_unpack_v.argtypes = [_I, _P, _I, _P, _P]
    L.tqo_encode.restype = _I
    L.tqo_encode.argtypes = [_I, _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I64,
                             _P, _P, _P, _P, _P, _P, _P]
    L.tqo_decode.restype = _I
    L.tqo_decode.argtypes = [_I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _P, _P]
    L.tqo_decode_explicit.restype = _I
    L.tqo_decode_explicit.argtypes = L.tqo_decode.argtypes


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars

def fp16_rne(x: float) -> int:
    return int(lib().tqo_fp16_rne(float(x)))


def fp16_value(h: int) -> float:
    return float(lib().tqo_fp16_value(int(h)))


def hadamard_entry(i: int, j: int) -> int:
    return int(lib().tqo_hadamard_entry(int(i), int(j)))


# ---------------------------------------------------------------- codebook

def lloyd_max8():
    """Returns (centroids[8], thresholds[7], mse, iterations), all fp64."""
    c = np.zeros(8, np.float64)
    t = np.zeros(7, np.float64)
    mse = np.zeros(1, np.float64)
    it = lib().tqo_lloyd_max8(_ptr(c), _ptr(t), _ptr(mse))
    return c, t, float(mse[0]), int(it)


_CB = None


def codebook():
    global _CB
    if _CB is None:
        _CB = lloyd_max8()
    return _CB


# ---------------------------------------------------------------- rotation

def rotate(D: np.ndarray, x: np.ndarray) -> np.ndarray:
    d = len(D)
    D = _c(D, np.int8)
    x = _c(x, np.float64)
    y = np.zeros(d, np.float64)
    lib().tqo_rotate(d, _ptr(D), _ptr(x), _ptr(y))
    return y


def rotate_t(D: np.ndarray, y: np.ndarray) -> np.ndarray:
    d = len(D)
    D = _c(D, np.int8)
    y = _c(y, np.float64)
    x = np.zeros(d, np.float64)
    lib().tqo_rotate_t(d, _ptr(D), _ptr(y), _ptr(x))
    return x


# ---------------------------------------------------------------- encode

def encode_vector(is_k: bool, D, S, x, codes_in=None, centroids=None, thresholds=None):
    """Encode one vector; returns dict(codes, signs, n, gamma, z, p)."""
    d = len(D)
    c, t = (centroids, thresholds) if centroids is not None else codebook()[:2]
    D = _c(D, np.int8)
    S = _c(S, np.float32)
    x = _c(x, np.float64)
    c = _c(c, np.float64)
    t = _c(t, np.float64)
    ci = None if codes_in is None else _c(codes_in, np.uint8)
    codes = np.zeros(d, np.uint8)
    signs = np.zeros(d, np.uint8)
    n = np.zeros(1)
    g = np.zeros(1)
    z = np.zeros(d)
    p = np.zeros(d)
    lib().tqo_encode_vector(int(is_k), d, _ptr(D), _ptr(S), _ptr(c), _ptr(t), _ptr(x), _ptr(ci),
                            _ptr(codes), _ptr(signs), _ptr(n), _ptr(g), _ptr(z), _ptr(p))
    return dict(codes=codes, signs=signs, n=float(n[0]), gamma=float(g[0]), z=z, p=p)


def record_bytes(is_k: bool, d: int) -> int:
    return int(lib().tqo_k_record_bytes(d) if is_k else lib().tqo_v_record_bytes(d))


def encode(is_k: bool, D, S, x: np.ndarray, slots: np.ndarray, pool: np.ndarray,
           codes_in=None, want_details=False, centroids=None, thresholds=None):
    """Encode x[N][H][d] (fp32 values) into ``pool`` (uint8, modified in place).

    pool is [num_blocks][H][record_bytes]; slots[N] = block*16 + offset.
    With want_details, returns dict(codes, signs, n, gamma, z, p) per vector.
    """
    N, H, d = x.shape
    c, t = (centroids, thresholds) if centroids is not None else codebook()[:2]
    D = _c(D, np.int8)
    S = _c(S, np.float32)
    x = _c(x, np.float32)
    slots = _c(slots, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    rec = record_bytes(is_k, d)
    assert pool.size % (H * rec) == 0
    num_blocks = pool.size // (H * rec)
    ci = None if codes_in is None else _c(codes_in, np.uint8)
    det = None
    if want_details:
        det = dict(codes=np.zeros((N, H, d), np.uint8), signs=np.zeros((N, H, d), np.uint8),
                   n=np.zeros((N, H)), gamma=np.zeros((N, H)),
                   z=np.zeros((N, H, d)), p=np.zeros((N, H, d)) if is_k else None)
    rc = lib().tqo_encode(int(is_k), d, _ptr(D), _ptr(S), _ptr(_c(c, np.float64)),
                          _ptr(_c(t, np.float64)), _ptr(x), N, H, _ptr(slots), _ptr(pool),
                          num_blocks, _ptr(ci),
                          _ptr(det["codes"]) if det else None,
                          _ptr(det["signs"]) if det else None,
                          _ptr(det["n"]) if det else None,
                          _ptr(det["gamma"]) if det else None,
                          _ptr(det["z"]) if det else None,
                          _ptr(det["p"]) if det and is_k else None)
    if rc != 0:
        raise ValueError("oracle encode: slot outside the pool")
    return det


def unpack(is_k: bool, d: int, pool: np.ndarray, H: int, slots: np.ndarray):
    """Read back codes/signs/fp16 norms for (slot, head) pairs: arrays [N][H]..."""
    rec = record_bytes(is_k, d)
    N = len(slots)
    codes = np.zeros((N, H, d), np.uint8)
    signs = np.zeros((N, H, d), np.uint8)
    n16 = np.zeros((N, H), np.uint16)
    g16 = np.zeros((N, H), np.uint16)
    pool = _c(pool, np.uint8).reshape(-1)
    L = lib()
    for k, s in enumerate(np.asarray(slots, np.int64)):
        blk, off = int(s) // BLOCK, int(s) % BLOCK
        for h in range(H):
            r = pool[(blk * H + h) * rec:(blk * H + h + 1) * rec]
            r = np.ascontiguousarray(r)
            cc = np.zeros(d, np.uint8)
            ss = np.zeros(d, np.uint8)
            a = np.zeros(1, np.uint16)
            b = np.zeros(1, np.uint16)
            if is_k:
                L.tqo_unpack_k(d, _ptr(r), off, _ptr(cc), _ptr(ss), _ptr(a), _ptr(b))
            else:
                L.tqo_unpack_v(d, _ptr(r), off, _ptr(cc), _ptr(a))
            codes[k, h] = cc
            signs[k, h] = ss
            n16[k, h] = a[0]
            g16[k, h] = b[0]
    return dict(codes=codes, signs=signs, n16=n16, g16=g16)


def bitpos(is_k: bool, d: int, t: int, i: int, p: int):
    """Position of bit p of slot t's field for coordinate i in a record: (word, bit) of the
    little-endian 32-bit words of the cell region.  p = 0..2: cell bit p; p = 3: QJL sign (K)."""
    w = np.zeros(1, np.int32)
    b = np.zeros(1, np.int32)
    (lib().tqo_k_bitpos if is_k else lib().tqo_v_bitpos)(d, t, i, p, _ptr(w), _ptr(b))
    return int(w[0]), int(b[0])


def slot_owner(is_k: bool, d: int) -> np.ndarray:
    """Byte offset within a record -> the slot whose fields or norms it holds (-1: none)."""
    owner = np.full(record_bytes(is_k, d), -1, np.int64)
    for t in range(16):
        for i in range(d):
            for p in range(4 if is_k else 3):
                w, b = bitpos(is_k, d, t, i, p)
                owner[w * 4 + b // 8] = t
    nb = 4 if is_k else 2
    base = (8 if is_k else 6) * d
    for t in range(16):
        owner[base + nb * t: base + nb * (t + 1)] = t
    return owner


# ---------------------------------------------------------------- decode

def decode(D, S, q: np.ndarray, Hkv: int, kpool, vpool, block_table, ctx_lens,
           explicit=False, centroids=None):
    """q[B][Hq][d] (fp32 values) -> out[B][Hq][d] fp64."""
    B, Hq, d = q.shape
    c = centroids if centroids is not None else codebook()[0]
    bt = _c(block_table, np.int32)
    out = np.zeros((B, Hq, d), np.float64)
    fn = lib().tqo_decode_explicit if explicit else lib().tqo_decode
    rc = fn(d, _ptr(_c(D, np.int8)), _ptr(_c(S, np.float32)), _ptr(_c(c, np.float64)),
            _ptr(_c(q, np.float32)), B, Hq, Hkv, _ptr(_c(kpool, np.uint8)),
            _ptr(_c(vpool, np.uint8)), _ptr(bt), bt.shape[1], _ptr(_c(ctx_lens, np.int32)),
            _ptr(out))
    if rc != 0:
        raise ValueError("oracle decode: Hq must be a multiple of Hkv")
    return out


def decode_mq(D, S, q: np.ndarray, Hkv: int, kpool, vpool, block_table, ctx_lens, explicit=False,
              centroids=None):
    """Multi-query decode: q[B][Q][Hq][d] -> out[B][Q][Hq][d] fp64.  The Q queries verify the
    last Q of the ctx_lens[b] cached tokens (speculative / multi-token-prediction decoding,
    SwiftLM README "Performance: MTP Speculative Decoding"), so query i sees the tokens up to
    itself: it is the single-query decode of the first ctx_lens[b] - (Q - 1 - i) tokens."""
    B, Q, Hq, d = q.shape
    out = np.zeros((B, Q, Hq, d), np.float64)
    lens = np.asarray(ctx_lens, np.int64)
    for i in range(Q):
        li = np.maximum(lens - (Q - 1 - i), 0).astype(np.int32)
        out[:, i] = decode(D, S, np.ascontiguousarray(q[:, i]), Hkv, kpool, vpool, block_table, li,
                           explicit=explicit, centroids=centroids)
    return out


def dequant(is_k: bool, D, S, pool, H: int, block_ids, centroids=None):
    """Dense vectors of whole blocks: [len(block_ids) * 16][H][d] fp64 (SwiftLM README,
    "TurboQuantization: KV Cache Compression" -> "The Algorithm", each step undone):
      K: n  Pi^T ( c[cell]/sqrt d + sqrt(pi/2)/d gamma S^T (2 sign - 1) )
      V: nv Pi^T ( c[cell]/sqrt d )"""
    d = len(D)
    c = np.asarray(codebook()[0] if centroids is None else centroids, np.float64)
    ids = np.asarray(block_ids, np.int64)
    slots = (ids[:, None] * BLOCK + np.arange(BLOCK)).reshape(-1)
    u = unpack(is_k, d, pool, H, slots)
    f16 = lambda h: np.asarray(h, np.uint16).view(np.float16).astype(np.float64)
    y = c[u["codes"]] / np.sqrt(d)                                   # [N][H][d]
    if is_k:
        bt = 2.0 * u["signs"].astype(np.float64) - 1.0
        y = y + np.sqrt(np.pi / 2) / d * f16(u["g16"])[..., None] * (bt @ np.asarray(S, np.float64))
    N = len(slots)
    out = np.zeros((N, H, d), np.float64)
    n = f16(u["n16"])
    for i in range(N):
        for h in range(H):
            out[i, h] = n[i, h] * rotate_t(D, y[i, h])
    return out


def decode_hybrid(D, S, q: np.ndarray, Hkv: int, kpool, vpool, block_table, ctx_lens, win_k, win_v, win_lens):
    """Attention over a hybrid cache (SwiftLM README: compression starts past 2048 tokens, and
    attention covers the uncompressed recent window together with the compressed history):
    one softmax over the ctx_lens[b] compressed tokens (their dequantised K / V, the decode's
    estimator) and the win_lens[b] window rows win_k[b][j] / win_v[b][j] taken as given.
    q[B][Hq][d] -> out[B][Hq][d] fp64."""
    B, Hq, d = q.shape
    G = Hq // Hkv
    out = np.zeros((B, Hq, d), np.float64)
    for b in range(B):
        L, W = int(ctx_lens[b]), int(win_lens[b])
        nb = -(-L // BLOCK)
        Kc = dequant(True, D, S, kpool, Hkv, block_table[b, :nb])[:L] if L > 0 else np.zeros((0, Hkv, d))
        Vc = dequant(False, D, S, vpool, Hkv, block_table[b, :nb])[:L] if L > 0 else np.zeros((0, Hkv, d))
        Kw = np.asarray(win_k[b, :W], np.float64)
        Vw = np.asarray(win_v[b, :W], np.float64)
        for h in range(Hq):
            kv = h // G
            keys = np.concatenate([Kc[:, kv], Kw[:, kv]])
            vals = np.concatenate([Vc[:, kv], Vw[:, kv]])
            if len(keys) == 0:
                continue
            s = keys @ np.asarray(q[b, h], np.float64) / np.sqrt(d)
            p = np.exp(s - s.max())
            out[b, h] = (p[:, None] * vals).sum(0) / p.sum()
    return out



def hybrid_append(D, S, k_new, v_new, win_k, win_v, win_lens, ctx_lens, block_table, kpool, vpool):
    """One new token per sequence into a hybrid cache (SwiftLM README, "TurboQuantization: KV Cache
    Compression": compression starts at 2048 tokens, the most recent tokens stay uncompressed).

    Reading taken: while uncompressed, token p of a sequence is kept in window slot p mod W
    (W = win_k.shape[1]); tokens 0 .. ctx_lens[b] - 1 are compressed, the next win_lens[b] are in
    the window.  A full window first compresses its oldest token, position ctx_lens[b], into the
    paged pools at that history position (the K and V encodes of this module); the new token then
    takes that slot.  Otherwise the new token goes into slot win_lens[b].  A state this step does
    not produce (lengths out of range, or a window that is not full while ctx_lens[b] mod W != 0)
    is left as it is, and so is a full window whose leaving token's history position has no valid
    block (past the block table, or an id outside the pool): the step cannot be completed there.
    k_new, v_new [B][H][d]; win_k, win_v [B][W][H][d]; kpool / vpool are updated in place.
    Returns (win_k, win_v, win_lens, ctx_lens), updated copies."""
    win_k, win_v = np.array(win_k, copy=True), np.array(win_v, copy=True)
    win_lens = np.array(win_lens, np.int32, copy=True)
    ctx_lens = np.array(ctx_lens, np.int32, copy=True)
    B, W = win_k.shape[:2]
    nblk, mb = kpool.shape[0], block_table.shape[1]
    for b in range(B):
        L, n = int(ctx_lens[b]), int(win_lens[b])
        if not (L >= 0 and 0 <= n <= W and (n == W or L % W == 0)):
            continue
        if n == W:
            old = L % W
            blk = int(block_table[b, L // BLOCK]) if L // BLOCK < mb else -1
            if not 0 <= blk < nblk:
                continue
            slot = np.array([blk * BLOCK + L % BLOCK], np.int64)
            encode(True, D, S, np.asarray(win_k[b, old][None], np.float32), slot, kpool)
            encode(False, D, S, np.asarray(win_v[b, old][None], np.float32), slot, vpool)
            win_k[b, old], win_v[b, old] = k_new[b], v_new[b]
            ctx_lens[b] = L + 1
        else:
            win_k[b, n], win_v[b, n] = k_new[b], v_new[b]
            win_lens[b] = n + 1
    return win_k, win_v, win_lens, ctx_lens
