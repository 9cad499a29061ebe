"""TurboQuant compressed KV cache on GB300: Python binding of libtq.so.

Thin ctypes marshalling over the C ABI in include/tq.h; every step of the
path runs in the library's CUDA kernels.  PyTorch supplies device memory and
the current stream.  Importing works without a GPU; calling a compute entry
point without the built library raises immediately (there is no fallback).

Entry points (same names as the C ABI, minus the ``tq_`` prefix):
  codebook_init, encode_k, encode_v, paged_append, decode_attn,
  params_bytes, k_record_bytes, v_record_bytes, decode_workspace_bytes,
  the decode variants (decode_attn_mq, decode_step, decode_attn_hybrid, ...),
  dequant_k / dequant_v, and the group-quantised comparator (gq_*).
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libtq.so")

BLOCK_SIZE = 16
DTYPE_F32 = 0
DTYPE_BF16 = 1
STATUS_BAD_SLOT = 1
STATUS_BAD_PARAMS = 2
STATUS_TIMEOUT = 4

_lib = None


class TQError(RuntimeError):
    pass


def load_library(path: str | None = None):
    """Load libtq.so (built by turboquant_compressed_kv_gb300.build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise TQError(f"libtq.so not found at {p}; build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(p)
    _declare(L)
    if path is None:
        _lib = L
    return L


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


def _declare(L):
    L.tq_k_record_bytes.restype = _SZ
    L.tq_k_record_bytes.argtypes = [_I]
    L.tq_v_record_bytes.restype = _SZ
    L.tq_v_record_bytes.argtypes = [_I]
    L.tq_params_bytes.restype = _SZ
    L.tq_params_bytes.argtypes = [_I]
    L.tq_error_string.restype = ctypes.c_char_p
    L.tq_error_string.argtypes = [_I]
    L.tq_codebook_init.restype = _I
    L.tq_codebook_init.argtypes = [_I, _P, _P, _P, _SZ, _P, _P]
    for name in ("tq_encode_k", "tq_encode_v"):
        f = getattr(L, name)
        f.restype = _I
        f.argtypes = [_P, _I, _P, _I, _I64, _I, _P, _P, _I64, _P, _P]
    L.tq_paged_append.restype = _I
    L.tq_paged_append.argtypes = [_P, _I, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P, _I64, _P, _P]
    L.tq_decode_workspace_bytes.restype = _SZ
    L.tq_decode_workspace_bytes.argtypes = [_I, _I, _I, _I]
    L.tq_decode_attn.restype = _I
    L.tq_decode_attn.argtypes = [_P, _I, _P, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _SZ,
                                 _P, _P]
    L.tq_decode_qprep.restype = _I
    L.tq_decode_qprep.argtypes = [_P, _I, _P, _I, _I, _I, _I, _P, _I, _P, _SZ, _P]
    L.tq_decode_splitk.restype = _I
    L.tq_decode_splitk.argtypes = [_P, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _SZ, _P, _P]
    L.tq_decode_step.restype = _I
    L.tq_decode_step.argtypes = [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _P, _P, _I64, _P, _P, _SZ, _P,
                                 _P]
    L.tq_decode_workspace_bytes_mq.restype = _SZ
    L.tq_decode_workspace_bytes_mq.argtypes = [_I, _I, _I, _I, _I]
    L.tq_decode_attn_mq.restype = _I
    L.tq_decode_attn_mq.argtypes = [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _SZ,
                                    _P, _P]
    L.tq_decode_step_mq.restype = _I
    L.tq_decode_step_mq.argtypes = [_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P, _I, _P, _P, _I64, _P, _P,
                                    _SZ, _P, _P]
    for name in ("tq_dequant_k", "tq_dequant_v"):
        f = getattr(L, name)
        f.restype = _I
        f.argtypes = [_P, _I, _P, _I64, _I, _P, _I, _P, _I, _P, _P]
    L.tq_decode_workspace_bytes_hybrid.restype = _SZ
    L.tq_decode_workspace_bytes_hybrid.argtypes = [_I, _I, _I, _I, _I]
    L.tq_decode_attn_hybrid.restype = _I
    L.tq_decode_attn_hybrid.argtypes = [_P, _I, _P, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _I, _I, _P,
                                        _P, _P, _SZ, _P, _P]
    L.tq_selftest_wait_timeout.restype = _I
    L.tq_selftest_wait_timeout.argtypes = [_P, _P]
    L.tq_hybrid_append_scratch_bytes.restype = _SZ
    L.tq_hybrid_append_scratch_bytes.argtypes = [_I, _I, _I, _I]
    L.tq_hybrid_append.restype = _I
    L.tq_hybrid_append.argtypes = [_P, _I, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _I, _P, _P, _P, _I64, _P, _SZ,
                                   _P, _P]
    L.tq_decode_attn_noalloc.restype = _I
    L.tq_decode_attn_noalloc.argtypes = [_P, _I, _P, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _P]
    L.tq_gq_record_bytes.restype = _SZ
    L.tq_gq_record_bytes.argtypes = [_I, _I, _I]
    L.tq_gq_encode.restype = _I
    L.tq_gq_encode.argtypes = [_I, _I, _I, _P, _I, _I64, _I, _P, _P, _I64, _P, _P]
    L.tq_gq_decode_workspace_bytes.restype = _SZ
    L.tq_gq_decode_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
    L.tq_gq_decode_attn.restype = _I
    L.tq_gq_decode_attn.argtypes = [_I, _I, _I, _P, _I, _I, _I, _I, _P, _P, _I64, _P, _I, _P, _I, _P, _P, _SZ, _P,
                                    _P]



def _check(rc: int, what: str):
    if rc != 0:
        msg = load_library().tq_error_string(rc).decode()
        raise TQError(f"{what} failed: {msg} (code {rc})")


# ---------------------------------------------------------------- sizes

def params_bytes(d: int) -> int:
    return int(load_library().tq_params_bytes(d))


def k_record_bytes(d: int) -> int:
    return int(load_library().tq_k_record_bytes(d))


def v_record_bytes(d: int) -> int:
    return int(load_library().tq_v_record_bytes(d))


def decode_workspace_bytes(d: int, batch: int, n_q_heads: int, max_ctx: int) -> int:
    return int(load_library().tq_decode_workspace_bytes(d, batch, n_q_heads, max_ctx))


def decode_workspace_bytes_mq(d: int, batch: int, q_len: int, n_q_heads: int, max_ctx: int) -> int:
    return int(load_library().tq_decode_workspace_bytes_mq(d, batch, q_len, n_q_heads, max_ctx))


# ---------------------------------------------------------------- marshalling helpers

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TQError(f"unsupported input dtype {t.dtype} (float32 or bfloat16)")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise TQError("all tensors must be CUDA tensors")
        if t is not None and not t.is_contiguous():
            raise TQError("all tensors must be contiguous")


def _on_device(fn):
    """Run a wrapper with the device of its tensor arguments current, so that the library takes
    that device's scratch and default stream; tensors (or a stream) on different devices are an
    error."""
    import functools

    @functools.wraps(fn)
    def call(*args, **kwargs):
        torch = _torch()
        tensor = torch.Tensor
        devs = {a.device for a in args if isinstance(a, tensor) and a.is_cuda}
        devs.update(a.device for a in kwargs.values() if isinstance(a, tensor) and a.is_cuda)
        if len(devs) > 1:
            raise TQError(f"{fn.__name__}: tensors on more than one device ({sorted(map(str, devs))})")
        if not devs:
            return fn(*args, **kwargs)
        dev = devs.pop()
        st = kwargs.get("stream")
        if st is not None and st.device != dev:
            raise TQError(f"{fn.__name__}: the stream is on {st.device}, the tensors on {dev}")
        if torch.cuda.current_device() == dev.index:   # already current: no device switch
            return fn(*args, **kwargs)
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return call


def empty_pool(num_blocks: int, n_kv_heads: int, d: int, kind: str, device="cuda"):
    """Zeroed K or V pool tensor uint8[num_blocks][n_kv_heads][record_bytes]."""
    torch = _torch()
    rec = k_record_bytes(d) if kind == "k" else v_record_bytes(d)
    return torch.zeros((num_blocks, n_kv_heads, rec), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- entry points

def codebook_init(d: int, D, S, device="cuda", stream=None):
    """tq_codebook_init: returns (params uint8 device tensor, centroids list[8]).

    D: int8[d] of +-1 (host array or CPU tensor); S: float32[d][d] (host)."""
    import numpy as np
    torch = _torch()
    Dn = np.ascontiguousarray(np.asarray(D.cpu() if hasattr(D, "cpu") else D), dtype=np.int8)
    Sn = np.ascontiguousarray(np.asarray(S.cpu() if hasattr(S, "cpu") else S), dtype=np.float32)
    if Dn.shape != (d,) or Sn.shape != (d, d):
        raise TQError("D must be [d] and S must be [d][d]")
    nb = params_bytes(d)
    if nb == 0:
        raise TQError(f"unsupported head_dim {d}")
    params = torch.empty(nb, dtype=torch.uint8, device=device)
    cent = (ctypes.c_double * 8)()
    with torch.cuda.device(params.device):
        rc = load_library().tq_codebook_init(d, Dn.ctypes.data_as(_P), Sn.ctypes.data_as(_P), _ptr(params), nb,
                                             cent, _stream(stream))
    _check(rc, "tq_codebook_init")
    return params, [float(x) for x in cent]


@_on_device
def encode_k(params, d: int, k, slot_mapping, k_pool, status=None, stream=None):
    """tq_encode_k: k [n_tokens][n_kv_heads][d] (f32/bf16), slot_mapping int64[n_tokens]."""
    _need_cuda(params, k, slot_mapping, k_pool, status)
    n, h = k.shape[0], k.shape[1]
    rc = load_library().tq_encode_k(_ptr(params), d, _ptr(k), _dtype_code(k), n, h, _ptr(slot_mapping),
                                    _ptr(k_pool), k_pool.shape[0], _ptr(status), _stream(stream))
    _check(rc, "tq_encode_k")


@_on_device
def encode_v(params, d: int, v, slot_mapping, v_pool, status=None, stream=None):
    """tq_encode_v: v [n_tokens][n_kv_heads][d] (f32/bf16), slot_mapping int64[n_tokens]."""
    _need_cuda(params, v, slot_mapping, v_pool, status)
    n, h = v.shape[0], v.shape[1]
    rc = load_library().tq_encode_v(_ptr(params), d, _ptr(v), _dtype_code(v), n, h, _ptr(slot_mapping),
                                    _ptr(v_pool), v_pool.shape[0], _ptr(status), _stream(stream))
    _check(rc, "tq_encode_v")


@_on_device
def paged_append(params, d: int, k_new, v_new, block_table, ctx_lens, k_pool, v_pool, status=None, stream=None):
    """tq_paged_append: one token per sequence at slot ctx_lens[b] (lengths before the append)."""
    _need_cuda(params, k_new, v_new, block_table, ctx_lens, k_pool, v_pool, status)
    b, h = k_new.shape[0], k_new.shape[1]
    rc = load_library().tq_paged_append(_ptr(params), d, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), b, h,
                                        _ptr(block_table), block_table.shape[1], _ptr(ctx_lens), _ptr(k_pool),
                                        _ptr(v_pool), k_pool.shape[0], _ptr(status), _stream(stream))
    _check(rc, "tq_paged_append")


@_on_device
def decode_attn(params, d: int, q, n_kv_heads: int, k_pool, v_pool, block_table, ctx_lens, max_ctx: int,
                out=None, workspace=None, status=None, stream=None):
    """tq_decode_attn: q [batch][n_q_heads][d] -> out float32 [batch][n_q_heads][d]."""
    torch = _torch()
    _need_cuda(params, q, k_pool, v_pool, block_table, ctx_lens, out, workspace, status)
    B, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:   # (the library checks a given workspace's size itself)
        need = decode_workspace_bytes(d, B, Hq, max_ctx)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().tq_decode_attn(_ptr(params), d, _ptr(q), _dtype_code(q), B, Hq, n_kv_heads,
                                       _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
                                       block_table.shape[1], _ptr(ctx_lens), max_ctx, _ptr(out),
                                       _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check(rc, "tq_decode_attn")
    return out


# ---------------------------------------------------------------- decode stages

@_on_device
def decode_qprep(params, d: int, q, n_kv_heads: int, ctx_lens, max_ctx: int, workspace, stream=None):
    """tq_decode_qprep: qbar = Pi q, u = S qbar and the pass's work schedule into the workspace."""
    _need_cuda(params, q, ctx_lens, workspace)
    B, Hq = q.shape[0], q.shape[1]
    rc = load_library().tq_decode_qprep(_ptr(params), d, _ptr(q), _dtype_code(q), B, Hq, n_kv_heads,
                                        _ptr(ctx_lens), max_ctx, _ptr(workspace), workspace.numel(),
                                        _stream(stream))
    _check(rc, "tq_decode_qprep")


@_on_device
def decode_splitk(params, d: int, batch: int, n_q_heads: int, n_kv_heads: int, k_pool, v_pool, block_table,
                  ctx_lens, max_ctx: int, out, workspace, status=None, stream=None):
    """tq_decode_splitk: the split-K pass over the compressed cache, merged into out."""
    _need_cuda(params, k_pool, v_pool, block_table, ctx_lens, out, workspace, status)
    rc = load_library().tq_decode_splitk(_ptr(params), d, batch, n_q_heads, n_kv_heads, _ptr(k_pool),
                                         _ptr(v_pool), k_pool.shape[0], _ptr(block_table), block_table.shape[1],
                                         _ptr(ctx_lens), max_ctx, _ptr(out), _ptr(workspace), workspace.numel(),
                                         _ptr(status), _stream(stream))
    _check(rc, "tq_decode_splitk")


@_on_device
def decode_step(params, d: int, k_new, v_new, q, n_kv_heads: int, k_pool, v_pool, block_table, pre_lens,
                max_ctx: int, out=None, workspace=None, status=None, stream=None):
    """tq_decode_step: append (k_new, v_new) at position pre_lens[b], then attend pre_lens[b] + 1 tokens."""
    torch = _torch()
    _need_cuda(params, k_new, v_new, q, k_pool, v_pool, block_table, pre_lens, out, workspace, status)
    B, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:   # (the library checks a given workspace's size itself)
        need = decode_workspace_bytes(d, B, Hq, max_ctx)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TQError("k_new, v_new and q must share one dtype")
    rc = load_library().tq_decode_step(_ptr(params), d, _ptr(k_new), _ptr(v_new), _ptr(q), _dtype_code(q), B, Hq,
                                       n_kv_heads, _ptr(block_table), block_table.shape[1], _ptr(pre_lens), max_ctx,
                                       _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(out), _ptr(workspace),
                                       workspace.numel(), _ptr(status), _stream(stream))
    _check(rc, "tq_decode_step")
    return out


def _dequant(is_k: bool, params, d: int, pool, block_ids, out_dtype, out, status, stream):
    torch = _torch()
    _need_cuda(params, pool, block_ids, out, status)
    n, H = block_ids.numel(), pool.shape[1]
    if out is None:
        out = torch.empty((n * 16, H, d), dtype=out_dtype, device=pool.device)
    name = "tq_dequant_k" if is_k else "tq_dequant_v"
    rc = getattr(load_library(), name)(_ptr(params), d, _ptr(pool), pool.shape[0], H, _ptr(block_ids), n, _ptr(out),
                                       _dtype_code(out), _ptr(status), _stream(stream))
    _check(rc, name)
    return out


@_on_device
def dequant_k(params, d: int, k_pool, block_ids, out_dtype=None, out=None, status=None, stream=None):
    """tq_dequant_k: dense K [len(block_ids) * 16][n_kv_heads][d] of whole paged blocks."""
    return _dequant(True, params, d, k_pool, block_ids, out_dtype or _torch().bfloat16, out, status, stream)


@_on_device
def dequant_v(params, d: int, v_pool, block_ids, out_dtype=None, out=None, status=None, stream=None):
    """tq_dequant_v: dense V [len(block_ids) * 16][n_kv_heads][d] of whole paged blocks."""
    return _dequant(False, params, d, v_pool, block_ids, out_dtype or _torch().bfloat16, out, status, stream)


@_on_device
def decode_attn_hybrid(params, d: int, q, n_kv_heads: int, k_pool, v_pool, block_table, ctx_lens, max_ctx: int,
                       win_k, win_v, win_lens, out=None, workspace=None, status=None, stream=None):
    """tq_decode_attn_hybrid: one softmax over the compressed history (ctx_lens[b] tokens) and the
    uncompressed window rows win_k/win_v [batch][win_cap][n_kv_heads][d] (win_lens[b] of them)."""
    torch = _torch()
    _need_cuda(params, q, k_pool, v_pool, block_table, ctx_lens, win_k, win_v, win_lens, out, workspace, status)
    B, Hq = q.shape[0], q.shape[1]
    cap = win_k.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    need = int(load_library().tq_decode_workspace_bytes_hybrid(d, B, Hq, max_ctx, cap))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().tq_decode_attn_hybrid(_ptr(params), d, _ptr(q), _dtype_code(q), B, Hq, n_kv_heads,
                                              _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
                                              block_table.shape[1], _ptr(ctx_lens), max_ctx, _ptr(win_k),
                                              _ptr(win_v), _dtype_code(win_k), cap, _ptr(win_lens), _ptr(out),
                                              _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check(rc, "tq_decode_attn_hybrid")
    return out


@_on_device
def selftest_wait_timeout(status, stream=None):
    """tq_selftest_wait_timeout: one bounded wait that runs out; ORs STATUS_TIMEOUT into status."""
    _need_cuda(status)
    _check(load_library().tq_selftest_wait_timeout(_ptr(status), _stream(stream)), "tq_selftest_wait_timeout")


@_on_device
def hybrid_append(params, d: int, k_new, v_new, win_k, win_v, win_lens, block_table, ctx_lens, k_pool, v_pool,
                  scratch=None, status=None, stream=None):
    """tq_hybrid_append: k_new / v_new [batch][n_kv_heads][d] into the window win_k / win_v
    [batch][win_cap][n_kv_heads][d] (same dtype); a full window first moves its oldest token into
    the paged pools at history position ctx_lens[b].  win_lens and ctx_lens are updated in place."""
    torch = _torch()
    _need_cuda(params, k_new, v_new, win_k, win_v, win_lens, block_table, ctx_lens, k_pool, v_pool, scratch, status)
    B, H = k_new.shape[0], k_new.shape[1]
    if _dtype_code(k_new) != _dtype_code(win_k):
        raise TQError("hybrid_append: the new rows and the window must have the same dtype")
    need = int(load_library().tq_hybrid_append_scratch_bytes(d, B, H, _dtype_code(k_new)))
    if scratch is None:
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=k_new.device)
    rc = load_library().tq_hybrid_append(_ptr(params), d, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), B, H,
                                         _ptr(win_k), _ptr(win_v), win_k.shape[1], _ptr(win_lens), _ptr(block_table),
                                         block_table.shape[1], _ptr(ctx_lens), _ptr(k_pool), _ptr(v_pool),
                                         k_pool.shape[0], _ptr(scratch), scratch.numel(), _ptr(status),
                                         _stream(stream))
    _check(rc, "tq_hybrid_append")


@_on_device
def decode_attn_mq(params, d: int, q, n_kv_heads: int, k_pool, v_pool, block_table, ctx_lens, max_ctx: int,
                   out=None, workspace=None, status=None, stream=None):
    """tq_decode_attn_mq: q [batch][q_len][n_q_heads][d] -> out float32 of the same shape.

    ctx_lens counts the q_len new tokens; query i attends ctx_lens[b] - (q_len - 1 - i) tokens."""
    torch = _torch()
    _need_cuda(params, q, k_pool, v_pool, block_table, ctx_lens, out, workspace, status)
    B, Q, Hq = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, Q, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:   # (the library checks a given workspace's size itself)
        need = decode_workspace_bytes_mq(d, B, Q, Hq, max_ctx)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().tq_decode_attn_mq(_ptr(params), d, _ptr(q), _dtype_code(q), B, Q, Hq, n_kv_heads,
                                          _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
                                          block_table.shape[1], _ptr(ctx_lens), max_ctx, _ptr(out),
                                          _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check(rc, "tq_decode_attn_mq")
    return out


@_on_device
def decode_step_mq(params, d: int, k_new, v_new, q, n_kv_heads: int, k_pool, v_pool, block_table, pre_lens,
                   max_ctx: int, out=None, workspace=None, status=None, stream=None):
    """tq_decode_step_mq: append k_new/v_new [batch][q_len][n_kv_heads][d] at pre_lens[b] + i, then
    query i of q [batch][q_len][n_q_heads][d] attends pre_lens[b] + 1 + i tokens."""
    torch = _torch()
    _need_cuda(params, k_new, v_new, q, k_pool, v_pool, block_table, pre_lens, out, workspace, status)
    B, Q, Hq = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, Q, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:   # (the library checks a given workspace's size itself)
        need = decode_workspace_bytes_mq(d, B, Q, Hq, max_ctx)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TQError("k_new, v_new and q must share one dtype")
    rc = load_library().tq_decode_step_mq(_ptr(params), d, _ptr(k_new), _ptr(v_new), _ptr(q), _dtype_code(q), B,
                                          Q, Hq, n_kv_heads, _ptr(block_table), block_table.shape[1],
                                          _ptr(pre_lens), max_ctx, _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                          _ptr(out), _ptr(workspace), workspace.numel(), _ptr(status),
                                          _stream(stream))
    _check(rc, "tq_decode_step_mq")
    return out


@_on_device
def decode_attn_noalloc(params, d: int, q, n_kv_heads: int, k_pool, v_pool, block_table, ctx_lens, max_ctx: int,
                        out=None, status=None, stream=None):
    """tq_decode_attn_noalloc: decode attention with the library's fixed scratch instead of a workspace.

    For callers that cannot allocate device memory while decoding; shapes whose
    workspace would exceed 16 MiB are rejected.  Calls that overlap on the GPU
    share the scratch and race."""
    torch = _torch()
    _need_cuda(params, q, k_pool, v_pool, block_table, ctx_lens, out, status)
    B, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    rc = load_library().tq_decode_attn_noalloc(_ptr(params), d, _ptr(q), _dtype_code(q), B, Hq, n_kv_heads,
                                               _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(block_table),
                                               block_table.shape[1], _ptr(ctx_lens), max_ctx, _ptr(out),
                                               _ptr(status), _stream(stream))
    _check(rc, "tq_decode_attn_noalloc")
    return out


# ---------------------------------------------------------------- group-quantised comparator

def gq_record_bytes(d: int, bits: int, group: int = 64) -> int:
    """tq_gq_record_bytes: bytes of one (block, kv head) record of the group-quantised cache."""
    return load_library().tq_gq_record_bytes(d, bits, group)


def gq_empty_pool(num_blocks: int, n_kv_heads: int, d: int, bits: int, group: int = 64, device="cuda"):
    """Zeroed group-quantised pool tensor uint8[num_blocks][n_kv_heads][record_bytes]."""
    torch = _torch()
    rec = gq_record_bytes(d, bits, group)
    if rec == 0:
        raise TQError(f"unsupported group-quantised format d={d} bits={bits} group={group}")
    return torch.zeros((num_blocks, n_kv_heads, rec), dtype=torch.uint8, device=device)


@_on_device
def gq_encode(d: int, bits: int, group: int, x, slot_mapping, pool, status=None, stream=None):
    """tq_gq_encode: x [n_tokens][n_kv_heads][d] (f32/bf16) into slot slot_mapping[token] of pool."""
    _need_cuda(x, slot_mapping, pool, status)
    n, h = x.shape[0], x.shape[1]
    rc = load_library().tq_gq_encode(d, bits, group, _ptr(x), _dtype_code(x), n, h, _ptr(slot_mapping), _ptr(pool),
                                     pool.shape[0], _ptr(status), _stream(stream))
    _check(rc, "tq_gq_encode")


def gq_decode_workspace_bytes(d: int, batch: int, n_q_heads: int, n_kv_heads: int, max_ctx: int) -> int:
    return load_library().tq_gq_decode_workspace_bytes(d, batch, n_q_heads, n_kv_heads, max_ctx)


@_on_device
def gq_decode_attn(d: int, bits: int, group: int, q, n_kv_heads: int, k_pool, v_pool, block_table, ctx_lens,
                   max_ctx: int, out=None, workspace=None, status=None, stream=None):
    """tq_gq_decode_attn: q [batch][n_q_heads][d] -> out float32 [batch][n_q_heads][d]."""
    torch = _torch()
    _need_cuda(q, k_pool, v_pool, block_table, ctx_lens, out, workspace, status)
    B, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    need = gq_decode_workspace_bytes(d, B, Hq, n_kv_heads, max_ctx)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().tq_gq_decode_attn(d, bits, group, _ptr(q), _dtype_code(q), B, Hq, n_kv_heads, _ptr(k_pool),
                                          _ptr(v_pool), k_pool.shape[0], _ptr(block_table), block_table.shape[1],
                                          _ptr(ctx_lens), max_ctx, _ptr(out), _ptr(workspace), workspace.numel(),
                                          _ptr(status), _stream(stream))
    _check(rc, "tq_gq_decode_attn")
    return out
