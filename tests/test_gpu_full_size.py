"""Full-size decode parity on the benchmark-sized workloads, sampled by (sequence, kv head).

The whole batch is prefilled on the device (synth.kv_tokens_device) and decoded in one call, at
the sizes and launch configuration the benchmark uses.  For sampled (sequence, kv head) units
(every kv head of one sequence, plus units of other sequences), the oracle encodes every token of the unit itself (synth.kv_tokens, seeded) into a
one-unit cache; those records are written over the unit's slots in the device pools, and the
oracle decodes the unit's query heads.  A unit's attention reads only its own records, so the
device output of the sampled heads must match the oracle's within the attention tolerance.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import turboquant_compressed_kv_gb300 as tq
from turboquant_compressed_kv_gb300 import synth
from turboquant_compressed_kv_gb300.cache import PagedCache, to_device
from tests import parity

DEV = "cuda"
pytestmark = pytest.mark.gpu


def _oracle_unit(w, cache, b, kvh):
    """Oracle-written records of unit (b, kvh), as [blocks][1][record] arrays, and the unit's block ids."""
    d, L = w.head_dim, w.ctx_lens[b]
    K, V = synth.kv_tokens(w, b, 0, L)
    nb = (L + 15) // 16
    kp = np.zeros((nb, 1, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nb, 1, oracle.record_bytes(False, d)), np.uint8)
    slots = np.arange(L, dtype=np.int64)              # identity block table of the one-unit cache
    oracle.encode(True, cache.D, cache.S, np.ascontiguousarray(K[:, kvh:kvh + 1]), slots, kp)
    oracle.encode(False, cache.D, cache.S, np.ascontiguousarray(V[:, kvh:kvh + 1]), slots, vp)
    return kp, vp, cache.block_table_np[b, :nb]


@pytest.mark.parametrize("name,units", [
    # 16 x 32/8 heads, d=128, 4096 tokens: every kv head of sequence 9, and units of three others
    ("llama8b_decode", [(9, h) for h in range(8)] + [(0, 0), (6, 3), (15, 7)]),
    # 64 x 32/4 heads, d=128, 512..32768 tokens: every kv head of sequence 41, and three others
    ("ragged", [(41, h) for h in range(4)] + [(3, 1), (20, 2), (63, 0)]),
    # 4 x 16/8 heads, d=256, 131072 tokens (about 8 s of oracle encode per unit)
    ("long256", [(2, 6), (0, 1)]),
])
def test_full_size_sampled_parity(name, units):
    w = synth.workload(name)
    w = dataclasses.replace(w, prefill_lens=list(w.ctx_lens), append=False)
    d, B, Hq, Hkv, G = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads, w.group
    tq.load_library()
    cache = PagedCache.create(w, DEV)
    cache.prefill_device()
    refs = {}
    for b, kvh in units:
        kp, vp, blocks = _oracle_unit(w, cache, b, kvh)
        idx = torch.from_numpy(blocks.astype(np.int64)).to(DEV)
        cache.k_pool[idx, kvh] = torch.from_numpy(kp[:, 0]).to(DEV)
        cache.v_pool[idx, kvh] = torch.from_numpy(vp[:, 0]).to(DEV)
        refs[(b, kvh)] = (kp, vp)
    q = synth.queries(w)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn(cache.params, d, to_device(q, w.dtype, DEV), Hkv, cache.k_pool, cache.v_pool,
                         cache.block_table, ctx, max(w.ctx_lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    for (b, kvh), (kp, vp) in refs.items():
        L = w.ctx_lens[b]
        nb = kp.shape[0]
        qu = np.ascontiguousarray(q[b:b + 1, kvh * G:(kvh + 1) * G])
        ref = oracle.decode(cache.D, cache.S, qu, 1, kp, vp, np.arange(nb, dtype=np.int32)[None],
                            np.array([L], np.int32))
        worst = parity.check_attention(o[b:b + 1, kvh * G:(kvh + 1) * G], ref)
        print(f"{name} unit ({b}, {kvh}): worst max-abs {worst[0]:.3e}, worst relative {worst[1]:.3e}")


@pytest.mark.parametrize("name", ["prefill", "prefill256"])
def test_full_size_encode_sampled_parity(name):
    """The prefill encodes at their full size (prefill: 8 x 32768 tokens x 8 kv heads, d=128, bf16,
    2% of K channels x 10; prefill256: 4 x 32768 tokens x 8 kv heads, d=256, bf16, lognormal K
    scales), in the launch configuration the benchmark times: the whole batch is encoded in one
    tq_encode_k and one tq_encode_v call, then 512 sampled tokens (every kv head, K and V) are
    compared with the oracle's encode of the same input rows, read back from the device."""
    w = synth.workload(name)
    d, Hkv = w.head_dim, w.n_kv_heads
    tq.load_library()
    cache = PagedCache.create(w, DEV)
    Ks, Vs, slots = [], [], []
    for b in range(w.batch):
        K, V = synth.kv_tokens_device(w, b, 0, w.prefill_lens[b], DEV)
        Ks.append(K)
        Vs.append(V)
        slots.append(synth.slots_for(cache.block_table_np, b, 0, w.prefill_lens[b]))
    K, V = torch.cat(Ks), torch.cat(Vs)
    del Ks, Vs
    sl = np.concatenate(slots)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.encode_k(cache.params, d, K, torch.from_numpy(sl).to(DEV), cache.k_pool, status=status)
    tq.encode_v(cache.params, d, V, torch.from_numpy(sl).to(DEV), cache.v_pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pick = np.sort(np.random.default_rng(12).choice(K.shape[0], 512, replace=False))
    idx = torch.from_numpy(pick).to(DEV)
    xk = K[idx].float().cpu().numpy()
    xv = V[idx].float().cpu().numpy()
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    sk = parity.check_encode(True, cache.D, cache.S, xk, sl[pick], kp, pool_fill=0)
    sv = parity.check_encode(False, cache.D, cache.S, xv, sl[pick], vp, pool_fill=0)
    print(f"{name} encode, 512 tokens x {Hkv} heads: K {sk}, V {sv}")


def test_full_size_dequant_sampled_parity():
    """The prefill dequantisation at its full size (131,072 (block, kv head) records of each pool
    back to bf16 and fp32), in the launch configuration the benchmark times: one tq_dequant_k and
    one tq_dequant_v over every block of the cache; 64 sampled blocks (every slot and kv head) are
    compared with the oracle's reconstruction of the same records read back from the device."""
    w = synth.workload("prefill")
    d, Hkv = w.head_dim, w.n_kv_heads
    tq.load_library()
    cache = PagedCache.create(w, DEV)
    cache.prefill_device()
    ids = torch.cat([cache.block_table[b, :w.prefill_lens[b] // 16] for b in range(w.batch)]).contiguous()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pick = np.sort(np.random.default_rng(13).choice(ids.numel(), 64, replace=False))
    ids_np = ids.cpu().numpy()
    for is_k, fn, pool in ((True, tq.dequant_k, cache.k_pool), (False, tq.dequant_v, cache.v_pool)):
        pool_np = pool.cpu().numpy()
        ref = oracle.dequant(is_k, cache.D, cache.S, pool_np, Hkv, ids_np[pick]).reshape(64, 16, Hkv, d)
        for out_dtype, tol in ((torch.float32, None), (torch.bfloat16, 2.0 ** -8)):
            o = fn(cache.params, d, pool, ids, out_dtype=out_dtype, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            g = o.view(ids.numel(), 16, Hkv, d)[torch.from_numpy(pick).to(DEV)].float().cpu().numpy().astype(np.float64)
            del o
            if tol is None:
                err = np.linalg.norm(g - ref, axis=-1) / np.maximum(np.linalg.norm(ref, axis=-1), 1e-30)
                assert err.max() < 1e-5, (is_k, err.max())
            else:   # one bf16 rounding of the exact value (plus the fp32 error above)
                assert np.all(np.abs(g - ref) <= np.abs(ref) * tol + 1e-5 * np.linalg.norm(ref, axis=-1, keepdims=True)), is_k


def test_full_size_hybrid_sampled_parity():
    """Hybrid attention at the benchmark's size (16 sequences x 32/8 heads, d=128: 30720 compressed
    tokens plus a 2048-row bf16 window each), in one tq_decode_attn_hybrid call; for two sampled
    sequences (all 32 query heads) the oracle decodes the same packed records and window rows,
    read back from the device."""
    w0 = synth.workload("llama8b_decode")
    history, window = 30720, 2048
    w = dataclasses.replace(w0, ctx_lens=[history] * w0.batch, prefill_lens=[history] * w0.batch, append=False)
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    tq.load_library()
    cache = PagedCache.create(w, DEV)
    cache.prefill_device()
    g = torch.Generator(device=DEV).manual_seed(99)
    wk = torch.randn((B, window, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    wv = torch.randn((B, window, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    wl = torch.tensor([window - 3 * b for b in range(B)], dtype=torch.int32, device=DEV)   # some windows not full
    q = synth.queries(w)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn_hybrid(cache.params, d, to_device(q, w.dtype, DEV), Hkv, cache.k_pool, cache.v_pool,
                                cache.block_table, ctx, history, wk, wv, wl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    for b in (5, 14):
        ref = oracle.decode_hybrid(cache.D, cache.S, q[b:b + 1], Hkv, kp, vp, cache.block_table_np[b:b + 1],
                                   np.array([history], np.int32), wk[b:b + 1].float().cpu().numpy(),
                                   wv[b:b + 1].float().cpu().numpy(), wl[b:b + 1].cpu().numpy())
        worst = parity.check_attention(o[b:b + 1], ref)
        print(f"hybrid sequence {b}: worst max-abs {worst[0]:.3e}, worst relative {worst[1]:.3e}")


@pytest.mark.parametrize("q_len", [1, 2])
def test_full_size_step_sampled_parity(q_len):
    """The decode step at the benchmark's size (16 sequences x 32/8 heads, d=128, 4096 attended
    tokens): q_len = 1 is the benchmark's step (tq_decode_step: append one token, attend), q_len = 2
    the speculative-verify step (tq_decode_step_mq: append two draft tokens, two causal queries).
    For two sampled sequences the appended records are checked against the oracle's encode of the
    new rows, and the queries against the oracle's decode of the same packed cache."""
    w0 = synth.workload("llama8b_decode")
    w = dataclasses.replace(w0, prefill_lens=[L - q_len for L in w0.ctx_lens])
    d, B, Hq, Hkv = w.head_dim, w.batch, w.n_q_heads, w.n_kv_heads
    tq.load_library()
    cache = PagedCache.create(w, DEV)
    cache.prefill_device()
    g = torch.Generator(device=DEV).manual_seed(1234)
    k_new = torch.randn((B, q_len, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn((B, q_len, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn((B, q_len, Hq, d), generator=g, device=DEV).to(torch.bfloat16)
    pre = torch.tensor(w.prefill_lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if q_len == 1:
        out = tq.decode_step(cache.params, d, k_new[:, 0].contiguous(), v_new[:, 0].contiguous(),
                             q[:, 0].contiguous(), Hkv, cache.k_pool, cache.v_pool, cache.block_table, pre,
                             max(w.ctx_lens), status=status)[:, None]
    else:
        out = tq.decode_step_mq(cache.params, d, k_new, v_new, q, Hkv, cache.k_pool, cache.v_pool,
                                cache.block_table, pre, max(w.ctx_lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    kp, vp = cache.k_pool.cpu().numpy(), cache.v_pool.cpu().numpy()
    for b in (2, 11):
        P = w.prefill_lens[b]
        slots = synth.slots_for(cache.block_table_np, b, P, q_len)
        parity.check_encode(True, cache.D, cache.S, k_new[b].float().cpu().numpy(), slots, kp, pool_fill=0)
        parity.check_encode(False, cache.D, cache.S, v_new[b].float().cpu().numpy(), slots, vp, pool_fill=0)
        ref = oracle.decode_mq(cache.D, cache.S, q[b:b + 1].float().cpu().numpy(), Hkv, kp, vp,
                               cache.block_table_np[b:b + 1], np.array([P + q_len], np.int32))
        worst = parity.check_attention(o[b], ref[0])
        print(f"step (q_len {q_len}) sequence {b}: worst max-abs {worst[0]:.3e}, worst relative {worst[1]:.3e}")
