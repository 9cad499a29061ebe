"""Device-side paged cache for a synthetic workload, filled through the C ABI.

PagedCache owns the pools, block table and lengths of one workload (torch
tensors on one device) and prefills them by calling tq_encode_k/tq_encode_v
sequence by sequence, so the host never holds more than one sequence of
inputs.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import turboquant_compressed_kv_gb300 as tq
from turboquant_compressed_kv_gb300 import synth


def to_device(a: np.ndarray, dtype: str, device):
    """Upload fp32 values already rounded to `dtype` (so the cast is exact)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(device, non_blocking=False)


@dataclasses.dataclass
class PagedCache:
    w: synth.Workload
    params: object
    k_pool: object
    v_pool: object
    block_table: object       # device int32 [B][max_blocks]
    block_table_np: np.ndarray
    num_blocks: int
    D: np.ndarray
    S: np.ndarray

    @classmethod
    def create(cls, w: synth.Workload, device="cuda"):
        import torch
        d = w.head_dim
        D = synth.rotation_signs(d)
        S = synth.qjl_matrix(d)
        params, _ = tq.codebook_init(d, D, S, device=device)
        bt, nblk = synth.block_tables(w)
        kp = tq.empty_pool(nblk, w.n_kv_heads, d, "k", device)
        vp = tq.empty_pool(nblk, w.n_kv_heads, d, "v", device)
        return cls(w, params, kp, vp, torch.from_numpy(bt).to(device), bt, nblk, D, S)

    def prefill(self, chunk: int = 65536):
        """Encode tokens [0, prefill_lens[b]) of every sequence into the pools."""
        import torch
        w = self.w
        dev = self.k_pool.device
        for b in range(w.batch):
            L = w.prefill_lens[b]
            for s0 in range(0, L, chunk):
                n = min(chunk, L - s0)
                K, V = synth.kv_tokens(w, b, s0, n)
                slots = torch.from_numpy(synth.slots_for(self.block_table_np, b, s0, n)).to(dev)
                tq.encode_k(self.params, w.head_dim, to_device(K, w.dtype, dev), slots, self.k_pool)
                tq.encode_v(self.params, w.head_dim, to_device(V, w.dtype, dev), slots, self.v_pool)
        torch.cuda.synchronize(dev)

    def prefill_device(self, chunk: int = 65536):
        """Like prefill, with inputs drawn on the device (synth.kv_tokens_device)."""
        import torch
        w = self.w
        dev = self.k_pool.device
        for b in range(w.batch):
            L = w.prefill_lens[b]
            for s0 in range(0, L, chunk):
                n = min(chunk, L - s0)
                K, V = synth.kv_tokens_device(w, b, s0, n, dev)
                slots = torch.from_numpy(synth.slots_for(self.block_table_np, b, s0, n)).to(dev)
                tq.encode_k(self.params, w.head_dim, K, slots, self.k_pool)
                tq.encode_v(self.params, w.head_dim, V, slots, self.v_pool)
        torch.cuda.synchronize(dev)

    def append_inputs(self, step: int = 0):
        """The token appended by the decode step (position prefill_lens[b]): K/V [B][Hkv][d]."""
        w = self.w
        K = np.empty((w.batch, w.n_kv_heads, w.head_dim), np.float32)
        V = np.empty_like(K)
        for b in range(w.batch):
            kb, vb = synth.kv_tokens(w, b, w.prefill_lens[b], 1)
            K[b], V[b] = kb[0], vb[0]
        return K, V
