"""tq_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (a runtime that reserved all GPU memory up front, or a
decode loop that must not call cudaMalloc).  It must give what tq_decode_attn
gives with a caller workspace, call after call, although every call reuses
the same fixed scratch array inside the library.

This file is collected last on purpose, and it builds all its own inputs, so
it passes both alone in a fresh process and after the other tests."""
import numpy as np
import pytest

from tests import parity

torch = pytest.importorskip("torch")
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cache(d, Hkv, lens, seed):
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    need = [max(1, -(-L // 16)) for L in lens]
    nblk = sum(need) + 2
    perm = np.random.default_rng(seed).permutation(nblk)
    bt = np.zeros((len(lens), max(need)), np.int32)
    k0 = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k0:k0 + n]
        k0 += n
    kp = tq.empty_pool(nblk, Hkv, d, "k", DEV)
    vp = tq.empty_pool(nblk, Hkv, d, "v", DEV)
    rng = np.random.default_rng(seed + 1)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        K = rng.standard_normal((L, Hkv, d)).astype(np.float32) * 2
        V = rng.standard_normal((L, Hkv, d)).astype(np.float32)
        sl = torch.from_numpy(synth.slots_for(bt, b, 0, L)).to(DEV)
        tq.encode_k(params, d, torch.from_numpy(K).to(DEV), sl, kp)
        tq.encode_v(params, d, torch.from_numpy(V).to(DEV), sl, vp)
    return params, torch.from_numpy(bt).to(DEV), kp, vp


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (256, 8, 4)])
def test_noalloc_matches_workspace_decode_on_two_calls(d, Hq, Hkv):
    lens = [1, 600, 4096, 0, 1500]
    params, bt, kp, vp = _cache(d, Hkv, lens, seed=d)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    rng = np.random.default_rng(3)
    for call in range(2):
        q = torch.from_numpy(rng.standard_normal((len(lens), Hq, d)).astype(np.float32)).to(DEV)
        q = q.to(torch.bfloat16) if call == 1 else q
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        got = tq.decode_attn_noalloc(params, d, q, Hkv, kp, vp, bt, ctx, max(lens), status=status)
        want = tq.decode_attn(params, d, q, Hkv, kp, vp, bt, ctx, max(lens))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        parity.check_attention(got.cpu().numpy(), want.cpu().numpy().astype(np.float64))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    d, Hq, Hkv, B = 128, 32, 8, 64
    params, bt1, kp, vp = _cache(d, Hkv, [16], seed=5)
    # the query packs of 64 x 32 heads alone exceed the fixed scratch
    assert tq.decode_workspace_bytes(d, B, Hq, 16) > 16 << 20
    bt = bt1[:1].repeat(B, 1)
    q = torch.zeros((B, Hq, d), device=DEV)
    ctx = torch.full((B,), 16, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError, match="workspace"):
        tq.decode_attn_noalloc(params, d, q, Hkv, kp, vp, bt, ctx, 16)
