"""tq_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (a runtime that reserved all GPU memory up front, or a
decode loop that must not call cudaMalloc).  It runs the same kernels as
tq_decode_attn with a caller workspace, so its output must be identical to
that call's, bit for bit, call after call, although every call reuses the
same fixed scratch array inside the library (left holding whatever the last
call wrote).

This file is collected last on purpose, and it builds all its own inputs, so
it passes both alone in a fresh process and after the other tests."""
import numpy as np
import pytest

from tests import parity

torch = pytest.importorskip("torch")
import oracle  # noqa: E402
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _table(lens, seed):
    need = [max(1, -(-L // 16)) for L in lens]
    nblk = sum(need) + 2
    perm = np.random.default_rng(seed).permutation(nblk)
    bt = np.zeros((len(lens), max(need)), np.int32)
    k0 = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k0:k0 + n]
        k0 += n
    return bt, nblk


def _cache(d, Hkv, lens, seed):
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    bt, nblk = _table(lens, seed)
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


def _both(params, d, q, Hkv, kp, vp, bt, ctx, max_ctx):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tq.decode_attn_noalloc(params, d, q, Hkv, kp, vp, bt, ctx, max_ctx, status=status)
    want = tq.decode_attn(params, d, q, Hkv, kp, vp, bt, ctx, max_ctx)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return got, want


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (256, 8, 4)])
def test_noalloc_equals_workspace_decode_on_two_calls(d, Hq, Hkv):
    lens = [1, 600, 4096, 0, 1500]
    params, bt, kp, vp = _cache(d, Hkv, lens, seed=d)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    rng = np.random.default_rng(3)
    for call in range(2):
        q = torch.from_numpy(rng.standard_normal((len(lens), Hq, d)).astype(np.float32)).to(DEV)
        q = q.to(torch.bfloat16) if call == 1 else q
        got, want = _both(params, d, q, Hkv, kp, vp, bt, ctx, max(lens))
        assert torch.equal(got, want)


def test_noalloc_after_a_larger_call_that_left_garbage():
    """A larger call (more sequences, longer contexts, a NaN query) fills the scratch with packs and
    partials of its own; the smaller call after it must read none of them."""
    d, Hq, Hkv = 128, 16, 4
    big = [4000, 3000, 17, 2500, 0, 3900, 1024, 2048]
    params, bt, kp, vp = _cache(d, Hkv, big, seed=11)
    ctx = torch.tensor(big, dtype=torch.int32, device=DEV)
    q_nan = torch.full((len(big), Hq, d), float("nan"), device=DEV)
    tq.decode_attn_noalloc(params, d, q_nan, Hkv, kp, vp, bt, ctx, max(big))
    q_big = torch.from_numpy(np.random.default_rng(5).standard_normal((len(big), Hq, d)).astype(np.float32)).to(DEV)
    got, want = _both(params, d, q_big, Hkv, kp, vp, bt, ctx, max(big))
    assert torch.equal(got, want)
    tq.decode_attn_noalloc(params, d, q_nan, Hkv, kp, vp, bt, ctx, max(big))   # garbage again
    small = [700, 33]
    ctx_s = torch.tensor(small, dtype=torch.int32, device=DEV)
    q_s = torch.from_numpy(np.random.default_rng(6).standard_normal((2, Hq, d)).astype(np.float32)).to(DEV)
    got, want = _both(params, d, q_s, Hkv, kp, vp, bt[:2], ctx_s, 4000)
    assert torch.isfinite(got).all()
    assert torch.equal(got, want)


def test_noalloc_matches_the_oracle_on_an_oracle_written_cache():
    """The cache is written by the oracle's encoder (no GPU encode involved); the no-allocation
    decode must match the oracle's decode of the same records within the attention tolerance."""
    d, Hq, Hkv = 128, 8, 2
    lens = [300, 47, 0, 129]
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    bt, nblk = _table(lens, seed=21)
    kp = np.zeros((nblk, Hkv, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nblk, Hkv, oracle.record_bytes(False, d)), np.uint8)
    rng = np.random.default_rng(22)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        sl = synth.slots_for(bt, b, 0, L)
        oracle.encode(True, D, S, (rng.standard_normal((L, Hkv, d)) * 2).astype(np.float32), sl, kp)
        oracle.encode(False, D, S, rng.standard_normal((L, Hkv, d)).astype(np.float32), sl, vp)
    q = rng.standard_normal((len(lens), Hq, d)).astype(np.float32)
    ref = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32))
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tq.decode_attn_noalloc(params, d, torch.from_numpy(q).to(DEV), Hkv, torch.from_numpy(kp).to(DEV),
                                 torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV),
                                 torch.tensor(lens, dtype=torch.int32, device=DEV), max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    parity.check_attention(got.cpu().numpy(), ref)


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
