"""GPU parity of the group-quantised comparator (tq_gq_*) against its oracle (oracle/gq.py).

The codes, fp16 scales and biases are integers decided in fp32 on both sides, so the packed
pools must be byte-identical; decode attention is held to the same tolerance as TurboQuant's
(tests/parity.py), with both sides reading the same packed cache.
"""
import numpy as np
import pytest

from oracle import gq
from tests import parity

torch = pytest.importorskip("torch")
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
FILL = 0xA5


def _upload(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).to(DEV)


def _inputs(N, H, d, dtype, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, H, d)).astype(np.float32)
    x *= rng.lognormal(0, 1, (1, H, d)).astype(np.float32)
    x[:, :, 3] *= 20
    if N > 4:
        x[2] = 0.0                       # an all-zero vector: scale 0, codes 0
        x[3, :, :] = 1.5                 # constant groups
    return synth.round_dtype(x, dtype)


@pytest.mark.parametrize("d,bits,group", [(128, 4, 64), (128, 8, 64), (128, 4, 32), (128, 8, 128),
                                          (256, 4, 64), (256, 8, 32), (256, 4, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gq_encode_parity(d, bits, group, dtype):
    N, H, nb = 300, 3, 24
    x = _inputs(N, H, d, dtype, seed=d + bits + group)
    rng = np.random.default_rng(7)
    slots = rng.permutation(nb * 16)[:N].astype(np.int64)
    slots[::37] = -1                     # padding
    rec = gq.record_bytes(d, bits, group)
    assert tq.gq_record_bytes(d, bits, group) == rec
    pool = torch.full((nb, H, rec), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.gq_encode(d, bits, group, _upload(x, dtype), torch.from_numpy(slots).to(DEV), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = np.full(nb * H * rec, FILL, np.uint8)
    c, s, z = gq.encode(x, bits, group)
    gq.pack(c, s, z, slots, ref, H, bits, group)
    got = pool.cpu().numpy().reshape(-1)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


def test_gq_encode_flags_bad_slots():
    d, H, nb = 128, 2, 4
    x = _inputs(8, H, d, "bf16", seed=1)
    slots = np.array([0, 5, nb * 16, -3, 17, nb * 16 + 40, 2, 63], np.int64)
    rec = gq.record_bytes(d, 4, 64)
    pool = torch.full((nb, H, rec), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.gq_encode(d, 4, 64, _upload(x, "bf16"), torch.from_numpy(slots).to(DEV), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & tq.STATUS_BAD_SLOT
    ref = np.full(nb * H * rec, FILL, np.uint8)
    c, s, z = gq.encode(x, 4, 64)
    keep = slots < nb * 16
    gq.pack(c[keep], s[keep], z[keep], slots[keep], ref, H, 4, 64)
    assert np.array_equal(pool.cpu().numpy().reshape(-1), ref)


def _gq_cache(d, Hkv, lens, bits, group, dtype, seed, spare=3):
    """Paged group-quantised cache written by the oracle and uploaded."""
    B = len(lens)
    need = [max(1, -(-L // 16)) for L in lens]
    mb = max(need)
    nblk = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(nblk)
    bt = np.zeros((B, mb), np.int32)
    k0 = 0
    for b in range(B):
        bt[b, :need[b]] = perm[k0:k0 + need[b]]
        k0 += need[b]
    rec = gq.record_bytes(d, bits, group)
    kp = np.zeros(nblk * Hkv * rec, np.uint8)
    vp = np.zeros_like(kp)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        K = _inputs(L, Hkv, d, dtype, seed=seed * 100 + b)
        V = _inputs(L, Hkv, d, dtype, seed=seed * 100 + b + 50)
        sl = synth.slots_for(bt, b, 0, L)
        gq.pack(*gq.encode(K, bits, group), sl, kp, Hkv, bits, group)
        gq.pack(*gq.encode(V, bits, group), sl, vp, Hkv, bits, group)
    return bt, kp.reshape(nblk, Hkv, rec), vp.reshape(nblk, Hkv, rec)


@pytest.mark.parametrize("d,Hq,Hkv,bits,group", [
    (128, 4, 1, 4, 64), (128, 8, 2, 8, 64), (128, 16, 2, 4, 32), (128, 3, 3, 8, 128),
    (128, 12, 2, 4, 64), (256, 4, 2, 4, 64), (256, 2, 2, 8, 32)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gq_decode_parity(d, Hq, Hkv, bits, group, dtype):
    lens = [1, 17, 300, 0, 129, 700, 128]
    bt, kp, vp = _gq_cache(d, Hkv, lens, bits, group, dtype, seed=Hq + d + bits)
    B = len(lens)
    q = synth.round_dtype(np.random.default_rng(9).standard_normal((B, Hq, d)).astype(np.float32), dtype)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.gq_decode_attn(d, bits, group, _upload(q, dtype), Hkv, torch.from_numpy(kp).to(DEV),
                            torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV), ctx, max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    ref = gq.decode(q, Hkv, kp, vp, bt, np.array(lens, np.int32), bits, group)
    assert np.all(o[lens.index(0)] == 0)
    parity.check_attention(o, ref)


def test_gq_gpu_encode_then_decode():
    """The whole comparator on the device: encode K and V, decode, against the oracle
    decoding the pools the GPU wrote."""
    d, Hq, Hkv, bits, group = 128, 8, 2, 4, 64
    lens = [200, 33, 1000]
    B, nblk = len(lens), 200
    rng = np.random.default_rng(3)
    bt = rng.permutation(nblk)[:B * 63].reshape(B, 63).astype(np.int32)
    rec = gq.record_bytes(d, bits, group)
    kp = torch.zeros((nblk, Hkv, rec), dtype=torch.uint8, device=DEV)
    vp = torch.zeros_like(kp)
    for b, L in enumerate(lens):
        K = _inputs(L, Hkv, d, "bf16", seed=20 + b)
        V = _inputs(L, Hkv, d, "bf16", seed=40 + b)
        sl = torch.from_numpy(synth.slots_for(bt, b, 0, L)).to(DEV)
        tq.gq_encode(d, bits, group, _upload(K, "bf16"), sl, kp)
        tq.gq_encode(d, bits, group, _upload(V, "bf16"), sl, vp)
    q = synth.round_dtype(rng.standard_normal((B, Hq, d)).astype(np.float32), "bf16")
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.gq_decode_attn(d, bits, group, _upload(q, "bf16"), Hkv, kp, vp, torch.from_numpy(bt).to(DEV), ctx,
                            max(lens))
    torch.cuda.synchronize()
    ref = gq.decode(q, Hkv, kp.cpu().numpy(), vp.cpu().numpy(), bt, np.array(lens, np.int32), bits, group)
    parity.check_attention(out.cpu().numpy(), ref)


def test_gq_decode_bad_block_id_is_flagged():
    d, Hq, Hkv, bits, group = 128, 4, 1, 8, 64
    lens = [40, 40]
    bt, kp, vp = _gq_cache(d, Hkv, lens, bits, group, "bf16", seed=5)
    bt[1, 1] = kp.shape[0] + 7            # sequence 1, tokens 16..31: outside the pool
    q = synth.round_dtype(np.random.default_rng(2).standard_normal((2, Hq, d)).astype(np.float32), "bf16")
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.gq_decode_attn(d, bits, group, _upload(q, "bf16"), Hkv, torch.from_numpy(kp).to(DEV),
                            torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV), ctx, max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & tq.STATUS_BAD_SLOT
    o = out.cpu().numpy()
    assert np.isfinite(o).all()
    ref = gq.decode(q[:1], Hkv, kp, vp, bt[:1], np.array(lens[:1], np.int32), bits, group)
    parity.check_attention(o[:1], ref)     # the other sequence is untouched


def test_gq_rejects_bad_arguments():
    x = torch.zeros((4, 1, 128), dtype=torch.bfloat16, device=DEV)
    sl = torch.zeros(4, dtype=torch.int64, device=DEV)
    pool = torch.zeros((1, 1, gq.record_bytes(128, 4, 64)), dtype=torch.uint8, device=DEV)
    for bits, group in ((3, 64), (4, 48), (8, 256)):
        with pytest.raises(tq.TQError):
            tq.gq_encode(128, bits, group, x, sl, pool)
    with pytest.raises(tq.TQError):
        tq.gq_encode(96, 4, 32, x, sl, pool)
