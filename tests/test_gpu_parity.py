"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Small cases run the oracle on every output; they span several paged blocks
and context splits with ragged tails.  Tolerances are in tests/parity.py.
"""
import math

import numpy as np
import pytest

import oracle
from tests import parity

torch = pytest.importorskip("torch")
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
FILL = 0xA5


def _params(d):
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    params, cent = tq.codebook_init(d, D, S, device=DEV)
    return D, S, params, cent


def _upload(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).to(DEV)


def _inputs(N, H, d, dtype, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, H, d)).astype(np.float32)
    if outliers:
        x *= rng.lognormal(0, 1, (1, H, d)).astype(np.float32)
        x[:, :, 3] *= 20
    if N > 2:
        x[1] = 0.0          # zero vectors
    return synth.round_dtype(x, dtype)


def _slot_owner(is_k, d):
    """byte offset within a record -> owning slot (from the oracle's layout)."""
    owner = oracle.slot_owner(is_k, d)
    assert (owner >= 0).all()
    return owner


# ------------------------------------------------------------------ codebook

@pytest.mark.parametrize("d", [128, 256])
def test_codebook_on_device(d):
    _, _, params, cent = _params(d)
    c, t, _, _ = oracle.codebook()
    # both sides stop a linearly convergent iteration at a step below 1e-15;
    # the fp32 values the kernels use must be identical (checked below)
    np.testing.assert_allclose(cent, c, rtol=0, atol=1e-12)
    hdr = params[:256].cpu().numpy()
    cf = hdr[16:48].view(np.float32)
    tf = hdr[48:80].view(np.float32)
    np.testing.assert_array_equal(cf, c.astype(np.float32))
    np.testing.assert_array_equal(tf[:7], t.astype(np.float32))
    # S is held at binary16 precision: the test matrix is binary16 already, so it is stored as is
    S = synth.qjl_matrix(d)
    assert np.array_equal(S.astype(np.float16).astype(np.float32), S)
    off = 256 + 4 * d
    sp = params[off:off + 4 * d * d].cpu().numpy().view(np.float32).reshape(d, d)
    np.testing.assert_array_equal(sp, S)


# ------------------------------------------------------------------ encode

@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("is_k", [True, False])
def test_encode_parity(d, dtype, is_k):
    H, N, nblk = 3, 203, 20
    D, S, params, _ = _params(d)
    x = _inputs(N, H, d, dtype, seed=d + (7 if is_k else 0))
    slots = np.random.default_rng(1).permutation(nblk * 16)[:N].astype(np.int64)
    rec = tq.k_record_bytes(d) if is_k else tq.v_record_bytes(d)
    pool = torch.full((nblk, H, rec), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn = tq.encode_k if is_k else tq.encode_v
    fn(params, d, _upload(x, dtype), torch.from_numpy(slots).to(DEV), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gp = pool.cpu().numpy()
    st = parity.check_encode(is_k, D, S, x, slots, gp, pool_fill=FILL)
    assert st["entries"] == N * H * d
    # bytes of slots that were not written keep the fill pattern
    owner = _slot_owner(is_k, d)
    written = np.zeros((nblk, 16), bool)
    written[slots // 16, slots % 16] = True
    for blk in range(nblk):
        untouched = ~written[blk][owner]
        assert np.all(gp[blk][:, untouched] == FILL)


@pytest.mark.parametrize("d,H", [(128, 8), (128, 2), (128, 3), (256, 8), (256, 4)])
def test_encode_v_whole_blocks_and_exceptions(d, H):
    """Bulk V encodes whose 16-token blocks map to whole records in token order take the
    assembled-record path; blocks broken in several ways must still match the oracle: two tokens
    swapped, a block shifted off the 16-slot alignment, a ragged last tile, and (H = 3) every tile."""
    D, S, params, _ = _params(d)
    nb_tok = 24                                          # 16-token blocks of input
    N = 16 * nb_tok + 5
    nblk = nb_tok + 8
    perm = np.random.default_rng(H).permutation(nblk)
    slots = np.concatenate([perm[t // 16] * 16 + np.arange(16) for t in range(0, 16 * (nb_tok + 1), 16)])[:N]
    slots = slots.astype(np.int64)
    slots[[16 * 3 + 2, 16 * 3 + 9]] = slots[[16 * 3 + 9, 16 * 3 + 2]]   # block 3: two tokens swapped
    slots[16 * 7:16 * 8] = perm[nb_tok + 2] * 16 + (np.arange(16) + 5) % 16   # block 7: rotated offsets
    slots[16 * 11:16 * 12] = -1                                           # block 11: padding, skipped
    x = _inputs(N, H, d, "bf16", seed=H + 100 + d, outliers=False)
    pool = torch.full((nblk, H, tq.v_record_bytes(d)), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.encode_v(params, d, _upload(x, "bf16"), torch.from_numpy(slots).to(DEV), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gp = pool.cpu().numpy()
    ok = slots >= 0
    parity.check_encode(False, D, S, x[ok], slots[ok], gp, pool_fill=FILL)
    owner = _slot_owner(False, d)
    written = np.zeros((nblk, 16), bool)
    written[slots[ok] // 16, slots[ok] % 16] = True
    for blk in range(nblk):
        assert np.all(gp[blk][:, ~written[blk][owner]] == FILL)


def test_encode_skips_bad_slots_and_flags():
    d, H = 128, 2
    D, S, params, _ = _params(d)
    x = _inputs(5, H, d, "f32", seed=3)
    slots = np.array([0, 17, -1, 10_000, 33], np.int64)
    pool = torch.full((4, H, tq.k_record_bytes(d)), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.encode_k(params, d, _upload(x, "f32"), torch.from_numpy(slots).to(DEV), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & tq.STATUS_BAD_SLOT
    ok = np.array([0, 1, 4])
    parity.check_encode(True, D, S, x[ok], slots[ok], pool.cpu().numpy(), pool_fill=FILL)


@pytest.mark.parametrize("d", [128, 256])
def test_paged_append_parity(d):
    H, B = 2, 6
    D, S, params, _ = _params(d)
    lens = np.array([0, 15, 16, 33, 100, -1], np.int32)      # -1: skipped
    mb = 8
    bt = np.random.default_rng(5).permutation(B * mb).reshape(B, mb).astype(np.int32)
    nblk = B * mb
    kp = torch.full((nblk, H, tq.k_record_bytes(d)), FILL, dtype=torch.uint8, device=DEV)
    vp = torch.full((nblk, H, tq.v_record_bytes(d)), FILL, dtype=torch.uint8, device=DEV)
    k = _inputs(B, H, d, "bf16", seed=11)
    v = _inputs(B, H, d, "bf16", seed=12)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.paged_append(params, d, _upload(k, "bf16"), _upload(v, "bf16"), torch.from_numpy(bt).to(DEV),
                    torch.from_numpy(lens).to(DEV), kp, vp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.array([b for b in range(B) if lens[b] >= 0])
    slots = np.array([bt[b, lens[b] // 16] * 16 + lens[b] % 16 for b in sel], np.int64)
    parity.check_encode(True, D, S, k[sel], slots, kp.cpu().numpy(), pool_fill=FILL)
    parity.check_encode(False, D, S, v[sel], slots, vp.cpu().numpy(), pool_fill=FILL)
    for pool, is_k in ((kp, True), (vp, False)):
        gp = pool.cpu().numpy()
        owner = _slot_owner(is_k, d)
        written = np.zeros((nblk, 16), bool)
        written[slots // 16, slots % 16] = True
        for blk in range(nblk):
            assert np.all(gp[blk][:, ~written[blk][owner]] == FILL)


# ------------------------------------------------------------------ decode

def _build_cache(d, Hkv, lens, dtype, seed, spare=3):
    """Paged cache written by the oracle (CPU) and uploaded: the GPU decode and
    the oracle decode then read the very same packed records."""
    D, S, params, _ = _params(d)
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
    kp = np.zeros((nblk, Hkv, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nblk, Hkv, oracle.record_bytes(False, d)), np.uint8)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        K = _inputs(L, Hkv, d, dtype, seed=seed * 100 + b)
        V = _inputs(L, Hkv, d, dtype, seed=seed * 100 + b + 50, outliers=False)
        sl = synth.slots_for(bt, b, 0, L)
        oracle.encode(True, D, S, K, sl, kp)
        oracle.encode(False, D, S, V, sl, vp)
    return D, S, params, bt, kp, vp


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 4, 1), (128, 8, 2), (128, 16, 2), (128, 3, 3), (256, 4, 2)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_parity(d, Hq, Hkv, dtype):
    lens = [1, 17, 512, 513, 1100, 0, 16, 700]
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, dtype, seed=Hq + d)
    B = len(lens)
    q = synth.round_dtype(np.random.default_rng(9).standard_normal((B, Hq, d)).astype(np.float32), dtype)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn(params, d, _upload(q, dtype), Hkv, torch.from_numpy(kp).to(DEV),
                         torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV), ctx, max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    ref = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32))
    assert np.all(o[lens.index(0)] == 0)
    parity.check_attention(o, ref)


@pytest.mark.parametrize("d,Hq,Hkv,lens", [
    (128, 16, 4, [9000, 3000, 12000, 700, 5000, 1, 129, 128]),   # more chunks than resident CTAs
    (128, 32, 4, [7000, 2500, 10000, 300, 4100, 17]),             # groups of 8: 256-token chunks
    (256, 4, 2, [20000, 7000, 0, 33]),                            # d=256, long contexts
])
def test_decode_parity_many_chunks(d, Hq, Hkv, lens):
    """Contexts long enough that CTAs cover several chunks of one (sequence,
    kv head), several units, and units shared by many CTAs."""
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "bf16", seed=Hq + d + 7)
    B = len(lens)
    q = synth.round_dtype(np.random.default_rng(11).standard_normal((B, Hq, d)).astype(np.float32), "bf16")
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn(params, d, _upload(q, "bf16"), Hkv, torch.from_numpy(kp).to(DEV),
                         torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV), ctx, max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32))
    parity.check_attention(out.cpu().numpy(), ref)


def test_decode_stages_equal_decode_attn():
    """tq_decode_qprep then tq_decode_splitk give exactly tq_decode_attn's output."""
    d, Hq, Hkv = 128, 8, 2
    lens = [3000, 40, 0, 1500]
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "f32", seed=3)
    B = len(lens)
    q = _upload(np.random.default_rng(5).standard_normal((B, Hq, d)).astype(np.float32), "f32")
    kp, vp, bt = torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    want = tq.decode_attn(params, d, q, Hkv, kp, vp, bt, ctx, max(lens))
    ws = torch.empty(tq.decode_workspace_bytes(d, B, Hq, max(lens)), dtype=torch.uint8, device=DEV)
    got = torch.full((B, Hq, d), float("nan"), device=DEV)
    for _ in range(2):   # the second round reuses counters and schedule left by the first
        tq.decode_qprep(params, d, q, Hkv, ctx, max(lens), ws)
        tq.decode_splitk(params, d, B, Hq, Hkv, kp, vp, bt, ctx, max(lens), got, ws)
        torch.cuda.synchronize()
        assert torch.equal(got, want)


@pytest.mark.parametrize("d,Hq,Hkv,dtype", [(128, 8, 2, "bf16"), (128, 4, 4, "f32"), (256, 4, 2, "bf16")])
def test_decode_step_appends_then_attends(d, Hq, Hkv, dtype):
    """tq_decode_step on a cache of pre_lens[b] tokens equals the oracle's attention over
    pre_lens[b] + 1 tokens (the oracle encodes every token itself, the new one included),
    and equals tq_paged_append followed by tq_decode_attn bit for bit."""
    pre = [15, 600, -1, 129, 0, 1023]
    B = len(pre)
    full = [p + 1 if p >= 0 else 0 for p in pre]
    D, S, params, _ = _params(d)
    need = [max(1, -(-L // 16)) for L in full]
    nblk = sum(need) + 2
    perm = np.random.default_rng(17).permutation(nblk)
    bt = np.zeros((B, max(need)), np.int32)
    k0 = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k0:k0 + n]
        k0 += n
    kp_pre = np.zeros((nblk, Hkv, oracle.record_bytes(True, d)), np.uint8)
    vp_pre = np.zeros((nblk, Hkv, oracle.record_bytes(False, d)), np.uint8)
    kp_full, vp_full = kp_pre.copy(), vp_pre.copy()
    k_new = np.zeros((B, Hkv, d), np.float32)
    v_new = np.zeros((B, Hkv, d), np.float32)
    for b, L in enumerate(full):
        if L == 0:
            continue
        rng = np.random.default_rng([23, b])
        K = synth.round_dtype(rng.standard_normal((L, Hkv, d)).astype(np.float32) * 2, dtype)
        V = synth.round_dtype(rng.standard_normal((L, Hkv, d)).astype(np.float32), dtype)
        sl = synth.slots_for(bt, b, 0, L)
        oracle.encode(True, D, S, K, sl, kp_full)
        oracle.encode(False, D, S, V, sl, vp_full)
        if L > 1:
            oracle.encode(True, D, S, K[:-1], sl[:-1], kp_pre)
            oracle.encode(False, D, S, V[:-1], sl[:-1], vp_pre)
        k_new[b], v_new[b] = K[-1], V[-1]
    q = synth.round_dtype(np.random.default_rng(29).standard_normal((B, Hq, d)).astype(np.float32), dtype)
    max_ctx = max(full)
    dq, dk, dv = _upload(q, dtype), _upload(k_new, dtype), _upload(v_new, dtype)
    dbt = torch.from_numpy(bt).to(DEV)
    pre_t = torch.tensor(pre, dtype=torch.int32, device=DEV)
    kp1, vp1 = torch.from_numpy(kp_pre).to(DEV), torch.from_numpy(vp_pre).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_step(params, d, dk, dv, dq, Hkv, kp1, vp1, dbt, pre_t, max_ctx, status=status)
    kp2, vp2 = torch.from_numpy(kp_pre).to(DEV), torch.from_numpy(vp_pre).to(DEV)
    tq.paged_append(params, d, dk, dv, dbt, pre_t, kp2, vp2)
    full_t = torch.tensor(full, dtype=torch.int32, device=DEV)
    want = tq.decode_attn(params, d, dq, Hkv, kp2, vp2, dbt, full_t, max_ctx)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kp1, kp2) and torch.equal(vp1, vp2)
    assert torch.equal(out, want)
    ref = oracle.decode(D, S, q, Hkv, kp_full, vp_full, bt, np.array(full, np.int32))
    o = out.cpu().numpy()
    assert np.all(o[pre.index(-1)] == 0)
    parity.check_attention(o, ref)


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (256, 16, 8)])
def test_decode_step_in_a_cuda_graph(d, Hq, Hkv):
    """The step captured once in a CUDA graph (both launches, the pass as a programmatic dependent
    of the prep) and replayed: each replay equals a direct tq_decode_step bit for bit, and the
    appended records are the same."""
    lens = [1000, 17, 4095, 250]   # none a multiple of 16: the new token lands in the sequence's own last block
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "bf16", seed=31)
    B = len(lens)
    rng = np.random.default_rng(37)
    dbt = torch.from_numpy(bt).to(DEV)
    pre = torch.tensor(lens, dtype=torch.int32, device=DEV)
    max_ctx = max(lens) + 1
    ws = torch.empty(tq.decode_workspace_bytes(d, B, Hq, max_ctx), dtype=torch.uint8, device=DEV)
    q = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=DEV)
    k_new = torch.empty((B, Hkv, d), dtype=torch.bfloat16, device=DEV)
    v_new = torch.empty_like(k_new)
    kp_g, vp_g = torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV)
    out_g = torch.empty((B, Hq, d), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # warm-up call (attribute setup) outside the capture
        tq.decode_step(params, d, k_new.zero_(), v_new.zero_(), q.zero_(), Hkv, kp_g.clone(), vp_g.clone(), dbt,
                       pre, max_ctx, out=out_g, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tq.decode_step(params, d, k_new, v_new, q, Hkv, kp_g, vp_g, dbt, pre, max_ctx, out=out_g, workspace=ws)
    for rep in range(3):
        q.copy_(torch.from_numpy(rng.standard_normal((B, Hq, d)).astype(np.float32)).to(torch.bfloat16))
        k_new.copy_(torch.from_numpy(rng.standard_normal((B, Hkv, d)).astype(np.float32)).to(torch.bfloat16))
        v_new.copy_(torch.from_numpy(rng.standard_normal((B, Hkv, d)).astype(np.float32)).to(torch.bfloat16))
        kp_d, vp_d = kp_g.clone(), vp_g.clone()
        torch.cuda.synchronize()
        g.replay()
        want = tq.decode_step(params, d, k_new, v_new, q, Hkv, kp_d, vp_d, dbt, pre, max_ctx)
        torch.cuda.synchronize()
        assert torch.equal(out_g, want), f"replay {rep}"
        assert torch.equal(kp_g, kp_d) and torch.equal(vp_g, vp_d)


@pytest.mark.parametrize("d,Hq,Hkv,Q", [(128, 8, 2, 2), (128, 4, 2, 4), (128, 3, 3, 3), (128, 2, 2, 8),
                                         (256, 4, 2, 2), (256, 1, 1, 5)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_mq_parity(d, Hq, Hkv, Q, dtype):
    """Multi-query decode: query i of Q attends the first ctx - (Q - 1 - i) tokens.  Lengths below Q
    leave the first queries with nothing to attend (out = 0)."""
    lens = [1, 17, 512, 513, 1100, 0, 16, 700, 2, 3]
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, dtype, seed=Hq + d + Q)
    B = len(lens)
    q = synth.round_dtype(np.random.default_rng(12).standard_normal((B, Q, Hq, d)).astype(np.float32), dtype)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn_mq(params, d, _upload(q, dtype), Hkv, torch.from_numpy(kp).to(DEV),
                            torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV), ctx, max(lens), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    ref = oracle.decode_mq(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32))
    for b, L in enumerate(lens):
        for i in range(Q):
            if L - (Q - 1 - i) <= 0:
                assert np.all(o[b, i] == 0)
    parity.check_attention(o.reshape(B * Q, Hq, d), ref.reshape(B * Q, Hq, d))


def test_decode_mq_single_query_is_decode_attn():
    """q_len = 1 through the multi-query entry point is tq_decode_attn, bit for bit."""
    d, Hq, Hkv = 128, 8, 2
    lens = [3000, 40, 0, 1500]
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "bf16", seed=31)
    B = len(lens)
    q = _upload(np.random.default_rng(6).standard_normal((B, 1, Hq, d)).astype(np.float32), "bf16")
    kp, vp, bt = torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    a = tq.decode_attn_mq(params, d, q, Hkv, kp, vp, bt, ctx, max(lens))
    b = tq.decode_attn(params, d, q[:, 0].contiguous(), Hkv, kp, vp, bt, ctx, max(lens))
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


@pytest.mark.parametrize("d,Hq,Hkv,Q,dtype", [(128, 8, 2, 2, "bf16"), (128, 2, 2, 4, "f32"), (256, 4, 2, 2, "bf16")])
def test_decode_step_mq_appends_then_attends(d, Hq, Hkv, Q, dtype):
    """tq_decode_step_mq on a cache of pre_lens[b] tokens: the Q new tokens land at pre_lens[b] + i
    (bit-exact against one tq_paged_append per token), the Q queries then equal tq_decode_attn_mq
    over pre_lens + Q tokens bit for bit, and the oracle's multi-query attention within tolerance."""
    pre = [15, 600, -1, 129, 0, 1022]
    B = len(pre)
    full = [p + Q if p >= 0 else 0 for p in pre]
    D, S, params, _ = _params(d)
    need = [max(1, -(-L // 16)) for L in full]
    nblk = sum(need) + 2
    perm = np.random.default_rng(19).permutation(nblk)
    bt = np.zeros((B, max(need)), np.int32)
    k0 = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k0:k0 + n]
        k0 += n
    kp_pre = np.zeros((nblk, Hkv, oracle.record_bytes(True, d)), np.uint8)
    vp_pre = np.zeros((nblk, Hkv, oracle.record_bytes(False, d)), np.uint8)
    kp_full, vp_full = kp_pre.copy(), vp_pre.copy()
    k_new = np.zeros((B, Q, Hkv, d), np.float32)
    v_new = np.zeros((B, Q, Hkv, d), np.float32)
    for b, L in enumerate(full):
        if L == 0:
            continue
        rng = np.random.default_rng([29, b])
        K = synth.round_dtype(rng.standard_normal((L, Hkv, d)).astype(np.float32) * 2, dtype)
        V = synth.round_dtype(rng.standard_normal((L, Hkv, d)).astype(np.float32), dtype)
        sl = synth.slots_for(bt, b, 0, L)
        oracle.encode(True, D, S, K, sl, kp_full)
        oracle.encode(False, D, S, V, sl, vp_full)
        if L > Q:
            oracle.encode(True, D, S, K[:-Q], sl[:-Q], kp_pre)
            oracle.encode(False, D, S, V[:-Q], sl[:-Q], vp_pre)
        k_new[b], v_new[b] = K[-Q:], V[-Q:]
    q = synth.round_dtype(np.random.default_rng(37).standard_normal((B, Q, Hq, d)).astype(np.float32), dtype)
    max_ctx = max(full)
    dq, dk, dv = _upload(q, dtype), _upload(k_new, dtype), _upload(v_new, dtype)
    dbt = torch.from_numpy(bt).to(DEV)
    pre_t = torch.tensor(pre, dtype=torch.int32, device=DEV)
    kp1, vp1 = torch.from_numpy(kp_pre).to(DEV), torch.from_numpy(vp_pre).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_step_mq(params, d, dk, dv, dq, Hkv, kp1, vp1, dbt, pre_t, max_ctx, status=status)
    kp2, vp2 = torch.from_numpy(kp_pre).to(DEV), torch.from_numpy(vp_pre).to(DEV)
    for i in range(Q):
        pos = torch.tensor([p + i if p >= 0 else -1 for p in pre], dtype=torch.int32, device=DEV)
        tq.paged_append(params, d, dk[:, i].contiguous(), dv[:, i].contiguous(), dbt, pos, kp2, vp2)
    full_t = torch.tensor(full, dtype=torch.int32, device=DEV)
    want = tq.decode_attn_mq(params, d, dq, Hkv, kp2, vp2, dbt, full_t, max_ctx)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kp1, kp2) and torch.equal(vp1, vp2)
    assert torch.equal(out, want)
    ref = oracle.decode_mq(D, S, q, Hkv, kp_full, vp_full, bt, np.array(full, np.int32))
    o = out.cpu().numpy()
    assert np.all(o[pre.index(-1)] == 0)
    parity.check_attention(o.reshape(B * Q, Hq, d), ref.reshape(B * Q, Hq, d))


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("is_k", [True, False])
def test_dequant_parity(d, is_k):
    """Dense K / V of whole blocks against the oracle's reconstruction: fp32 output within 1e-5
    relative per vector, bf16 output within one bf16 rounding of the fp32 result; a bad block
    id gives zero rows and sets the status."""
    Hkv = 3
    lens = [40, 70, 16]
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "f32", seed=41 + d)
    pool_np = kp if is_k else vp
    pool = torch.from_numpy(pool_np).to(DEV)
    ids_np = np.concatenate([bt[b, :-(-L // 16)] for b, L in enumerate(lens)]).astype(np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    fn = tq.dequant_k if is_k else tq.dequant_v
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o32 = fn(params, d, pool, ids, out_dtype=torch.float32, status=status)
    o16 = fn(params, d, pool, ids, out_dtype=torch.bfloat16, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.dequant(is_k, D, S, pool_np, Hkv, ids_np)
    g = o32.cpu().numpy().astype(np.float64)
    err = np.linalg.norm(g - ref, axis=-1) / np.maximum(np.linalg.norm(ref, axis=-1), 1e-30)
    assert err.max() < 1e-5, err.max()
    b16 = o16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(b16 - g) <= np.abs(g) * 2.0 ** -8 + 1e-30)
    # an id outside the pool: zero rows, status flagged
    bad = torch.tensor([ids_np[0], pool.shape[0] + 5], dtype=torch.int32, device=DEV)
    ob = fn(params, d, pool, bad, out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1            # TQ_STATUS_BAD_SLOT
    assert torch.all(ob[16:] == 0) and torch.equal(ob[:16], o32[:16])


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 8, 2), (128, 4, 4), (128, 16, 2), (256, 4, 2)])
@pytest.mark.parametrize("wdtype", ["f32", "bf16"])
def test_decode_hybrid_parity(d, Hq, Hkv, wdtype):
    """One softmax over the compressed history and an uncompressed window (ragged lengths, an
    empty history, an empty window, both empty) against the oracle; win_cap = 0 is
    tq_decode_attn bit for bit."""
    lens = [600, 0, 17, 1500, 33, 0]
    wl = [300, 129, 0, 128, 5, 0]
    cap = 300
    D, S, params, bt, kp, vp = _build_cache(d, Hkv, lens, "bf16", seed=Hq + d + 5)
    B = len(lens)
    rng = np.random.default_rng(51)
    q = synth.round_dtype(rng.standard_normal((B, Hq, d)).astype(np.float32), "bf16")
    wk = synth.round_dtype(rng.standard_normal((B, cap, Hkv, d)).astype(np.float32) * 2, wdtype)
    wv = synth.round_dtype(rng.standard_normal((B, cap, Hkv, d)).astype(np.float32), wdtype)
    dkp, dvp, dbt = torch.from_numpy(kp).to(DEV), torch.from_numpy(vp).to(DEV), torch.from_numpy(bt).to(DEV)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    wlt = torch.tensor(wl, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dq = _upload(q, "bf16")
    out = tq.decode_attn_hybrid(params, d, dq, Hkv, dkp, dvp, dbt, ctx, max(lens), _upload(wk, wdtype),
                                _upload(wv, wdtype), wlt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out.cpu().numpy()
    ref = oracle.decode_hybrid(D, S, q, Hkv, kp, vp, bt, lens, wk, wv, wl)
    assert np.all(o[5] == 0)
    parity.check_attention(o, ref)
    # no window at all: exactly the compressed decode
    e = torch.zeros((B, 0, Hkv, d), dtype=torch.float32, device=DEV)
    o0 = tq.decode_attn_hybrid(params, d, dq, Hkv, dkp, dvp, dbt, ctx, max(lens), e, e, wlt)
    want = tq.decode_attn(params, d, dq, Hkv, dkp, dvp, dbt, ctx, max(lens))
    torch.cuda.synchronize()
    assert torch.equal(o0, want)


def test_tiny_workload_end_to_end():
    """1 sequence, 1 head, d=128, 256 fp32 tokens with 20x outlier channels:
    GPU encode vs oracle encode, then GPU decode vs oracle decode of the
    oracle-written cache."""
    w = synth.workload("tiny")
    from turboquant_compressed_kv_gb300.cache import PagedCache
    cache = PagedCache.create(w, DEV)
    cache.prefill()
    K, V = synth.kv_tokens(w, 0, 0, 256)
    slots = synth.slots_for(cache.block_table_np, 0, 0, 256)
    parity.check_encode(True, cache.D, cache.S, K, slots, cache.k_pool.cpu().numpy())
    parity.check_encode(False, cache.D, cache.S, V, slots, cache.v_pool.cpu().numpy())
    kp = np.zeros(tuple(cache.k_pool.shape), np.uint8)
    vp = np.zeros(tuple(cache.v_pool.shape), np.uint8)
    oracle.encode(True, cache.D, cache.S, K, slots, kp)
    oracle.encode(False, cache.D, cache.S, V, slots, vp)
    q = synth.queries(w)
    out = tq.decode_attn(cache.params, 128, _upload(q, "f32"), 1, torch.from_numpy(kp).to(DEV),
                         torch.from_numpy(vp).to(DEV), cache.block_table,
                         torch.tensor([256], dtype=torch.int32, device=DEV), 256)
    ref = oracle.decode(cache.D, cache.S, q, 1, kp, vp, cache.block_table_np, np.array([256], np.int32))
    parity.check_attention(out.cpu().numpy(), ref)


def test_decode_rejects_bad_arguments():
    d = 128
    _, _, params, _ = _params(d)
    q = torch.zeros((1, 4, d), device=DEV)
    kp = tq.empty_pool(1, 1, d, "k", DEV)
    vp = tq.empty_pool(1, 1, d, "v", DEV)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=DEV)
    ctx = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError, match="multiple"):
        tq.decode_attn(params, d, q, 3, kp, vp, bt, ctx, 16)
    with pytest.raises(tq.TQError, match="head_dim"):
        tq.decode_attn(params, 64, q, 1, kp, vp, bt, ctx, 16)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError, match="workspace"):
        tq.decode_attn(params, d, q, 1, kp, vp, bt, ctx, 16, workspace=ws)


def test_decode_bad_block_id_is_flagged():
    d = 128
    D, S, params, bt, kp, vp = _build_cache(d, 1, [40], "f32", seed=2)
    kp = torch.from_numpy(kp).to(DEV)
    vp = torch.from_numpy(vp).to(DEV)
    bt_bad = bt.copy()
    bt_bad[0, 1] = 10_000
    q = np.random.default_rng(0).standard_normal((1, 2, d)).astype(np.float32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = tq.decode_attn(params, d, _upload(q, "f32"), 1, kp, vp, torch.from_numpy(bt_bad).to(DEV),
                         torch.tensor([40], dtype=torch.int32, device=DEV), 40, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & tq.STATUS_BAD_SLOT
    assert np.all(np.isfinite(out.cpu().numpy()))
