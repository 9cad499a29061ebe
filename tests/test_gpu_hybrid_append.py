"""GPU parity of the hybrid-cache upkeep (tq_hybrid_append) against the oracle's restatement.

Sequences start in different window states (empty, partly filled, full with and without a
compressed history, and one state the upkeep never produces); several appends follow.  After each
one the window rows and both lengths must equal the oracle's exactly; the tokens that left the
window must be encoded into the pools as the oracle encodes them (tolerances of tests/parity.py),
with every other pool byte untouched; hybrid attention over the result must match the oracle's.
"""
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


def _up(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).to(DEV)


def _down(t):
    return t.float().cpu().numpy()


def _slot_owner(is_k, d):
    """byte offset within a record -> owning slot (from the oracle's layout)."""
    owner = oracle.slot_owner(is_k, d)
    assert (owner >= 0).all()
    return owner


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (128, "f32"), (256, "bf16")])
def test_hybrid_append_parity(d, dtype):
    H, W, steps = 2, 4, 5
    # (history length, window length): empty, partly filled, full with no history, full with a
    # history ending inside a block, full at a block boundary, full with the leaving token's
    # position past the block table (left unchanged), and a state the upkeep never makes
    init = [(0, 0), (0, 2), (0, 4), (9, 4), (16, 4), (48, 4), (3, 1)]
    B, mb = len(init), 3
    rng = np.random.default_rng(7)
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    nblk = B * mb
    bt = rng.permutation(nblk).reshape(B, mb).astype(np.int32)
    win_k = synth.round_dtype(rng.standard_normal((B, W, H, d)).astype(np.float32), dtype)
    win_v = synth.round_dtype(rng.standard_normal((B, W, H, d)).astype(np.float32), dtype)
    win_k0, win_v0 = win_k.copy(), win_v.copy()
    ctx = np.array([c for c, _ in init], np.int32)
    wl = np.array([w for _, w in init], np.int32)
    kp_o = np.full((nblk, H, oracle.record_bytes(True, d)), FILL, np.uint8)
    vp_o = np.full((nblk, H, oracle.record_bytes(False, d)), FILL, np.uint8)

    g_wk, g_wv = _up(win_k, dtype), _up(win_v, dtype)
    g_ctx, g_wl = torch.from_numpy(ctx).to(DEV), torch.from_numpy(wl).to(DEV)
    g_bt = torch.from_numpy(bt).to(DEV)
    g_kp = torch.full(kp_o.shape, FILL, dtype=torch.uint8, device=DEV)
    g_vp = torch.full(vp_o.shape, FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    left_k, left_v, left_slots = [], [], []
    for step in range(steps):
        kn = synth.round_dtype(rng.standard_normal((B, H, d)).astype(np.float32), dtype)
        vn = synth.round_dtype(rng.standard_normal((B, H, d)).astype(np.float32), dtype)
        if step == 1:
            kn[0] = 0.0     # a zero vector enters the window and later leaves it
        for b in range(B):   # the rows that leave the window in this step, by the oracle's state
            L, n = int(ctx[b]), int(wl[b])
            if L >= 0 and n == W and L // 16 < mb:
                left_k.append(win_k[b, L % W].copy())
                left_v.append(win_v[b, L % W].copy())
                left_slots.append(int(bt[b, L // 16]) * 16 + L % 16)
        win_k, win_v, wl, ctx = oracle.hybrid_append(D, S, kn, vn, win_k, win_v, wl, ctx, bt, kp_o, vp_o)
        tq.hybrid_append(params, d, _up(kn, dtype), _up(vn, dtype), g_wk, g_wv, g_wl, g_bt, g_ctx, g_kp, g_vp,
                         status=status)
        torch.cuda.synchronize()
        assert np.array_equal(g_ctx.cpu().numpy(), ctx) and np.array_equal(g_wl.cpu().numpy(), wl), step
        assert np.array_equal(_down(g_wk), win_k) and np.array_equal(_down(g_wv), win_v), step
    assert int(status.item()) == tq.STATUS_BAD_SLOT     # the last two sequences' states, left unchanged
    assert (ctx[-2], wl[-2]) == (48, 4) and (ctx[-1], wl[-1]) == (3, 1)
    assert np.array_equal(_down(g_wk)[-2], win_k0[-2]) and np.array_equal(_down(g_wv)[-2], win_v0[-2])

    # the tokens that left the window, against the oracle's encode of the same rows
    slots = np.array(left_slots, np.int64)
    assert len(slots) == 1 + 3 + 3 * steps   # sequence 0 once, sequence 1 from its third step, 2-4 every step
    kp_g, vp_g = g_kp.cpu().numpy(), g_vp.cpu().numpy()
    parity.check_encode(True, D, S, np.stack(left_k), slots, kp_g, pool_fill=FILL)
    parity.check_encode(False, D, S, np.stack(left_v), slots, vp_g, pool_fill=FILL)
    for pool, is_k in ((kp_g, True), (vp_g, False)):
        owner = _slot_owner(is_k, d)
        written = np.zeros((nblk, 16), bool)
        written[slots // 16, slots % 16] = True
        for blk in range(nblk):   # bytes of slots nothing was encoded into keep the fill
            assert np.all(pool[blk][:, ~written[blk][owner]] == FILL)

    # hybrid attention over the result (the five sequences the upkeep advanced)
    n = B - 2
    Hq = 2 * H
    q = synth.round_dtype(rng.standard_normal((n, Hq, d)).astype(np.float32), dtype)
    out = tq.decode_attn_hybrid(params, d, _up(q, dtype), H, g_kp, g_vp, g_bt[:n].contiguous(),
                                g_ctx[:n].contiguous(), int(ctx[:n].max()), g_wk[:n].contiguous(),
                                g_wv[:n].contiguous(), g_wl[:n].contiguous())
    torch.cuda.synchronize()
    ref = oracle.decode_hybrid(D, S, q, H, kp_g, vp_g, bt[:n], ctx[:n], win_k[:n], win_v[:n], wl[:n])
    parity.check_attention(out.cpu().numpy(), ref)


def test_hybrid_append_rejects_bad_arguments():
    d, H, W, B = 128, 2, 4, 2
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    kn = torch.zeros((B, H, d), dtype=torch.bfloat16, device=DEV)
    wk = torch.zeros((B, W, H, d), dtype=torch.bfloat16, device=DEV)
    lens = torch.zeros(B, dtype=torch.int32, device=DEV)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=DEV)
    kp = torch.zeros((2, H, tq.k_record_bytes(d)), dtype=torch.uint8, device=DEV)
    vp = torch.zeros((2, H, tq.v_record_bytes(d)), dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError):    # the window's dtype differs from the new rows'
        tq.hybrid_append(params, d, kn, kn, wk.float(), wk.float(), lens, bt, lens.clone(), kp, vp)
    with pytest.raises(tq.TQError):    # scratch too small
        tq.hybrid_append(params, d, kn, kn, wk, wk, lens, bt, lens.clone(), kp, vp,
                         scratch=torch.empty(16, dtype=torch.uint8, device=DEV))
    L = tq.load_library()
    rc = L.tq_hybrid_append(None, d, None, None, 1, B, H, None, None, 0, None, None, 1, None, None, None, 2, None, 0,
                            None, None)
    assert rc == -1   # win_cap 0: TQ_ERR_INVALID
