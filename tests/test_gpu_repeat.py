"""Back-to-back decode steps are repeatable bit for bit.

A serving loop issues decode steps back to back on the same stream, alternating between caches
(layers), with every launch of one step free to overlap the launches around it as the library
allows.  Running the same sequence of steps twice, from identical caches, must give identical
outputs and identical caches: the split of the context over CTAs, the order of every sum and the
records the steps append are functions of the inputs alone, whatever the launches' timing."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cache(d, Hkv, lens, seed):
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, _ = tq.codebook_init(d, D, S, device=DEV)
    need = [-(-(L + 1) // 16) for L in lens]   # room for the appended token
    nblk = sum(need) + 3
    perm = np.random.default_rng(seed).permutation(nblk)
    bt = np.zeros((len(lens), max(need)), np.int32)
    k0 = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k0:k0 + n]
        k0 += n
    kp = tq.empty_pool(nblk, Hkv, d, "k", DEV)
    vp = tq.empty_pool(nblk, Hkv, d, "v", DEV)
    g = torch.Generator(device=DEV).manual_seed(seed)
    for b, L in enumerate(lens):
        K = (torch.randn((L, Hkv, d), generator=g, device=DEV) * 2).to(torch.bfloat16)
        V = torch.randn((L, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
        sl = torch.from_numpy(synth.slots_for(bt, b, 0, L)).to(DEV)
        tq.encode_k(params, d, K, sl, kp)
        tq.encode_v(params, d, V, sl, vp)
    return params, torch.from_numpy(bt).to(DEV), kp, vp


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 4), (128, 16, 4), (256, 8, 4)])
def test_back_to_back_steps_repeat_bit_for_bit(d, Hq, Hkv):
    lens = [6000, 700, 12000, 33, 2048, 9000, 4096, 15]
    B = len(lens)
    params, bt, kp0, vp0 = _cache(d, Hkv, lens, seed=d + Hq)
    g = torch.Generator(device=DEV).manual_seed(7)
    q = torch.randn((B, Hq, d), generator=g, device=DEV).to(torch.bfloat16)
    k_new = torch.randn((B, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    v_new = torch.randn((B, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    pre = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ctx = pre + 1
    max_ctx = max(lens) + 1
    ws = torch.empty(tq.decode_workspace_bytes(d, B, Hq, max_ctx), dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run():
        pools = [(kp0.clone(), vp0.clone()) for _ in range(2)]
        outs = []
        for i in range(24):
            kp, vp = pools[i % 2]
            out = torch.empty((B, Hq, d), dtype=torch.float32, device=DEV)
            tq.decode_step(params, d, k_new, v_new, q, Hkv, kp, vp, bt, pre, max_ctx, out=out, workspace=ws,
                           status=status)
            outs.append(out)
        for kp, vp in pools:
            outs.append(tq.decode_attn(params, d, q, Hkv, kp, vp, bt, ctx, max_ctx, workspace=ws, status=status))
        torch.cuda.synchronize()
        return outs, pools

    outs1, pools1 = run()
    outs2, pools2 = run()
    assert int(status.item()) == 0
    for a, b in zip(outs1, outs2):
        assert torch.isfinite(a).all()
        assert torch.equal(a, b)
    for (ka, va), (kb, vb) in zip(pools1, pools2):
        assert torch.equal(ka, kb) and torch.equal(va, vb)
    # every step attended the same tokens: all step outputs equal the attention over the final caches
    for a in outs1[:24]:
        assert torch.equal(a, outs1[24])
