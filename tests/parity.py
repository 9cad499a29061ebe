"""Comparison helpers between the CUDA library and the fp64 oracle.

Tolerances (written here once, used by every parity test):
  * cells and sign bits are integers decided from floating point: they must be
    bit-identical except where the oracle's fp64 value lies within 1e-6 of the
    decision point (a Lloyd-Max threshold for a cell, 0 for a QJL sign); such
    near-threshold entries are counted and must be at most 1e-5 of all entries;
    the expected rate is about 4e-6 per entry, so a small test (under 400K
    entries, where 1e-5 of them is below 4) allows up to 4 as a Poisson floor;
  * fp16 norms: within 1 ulp;
  * attention output, with the oracle and the GPU both decoding the same
    packed cache (written by the oracle and uploaded to the device):
    per (sequence, query head) max|o_gpu - o_ref| <= 2e-3 and
    ||o_gpu - o_ref||_2 / ||o_ref||_2 <= 1e-3.
"""
from __future__ import annotations

import numpy as np

import oracle

NEAR = 1e-6
NEAR_FRACTION = 1e-5
NEAR_FLOOR = 4
ATT_MAX_ABS = 2e-3
ATT_REL = 1e-3


def fp16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in units in the last place for same-sign binary16 bit patterns."""
    a = a.astype(np.int64)
    b = b.astype(np.int64)
    return np.abs(a - b)


def check_encode(is_k, D, S, x, slots, gpu_pool, pool_fill=0xA5):
    """Compare a GPU-encoded pool with the oracle on the vectors x[N][H][d] at slots."""
    N, H, d = x.shape
    c, t, _, _ = oracle.codebook()
    g = oracle.unpack(is_k, d, gpu_pool, H, slots)
    ref = oracle.encode(is_k, D, S, x, slots, np.full_like(gpu_pool, pool_fill), want_details=True)
    margin = np.min(np.abs(ref["z"][..., None] - t), axis=-1)
    # a zero vector has z = 0 exactly on the middle threshold: a deterministic
    # tie (upper cell) on both sides, so it is compared exactly, not counted
    near = (margin < NEAR) & (ref["n"] > 0)[..., None]
    n_near = int(near.sum())
    assert n_near <= max(NEAR_FLOOR, NEAR_FRACTION * near.size), f"{n_near} near-threshold cells"
    bad = (g["codes"] != ref["codes"]) & ~near
    assert not bad.any(), f"{int(bad.sum())} cells differ away from thresholds"
    # norms
    n16_ref = np.vectorize(oracle.fp16_rne)(ref["n"]).astype(np.uint16)
    assert fp16_ulp_diff(g["n16"], n16_ref).max() <= 1
    stats = dict(entries=near.size, near=n_near, cell_mismatch=int((g["codes"] != ref["codes"]).sum()))
    if is_k:
        # QJL bits and gamma given the GPU's own cells
        ref2 = oracle.encode(True, D, S, x, slots, np.full_like(gpu_pool, pool_fill), codes_in=g["codes"],
                             want_details=True)
        pnear = np.abs(ref2["p"] / 1.0) < NEAR
        assert int(pnear.sum()) <= max(NEAR_FLOOR, NEAR_FRACTION * pnear.size), f"{int(pnear.sum())} near-zero QJL projections"
        sbad = (g["signs"] != ref2["signs"]) & ~pnear
        assert not sbad.any(), f"{int(sbad.sum())} QJL sign bits differ away from zero"
        g16_ref = np.vectorize(oracle.fp16_rne)(ref2["gamma"]).astype(np.uint16)
        assert fp16_ulp_diff(g["g16"], g16_ref).max() <= 1
        stats["sign_near"] = int(pnear.sum())
        stats["sign_mismatch"] = int((g["signs"] != ref2["signs"]).sum())
    return stats


def check_attention(o_gpu: np.ndarray, o_ref: np.ndarray):
    """Per (seq, q head) bounds; returns (worst max-abs, worst relative)."""
    B, Hq, d = o_ref.shape
    worst_abs = 0.0
    worst_rel = 0.0
    for b in range(B):
        for h in range(Hq):
            diff = o_gpu[b, h].astype(np.float64) - o_ref[b, h]
            a = float(np.max(np.abs(diff)))
            nr = float(np.linalg.norm(o_ref[b, h]))
            r = float(np.linalg.norm(diff) / nr) if nr > 0 else float(np.linalg.norm(diff))
            worst_abs = max(worst_abs, a)
            worst_rel = max(worst_rel, r)
            assert a <= ATT_MAX_ABS and r <= ATT_REL, f"(b={b}, h={h}) max-abs {a:.3e} rel {r:.3e}"
    return worst_abs, worst_rel
