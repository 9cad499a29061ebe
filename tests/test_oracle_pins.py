"""Pins of the fp64 oracle against facts fixed outside it.

Each test checks the oracle against something it cannot have copied:
a printed table, a closed form, a library routine, an invariant of the
mathematics, or brute force on tiny inputs.  None needs a GPU.
"""
import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.stats

import oracle
from turboquant_compressed_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [float(x) for x in v]
    return out


# ------------------------------------------------------------------ codebook

def test_codebook_matches_max_1960_table():
    g = _golden("lloyd_max_gaussian_8.txt")
    c, t, mse, it = oracle.lloyd_max8()
    assert it > 0
    np.testing.assert_allclose(c[4:], g["levels"], atol=1e-3)
    np.testing.assert_allclose(t[3:], g["thresholds"], atol=1e-3)
    assert abs(mse - g["mse"][0]) < 1e-4


def test_codebook_symmetry_and_midpoints():
    c, t, _, _ = oracle.lloyd_max8()
    assert t[3] == 0.0
    np.testing.assert_array_equal(c[::-1], -c)
    np.testing.assert_allclose(t, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    assert np.all(np.diff(c) > 0)


def test_codebook_is_a_fixed_point_by_numerical_integration():
    """Centroid condition checked with scipy quadrature, not the closed form."""
    c, t, mse, _ = oracle.lloyd_max8()
    edges = [-np.inf] + list(t) + [np.inf]
    pdf = scipy.stats.norm.pdf
    err = 0.0
    for j in range(8):
        a, b = edges[j], edges[j + 1]
        m0 = scipy.integrate.quad(pdf, a, b, epsabs=1e-14, epsrel=1e-13)[0]
        m1 = scipy.integrate.quad(lambda x: x * pdf(x), a, b, epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(m1 / m0 - c[j]) < 1e-10
        err += scipy.integrate.quad(lambda x: (x - c[j]) ** 2 * pdf(x), a, b,
                                    epsabs=1e-14, epsrel=1e-13)[0]
    assert abs(err - mse) < 1e-10


def test_codebook_beats_perturbations():
    """Lloyd-Max is a local minimum of the distortion: nudging any level raises it."""
    c, t, mse, _ = oracle.lloyd_max8()
    pdf = scipy.stats.norm.pdf

    def distortion(levels):
        levels = np.sort(levels)
        th = 0.5 * (levels[:-1] + levels[1:])
        edges = [-np.inf] + list(th) + [np.inf]
        return sum(scipy.integrate.quad(lambda x: (x - levels[j]) ** 2 * pdf(x),
                                        edges[j], edges[j + 1])[0] for j in range(8))

    base = distortion(c)
    assert abs(base - mse) < 1e-9
    for j in range(8):
        for eps in (1e-3, -1e-3):
            cc = c.copy()
            cc[j] += eps
            assert distortion(cc) > base


# ------------------------------------------------------------------ fp16

def test_fp16_rne_matches_numpy_conversion():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000),
        rng.uniform(0, 1, 500) * 2.0 ** -24 * 4,      # subnormals
        np.array([0.0, -0.0, 65504.0, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -26,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0]),
    ])
    for v in vals:
        want = np.array([v], np.float64).astype(np.float16).view(np.uint16)[0]
        assert oracle.fp16_rne(v) == want, v
        if np.isfinite(np.float16(v)):
            assert oracle.fp16_value(want) == float(np.float16(v))


# ------------------------------------------------------------------ rotation

@pytest.mark.parametrize("d", [128, 256])
def test_hadamard_orthogonal_integer(d):
    H = np.array([[oracle.hadamard_entry(i, j) for j in range(d)] for i in range(d)])
    np.testing.assert_array_equal(H @ H.T, d * np.eye(d, dtype=H.dtype))
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(d))


@pytest.mark.parametrize("d", [128, 256])
def test_rotation_matches_library_hadamard(d):
    D = synth.rotation_signs(d)
    rng = np.random.default_rng(0)
    for _ in range(3):
        x = rng.standard_normal(d)
        want = scipy.linalg.hadamard(d) @ (D * x) / math.sqrt(d)
        y = oracle.rotate(D, x)
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
        np.testing.assert_allclose(oracle.rotate_t(D, y), x, rtol=0, atol=1e-12)


def test_rotation_spreads_outliers():
    """Two channels at 20x: after the rotation no coordinate keeps the spike."""
    d = 128
    D = synth.rotation_signs(d)
    w = synth.workload("tiny")
    K, _ = synth.kv_tokens(w, 0, 0, 256)
    before, after = [], []
    for x in K[:, 0, :].astype(np.float64):
        xh = x / np.linalg.norm(x)
        before.append(np.max(np.abs(xh)))
        after.append(np.max(np.abs(oracle.rotate(D, xh))))
    assert np.mean(before) > 0.6          # the 20x channels dominate
    assert np.mean(after) < 3.5 * math.sqrt(2 * math.log(d) / d)


# ------------------------------------------------------------------ quantiser

def test_code_is_nearest_centroid():
    """Threshold counting equals brute-force nearest-centroid search."""
    c, t, _, _ = oracle.lloyd_max8()
    d = 128
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal(d) * rng.lognormal(0, 1, d)
        r = oracle.encode_vector(False, D, S, x)
        near = np.argmin(np.abs(r["z"][:, None] - c[None, :]), axis=1)
        margin = np.min(np.abs(r["z"][:, None] - t[None, :]), axis=1)
        ok = margin > 1e-6
        np.testing.assert_array_equal(r["codes"][ok], near[ok])
        np.testing.assert_allclose(r["z"], math.sqrt(d) * oracle.rotate(D, x / np.linalg.norm(x)),
                                   atol=1e-12)


def test_quantiser_distortion_matches_mse():
    """E||xhat - Pi^T yhat||^2 ~ Lloyd-Max MSE (the rotated coordinates are near N(0,1/d))."""
    c, _, mse, _ = oracle.lloyd_max8()
    d = 128
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    rng = np.random.default_rng(2)
    errs, cells = [], np.zeros(8)
    for _ in range(400):
        x = rng.standard_normal(d)
        r = oracle.encode_vector(True, D, S, x)
        yhat = c[r["codes"]] / math.sqrt(d)
        xr = oracle.rotate_t(D, yhat)
        errs.append(np.sum((x / np.linalg.norm(x) - xr) ** 2))
        assert abs(r["gamma"] ** 2 - errs[-1]) < 1e-12      # gamma = ||r|| in either domain
        cells += np.bincount(r["codes"], minlength=8)
    assert abs(np.mean(errs) - mse) / mse < 0.05
    edges = np.concatenate([[-np.inf], oracle.lloyd_max8()[1], [np.inf]])
    probs = np.diff(scipy.stats.norm.cdf(edges))
    np.testing.assert_allclose(cells / cells.sum(), probs, atol=0.01)


def test_encode_scale_invariance_and_zero_vector():
    d = 128
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    x = np.random.default_rng(3).standard_normal(d)
    a = oracle.encode_vector(True, D, S, x)
    b = oracle.encode_vector(True, D, S, 8.0 * x)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["signs"], b["signs"])
    assert b["n"] == 8.0 * a["n"] and abs(a["gamma"] - b["gamma"]) < 1e-15
    z = oracle.encode_vector(True, D, S, np.zeros(d))
    assert z["n"] == 0.0
    assert np.all(z["codes"] == 4)          # z = 0 sits on the middle threshold: upper cell


def test_qjl_given_codes_mode():
    d = 128
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    x = np.random.default_rng(4).standard_normal(d)
    a = oracle.encode_vector(True, D, S, x)
    b = oracle.encode_vector(True, D, S, x, codes_in=a["codes"])
    np.testing.assert_array_equal(a["signs"], b["signs"])
    codes = a["codes"].copy()
    codes[0] = (codes[0] + 1) % 8
    c = oracle.encode_vector(True, D, S, x, codes_in=codes)
    assert c["codes"][0] == codes[0]
    assert abs(c["gamma"] - a["gamma"]) > 1e-6


def test_qjl_inner_product_estimator_is_unbiased():
    """Over many Gaussian S, sqrt(pi/2)/m * gamma * <S qbar, sign(S r)> averages to <qbar, r>."""
    d = 128
    c, _, _, _ = oracle.lloyd_max8()
    D = synth.rotation_signs(d)
    rng = np.random.default_rng(6)
    x = rng.standard_normal(d)
    q = rng.standard_normal(d)
    qbar = oracle.rotate(D, q)
    ests = []
    r_true = None
    for s in range(1500):
        S = np.random.default_rng([77, s]).standard_normal((d, d)).astype(np.float32)
        e = oracle.encode_vector(True, D, S, x)
        y = oracle.rotate(D, x / np.linalg.norm(x))
        r = y - c[e["codes"]] / math.sqrt(d)
        if r_true is None:
            r_true = r
        bt = 2.0 * e["signs"] - 1.0
        u = S.astype(np.float64) @ qbar
        ests.append(math.sqrt(math.pi / 2) / d * e["gamma"] * np.dot(u, bt))
        np.testing.assert_array_equal(bt, np.where(S.astype(np.float64) @ r >= 0, 1.0, -1.0))
    ests = np.array(ests)
    truth = float(np.dot(qbar, r_true))
    se = ests.std(ddof=1) / math.sqrt(len(ests))
    assert abs(ests.mean() - truth) < 5 * se
    # variance of a single-sketch estimate: (pi/2 ||r||^2||q||^2 - <q,r>^2)/m  (closed form)
    var_pred = (math.pi / 2 * np.dot(r_true, r_true) * np.dot(qbar, qbar) - truth ** 2) / d
    assert 0.8 < ests.var(ddof=1) / var_pred < 1.25


# ------------------------------------------------------------------ bits

def test_bits_per_dim():
    for d in (128, 256):
        kb = oracle.record_bytes(True, d) * 8 / (16 * d)
        vb = oracle.record_bytes(False, d) * 8 / (16 * d)
        if d == 128:
            assert kb == 4.25 and vb == 3.125
            assert abs((kb + vb) / 2 - 3.6) < 0.1
            assert abs(16 / ((kb + vb) / 2) - 4.339) < 1e-3
        else:
            assert kb == 4.125 and vb == 3.0625


@pytest.mark.parametrize("is_k", [True, False])
@pytest.mark.parametrize("d", [128, 256])
def test_layout_is_a_bijection(is_k, d):
    """Every (slot, coordinate, field bit) has its own bit of the record's cell region, and the
    region is used in full: 4 bits per coordinate for K (4.25 bits/dim with the norms at d=128),
    3 for V (3.125)."""
    nbits = 4 if is_k else 3
    seen = set()
    for t in range(16):
        for i in range(d):
            for p in range(nbits):
                w, b = oracle.bitpos(is_k, d, t, i, p)
                assert 0 <= b < 32 and 0 <= w * 32 + b < 16 * d * nbits
                seen.add(w * 32 + b)
    assert len(seen) == 16 * d * nbits


@pytest.mark.parametrize("is_k", [True, False])
@pytest.mark.parametrize("d", [128, 256])
def test_layout_bytes_have_one_owner(is_k, d):
    """A byte of a record holds fields of one slot only, so slots are written independently."""
    owner = oracle.slot_owner(is_k, d)
    assert (owner >= 0).all()
    for t in range(16):
        for i in range(0, d, 7):
            for p in range(4 if is_k else 3):
                w, b = oracle.bitpos(is_k, d, t, i, p)
                assert owner[w * 4 + b // 8] == t


def test_pack_unpack_roundtrip():
    d, H = 128, 2
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((40, H, d)).astype(np.float32)
    slots = rng.permutation(64)[:40].astype(np.int64)
    for is_k in (True, False):
        pool = np.zeros((4, H, oracle.record_bytes(is_k, d)), np.uint8)
        det = oracle.encode(is_k, D, S, x, slots, pool, want_details=True)
        back = oracle.unpack(is_k, d, pool, H, slots)
        np.testing.assert_array_equal(back["codes"], det["codes"])
        if is_k:
            np.testing.assert_array_equal(back["signs"], det["signs"])
        for k in range(40):
            for h in range(H):
                assert back["n16"][k, h] == oracle.fp16_rne(det["n"][k, h])
                if is_k:
                    assert back["g16"][k, h] == oracle.fp16_rne(det["gamma"][k, h])


# ------------------------------------------------------------------ attention

def _small_cache(d, B, Hkv, lens, seed=0, same_key=False):
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    rng = np.random.default_rng(seed)
    nb = [max(1, -(-L // 16)) for L in lens]
    mb = max(nb)
    perm = rng.permutation(sum(nb) + 3)
    bt = np.zeros((B, mb), np.int32)
    k = 0
    for b in range(B):
        bt[b, :nb[b]] = perm[k:k + nb[b]]
        k += nb[b]
    nblk = sum(nb) + 3
    kp = np.zeros((nblk, Hkv, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nblk, Hkv, oracle.record_bytes(False, d)), np.uint8)
    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        K = rng.standard_normal((L, Hkv, d)).astype(np.float32) * 3
        V = rng.standard_normal((L, Hkv, d)).astype(np.float32)
        if same_key:
            K[:] = K[0]
        slots = (bt[b, np.arange(L) // 16].astype(np.int64) * 16 + np.arange(L) % 16)
        oracle.encode(True, D, S, K, slots, kp)
        oracle.encode(False, D, S, V, slots, vp)
    return D, S, bt, kp, vp


@pytest.mark.parametrize("d", [128, 256])
def test_two_attention_formulations_agree(d):
    B, Hq, Hkv = 2, 4, 2
    lens = [37, 20]
    D, S, bt, kp, vp = _small_cache(d, B, Hkv, lens)
    q = np.random.default_rng(9).standard_normal((B, Hq, d)).astype(np.float32)
    a = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32))
    b = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array(lens, np.int32), explicit=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def _dequant_v(D, det_codes, n16, d):
    c = oracle.codebook()[0]
    return oracle.fp16_value(n16) * oracle.rotate_t(D, c[det_codes] / math.sqrt(d))


def test_attention_special_cases():
    d, Hkv = 128, 1
    # one cached token: output is that token's dequantised value
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [1], seed=3)
    q = np.random.default_rng(1).standard_normal((1, 2, d)).astype(np.float32)
    o = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array([1], np.int32))
    u = oracle.unpack(False, d, vp, Hkv, np.array([bt[0, 0] * 16], np.int64))
    want = _dequant_v(D, u["codes"][0, 0], u["n16"][0, 0], d)
    np.testing.assert_allclose(o[0, 0], want, atol=1e-12)
    np.testing.assert_allclose(o[0, 1], want, atol=1e-12)
    # all keys equal: plain mean of the dequantised values
    L = 23
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [L], seed=4, same_key=True)
    o = oracle.decode(D, S, q[:, :1], Hkv, kp, vp, bt, np.array([L], np.int32))
    slots = bt[0, np.arange(L) // 16].astype(np.int64) * 16 + np.arange(L) % 16
    u = oracle.unpack(False, d, vp, Hkv, slots)
    mean = np.mean([_dequant_v(D, u["codes"][j, 0], u["n16"][j, 0], d) for j in range(L)], axis=0)
    np.testing.assert_allclose(o[0, 0], mean, atol=1e-12)
    # empty context: zeros
    o = oracle.decode(D, S, q[:, :1], Hkv, kp, vp, bt, np.array([0], np.int32))
    assert np.all(o == 0)


def test_multi_query_decode_is_causal_over_the_new_tokens():
    """decode_mq: query i of Q sees the cache up to token L - Q + i.  Pinned against a brute-force
    softmax over the explicitly dequantised keys and values of the oracle's second formulation,
    and by causality: rewriting the last cached token moves only the last query."""
    d, Hkv, Hq, L, Q = 128, 2, 4, 40, 3
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [L], seed=8)
    q = np.random.default_rng(4).standard_normal((1, Q, Hq, d)).astype(np.float32)
    o = oracle.decode_mq(D, S, q, Hkv, kp, vp, bt, np.array([L], np.int32))
    assert o.shape == (1, Q, Hq, d)
    # query 0 of a Q = 1 call is the single-query decode
    o1 = oracle.decode_mq(D, S, q[:, -1:], Hkv, kp, vp, bt, np.array([L], np.int32))
    np.testing.assert_array_equal(o1[:, 0], oracle.decode(D, S, np.ascontiguousarray(q[:, -1]), Hkv, kp, vp, bt,
                                                          np.array([L], np.int32)))
    # brute force: dequantise every token (K with its QJL term) and run a plain softmax per prefix
    slots = bt[0, np.arange(L) // 16].astype(np.int64) * 16 + np.arange(L) % 16
    uk = oracle.unpack(True, d, kp, Hkv, slots)
    uv = oracle.unpack(False, d, vp, Hkv, slots)
    c = oracle.codebook()[0]
    Sd = S.astype(np.float64)
    G = Hq // Hkv
    for h in range(Hq):
        kv = h // G
        keys = np.array([oracle.fp16_value(uk["n16"][t, kv]) * oracle.rotate_t(
            D, c[uk["codes"][t, kv]] / math.sqrt(d) + math.sqrt(math.pi / 2) / d * oracle.fp16_value(
                uk["g16"][t, kv]) * (Sd.T @ (2.0 * uk["signs"][t, kv] - 1))) for t in range(L)])
        vals = np.array([_dequant_v(D, uv["codes"][t, kv], uv["n16"][t, kv], d) for t in range(L)])
        for i in range(Q):
            n = L - (Q - 1 - i)
            s = keys[:n] @ q[0, i, h].astype(np.float64) / math.sqrt(d)
            p = np.exp(s - s.max())
            want = (p[:, None] * vals[:n]).sum(0) / p.sum()
            np.testing.assert_allclose(o[0, i, h], want, rtol=1e-10, atol=1e-10)
    # causality: a different last token changes query Q-1 only
    kp2, vp2 = kp.copy(), vp.copy()
    x = np.random.default_rng(77).standard_normal((1, Hkv, d)).astype(np.float32)
    oracle.encode(True, D, S, x, slots[-1:], kp2)
    oracle.encode(False, D, S, x, slots[-1:], vp2)
    o2 = oracle.decode_mq(D, S, q, Hkv, kp2, vp2, bt, np.array([L], np.int32))
    np.testing.assert_array_equal(o2[:, :Q - 1], o[:, :Q - 1])
    assert np.abs(o2[:, Q - 1] - o[:, Q - 1]).max() > 1e-6
    # a query with no token before it gets zeros
    o3 = oracle.decode_mq(D, S, q, Hkv, kp, vp, bt, np.array([1], np.int32))
    assert np.all(o3[:, :Q - 1] == 0) and np.abs(o3[:, Q - 1]).max() > 0


def test_dequant_gives_the_decode_attention():
    """Attention by a plain softmax over the dequantised K and V (numpy) equals the oracle's
    rotated-domain decode (C) to 1e-12, and V's reconstruction error on Gaussian vectors is the
    codebook MSE."""
    d, Hkv, Hq, L = 128, 2, 4, 45
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [L], seed=12)
    nb = -(-L // 16)
    K = oracle.dequant(True, D, S, kp, Hkv, bt[0, :nb])[:L]
    V = oracle.dequant(False, D, S, vp, Hkv, bt[0, :nb])[:L]
    q = np.random.default_rng(6).standard_normal((1, Hq, d)).astype(np.float32)
    o = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array([L], np.int32))
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        s = K[:, kv] @ q[0, h].astype(np.float64) / math.sqrt(d)
        p = np.exp(s - s.max())
        np.testing.assert_allclose(o[0, h], (p[:, None] * V[:, kv]).sum(0) / p.sum(), rtol=1e-12, atol=1e-12)
    # V: E ||v - v~||^2 / ||v||^2 over Gaussian vectors is the Lloyd-Max MSE of N(0,1)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((64, 1, d)).astype(np.float32)
    pool = np.zeros((4, 1, oracle.record_bytes(False, d)), np.uint8)
    oracle.encode(False, D, S, x, np.arange(64, dtype=np.int64), pool)
    xr = oracle.dequant(False, D, S, pool, 1, np.arange(4))
    err = np.sum((xr[:, 0] - x[:, 0]) ** 2, axis=1) / np.sum(x[:, 0].astype(np.float64) ** 2, axis=1)
    mse = oracle.codebook()[2]
    assert abs(err.mean() / mse - 1) < 0.1, (err.mean(), mse)


def test_hybrid_attention_merges_history_and_window():
    """decode_hybrid (one softmax over dequantised history and raw window rows) equals the
    log-sum-exp merge of the rotated-domain decode over the history and a plain softmax over the
    window; an empty window gives the decode; the order of window slots does not matter."""
    d, Hkv, Hq, L, W = 128, 2, 4, 37, 11
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [L], seed=21)
    rng = np.random.default_rng(22)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    wk = rng.standard_normal((1, W + 3, Hkv, d)).astype(np.float32) * 2
    wv = rng.standard_normal((1, W + 3, Hkv, d)).astype(np.float32)
    o = oracle.decode_hybrid(D, S, q, Hkv, kp, vp, bt, [L], wk, wv, [W])
    oc = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array([L], np.int32))
    np.testing.assert_allclose(oracle.decode_hybrid(D, S, q, Hkv, kp, vp, bt, [L], wk, wv, [0]), oc, rtol=1e-12,
                               atol=1e-12)
    # the merge: lse of the history from its scores, the window by a plain softmax
    nb = -(-L // 16)
    Kc = oracle.dequant(True, D, S, kp, Hkv, bt[0, :nb])[:L]
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        sc = Kc[:, kv] @ q[0, h].astype(np.float64) / math.sqrt(d)
        sw = wk[0, :W, kv].astype(np.float64) @ q[0, h].astype(np.float64) / math.sqrt(d)
        M = max(sc.max(), sw.max())
        ec, ew = np.exp(sc - M).sum(), np.exp(sw - M)
        want = (oc[0, h] * ec + (ew[:, None] * wv[0, :W, kv]).sum(0)) / (ec + ew.sum())
        np.testing.assert_allclose(o[0, h], want, rtol=1e-11, atol=1e-12)
    perm = rng.permutation(W)
    o2 = oracle.decode_hybrid(D, S, q, Hkv, kp, vp, bt, [L], wk[:, perm], wv[:, perm], [W])
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)


def test_attention_ignores_physical_block_order():
    d, Hkv = 128, 2
    D, S, bt, kp, vp = _small_cache(d, 1, Hkv, [50], seed=5)
    q = np.random.default_rng(2).standard_normal((1, 4, d)).astype(np.float32)
    o1 = oracle.decode(D, S, q, Hkv, kp, vp, bt, np.array([50], np.int32))
    # move every block to a new physical id
    nblk = kp.shape[0]
    perm = np.random.default_rng(3).permutation(nblk)
    kp2 = np.zeros_like(kp)
    vp2 = np.zeros_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = perm[bt].astype(np.int32)
    o2 = oracle.decode(D, S, q, Hkv, kp2, vp2, bt2, np.array([50], np.int32))
    np.testing.assert_array_equal(o1, o2)


def test_attention_close_to_uncompressed():
    """Information only in spirit, but a gross error would show: cosine > 0.9."""
    d, Hkv, L = 128, 1, 200
    D = synth.rotation_signs(d)
    S = synth.qjl_matrix(d)
    rng = np.random.default_rng(11)
    K = rng.standard_normal((L, 1, d)).astype(np.float32)
    V = rng.standard_normal((L, 1, d)).astype(np.float32)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    kp = np.zeros((13, 1, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((13, 1, oracle.record_bytes(False, d)), np.uint8)
    slots = np.arange(L, dtype=np.int64)
    oracle.encode(True, D, S, K, slots, kp)
    oracle.encode(False, D, S, V, slots, vp)
    bt = np.arange(13, dtype=np.int32)[None]
    o = oracle.decode(D, S, q, 1, kp, vp, bt, np.array([L], np.int32))[0, 0]
    s = K[:, 0].astype(np.float64) @ q[0, 0] / math.sqrt(d)
    p = np.exp(s - s.max())
    p /= p.sum()
    ref = p @ V[:, 0].astype(np.float64)
    cos = np.dot(o, ref) / np.linalg.norm(o) / np.linalg.norm(ref)
    assert cos > 0.9


# ------------------------------------------------------------------ group-quantised comparator

from oracle import gq  # noqa: E402


def _gq_data(N, H, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, H, d)).astype(np.float32)
    x *= rng.lognormal(0, 1, (1, H, d)).astype(np.float32)
    x[:, :, 5] *= 10
    return x


@pytest.mark.parametrize("bits,group", [(4, 64), (4, 32), (8, 64), (8, 128)])
def test_gq_codes_are_the_nearest_grid_level(bits, group):
    """Brute force: each code is the index of the nearest of the 2^bits levels
    bias + scale k, over all k (clamping included), except where two levels are
    equally near to 1e-6 of a step."""
    x = _gq_data(40, 2, 128, 3)
    codes, s16, z16 = gq.encode(x, bits, group)
    s = s16.view(np.float16).astype(np.float64)
    z = z16.view(np.float16).astype(np.float64)
    xg = x.astype(np.float64).reshape(40, 2, 128 // group, group)
    k = np.arange(2 ** bits, dtype=np.float64)
    lv = z[..., None, None] + s[..., None, None] * k              # [N][H][ng][1][levels]
    dist = np.abs(xg[..., None] - lv)
    best = dist.argmin(-1)
    srt = np.sort(dist, -1)
    clear = (srt[..., 1] - srt[..., 0]) > 1e-6 * s[..., None]
    cg = codes.reshape(best.shape)
    assert clear.mean() > 0.999
    np.testing.assert_array_equal(cg[clear], best[clear])


@pytest.mark.parametrize("bits", [4, 8])
def test_gq_scale_and_bias_span_the_group(bits):
    """scale and bias are the fp16 roundings of (max - min)/(2^bits - 1) and min (relative
    error <= 2^-11), and the group's minimum and maximum get the end codes."""
    x = _gq_data(30, 3, 128, 4)
    codes, s16, z16 = gq.encode(x, bits, 64)
    s = s16.view(np.float16).astype(np.float64)
    z = z16.view(np.float16).astype(np.float64)
    xg = x.astype(np.float64).reshape(30, 3, 2, 64)
    lo, hi = xg.min(-1), xg.max(-1)
    np.testing.assert_array_less(np.abs(s - (hi - lo) / (2 ** bits - 1)), 2 ** -11 * (hi - lo) / (2 ** bits - 1) + 1e-12)
    np.testing.assert_array_less(np.abs(z - lo), 2 ** -11 * np.abs(lo) + 1e-12)
    cg = codes.reshape(30, 3, 2, 64)
    assert (np.take_along_axis(cg, xg.argmin(-1)[..., None], -1) == 0).all()
    assert (np.take_along_axis(cg, xg.argmax(-1)[..., None], -1) == 2 ** bits - 1).all()


def test_gq_constant_group_gets_code_zero():
    x = np.full((1, 1, 128), 0.75, np.float32)
    codes, s16, z16 = gq.encode(x, 4, 64)
    assert (codes == 0).all() and (s16 == 0).all()
    np.testing.assert_array_equal(gq.decode_values(codes, s16, z16, 64), 0.75)


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 32)])
def test_gq_exact_grid_round_trip_and_attention(bits, group):
    """Vectors that lie on a grid exact in fp16 and fp32 (power-of-two step, bias a
    multiple of 1/8, both end levels present in every group) come back exactly, and
    the paged decode then equals textbook attention on the original vectors."""
    rng = np.random.default_rng(5)
    d, Hkv, Hq, lens = 128, 2, 6, [37, 0, 70]
    top = 2 ** bits - 1

    def grid(n):
        codes = rng.integers(0, top + 1, (n, Hkv, d // group, group))
        codes[..., 0], codes[..., 1] = 0, top
        step = 2.0 ** rng.integers(-6, -1, (n, Hkv, d // group, 1))
        base = rng.integers(-24, 24, (n, Hkv, d // group, 1)) / 8.0
        return (base + step * codes).reshape(n, Hkv, d).astype(np.float32), codes.reshape(n, Hkv, d)

    nb = 18
    rec = gq.record_bytes(d, bits, group)
    kp = np.zeros(nb * Hkv * rec, np.uint8)
    vp = np.zeros_like(kp)
    bt = rng.permutation(nb).astype(np.int32).reshape(3, 6)         # scattered physical blocks
    q = rng.standard_normal((3, Hq, d))
    refs = {}
    for b in (0, 2):
        L = lens[b]
        K, kc = grid(L)
        V, vc = grid(L)
        j = np.arange(L)
        slots = bt[b, j // 16].astype(np.int64) * 16 + j % 16
        ck, ks, kz = gq.encode(K, bits, group)
        cv, vs, vz = gq.encode(V, bits, group)
        np.testing.assert_array_equal(ck, kc)
        np.testing.assert_array_equal(gq.decode_values(ck, ks, kz, group), K)
        np.testing.assert_array_equal(gq.decode_values(cv, vs, vz, group), V)
        gq.pack(ck, ks, kz, slots, kp, Hkv, bits, group)
        gq.pack(cv, vs, vz, slots, vp, Hkv, bits, group)
        refs[b] = (K, V)
    out = gq.decode(q, Hkv, kp, vp, bt, np.array(lens, np.int32), bits, group)
    for b in (0, 2):
        K, V = refs[b]
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            s = K[:, kv].astype(np.float64) @ q[b, h] / np.sqrt(d)
            p = np.exp(s - s.max())
            ref = (p / p.sum()) @ V[:, kv].astype(np.float64)
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(out[1], 0.0)


def test_gq_bits_per_dim_match_the_stated_saving():
    """4.5 and 8.5 bits per coordinate at d = 128, group 64 (fp16 scale and bias per
    group): 3.6x and 1.9x smaller than fp16, the "~2-4x vs FP16" of the README table."""
    for bits, want in ((4, 4.5), (8, 8.5)):
        b = gq.record_bytes(128, bits, 64) * 8 / (16 * 128)
        assert b == want
        assert 1.8 <= 16 / b <= 4.0


# ------------------------------------------------------------------ hybrid cache upkeep

def _hybrid_run(d, H, W, T, bt, seed=0):
    """T appends, one token per step, into an empty hybrid cache of window W (one sequence)."""
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, H, d)).astype(np.float32)
    V = rng.standard_normal((T, H, d)).astype(np.float32)
    nblk = int(bt.max()) + 2
    kp = np.zeros((nblk, H, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((nblk, H, oracle.record_bytes(False, d)), np.uint8)
    wk = np.zeros((1, W, H, d), np.float32)
    wv = np.zeros_like(wk)
    wl, cl = np.zeros(1, np.int32), np.zeros(1, np.int32)
    for t in range(T):
        wk, wv, wl, cl = oracle.hybrid_append(D, S, K[t][None], V[t][None], wk, wv, wl, cl, bt, kp, vp)
    return D, S, K, V, kp, vp, wk, wv, int(wl[0]), int(cl[0])


def test_hybrid_append_keeps_the_last_window_tokens_and_compresses_the_rest():
    # 40 tokens through a window of 12: the first 28 are compressed at their positions, byte for byte
    # the records a direct encode of those tokens writes, and token p of the last 12 sits in slot p mod 12
    d, H, W, T = 128, 2, 12, 40
    bt = np.array([[5, 1, 3]], np.int32)
    D, S, K, V, kp, vp, wk, wv, wl, cl = _hybrid_run(d, H, W, T, bt)
    assert (cl, wl) == (T - W, W)
    for p in range(T - W, T):
        assert np.array_equal(wk[0, p % W], K[p]) and np.array_equal(wv[0, p % W], V[p])
    kd, vd = np.zeros_like(kp), np.zeros_like(vp)
    slots = synth.slots_for(bt, 0, 0, T - W)
    oracle.encode(True, D, S, K[:T - W], slots, kd)
    oracle.encode(False, D, S, V[:T - W], slots, vd)
    assert np.array_equal(kp, kd) and np.array_equal(vp, vd)


def test_hybrid_append_fills_the_window_before_compressing():
    d, H, W, T = 128, 1, 8, 5
    bt = np.array([[0]], np.int32)
    _, _, K, _, kp, vp, wk, _, wl, cl = _hybrid_run(d, H, W, T, bt)
    assert (cl, wl) == (0, T)
    assert np.array_equal(wk[0, :T], K) and not kp.any() and not vp.any()


def test_hybrid_append_attends_the_whole_sequence_while_it_fits_the_window():
    # no token has left the window: hybrid attention is the textbook softmax over all T tokens
    d, H, W, T = 128, 2, 16, 11
    bt = np.array([[0]], np.int32)
    D, S, K, V, kp, vp, wk, wv, wl, cl = _hybrid_run(d, H, W, T, bt, seed=3)
    q = np.random.default_rng(4).standard_normal((1, 2 * H, d))
    out = oracle.decode_hybrid(D, S, q, H, kp, vp, bt, np.array([cl]), wk, wv, np.array([wl]))
    for h in range(2 * H):
        s = K[:, h // 2].astype(np.float64) @ q[0, h] / np.sqrt(d)
        p = np.exp(s - s.max())
        ref = (p[:, None] * V[:, h // 2]).sum(0) / p.sum()
        assert np.max(np.abs(out[0, h] - ref)) < 1e-12


def test_hybrid_append_leaves_a_state_it_does_not_produce():
    # a window that is not full while the history length is not a multiple of the window
    d, H, W = 128, 1, 4
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    kp = np.zeros((2, H, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((2, H, oracle.record_bytes(False, d)), np.uint8)
    wk = np.ones((1, W, H, d), np.float32)
    x = np.full((1, H, d), 2.0, np.float32)
    wk2, _, wl, cl = oracle.hybrid_append(D, S, x, x, wk, wk, np.array([1], np.int32), np.array([3], np.int32),
                                          np.array([[0]], np.int32), kp, vp)
    assert np.array_equal(wk2, wk) and (int(wl[0]), int(cl[0])) == (1, 3) and not kp.any()


def test_hybrid_append_leaves_a_full_window_whose_token_has_no_block():
    # the leaving token's history position (16) is past the one-block table: nothing can move,
    # so neither the window nor the lengths change and the pools stay untouched
    d, H, W = 128, 1, 4
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    kp = np.zeros((2, H, oracle.record_bytes(True, d)), np.uint8)
    vp = np.zeros((2, H, oracle.record_bytes(False, d)), np.uint8)
    wk = np.arange(W * H * d, dtype=np.float32).reshape(1, W, H, d)
    x = np.full((1, H, d), 2.0, np.float32)
    for table in (np.array([[0]], np.int32), np.array([[0, 7]], np.int32)):   # past the table; id 7 outside the pool
        wk2, wv2, wl, cl = oracle.hybrid_append(D, S, x, x, wk, wk, np.array([W], np.int32),
                                                np.array([16], np.int32), table, kp, vp)
        assert np.array_equal(wk2, wk) and np.array_equal(wv2, wk)
        assert (int(wl[0]), int(cl[0])) == (W, 16) and not kp.any() and not vp.any()
