"""Failure detection on the GPU without a fault: a bounded device wait that runs out reports
TQ_STATUS_TIMEOUT through the status word, the kernel exits normally, and the context stays usable.
(Bad block ids and slots, the other device-side failures, are covered by the parity tests.)
"""
import time

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
import turboquant_compressed_kv_gb300 as tq  # noqa: E402
from turboquant_compressed_kv_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tq.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == tq.STATUS_TIMEOUT
    assert 0.3 < waited < 30.0, waited          # the wait's limit is about half a second
    # the context still runs kernels: the device codebook, then an encode checked against the oracle
    d = 128
    D, S = synth.rotation_signs(d), synth.qjl_matrix(d)
    params, cent = tq.codebook_init(d, D, S, device="cuda")
    assert np.max(np.abs(np.array(cent) - oracle.codebook()[0])) < 1e-12
    x = np.random.default_rng(0).standard_normal((16, 1, d)).astype(np.float32)
    slots = np.arange(16, dtype=np.int64)
    pool = tq.empty_pool(1, 1, d, "v", "cuda")
    status.zero_()
    tq.encode_v(params, d, torch.from_numpy(x).cuda(), torch.from_numpy(slots).cuda(), pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = oracle.unpack(False, d, pool.cpu().numpy(), 1, slots)
    ref = oracle.encode(False, D, S, x, slots, np.zeros_like(pool.cpu().numpy()), want_details=True)
    margin = np.min(np.abs(ref["z"][..., None] - oracle.codebook()[1]), axis=-1)
    assert np.all((g["codes"] == ref["codes"]) | (margin < 1e-6))


def test_selftest_wait_timeout_needs_a_status_word():
    assert tq.load_library().tq_selftest_wait_timeout(None, None) == -1   # TQ_ERR_INVALID
