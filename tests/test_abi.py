"""The C-ABI library loads on a machine without a GPU, exports every entry
point declared in include/tq.h, answers its size queries and rejects bad
arguments on the host before any launch.  No compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from turboquant_compressed_kv_gb300 import build
    build.build()
    import turboquant_compressed_kv_gb300 as tq
    return tq.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_sizes(lib):
    import turboquant_compressed_kv_gb300 as tq
    assert tq.k_record_bytes(128) == 1088 and tq.v_record_bytes(128) == 800
    assert tq.k_record_bytes(256) == 2112 and tq.v_record_bytes(256) == 1568
    assert tq.k_record_bytes(64) == 0 and tq.params_bytes(96) == 0
    assert tq.params_bytes(128) >= 128 * 128 * 4
    assert tq.decode_workspace_bytes(128, 16, 32, 4096) > 0
    assert tq.decode_workspace_bytes(100, 16, 32, 4096) == 0
    assert tq.decode_workspace_bytes_mq(128, 16, 1, 32, 4096) == tq.decode_workspace_bytes(128, 16, 32, 4096)
    assert tq.decode_workspace_bytes_mq(128, 16, 2, 32, 4096) == tq.decode_workspace_bytes(128, 16, 64, 4096)
    assert tq.decode_workspace_bytes_mq(128, 16, 0, 32, 4096) == 0


def test_host_side_argument_errors(lib):
    P = ctypes.c_void_p
    fake = P(16)    # never dereferenced: every call below fails its checks first
    assert lib.tq_encode_k(fake, 64, fake, 0, 10, 1, fake, fake, 4, None, None) == -2
    assert lib.tq_encode_k(fake, 128, fake, 7, 10, 1, fake, fake, 4, None, None) == -6
    assert lib.tq_encode_k(fake, 128, fake, 0, -1, 1, fake, fake, 4, None, None) == -1
    assert lib.tq_encode_k(fake, 128, fake, 0, 0, 1, fake, fake, 4, None, None) == 0    # empty: no-op
    assert lib.tq_encode_v(fake, 128, None, 0, 3, 1, fake, fake, 4, None, None) == -1
    assert lib.tq_encode_k(P(17), 128, fake, 0, 3, 1, fake, fake, 4, None, None) == -7
    args = [fake, 128, fake, 0, 2, 12, 8, fake, fake, 4, fake, 1, fake, 16, fake, fake, 1 << 30, None, None]
    assert lib.tq_decode_attn(*args) == -3                      # 12 % 8 != 0
    args[5], args[6] = 32, 2
    assert lib.tq_decode_attn(*args) == -3                      # group 16 > 8
    args[5], args[6] = 32, 8
    args[16] = 10
    assert lib.tq_decode_attn(*args) == -4                      # workspace too small
    mq = [fake, 128, fake, 0, 2, 3, 32, 8, fake, fake, 4, fake, 1, fake, 16, fake, fake, 1 << 30, None, None]
    assert lib.tq_decode_attn_mq(*mq) == -3                     # 3 queries x group 4 > 8
    mq[5] = 0
    assert lib.tq_decode_attn_mq(*mq) == -1                     # q_len 0
    mq[5], mq[17] = 2, 10
    assert lib.tq_decode_attn_mq(*mq) == -4                     # workspace too small
    assert lib.tq_paged_append(fake, 128, fake, fake, 0, 0, 8, fake, 4, fake, fake, fake, 4, None, None) == 0
    D = (ctypes.c_int8 * 128)(*([1] * 127 + [3]))
    S = (ctypes.c_float * (128 * 128))()
    assert lib.tq_codebook_init(128, D, S, fake, 1 << 20, None, None) == -1   # D entry not +-1
    assert lib.tq_codebook_init(128, D, S, fake, 16, None, None) == -4
    assert lib.tq_error_string(-3).decode().startswith("n_q_heads")
