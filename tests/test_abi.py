"""The C ABI library loads and exports every symbol include/dsa.h declares, and
its host-side argument checks return the documented codes (CPU only: no call
here reaches the GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_score_gb300 import build
    try:
        path = build.build()
    except RuntimeError as e:   # no nvcc on this machine
        pytest.skip(str(e))
    from sparse_attention_indexer_score_gb300 import dsa
    dsa._lib = None
    return dsa.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes_are_host_only(lib):
    a = lib.dsa_workspace_size(0, 64, 64, 128, 2048)
    b = lib.dsa_workspace_size(0, 128, 64, 128, 2048)
    assert a > 64 * 128 * 64 * 4 and b > a
    assert lib.dsa_topk_workspace_size(10, 64) >= 10 * 2048 * 4


def test_host_argument_checks(lib):
    # format, counts and strides are checked before anything touches the GPU
    assert lib.dsa_quantize_query(7, None, 4096, None, 32, 1, None, None, None) == -2
    assert lib.dsa_quantize_query(0, None, 4096, None, 32, -1, None, None, None) == -1
    assert lib.dsa_quantize_query(0, None, 4096, None, 32, 0, None, None, None) == 0
    assert lib.dsa_quantize_query(0, 16, 4000, 16, 32, 2, 16, 16, None) == -1
    assert lib.dsa_insert_key(0, 16, 128, 16, 16, 1e-6, 16, 1, 16, 4352, 1, None, None) == -1   # FP8 stride < 8448
    assert lib.dsa_insert_key(2, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == 0
    assert lib.dsa_decode_layout(None, 0, None, 0, -1, None, None, None) == -1
    assert lib.dsa_decode_layout(16, 1, 16, 2, 2, 16, 16, None) == -1        # fewer seq_lens than requests
    assert lib.dsa_score_paged(4, *([0] * 21)) == -2
    assert lib.dsa_selftest_wait_timeout(None, None) == -1
    assert lib.dsa_quantize_queries_rg(16, 4096, 128, 48, 1, 16, 16, None) == -2      # 48 heads
    assert lib.dsa_quantize_queries_rg(None, 0, 128, 64, 0, None, None, None) == 0    # no rows
    assert lib.dsa_quantize_queries_rg(16, 4096, 100, 32, 1, 16, 16, None) == -1     # head stride < 128
    assert lib.dsa_insert_key(4, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == -2
    assert lib.dsa_insert_key(3, 16, 128, 16, 16, 1e-6, 16, 0, 16, 4352, 1, None, None) == 0   # row-group MXFP4
    assert lib.dsa_insert_key(3, 16, 128, 16, 16, 1e-6, 16, 1, 16, 4352 - 16, 1, None, None) == -1
    assert lib.dsa_score_paged(3, 32, 32, 32, 4352 + 8, 1, 16, 1, 1, 16, 16, 1, 1, 1, None, 0, 4, None, 256,
                               10**9, None, None) == -1                         # row-group stride not a multiple of 16
    assert lib.dsa_score_paged(0, 16, 16, 16, 8448, 1, 16, 1, 1, 16, 16, 1, 0, 1, None, 0, 4, None, 256, 10**9,
                               None, None) == 0                                 # zero rows
    assert lib.dsa_score_paged(2, 32, 32, 32, 4352 + 8, 1, 16, 1, 1, 16, 16, 1, 1, 1, None, 0, 4, None, 256,
                               10**9, None, None) == -1                         # MXFP4 stride not a multiple of 16
    assert lib.dsa_topk(None, 10, None, 1, 20, 4, None, None, 0, None) == -1  # ld < width
