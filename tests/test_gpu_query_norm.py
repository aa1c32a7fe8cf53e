"""QueryNorm on GB300 through the C ABI: bit-exact against the oracle in both
summation orders (page *cutedsl.dsa.overlap*, ``QueryNorm``)."""

import numpy as np
import pytest

from dsa_case import bf16_tensor
from oracle.codecs import bf16_round
from oracle.query_norm import COLS, query_norm_cta, query_norm_tiled

pytestmark = pytest.mark.gpu


def _bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _rows(rng, batch):
    x = rng.standard_normal((batch, COLS)).astype(np.float32)
    if batch > 3:
        x[0] = 0.0                                # zero row: rr = 1/sqrt(eps)
        x[1] *= 1e18                              # large
        x[2] *= 1e-18                             # small
        x[3, ::5] *= 300.0                        # outliers
    return bf16_round(x)


@pytest.mark.parametrize("variant", ["row", "tiled"])
@pytest.mark.parametrize("batch", [1, 7, 8, 9, 64, 301])
def test_query_norm_bit_exact(cuda_lib, variant, batch):
    import torch
    rng = np.random.default_rng(batch)
    x = _rows(rng, batch)
    w = bf16_round((1 + 0.1 * rng.standard_normal(COLS)).astype(np.float32))
    stride = COLS + 64                            # q_a is the first part of a wider packed row
    xp = np.zeros((batch, stride), np.uint16)
    xp[:, :COLS] = _bits(x)
    xp[:, COLS:] = 0x7FC0                         # NaNs past q_a must not be read
    got = cuda_lib.query_norm(bf16_tensor(xp, "cuda"), bf16_tensor(_bits(w), "cuda"), 1e-6, variant)
    got = (got.view(torch.int16).cpu().numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
    want = (query_norm_cta if variant == "row" else query_norm_tiled)(x, w, 1e-6)
    assert np.array_equal(got, want)


def test_query_norm_auto_picks_by_batch(cuda_lib):
    import torch
    rng = np.random.default_rng(11)
    w = bf16_round((1 + 0.1 * rng.standard_normal(COLS)).astype(np.float32))
    for batch, oracle in ((63, query_norm_cta), (64, query_norm_tiled)):
        x = _rows(rng, batch)
        got = cuda_lib.query_norm(bf16_tensor(_bits(x), "cuda"), bf16_tensor(_bits(w), "cuda"), 1e-5)
        got = (got.view(torch.int16).cpu().numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(got, oracle(x, w, 1e-5))


def test_query_norm_argument_errors(cuda_lib):
    import torch
    x = torch.zeros((4, COLS), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(COLS, dtype=torch.bfloat16, device="cuda")
    lib = cuda_lib.lib()
    out = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.dsa_query_norm(x.data_ptr(), COLS, w.data_ptr(), 1e-6, -1, out.data_ptr(), COLS, 0, s) == -1
    assert lib.dsa_query_norm(x.data_ptr(), COLS - 8, w.data_ptr(), 1e-6, 4, out.data_ptr(), COLS, 0, s) == -1
    assert lib.dsa_query_norm(x.data_ptr(), COLS, w.data_ptr(), 1e-6, 4, out.data_ptr(), COLS, 2, s) == -1
    assert lib.dsa_query_norm(x.data_ptr() + 2, COLS, w.data_ptr(), 1e-6, 4, out.data_ptr(), COLS, 0, s) == -1
    assert lib.dsa_query_norm(x.data_ptr(), COLS, w.data_ptr(), 1e-6, 0, out.data_ptr(), COLS, 0, s) == 0
