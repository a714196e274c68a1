"""Inputs past 2^31 elements: element (and byte) offsets that no 32-bit index
holds. GATE and UP (or X) have 266,240 rows of 8192 values (8.7 GB each), so
rows from 262,144 on start beyond element 2^31. The rows repeat a block of
1024 seeded integer rows (copied on the device), so the expected output of
row r is the oracle's row r % 1024, exactly; sampled rows on both sides of
the 2^31 boundary and the last row are compared."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import integer_inputs, require_gpu
from transformer_linear_layer_tcgen05_gb300 import lin

pytestmark = pytest.mark.gpu

M, N, K = 266240, 2048, 8192
BLOCK = 1024
ROWS = [0, 1023, 131071, 262143, 262144, 262145, 263167, 265000, M - 1]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("form", ["matmul_residual_swiglu_a_w16", "matmul_residual"])
def test_rows_beyond_2_pow_31_elements(form):
    import torch
    base = integer_inputs(form, BLOCK, N, K, seed=31)
    reps = M // BLOCK
    dev = {}
    for k, v in base.items():
        t = torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
        dev[k] = t if k in ("W", "W16") else t.repeat(reps, 1)
    Y = torch.full((M, N), float("nan"), device="cuda")
    lin.run_form(form, dev, Y)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    got = Y[ROWS].cpu().numpy().astype(np.float64)
    ref, _ = oracle.reference(form, base, rows=[r % BLOCK for r in ROWS])
    assert np.array_equal(got, ref)
    del dev, Y
    torch.cuda.empty_cache()
