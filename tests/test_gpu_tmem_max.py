"""The forward's row maximum on fully visible key tiles comes from the TMEM
load itself (tcgen05.ld.red .max, include/mxa_testing.h mxa_test_tmem_max):
each row's values read back bit for bit, and the two 32-column maxima equal
numpy's on rows with mixed signs, all-negative rows, ties and large
magnitudes."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_tmem_load_with_max_matches_numpy():
    from block_scaled_mxfp8_gb300 import mxa

    rng = np.random.default_rng(7)
    x = (rng.standard_normal((128, 64)) * 30.0).astype(np.float32)
    x[1] = -np.abs(x[1]) - 1.0                         # all negative
    x[2] = 5.0                                         # all equal
    x[3, :32] = -3e38
    x[3, 17] = -2.5                                    # one large negative, one less negative
    x[4] = rng.standard_normal(64).astype(np.float32) * 1e30
    x[5, 31] = x[5, :32].max() + 1e-3                  # the last column of a half
    x[6, 0] = x[6, :32].max() + 1.0                    # the first column of a half
    xd = torch.from_numpy(x).cuda()
    out = torch.zeros(128, 3, dtype=torch.float32, device="cuda")
    assert mxa.mxa_test_tmem_max(xd, out) == mxa.MXA_OK
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.array_equal(o[:, 2], np.zeros(128, np.float32)), "values did not read back"
    assert np.array_equal(o[:, 0], x[:, :32].max(axis=1))
    assert np.array_equal(o[:, 1], x[:, 32:].max(axis=1))
