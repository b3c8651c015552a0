"""The block-scaled MMA rate probe (include/mxa_testing.h) that the
benchmark's tensor-core roofline is measured with: every CTA completes, the
device error word stays clear, and the rate per SM clock is positive and
below the instruction's own bound (N = 256 per 128 clocks is about 16.4
kFLOP per SM clock; twice that would mean the probe is not doing the work)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_mma_probe_runs_and_reports_a_plausible_rate():
    import bench
    from block_scaled_mxfp8_gb300 import mxa

    cyc = torch.zeros(4, dtype=torch.int64, device="cuda")
    assert mxa.mxa_test_mma_rate(0, cyc) == mxa.MXA_ERR_ARG
    r = bench.mma_probe(torch.device("cuda", 0), iters=2000)
    assert r is not None, "probe failed"
    print(r)
    assert 2000.0 < r["flop_per_sm_clk"] < 33000.0
    assert r["pflops"] > 0.5
    assert mxa.mxa_get_error() == mxa.MXA_OK


def test_ex2_probe_runs_and_reports_a_plausible_rate():
    """The exponential-unit probe behind the bench line's exp_unit fractions:
    arguments checked, every CTA completes, and the rate is positive and at
    most 64 per SM clock (the FLAMIA notes' sec. 7 quotes 32 for B300)."""
    import bench
    from block_scaled_mxfp8_gb300 import mxa

    cyc = torch.zeros(4, dtype=torch.int64, device="cuda")
    assert mxa.mxa_test_ex2_rate(0, cyc) == mxa.MXA_ERR_ARG
    r = bench.ex2_probe(torch.device("cuda", 0), iters=512)
    assert r is not None, "probe failed"
    print(r)
    assert 4.0 < r["ex2_per_sm_clk"] <= 64.0
    assert mxa.mxa_get_error() == mxa.MXA_OK
