"""The timeout report of the error contract (include/mxa.h: a kernel whose
bounded wait runs out records the device error word, mxa_get_error() reports
MXA_ERR_TIMEOUT and clears it).

The hook of include/mxa_testing.h runs the kernels' own bounded wait in a
one-warp kernel on a barrier that nothing arrives on, with a budget of about
half a millisecond; nothing asynchronous is in flight, so the kernel simply
returns after recording the error.  The context stays usable: the next
report is clean and a forward afterwards still matches the oracle."""
import math

import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import check_outputs, gpu_views, oracle_views, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    from block_scaled_mxfp8_gb300 import mxa

    torch.cuda.synchronize()
    assert mxa.mxa_get_error() == mxa.MXA_OK
    assert mxa.mxa_test_wait_timeout(-1) == mxa.MXA_ERR_ARG
    assert mxa.mxa_test_wait_timeout(1 << 20) == mxa.MXA_OK
    assert mxa.mxa_get_error() == mxa.MXA_ERR_TIMEOUT
    assert mxa.mxa_get_error() == mxa.MXA_OK  # the report cleared the word
    # a wait whose barrier does complete is not an error: the forward below
    # runs every kernel wait to completion
    w = inp.workload("tiny", causal=True)
    t = inp.tensors(w, with_grad=False)
    geo, gv = gpu_views(w, t, names=("q", "k", "v"))
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, True)
    torch.cuda.synchronize()
    assert mxa.mxa_get_error() == mxa.MXA_OK
    _, d = oracle_views(w, t, names=("q", "k", "v"))
    O, L = orc.attn_fwd_alg1(d["q"]["row"], d["k"]["row"], d["v"]["tok"], w.cu_seqlens.numpy(), True,
                             1.0 / math.sqrt(w.d))
    check_outputs("after timeout", {"O": to_np(o), "LSE": lse.cpu().numpy()}, {"O": O, "LSE": L})
