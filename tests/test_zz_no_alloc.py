"""mxa_bwd_noalloc: the backward without a caller workspace.

Some callers cannot allocate device memory (a framework whose caching
allocator owns all of it, a plugin host with a fixed budget), so they cannot
pass mxa_bwd a workspace; mxa_bwd_noalloc uses a statically sized device array
owned by the library instead.  This test calls it through the C ABI, twice in
a row, and checks both results against mxa_bwd with a caller workspace.  The
file is named to be collected last; it passes alone or after the others.
"""
import ctypes

import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp

from ._common import assert_close, to_np

pytestmark = pytest.mark.gpu


def _setup(w):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w)
    geo = mxa.Geometry.batched(w.B, w.L) if w.lengths is None else mxa.Geometry.packed(w.lengths)
    v = {k: mxa.quantize(t[k].cuda(), geo) for k in ("q", "k", "v", "do")}
    o, lse = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], geo, w.causal)
    views = {"q_row": v["q"][0], "k_row": v["k"][0], "v_row": v["v"][0], "g_row": v["do"][0],
             "q_tok": v["q"][1], "k_tok": v["k"][1], "g_tok": v["do"][1]}
    return geo, views, o, lse


@pytest.mark.parametrize("dq_mode", [0, 1])
def test_noalloc_matches_workspace_backward_twice(dq_mode):
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("noalloc", lengths=[300, 77, 512], Hq=4, Hkv=2, d=128, causal=True, seed=41)
    geo, views, o, lse = _setup(w)
    ref = mxa.bwd(views, o, lse, geo, w.causal, dq_mode=dq_mode)
    torch.cuda.synchronize()
    for _ in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in ref)
        p = mxa.bwd_params(views, o, lse, dq, dk, dv, geo, w.causal, dq_mode)
        assert mxa.mxa_bwd_workspace_bytes(p) <= mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
        st = mxa.lib().mxa_bwd_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == mxa.MXA_OK, mxa.status_str(st)
        torch.cuda.synchronize()
        mxa.check_error()
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            assert_close(name, to_np(got), to_np(want))
            if dq_mode == 0:  # the FP32 mode is deterministic: identical bits
                assert torch.equal(got, want), name


def test_noalloc_rejects_oversized_workspace_without_work():
    from block_scaled_mxfp8_gb300 import mxa

    # an FP16-mode call whose dQ accumulator alone exceeds the scratch array
    T, Hq, d = 1 << 16, 8, 128
    sh = mxa.c_shape(T, Hq, Hq, d, None, 1, T, T // 128, 1, 0.0)
    qv = mxa.c_qview(256, 256)
    p = mxa.c_bwd_params(sh, *[qv] * 7, 256, 256, 256, 256, 256, mxa.MXA_DQ_FP16_X512)
    assert mxa.mxa_bwd_workspace_bytes(p) > mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
    st = mxa.lib().mxa_bwd_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mxa.MXA_ERR_WORKSPACE
