"""mxa_bwd_noalloc: the backward without a caller workspace.

Some callers cannot allocate device memory (a framework whose caching
allocator owns all of it, a plugin host with a fixed budget), so they cannot
pass mxa_bwd a workspace; mxa_bwd_noalloc uses a statically sized device array
owned by the library instead.  These tests call it through the C ABI and
check its results against mxa_bwd with a caller workspace:
  * each target call follows a call on a different, larger packed shape
    (other lengths and seeds), so the array holds unrelated rows, tile lists
    and dS blocks when the target call starts; two target calls in a row;
  * every dQ mode that fits (FP32, FP16 x 2^9, FP16 per-row boost) and the
    strict dQ operand, bit for bit (all of them are deterministic and take
    mxa_bwd's full-workspace path here);
  * an FP32 call whose full workspace exceeds the array but whose smallest
    one fits: it forms dS again in the dQ kernel, dK and dV bit-identical to
    mxa_bwd's, dQ within the parity bar.
The file is named to be collected last; it passes alone or after the others.
"""
import ctypes

import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp

from ._common import assert_close, to_np

pytestmark = pytest.mark.gpu


def _setup(w, strict=False):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w)
    geo = mxa.Geometry.batched(w.B, w.L) if w.lengths is None else mxa.Geometry.packed(w.lengths)
    v = {k: mxa.quantize(t[k].cuda(), geo) for k in ("q", "k", "v", "do")}
    vkey = mxa.quantize_key(t["v"].cuda(), geo) if strict else None
    kkey = mxa.quantize_key(t["k"].cuda(), geo) if strict else None
    o, lse = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], geo, w.causal, v_key=vkey)
    views = {"q_row": v["q"][0], "k_row": v["k"][0], "v_row": v["v"][0], "g_row": v["do"][0],
             "q_tok": v["q"][1], "k_tok": v["k"][1], "g_tok": v["do"][1]}
    return geo, views, o, lse, kkey


def _noalloc(views, o, lse, geo, causal, dq_mode, kkey, like):
    from block_scaled_mxfp8_gb300 import mxa

    dq, dk, dv = (torch.full_like(x, float("nan")) for x in like)
    p = mxa.bwd_params(views, o, lse, dq, dk, dv, geo, causal, dq_mode, k_key=kkey)
    st = mxa.lib().mxa_bwd_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mxa.MXA_OK, mxa.status_str(st)
    torch.cuda.synchronize()
    mxa.check_error()
    return (dq, dk, dv), p


def _dirty_the_array(dq_mode):
    """A call on another packed shape (other lengths, seed and head count)
    that fills the scratch array with unrelated contents."""
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("noalloc_other", lengths=[700, 5, 260, 391], Hq=2, Hkv=1, d=128, causal=False, seed=61)
    geo, views, o, lse, _ = _setup(w)
    like = mxa.bwd(views, o, lse, geo, w.causal)
    _noalloc(views, o, lse, geo, w.causal, mxa.MXA_DQ_FP32, None, like)


@pytest.mark.parametrize("case", ["fp32", "fp16_x512", "fp16_row", "strict"])
def test_noalloc_matches_workspace_backward_after_other_calls(case):
    from block_scaled_mxfp8_gb300 import mxa

    dq_mode = {"fp32": 0, "fp16_x512": 1, "fp16_row": 2, "strict": 0}[case]
    strict = case == "strict"
    w = inp.make_custom("noalloc", lengths=[300, 77, 512], Hq=4, Hkv=2, d=128, causal=True, seed=41)
    geo, views, o, lse, kkey = _setup(w, strict)
    ref = mxa.bwd(views, o, lse, geo, w.causal, dq_mode=dq_mode, k_key=kkey)
    torch.cuda.synchronize()
    _dirty_the_array(dq_mode)
    for _ in range(2):
        got, p = _noalloc(views, o, lse, geo, w.causal, dq_mode, kkey, ref)
        assert mxa.mxa_bwd_workspace_bytes(p) <= mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
        for name, g, want in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(g, want), (case, name)


def test_noalloc_forms_ds_again_when_only_the_smallest_workspace_fits():
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("noalloc_big", B=1, L=4096, Hq=8, Hkv=4, d=128, causal=True, seed=62)
    geo, views, o, lse, _ = _setup(w)
    ref = mxa.bwd(views, o, lse, geo, w.causal)
    torch.cuda.synchronize()
    _dirty_the_array(0)
    for _ in range(2):
        got, p = _noalloc(views, o, lse, geo, w.causal, mxa.MXA_DQ_FP32, None, ref)
        assert mxa.mxa_bwd_workspace_min_bytes(p) <= mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
        assert mxa.mxa_bwd_workspace_bytes(p) > mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        assert_close("dQ (dS formed again)", to_np(got[0]), to_np(ref[0]))


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
