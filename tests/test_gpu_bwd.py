"""GPU backward vs the Algorithm 1 oracle on the same quantized operands
(dQ, dK, dV), with the direct oracle's error reported."""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import assert_close, check_outputs, gpu_views, oracle_views, to_np

pytestmark = pytest.mark.gpu

CASES = [
    (inp.workload("tiny", causal=False), 0),
    (inp.workload("tiny", causal=True), 0),
    (inp.workload("tiny", causal=True), 1),
    (inp.make_custom("d128_ragged_gqa_causal", lengths=[1, 129, 300, 64, 7], Hq=4, Hkv=2, d=128, causal=True,
                     seed=31), 0),
    (inp.make_custom("d128_ragged", lengths=[250, 33, 513], Hq=2, Hkv=1, d=128, causal=False, seed=32), 1),
    (inp.make_custom("tokblock_gqa", lengths=[100, 400, 37], Hq=4, Hkv=2, d=128, causal=True, mode="tokblock",
                     hadamard=True, seed=33), 0),
    # d = 64 with four query heads per kv head on packed documents, in the
    # FP32 and the per-row FP16 dQ modes; eight query heads per kv head (the
    # dK/dV CTA walks 8 heads x its query tiles)
    (inp.make_custom("d64_ragged_gqa4_causal", lengths=[300, 1, 129, 640], Hq=8, Hkv=2, d=64, causal=True,
                     seed=34), 0),
    (inp.make_custom("d64_ragged_gqa4_causal", lengths=[300, 1, 129, 640], Hq=8, Hkv=2, d=64, causal=True,
                     seed=34), 2),
    (inp.make_custom("d128_batched_gqa8", B=2, L=512, Hq=8, Hkv=1, d=128, causal=False, seed=35), 0),
    # equal documents, causal: the forward and dK/dV grids in their causal
    # launch order (40 and 20 (document, head) groups; the last 16 of each go
    # heaviest tile first across groups)
    (inp.make_custom("b5_gqa2_batched_causal", B=5, L=384, Hq=8, Hkv=4, d=128, causal=True, seed=37), 0),
    (inp.make_custom("b5_gqa2_batched_causal", B=5, L=384, Hq=8, Hkv=4, d=128, causal=True, seed=37), 1),
]


def run_bwd(w, dq_mode):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=True)
    geo, gv = gpu_views(w, t)
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
    views = {"q_row": gv["q"][0], "k_row": gv["k"][0], "v_row": gv["v"][0], "g_row": gv["do"][0],
             "q_tok": gv["q"][1], "k_tok": gv["k"][1], "g_tok": gv["do"][1]}
    dq, dk, dv = mxa.bwd(views, o, lse, geo, w.causal, dq_mode=dq_mode)
    torch.cuda.synchronize()
    mxa.check_error()
    _, d = oracle_views(w, t)
    cu = w.cu_seqlens.numpy()
    r = oracle_bwd(w, d)
    return t, (dq, dk, dv), r


def oracle_bwd(w, d, direct=False):
    """The Algorithm 1 oracle (direct=True: P and dS in fp64) on the decoded
    views d of workload w."""
    fn = orc.attn_bwd if direct else orc.attn_bwd_alg1
    return fn(d["q"]["row"], d["k"]["row"], d["v"]["tok"], d["v"]["row"], d["do"]["row"], d["q"]["tok"],
              d["k"]["tok"], d["do"]["tok"], w.cu_seqlens.numpy(), w.causal, 1.0 / math.sqrt(w.d))


@pytest.mark.parametrize("w,mode", CASES, ids=["%s%s_dq%s" % (c.name, "_causal" if c.causal else "", m)
                                                for c, m in CASES])
def test_bwd_matches_oracle(w, mode):
    t, (dq, dk, dv), r = run_bwd(w, mode)
    _, d = oracle_views(w, t)
    check_outputs("%s dq%d" % (w.name, mode), {"dQ": to_np(dq), "dK": to_np(dk), "dV": to_np(dv)}, r,
                  oracle_bwd(w, d, direct=True))


RECOMPUTE_CASES = [
    inp.workload("tiny", causal=True),
    inp.make_custom("d128_ragged_gqa_causal", lengths=[1, 129, 300, 64, 7], Hq=4, Hkv=2, d=128, causal=True,
                    seed=31),
]


@pytest.mark.parametrize("w", RECOMPUTE_CASES, ids=[c.name for c in RECOMPUTE_CASES])
def test_bwd_min_workspace_forms_ds_again(w):
    """FP32 mode with the smallest accepted workspace: the dQ kernel forms dS
    from S and dP again instead of reading the blocks the dK/dV pass emitted.
    Both paths quantize the same 32 x 32 blocks, so both meet the oracle bar,
    and dK, dV (computed identically) are bit-identical."""
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=True)
    geo, gv = gpu_views(w, t)
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
    views = {"q_row": gv["q"][0], "k_row": gv["k"][0], "v_row": gv["v"][0], "g_row": gv["do"][0],
             "q_tok": gv["q"][1], "k_tok": gv["k"][1], "g_tok": gv["do"][1]}
    full = mxa.bwd(views, o, lse, geo, w.causal)
    T, Hq, d = views["q_row"].codes.shape
    Hkv = views["k_row"].codes.shape[1]
    out = tuple(torch.empty((T, H, d), dtype=torch.bfloat16, device="cuda") for H in (Hq, Hkv, Hkv))
    p = mxa.bwd_params(views, o, lse, *out, geo, w.causal)
    need_min, need = mxa.mxa_bwd_workspace_min_bytes(p), mxa.mxa_bwd_workspace_bytes(p)
    assert 0 < need_min < need
    ws = torch.empty(need_min, dtype=torch.uint8, device="cuda")
    assert mxa.mxa_bwd(p, ws, need_min) == mxa.MXA_OK
    torch.cuda.synchronize()
    mxa.check_error()
    _, dd = oracle_views(w, t)
    r = oracle_bwd(w, dd)
    assert_close("dQ (dS formed again)", to_np(out[0]), r["dQ"])
    assert torch.equal(out[1], full[1]) and torch.equal(out[2], full[2])


def test_fp16_mode_small_workspace_takes_the_fused_kernel():
    """FP16 x 2^9 mode with a workspace that holds the fp16 dQ accumulator but
    not the emitted dS: the fused backward kernel (atomics into the fp16
    accumulator, order varies) -- same bar against the oracle; dK and dV are
    the same computation as with the full workspace, within the bar."""
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("d128_ragged_gqa_causal", lengths=[300, 77, 512], Hq=4, Hkv=2, d=128, causal=True,
                        seed=36)
    t = inp.tensors(w, with_grad=True)
    geo, gv = gpu_views(w, t)
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
    views = {"q_row": gv["q"][0], "k_row": gv["k"][0], "v_row": gv["v"][0], "g_row": gv["do"][0],
             "q_tok": gv["q"][1], "k_tok": gv["k"][1], "g_tok": gv["do"][1]}
    T, Hq, d = views["q_row"].codes.shape
    Hkv = views["k_row"].codes.shape[1]
    out = tuple(torch.empty((T, H, d), dtype=torch.bfloat16, device="cuda") for H in (Hq, Hkv, Hkv))
    p = mxa.bwd_params(views, o, lse, *out, geo, w.causal, mxa.MXA_DQ_FP16_X512)
    need_min, need = mxa.mxa_bwd_workspace_min_bytes(p), mxa.mxa_bwd_workspace_bytes(p)
    assert 0 < need_min < need
    ws = torch.empty(need_min, dtype=torch.uint8, device="cuda")
    assert mxa.mxa_bwd(p, ws, need_min) == mxa.MXA_OK
    torch.cuda.synchronize()
    mxa.check_error()
    _, dd = oracle_views(w, t)
    r = oracle_bwd(w, dd)
    for name, got, ref in (("dQ", out[0], r["dQ"]), ("dK", out[1], r["dK"]), ("dV", out[2], r["dV"])):
        assert_close(name + " (fused FP16 path)", to_np(got), ref)
