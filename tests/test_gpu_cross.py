"""GPU cross-attention (query and key/value documents of their own lengths)
against the Algorithm 1 oracle on the same quantized operands: O, LSE, dQ,
dK, dV (the direct oracle's error reported)."""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import check_outputs, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # name, query lengths, key lengths (None: equal documents), Hq, Hkv, d, seed
    ("packed_gqa", [100, 512, 7, 260], [900, 33, 1500, 129], 4, 2, 128, 91),
    ("batched_d64", [256, 256, 256], [640, 640, 640], 2, 2, 64, 92),
    ("doc_without_queries", [128, 0, 64], [300, 200, 50], 2, 1, 128, 93),
]


def _geo(lengths, equal):
    from block_scaled_mxfp8_gb300 import mxa

    if equal:
        return mxa.Geometry.batched(len(lengths), lengths[0])
    return mxa.Geometry.packed(lengths)


def _run(lq, lk, Hq, Hkv, d, seed):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.cross_tensors(lq, lk, Hq, Hkv, d, seed)
    equal = len(set(lq)) == 1 and len(set(lk)) == 1
    gq, gk = _geo(lq, equal), _geo(lk, equal)
    v = {nm: mxa.quantize(t[nm].cuda(), gq) for nm in ("q", "do")}
    v.update({nm: mxa.quantize(t[nm].cuda(), gk) for nm in ("k", "v")})
    o, lse = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], gq, False, kv_geo=gk)
    bv = {"q_row": v["q"][0], "k_row": v["k"][0], "v_row": v["v"][0], "g_row": v["do"][0],
          "q_tok": v["q"][1], "k_tok": v["k"][1], "g_tok": v["do"][1]}
    dq, dk, dv = mxa.bwd(bv, o, lse, gq, False, kv_geo=gk)
    o0, lse0 = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], gq, False, kv_geo=gk, use_list=False)
    torch.cuda.synchronize()
    mxa.check_error()
    return t, o, lse, dq, dk, dv, o0, lse0


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cross_attention_matches_oracle(case):
    name, lq, lk, Hq, Hkv, d, seed = case
    t, o, lse, dq, dk, dv, o0, lse0 = _run(lq, lk, Hq, Hkv, d, seed)
    # the work list only changes which CTA computes which tile
    assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))

    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    deq = {}
    for nm, cu in (("q", cq), ("do", cq), ("k", ck), ("v", ck)):
        rc, rs = orc.quant_row(t[nm])
        tc, ts = orc.quant_tok(t[nm], cu)
        deq[nm] = {"row": orc.dequant_row(rc, rs), "tok": orc.dequant_tok(tc, ts, cu)}
    alpha = 1.0 / math.sqrt(d)
    vw = (deq["q"]["row"], deq["k"]["row"], deq["v"]["tok"], deq["v"]["row"], deq["do"]["row"], deq["q"]["tok"],
          deq["k"]["tok"], deq["do"]["tok"])
    O, LSE = orc.attn_fwd_alg1(vw[0], vw[1], vw[2], cq, False, alpha, cu_k=ck)
    r = orc.attn_bwd_alg1(*vw, cq, False, alpha, cu_k=ck)
    rd = orc.attn_bwd_x(*vw, cq, ck, alpha)
    assert np.array_equal(np.nan_to_num(r["O"]), np.nan_to_num(O))
    got = {"O": to_np(o), "LSE": lse.cpu().numpy(), "dQ": to_np(dq), "dK": to_np(dk), "dV": to_np(dv)}
    check_outputs(name, got, dict(r, LSE=LSE), rd)
    # keys of a document without queries get zero gradients
    for b in range(len(lq)):
        if lq[b] == 0:
            assert not to_np(dk)[ck[b]:ck[b + 1]].any() and not to_np(dv)[ck[b]:ck[b + 1]].any()
