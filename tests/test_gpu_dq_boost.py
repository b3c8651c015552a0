"""GPU FP16 dQ reduction with a per-row boost (MXA_DQ_FP16_ROW; FLAMIA reading
notes sec. 4, the strict accumulator scale) against the oracle (Algorithm 1
variant for the gradients).

* The boost exponent beta_i of every query row, read from the workspace
  (documented layout: fp32 [Hq, T] after the D and LSE rows), equals the
  oracle's dq_row_boost on the same quantized views bit for bit -- an integer
  decided from exponents and code bits on both sides.
* dQ, dK, dV meet the parity bar of the other modes.
* Gradients 2^10 larger: the fixed 2^9 boost overflows fp16 (non-finite or
  far-off dQ), the per-row boost stays within the bar.
* Future perturbation: with the same G rows, every query row in a 32-token
  block strictly before the perturbed token keeps its dQ bit for bit in this
  mode too (deterministic fp16 sums in key-tile order, boosts that depend on
  the visible prefix only).
"""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import assert_close, check_outputs, gpu_views, metrics, oracle_views, to_np

pytestmark = pytest.mark.gpu

CASES = [
    inp.workload("tiny", causal=True),
    inp.make_custom("d128_ragged_gqa_causal", lengths=[1, 129, 300, 64, 7], Hq=4, Hkv=2, d=128, causal=True,
                    seed=31),
    inp.make_custom("d128_ragged", lengths=[250, 33, 513], Hq=2, Hkv=1, d=128, causal=False, seed=32),
    inp.make_custom("tokblock_gqa", lengths=[100, 400, 37], Hq=4, Hkv=2, d=128, causal=True, mode="tokblock",
                    hadamard=True, seed=33),
]


def _views(gv):
    return {"q_row": gv["q"][0], "k_row": gv["k"][0], "v_row": gv["v"][0], "g_row": gv["do"][0],
            "q_tok": gv["q"][1], "k_tok": gv["k"][1], "g_tok": gv["do"][1]}


def _gpu(w, t, mode):
    from block_scaled_mxfp8_gb300 import mxa

    geo, gv = gpu_views(w, t)
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
    views = _views(gv)
    T, Hq, d = views["q_row"].codes.shape
    Hkv = views["k_row"].codes.shape[1]
    out = tuple(torch.empty((T, H, d), dtype=torch.bfloat16, device="cuda") for H in (Hq, Hkv, Hkv))
    p = mxa.bwd_params(views, o, lse, *out, geo, w.causal, mode)
    ws = torch.empty(mxa.mxa_bwd_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    mxa.bwd(views, o, lse, geo, w.causal, dq_mode=mode, workspace=ws, out=out)
    torch.cuda.synchronize()
    mxa.check_error()
    beta = None
    if mode == mxa.MXA_DQ_FP16_ROW:
        rows = 2 * Hq * geo.ntiles * 128 * 4
        boost = ws[rows:rows + Hq * T * 4].view(torch.float32).reshape(Hq, T).cpu().numpy()
        beta = np.log2(boost.astype(np.float64))
        assert (beta == np.round(beta)).all(), "boosts are powers of two"
        beta = beta.astype(np.int32)
    return out, beta


def _oracle(w, t):
    _, d = oracle_views(w, t)
    cu = w.cu_seqlens.numpy()
    r = orc.attn_bwd_alg1(d["q"]["row"], d["k"]["row"], d["v"]["tok"], d["v"]["row"], d["do"]["row"],
                          d["q"]["tok"], d["k"]["tok"], d["do"]["tok"], cu, w.causal, 1.0 / math.sqrt(w.d))
    beta = orc.dq_row_boost(d["do"]["row"], d["v"]["row"], d["k"]["row"], cu, w.causal)
    return r, beta


@pytest.mark.parametrize("w", CASES, ids=[c.name + ("_causal" if c.causal else "") for c in CASES])
def test_row_boost_matches_oracle(w):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=True)
    (dq, dk, dv), beta = _gpu(w, t, mxa.MXA_DQ_FP16_ROW)
    r, beta_ref = _oracle(w, t)
    assert np.array_equal(beta, beta_ref), np.argwhere(beta != beta_ref)[:8]
    check_outputs(w.name + " dq2", {"dQ": to_np(dq), "dK": to_np(dk), "dV": to_np(dv)}, r)


def test_large_gradients_overflow_the_fixed_boost_only():
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("big_g", lengths=[300, 77, 200], Hq=4, Hkv=2, d=128, causal=True, seed=34)
    t = inp.tensors(w, with_grad=True)
    t["do"] = (t["do"].float() * 1024.0).to(torch.bfloat16)
    r, beta_ref = _oracle(w, t)
    assert np.abs(r["dQ"]).max() * 512 > 65504  # the fixed boost cannot hold these sums
    (dq2, _, _), beta = _gpu(w, t, mxa.MXA_DQ_FP16_ROW)
    assert np.array_equal(beta, beta_ref)
    assert torch.isfinite(dq2).all()
    assert_close("dQ", to_np(dq2), r["dQ"])
    (dq1, _, _), _ = _gpu(w, t, mxa.MXA_DQ_FP16_X512)
    bad = not torch.isfinite(dq1).all()
    if not bad:
        m = metrics(to_np(dq1), r["dQ"])
        bad = m["frac"] > 0.5
    assert bad, "the fixed 2^9 boost was expected to overflow"


def test_row_boost_future_perturbation_leaves_prefix_unchanged():
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.make_custom("prefix", lengths=[700, 300], Hq=4, Hkv=2, d=128, causal=True, seed=35)
    t = inp.tensors(w, with_grad=True)
    base, _ = _gpu(w, t, mxa.MXA_DQ_FP16_ROW)
    again, _ = _gpu(w, t, mxa.MXA_DQ_FP16_ROW)
    assert torch.equal(base[0], again[0]), "the per-row FP16 mode must be deterministic"
    rng = np.random.default_rng(78)
    for p in (130, 411, 650):
        tp = {k: x.clone() for k, x in t.items()}
        for k in ("q", "k", "v", "do"):
            tp[k][p:700] = (tp[k][p:700].float() * float(rng.choice([-64.0, 16.0, 0.25]))).to(torch.bfloat16)
        got, _ = _gpu(w, tp, mxa.MXA_DQ_FP16_ROW)
        keep = (p // 32) * 32  # rows of the blocks strictly before p's block
        assert torch.equal(got[0][:keep], base[0][:keep]), p
        assert torch.equal(got[0][700:], base[0][700:]), "the other document"
