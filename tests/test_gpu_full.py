"""Full-size workloads in the benchmark's launch configuration, checked on
sampled (document, kv-head) units that the oracle computes whole: the GPU
codes/scales of the unit bit-exact, and O, LSE, dQ, dK, dV of the unit within
the parity bar against the Algorithm 1 oracle (the direct oracle's error is
reported).  A gradient's max-abs bar is widened by the oracle's own movement
when its saved fp32 LSE moves one ulp (zero on rows of moderate scores; about
3e-2 on a head whose x50 outlier channels coincide in Q and K, where the
scores span thousands of nats and the LSE ulp is about 1e-4).  Quantization groups never cross heads or documents, so the
oracle quantizes just the unit's slice."""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import check_outputs, lse_spread, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _gpu_run(w, dq_mode=0):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w)
    geo = mxa.Geometry.batched(w.B, w.L) if w.lengths is None else mxa.Geometry.packed(w.lengths)
    tok = w.mode == "tokblock"
    v = {}
    for k in ("q", "k", "v", "do"):
        had = tok and w.hadamard and k in ("q", "k")
        v[k] = mxa.quantize(t[k].cuda(), geo, mode=mxa.MXA_SCALE_TOKBLOCK32 if tok else mxa.MXA_SCALE_MX32,
                            hadamard=had)
    o, lse = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], geo, w.causal)
    views = {"q_row": v["q"][0], "k_row": v["k"][0], "v_row": v["v"][0], "g_row": v["do"][0],
             "q_tok": v["q"][1], "k_tok": v["k"][1], "g_tok": v["do"][1]}
    dq, dk, dv = mxa.bwd(views, o, lse, geo, w.causal, dq_mode=dq_mode)
    torch.cuda.synchronize()
    mxa.check_error()
    return t, geo, v, (o, lse, dq, dk, dv)


def _check_unit(w, t, v, outs, b, hk):
    """Oracle on document b, kv head hk (and its query heads)."""
    from block_scaled_mxfp8_gb300 import mxa

    o, lse, dq, dk, dv = outs
    lens = w.doc_lengths
    s = int(sum(lens[:b]))
    n = lens[b]
    grp = w.Hq // w.Hkv
    hq = slice(hk * grp, (hk + 1) * grp)
    hkv = slice(hk, hk + 1)
    tb = sum((m + 127) // 128 for m in lens[:b])
    nt = (n + 127) // 128
    cu = np.array([0, n], np.int32)
    deq = {}
    for k, hs in (("q", hq), ("k", hkv), ("v", hkv), ("do", hq)):
        x = t[k][s:s + n, hs].contiguous()
        row, tok = v[k]
        if w.mode == "tokblock":
            had = w.hadamard and k in ("q", "k")
            c, sc = orc.quant_tokblock(x, cu, hadamard=had)
            assert np.array_equal(row.codes[s:s + n, hs].cpu().numpy(), c), k
            got = mxa.tok_scales_logical(tok.scales[hs, tb:tb + nt].contiguous(), [n], w.d)
            assert np.array_equal(got, np.broadcast_to(sc[:, None, :], got.shape)), k
            d_ = orc.dequant_tokblock(c, sc, cu)
            deq[k] = (d_, d_)
        else:
            rc, rs = orc.quant_row(x)
            tc, ts = orc.quant_tok(x, cu)
            assert np.array_equal(row.codes[s:s + n, hs].cpu().numpy(), rc), k
            assert np.array_equal(tok.codes[s:s + n, hs].cpu().numpy(), tc), k
            assert np.array_equal(mxa.row_scales_logical(row.scales[hs, tb:tb + nt].contiguous(), [n], w.d), rs), k
            assert np.array_equal(mxa.tok_scales_logical(tok.scales[hs, tb:tb + nt].contiguous(), [n], w.d), ts), k
            deq[k] = (orc.dequant_row(rc, rs), orc.dequant_tok(tc, ts, cu))
    args = (deq["q"][0], deq["k"][0], deq["v"][1], deq["v"][0], deq["do"][0], deq["q"][1], deq["k"][1], deq["do"][1],
            cu, w.causal, 1.0 / math.sqrt(w.d))
    r = orc.attn_bwd_alg1(*args)
    moved = [orc.attn_bwd_alg1(*args, lse_ulps=k) for k in (-1, 1)]
    rd = orc.attn_bwd(*args)
    got = {"O": to_np(o[s:s + n, hq]), "LSE": lse[hq, s:s + n].cpu().numpy().astype(np.float64),
           "dQ": to_np(dq[s:s + n, hq]), "dK": to_np(dk[s:s + n, hkv]), "dV": to_np(dv[s:s + n, hkv])}
    check_outputs("%s doc %d kvhead %d" % (w.name, b, hk), got, r, rd, spread=lse_spread(r, moved))


@pytest.mark.parametrize("causal", [False, True])
def test_llm_shape_b8_h32_l4096(causal):
    """The x50-outlier workload, forward and backward, on eight sampled
    (sequence, head) units spread over the batch and the heads."""
    w = inp.workload("llm", causal=causal)
    t, geo, v, outs = _gpu_run(w)
    for b, hk in ((0, 0), (1, 31), (2, 9), (3, 22), (4, 4), (5, 17), (6, 13), (7, 28)):
        _check_unit(w, t, v, outs, b, hk)


@pytest.mark.parametrize("dq_mode", [0, 1, 2])
def test_train_shape_b4_h16_l8192_causal(dq_mode):
    """FP32, FP16 x 2^9 and FP16 per-row-boost dQ accumulation at the
    training shape."""
    w = inp.workload("train")
    t, geo, v, outs = _gpu_run(w, dq_mode)
    _check_unit(w, t, v, outs, 3, 9)


def test_jagged_256_docs():
    w = inp.workload("jagged")
    t, geo, v, outs = _gpu_run(w)
    lens = np.array(w.doc_lengths)
    picks = [int(np.argmax(lens)), int(np.argmin(lens)), int(np.argsort(lens)[len(lens) // 2])]
    for b in picks:
        _check_unit(w, t, v, outs, b, b % w.Hkv)


def test_tokblock_gqa_packed():
    w = inp.workload("tokblock")
    t, geo, v, outs = _gpu_run(w)
    lens = np.array(w.doc_lengths)
    for b in (0, int(np.argmax(lens)), len(lens) - 1):
        _check_unit(w, t, v, outs, b, (3 * b) % w.Hkv)
