"""GPU per-key view and the strict causal forward (FLAMIA reading notes sec. 4:
each key of the diagonal tile carries its own power-of-two scale, folded into
the probability operand) against the oracle.

* mxa_quantize_key: codes and exponents bit for bit against the oracle's
  quant_key (exponents read through the tile-padded [H, NT, 128] layout).
* The folded forward: O and LSE against the Algorithm 1 oracle with the fold
  (key j's value row is its per-key view on query i's diagonal 128-token
  tile, its token view before it; the folded weights quantized per query and
  32 keys) at the parity bar of the other forward tests.
* The property: keys, values and queries after position p change, inside
  p's own 32-token block, and every row <= p keeps O and LSE bit for bit.
"""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import check_outputs, gpu_views, oracle_views, to_np

pytestmark = pytest.mark.gpu

CASES = [
    inp.workload("tiny", causal=True),
    inp.make_custom("d128_ragged_gqa_causal", lengths=[1, 129, 300, 64, 7, 515], Hq=4, Hkv=2, d=128, causal=True,
                    seed=41),
    inp.make_custom("d64_ragged", lengths=[256, 100, 383], Hq=2, Hkv=1, d=64, causal=True, seed=42),
    # packed documents with more list items (26 tiles x 8 heads) than SMs:
    # persistent CTAs take several items, so the next item's first S MMA
    # follows each diagonal tile's fold
    inp.make_custom("persist_list_gqa", lengths=[900, 5, 1000, 260, 700], Hq=8, Hkv=4, d=128, causal=True,
                    seed=48),
]


def _key_scales_logical(scales: torch.Tensor, lengths):
    """[H, NT, 128] tile-padded exponent bytes -> logical [T, H]."""
    s = scales.cpu().numpy()
    out, tb = [], 0
    for n in lengths:
        r = np.arange(n)
        out.append(s[:, tb + r // 128, r % 128].T)
        tb += (n + 127) // 128
    return np.concatenate(out, 0)


def _lengths(w):
    return list(w.lengths) if w.lengths is not None else [w.L] * w.B


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_quantize_key_bit_exact(w):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w)
    geo, _ = gpu_views(w, t, names=())
    key = mxa.quantize_key(t["v"].cuda().contiguous(), geo)
    torch.cuda.synchronize()
    codes, scales = orc.quant_key(t["v"])
    assert np.array_equal(key.codes.cpu().numpy(), codes)
    assert np.array_equal(_key_scales_logical(key.scales, _lengths(w)), scales)


def _fold_fwd(w, t, fold=True):
    from block_scaled_mxfp8_gb300 import mxa

    geo, gv = gpu_views(w, t)
    key = mxa.quantize_key(t["v"].cuda().contiguous(), geo) if fold else None
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, True, v_key=key)
    torch.cuda.synchronize()
    mxa.check_error()
    return o, lse


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_fold_forward_matches_oracle(w):
    t = inp.tensors(w)
    o, lse = _fold_fwd(w, t)
    _, d = oracle_views(w, t, names=("q", "k", "v"))
    vc, vs = orc.quant_key(t["v"])
    vk = orc.dequant_key(vc, vs)
    cu, alpha = w.cu_seqlens.numpy(), 1.0 / math.sqrt(w.d)
    O, L = orc.attn_fwd_alg1(d["q"]["row"], d["k"]["row"], d["v"]["tok"], cu, True, alpha, Vkey=vk, vkey_sf=vs)
    Od, _ = orc.attn_fwd_fold(d["q"]["row"], d["k"]["row"], d["v"]["tok"], vk, cu, alpha)
    check_outputs(w.name, {"O": to_np(o), "LSE": lse.cpu().numpy()}, {"O": O, "LSE": L}, {"O": Od})


def test_fold_forward_prefix_is_bit_identical_under_in_block_changes():
    w = inp.make_custom("fold_prefix", lengths=[600, 333], Hq=4, Hkv=2, d=128, causal=True, seed=43)
    t = inp.tensors(w)
    base = _fold_fwd(w, t)
    again = _fold_fwd(w, t)
    assert torch.equal(base[0], again[0]) and torch.equal(base[1], again[1]), "the forward must be deterministic"
    plain = _fold_fwd(w, t, fold=False)
    rng = np.random.default_rng(44)
    moved = 0
    for p in (35, 140, 255, 256, 300, 517):  # inside a 32-token block, tile starts and ends
        tp = {k: x.clone() for k, x in t.items()}
        gain = float(rng.choice([-300.0, 64.0, 1e-3]))
        for k in ("q", "k", "v"):
            tp[k][p + 1:600] = (tp[k][p + 1:600].float() * gain).to(torch.bfloat16)
        o, lse = _fold_fwd(w, tp)
        assert torch.equal(o[: p + 1], base[0][: p + 1]), p
        assert torch.equal(lse[:, : p + 1], base[1][:, : p + 1]), p
        assert torch.equal(o[600:], base[0][600:]) and torch.equal(lse[:, 600:], base[1][:, 600:])
        # control: without the fold the token view's groups straddle p, and
        # rows of p's block before p may move (rows of earlier blocks may not)
        o0, _ = _fold_fwd(w, tp, fold=False)
        blk = (p // 32) * 32
        assert torch.equal(o0[:blk], plain[0][:blk]), p
        moved += int(not torch.equal(o0[blk: p + 1], plain[0][blk: p + 1]))
    assert moved > 0, "the perturbations never reached the unfolded prefix: the check would not discriminate"


# ---------------------------------------------------------------- strict dQ

BWD_CASES = [
    inp.make_custom("d128_ragged_gqa_causal", lengths=[1, 129, 300, 64, 7, 515], Hq=4, Hkv=2, d=128, causal=True,
                    seed=45),
    inp.make_custom("d64_ragged", lengths=[256, 100, 383], Hq=2, Hkv=1, d=64, causal=True, seed=46),
    # equal documents: the dK/dV grid in its causal launch order (20 (document,
    # kv head) groups, the last 16 heaviest key tile first across groups)
    inp.make_custom("b5_gqa2_batched", B=5, L=384, Hq=8, Hkv=4, d=128, causal=True, seed=48),
]


def _strict_step(w, t, strict=True, dq_mode=0):
    """Folded forward, then the backward with (strict) or without the K fold
    and per-query dS scales, in dQ mode dq_mode.  -> (dq, dk, dv)."""
    from block_scaled_mxfp8_gb300 import mxa

    geo, gv = gpu_views(w, t)
    vkey = mxa.quantize_key(t["v"].cuda().contiguous(), geo)
    kkey = mxa.quantize_key(t["k"].cuda().contiguous(), geo) if strict else None
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, True, v_key=vkey)
    views = {"q_row": gv["q"][0], "k_row": gv["k"][0], "v_row": gv["v"][0], "g_row": gv["do"][0],
             "q_tok": gv["q"][1], "k_tok": gv["k"][1], "g_tok": gv["do"][1]}
    out = mxa.bwd(views, o, lse, geo, True, dq_mode=dq_mode, k_key=kkey)
    torch.cuda.synchronize()
    mxa.check_error()
    return out


@pytest.mark.parametrize("dq_mode", [0, 1, 2])
@pytest.mark.parametrize("w", BWD_CASES, ids=[c.name for c in BWD_CASES])
def test_strict_backward_matches_oracle(w, dq_mode):
    """Strict dQ in each accumulation mode: FP32, FP16 x 2^9, FP16 with the
    per-row boost."""
    t = inp.tensors(w, with_grad=True)
    dq, dk, dv = _strict_step(w, t, dq_mode=dq_mode)
    _, d = oracle_views(w, t)
    vc, vs = orc.quant_key(t["v"])
    kc, ks = orc.quant_key(t["k"])
    vk, kk = orc.dequant_key(vc, vs), orc.dequant_key(kc, ks)
    vw = (d["q"]["row"], d["k"]["row"], d["v"]["tok"], d["v"]["row"], d["do"]["row"], d["q"]["tok"], d["k"]["tok"],
          d["do"]["tok"])
    cu, alpha = w.cu_seqlens.numpy(), 1.0 / math.sqrt(w.d)
    r = orc.attn_bwd_alg1(*vw, cu, True, alpha, Vkey=vk, vkey_sf=vs, Kkey=kk, kkey_sf=ks)
    rd = orc.attn_bwd_fold(*vw, vk, kk, cu, alpha)
    check_outputs("%s strict dq%d" % (w.name, dq_mode), {"dQ": to_np(dq), "dK": to_np(dk), "dV": to_np(dv)}, r,
                  rd)


@pytest.mark.parametrize("dq_mode", [0, 1, 2])
def test_strict_dq_prefix_is_bit_identical_under_in_block_changes(dq_mode):
    w = inp.make_custom("strict_prefix", lengths=[600, 333], Hq=4, Hkv=2, d=128, causal=True, seed=47)
    t = inp.tensors(w, with_grad=True)
    base = _strict_step(w, t, dq_mode=dq_mode)
    again = _strict_step(w, t, dq_mode=dq_mode)
    assert torch.equal(base[0], again[0]), "the strict backward must be deterministic"
    plain = _strict_step(w, t, strict=False, dq_mode=dq_mode)
    rng = np.random.default_rng(48)
    moved = 0
    for p in (35, 140, 255, 300, 517):
        tp = {k: x.clone() for k, x in t.items()}
        gain = float(rng.choice([-300.0, 64.0, 1e-3]))
        for k in ("q", "k", "v", "do"):  # the incoming gradient of rows <= p stays fixed
            tp[k][p + 1:600] = (tp[k][p + 1:600].float() * gain).to(torch.bfloat16)
        dq, _, _ = _strict_step(w, tp, dq_mode=dq_mode)
        assert torch.equal(dq[: p + 1], base[0][: p + 1]), p
        assert torch.equal(dq[600:], base[0][600:])
        # control: with the folded forward but block-scaled dS and the token
        # view of K, rows of p's block before p may move, earlier blocks not
        dq0, _, _ = _strict_step(w, tp, strict=False, dq_mode=dq_mode)
        blk = (p // 32) * 32
        assert torch.equal(dq0[:blk], plain[0][:blk]), p
        moved += int(not torch.equal(dq0[blk: p + 1], plain[0][blk: p + 1]))
    assert moved > 0, "the perturbations never reached the unfolded prefix: the check would not discriminate"
