"""Causal safety in the token-block mode (FLAMIA notes sec. 3-4, sec. 10):
perturbing a future token must not change any earlier output.

Reading of "earlier": a token shares its block exponent with the other tokens
of its 32-token block, so the pages concede an in-block residual of up to 31
positions.  The assertion covers every query whose 32-token block lies
strictly before the perturbed token's block in the same document, and every
query of the other documents: O, LSE and dQ (with the incoming gradient G
fixed; FP32 mode, whose dQ sums run in a fixed order) bit for bit.  Two
identical runs are compared first (the pages' advice: measure the repeat
noise, then perturb only the future).
"""
import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp

pytestmark = pytest.mark.gpu


def _run(w, t, geo):
    from block_scaled_mxfp8_gb300 import mxa

    v = {}
    for k in ("q", "k", "v", "do"):
        v[k] = mxa.quantize(t[k], geo, mode=mxa.MXA_SCALE_TOKBLOCK32, hadamard=w.hadamard and k in ("q", "k"))
    o, lse = mxa.fwd(v["q"][0], v["k"][0], v["v"][1], geo, True)
    views = {"q_row": v["q"][0], "k_row": v["k"][0], "v_row": v["v"][0], "g_row": v["do"][0],
             "q_tok": v["q"][1], "k_tok": v["k"][1], "g_tok": v["do"][1]}
    dq, dk, dv = mxa.bwd(views, o, lse, geo, True)
    torch.cuda.synchronize()
    mxa.check_error()
    return o, lse, dq


def test_future_token_perturbation_leaves_prefix_unchanged():
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.workload("tokblock")
    t = {k: x.cuda() for k, x in inp.tensors(w).items()}
    geo = mxa.Geometry.packed(w.lengths)
    base = _run(w, t, geo)
    again = _run(w, t, geo)
    assert torch.equal(base[0], again[0]) and torch.equal(base[1], again[1]), "forward must be deterministic"
    assert torch.equal(base[2], again[2]), "FP32-mode dQ must be deterministic"

    rng = np.random.default_rng(77)
    lens = np.array(w.doc_lengths)
    starts = np.concatenate([[0], np.cumsum(lens)])
    trials = 0
    for _ in range(16):
        b = int(rng.integers(len(lens)))
        n = int(lens[b])
        if n < 70:
            continue
        p = int(rng.integers(64, n))  # doc-relative position, at least two blocks in
        gain = float(rng.choice([4.0, 8.0, 16.0, 64.0])) * float(rng.choice([-1.0, 1.0]))
        tp = {k: x.clone() for k, x in t.items()}
        pos = int(starts[b]) + p
        blk0 = int(starts[b]) + (p // 32) * 32
        for k in ("q", "k", "v"):
            amax = tp[k][blk0:blk0 + 32].float().abs().amax()
            tp[k][pos] = (gain * amax).to(torch.bfloat16)
        out = _run(w, tp, geo)
        keep = torch.ones(w.T, dtype=torch.bool, device="cuda")
        keep[blk0:int(starts[b + 1])] = False  # the perturbed block and everything after it in this document
        assert torch.equal(out[0][keep], base[0][keep]), ("O changed", b, p)
        assert torch.equal(out[1][:, keep], base[1][:, keep]), ("LSE changed", b, p)
        assert torch.equal(out[2][keep], base[2][keep]), ("dQ changed", b, p)
        # the perturbation does reach the suffix
        assert not torch.equal(out[0][~keep], base[0][~keep])
        trials += 1
    assert trials >= 8


def test_subnormal_crossing_perturbation():
    """A suffix value pushed to a tiny magnitude near the E4M3 subnormal range
    (FLAMIA notes sec. 10 test advice) leaves earlier blocks unchanged too."""
    from block_scaled_mxfp8_gb300 import mxa

    w = inp.workload("tokblock")
    t = {k: x.cuda() for k, x in inp.tensors(w).items()}
    geo = mxa.Geometry.packed(w.lengths)
    base = _run(w, t, geo)
    lens = np.array(w.doc_lengths)
    b = int(np.argmax(lens))
    s = int(np.concatenate([[0], np.cumsum(lens)])[b])
    p = 200
    tp = {k: x.clone() for k, x in t.items()}
    for k in ("q", "k", "v"):
        tp[k][s + p] = (tp[k][s + p].float() * 2.0 ** -20).to(torch.bfloat16)
    out = _run(w, tp, geo)
    blk0 = s + (p // 32) * 32
    keep = torch.ones(w.T, dtype=torch.bool, device="cuda")
    keep[blk0:s + int(lens[b])] = False
    assert torch.equal(out[0][keep], base[0][keep])
    assert torch.equal(out[1][:, keep], base[1][:, keep])
    assert torch.equal(out[2][keep], base[2][keep])
