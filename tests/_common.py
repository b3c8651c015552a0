"""Shared helpers of the GPU parity tests: run the CUDA path through the
C-ABI binding and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import math

import numpy as np
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

# Parity bar for floating-point outputs (O, LSE, dQ, dK, dV): cosine >= 0.999
# and max|err| <= 1e-2 * max|ref| against the oracle run on the same quantized
# operands -- the Algorithm 1 oracle (FLAMIA reading notes, sec. 5), which
# applies the roundings the method prescribes: the weights E4M3(2^4 p), O in
# bf16, dV's operand E4M3(2^8 P), dS per 32 x 32 block (and the strict
# operand where used).  What remains between it and the kernels is fp32
# against fp64 arithmetic (an E4M3 rounding decided differently at a near-tie,
# a block exponent at a 448 * 2^k boundary), the FP16 dQ partial sums (11
# significant bits per add) and the bf16 rounding of the gradients.  The
# error against the direct oracle (P and dS in fp64) and against the
# unquantized inputs is reported, not asserted.
COS_MIN = 0.999
MAXERR_FRAC = 1e-2


def metrics(got, ref):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    cos = float(got @ ref / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    maxerr = float(np.max(np.abs(got - ref)))
    maxref = float(np.max(np.abs(ref)))
    sqnr = 10 * math.log10(float(ref @ ref) / max(float((ref - got) @ (ref - got)), 1e-300))
    return {"cos": cos, "maxerr": maxerr, "maxref": maxref, "frac": maxerr / maxref, "sqnr_db": sqnr}


def assert_close(name, got, ref, cos_min=COS_MIN, frac=MAXERR_FRAC):
    m = metrics(got, ref)
    assert m["cos"] >= cos_min and m["frac"] <= frac, "%s: %s" % (name, m)
    return m


def geometry(w: inp.Workload):
    from block_scaled_mxfp8_gb300 import mxa

    if w.lengths is None:
        return mxa.Geometry.batched(w.B, w.L)
    return mxa.Geometry.packed(w.lengths)


def gpu_views(w: inp.Workload, t: dict, names=("q", "k", "v", "do")):
    """Quantize the named bf16 CPU tensors on the GPU.  Returns (geo, dict of
    name -> (row QView, tok QView))."""
    from block_scaled_mxfp8_gb300 import mxa

    geo = geometry(w)
    out = {}
    for nm in names:
        x = t[nm].cuda().contiguous()
        if w.mode == "tokblock":
            had = w.hadamard and nm in ("q", "k")
            out[nm] = mxa.quantize(x, geo, mode=mxa.MXA_SCALE_TOKBLOCK32, hadamard=had)
        else:
            out[nm] = mxa.quantize(x, geo)
    return geo, out


def oracle_views(w: inp.Workload, t: dict, names=("q", "k", "v", "do")):
    """Oracle quantization: name -> dict(row=(codes, scales_logical),
    tok=(codes, scales_logical)) and the dequantized fp64 arrays
    name -> dict(row=..., tok=...)."""
    cu = w.cu_seqlens.numpy()  # batched inputs are B documents of L tokens
    q, deq = {}, {}
    for nm in names:
        x = t[nm]
        if w.mode == "tokblock":
            had = w.hadamard and nm in ("q", "k")
            c, s = orc.quant_tokblock(x, cu, hadamard=had)
            q[nm] = {"blk": (c, s)}
            d = orc.dequant_tokblock(c, s, cu)
            deq[nm] = {"row": d, "tok": d}
        else:
            rc, rs = orc.quant_row(x)
            tc, ts = orc.quant_tok(x, cu)
            q[nm] = {"row": (rc, rs), "tok": (tc, ts)}
            deq[nm] = {"row": orc.dequant_row(rc, rs), "tok": orc.dequant_tok(tc, ts, cu)}
    return q, deq


def to_np(x: torch.Tensor):
    return x.detach().float().cpu().numpy().astype(np.float64)


def lse_spread(ref: dict, moved: list, names=("dQ", "dK", "dV")) -> dict:
    """How far the oracle's own gradients move, as a fraction of max|ref|,
    when the fp32 LSE that the backward rebuilds P from (Algorithm 1 step 08
    saves it in fp32) moves by one ulp either way: the results that an fp32
    LSE admits.  Rows whose scores span thousands of nats have an LSE ulp
    near 1e-4, enough to flip dS codes near their rounding ties."""
    out = {}
    for nm in names:
        mx = float(np.nanmax(np.abs(ref[nm])))
        out[nm] = max(float(np.nanmax(np.abs(m[nm] - ref[nm]))) / mx for m in moved)
    return out


def check_outputs(tag, got: dict, ref: dict, direct: dict | None = None, names=("O", "dQ", "dK", "dV"),
                  spread: dict | None = None):
    """Assert every named output against the Algorithm 1 oracle (ref) at the
    parity bar; print its error against the direct oracle too.  spread (from
    lse_spread) widens the max-abs bar of a gradient by the oracle's own
    movement under one ulp of its fp32 LSE -- zero except where the result
    is not fixed at fp32 resolution.  LSE (when present in got) must also
    agree to 1e-3 * max(1, max|LSE|)."""
    spread = spread or {}
    for nm in names:
        if nm not in got:
            continue
        line = "%s %s vs alg1 %s" % (tag, nm, metrics(got[nm], ref[nm]))
        if nm in spread:
            line += " lse-ulp spread %.4g" % spread[nm]
        if direct is not None and nm in direct:
            line += " | vs direct %s" % metrics(got[nm], direct[nm])
        print(line)
    for nm in names:
        if nm in got:
            assert_close("%s %s" % (tag, nm), got[nm], ref[nm], frac=MAXERR_FRAC + spread.get(nm, 0.0))
    if "LSE" in got:
        L = np.asarray(ref["LSE"], np.float64)
        err = float(np.nanmax(np.abs(np.asarray(got["LSE"], np.float64) - L)))
        assert err <= 1e-3 * max(1.0, float(np.nanmax(np.abs(L)))), (tag, "LSE", err)
