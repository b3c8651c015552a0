"""CPU oracle for MXFP8 block-scaled attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and this module imports
nothing from the product package.

The arithmetic lives in ``mxa_oracle.c`` (fp64, direct, untiled); this file
compiles it with gcc on first use and wraps it with ctypes + numpy.  Which
passage each function follows is stated in the C file and below.

Sources (page titles, sections):
  * "Flash Attention 4 + MXFP8 on Blackwell" write-up (aixai.ru):
    "Что такое MXFP8" (32-value groups, E8M0 scale).
  * "FLAMIA 阅读笔记": sec. 2 (attention and its backward, online softmax),
    sec. 3 (token blocks, Hadamard), sec. 4 (scale rule, two-value
    counterexample, scale doubling, the strict accumulator scale of the FP16
    dQ reduction), sec. 5 (P cap 2^(c+tau) <= 448, cosine example), sec. 6
    (visible-pair count).

Two attention oracles:
  * ``attn_fwd`` / ``attn_bwd`` (and the ``_x``, ``_fold`` variants): direct
    softmax attention in fp64 over the dequantized operands, P and dS kept in
    fp64 -- the "unquantized P" reference whose error is reported;
  * ``attn_fwd_alg1`` / ``attn_bwd_alg1``: the same direct computation with
    the roundings that the steps of Algorithm 1 (FLAMIA sec. 5) name -- the
    weights E4M3(2^4 p) against an integer reference maximum, O saved in
    bf16, dV's operand E4M3(2^8 P), U quantized per 32 x 32 block, the strict
    dQ operand -- each switchable (``RND_*``); the parity bar is asserted
    against this one.

Parity pins live in ``tests/test_oracle_*.py``.  Unpinned: none.  One
reading is recorded rather than derived from the pages: ``dq_row_boost``
restates the bound that the library documents for its per-row FP16 dQ
boost (the pages give only the shape b_i = 2^floor(log2(h / a_i))); its pins
check that the bound holds on exact backward values, so a GPU-vs-oracle
equality of the boost exponents compares the kernel with that stated
reading, not with a quantity the pages fix.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, OpenMP).  Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            sig = {
                "orc_e4m3_decode": (f64, [ctypes.c_uint8]),
                "orc_e4m3_encode": (ctypes.c_uint8, [f64]),
                "orc_e4m3_encode_array": (None, [P, i64, P]),
                "orc_ue8m0_decode": (f64, [ctypes.c_uint8]),
                "orc_mx_exponent": (i32, [f64]),
                "orc_block_offset": (i64, [P, i32, i64, i32]),
                "orc_total_blocks": (i64, [P, i32, i64]),
                "orc_visible_pairs": (i64, [P, i32, i64]),
                "orc_quant_row": (None, [P, i64, i32, i32, P, P]),
                "orc_quant_tok": (None, [P, i64, i32, i32, P, i32, P, P]),
                "orc_quant_tokblock": (None, [P, i64, i32, i32, P, i32, i32, P, P]),
                "orc_hadamard128_f32": (None, [P, P]),
                "orc_dequant_row": (None, [P, P, i64, i32, i32, P]),
                "orc_dequant_tok": (None, [P, P, i64, i32, i32, P, i32, P]),
                "orc_dequant_tokblock": (None, [P, P, i64, i32, i32, P, i32, P]),
                "orc_attn_fwd": (None, [P, P, P, i64, i32, i32, i32, P, i32, i32, f64, P, i64, P, P]),
                "orc_attn_bwd": (None, [P] * 8 + [i64, i32, i32, i32, P, i32, i32, f64, P, i32] + [P] * 6),
                "orc_rmsnorm_f32": (None, [P, i64, i32, i32, P, ctypes.c_float, P]),
                "orc_quant_row_f32": (None, [P, i64, i32, i32, P, P]),
                "orc_quant_tok_f32": (None, [P, i64, i32, i32, P, i32, P, P]),
                "orc_quant_tokblock_f32": (None, [P, i64, i32, i32, P, i32, i32, P, P]),
                "orc_attn_fwd_x": (None, [P, P, P, i64, i64, i32, i32, i32, P, P, i32, f64, P, P]),
                "orc_attn_bwd_x": (None, [P] * 8 + [i64, i64, i32, i32, i32, P, P, i32, f64] + [P] * 6),
                "orc_quant_key": (None, [P, i64, i32, i32, P, P]),
                "orc_attn_bwd_fold": (None, [P] * 10 + [i64, i32, i32, i32, P, i32, f64] + [P] * 6),
                "orc_attn_fwd_fold": (None, [P, P, P, P, i64, i32, i32, i32, P, i32, f64, P, P]),
                "orc_dq_row_boost": (None, [P, P, P, i64, i32, i32, i32, P, i32, i32, ctypes.c_float, P]),
                "orc_num_threads": (i32, []),
                "orc_e4m3_round": (f64, [f64]),
                "orc_e4m3_round_array": (None, [P, i64, P]),
                "orc_round_bf16": (f64, [f64]),
                "orc_round_bf16_array": (None, [P, i64, P]),
                "orc_attn_fwd_alg1": (None, [P] * 5 + [i64, i64, i32, i32, i32, P, P, i32, i32, f64, i32, i64, P,
                                                       i64, P, P]),
                "orc_attn_bwd_alg1": (None, [P] * 12 + [i64, i64, i32, i32, i32, P, P, i32, i32, f64, i32, i64, i32,
                                                        P, i32] + [P] * 6),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x):
    """bf16 tensor/array -> contiguous uint16 numpy array of its bit patterns."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16
    return x


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, 0
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, len(cu) - 1


# --------------------------------------------------------------------------
# formats ("Что такое MXFP8"; FLAMIA sec. 2 "两种硬件格式", sec. 4)
# --------------------------------------------------------------------------

def e4m3_decode(c: int) -> float:
    return _L().orc_e4m3_decode(int(c) & 0xFF)


def e4m3_encode(y: float) -> int:
    return int(_L().orc_e4m3_encode(float(y)))


def e4m3_encode_array(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64))
    out = np.empty(y.shape, np.uint8)
    _L().orc_e4m3_encode_array(_p(y), y.size, _p(out))
    return out


def ue8m0_decode(b: int) -> float:
    return _L().orc_ue8m0_decode(int(b) & 0xFF)


def mx_exponent(amax: float) -> int:
    """Smallest integer e with amax / 2^e <= 448 (FLAMIA sec. 4); 0 for an all-zero group."""
    return int(_L().orc_mx_exponent(float(amax)))


E4M3_TABLE = None


def e4m3_table() -> np.ndarray:
    """Decoded value of each of the 256 E4M3 codes (NaN for 0x7F / 0xFF)."""
    global E4M3_TABLE
    if E4M3_TABLE is None:
        E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return E4M3_TABLE


def block_offset(cu_seqlens, T: int, b: int) -> int:
    cu, nd = _cu(cu_seqlens)
    return int(_L().orc_block_offset(_p(cu), nd, T, b))


def total_blocks(cu_seqlens, T: int) -> int:
    cu, nd = _cu(cu_seqlens)
    return int(_L().orc_total_blocks(_p(cu), nd, T))


def visible_pairs(cu_seqlens, T: int) -> int:
    """Causal visible (query, key) pairs, sum n(n+1)/2 (FLAMIA sec. 6)."""
    cu, nd = _cu(cu_seqlens)
    return int(_L().orc_visible_pairs(_p(cu), nd, T))


# --------------------------------------------------------------------------
# quantizers
# --------------------------------------------------------------------------

def quant_row(x):
    """Row view: per (token, head, 32 channels).  x bf16 [T,H,d] ->
    (codes uint8 [T,H,d], scales uint8 [T,H,d/32])."""
    xu = _u16(x)
    T, H, d = xu.shape
    codes = np.empty((T, H, d), np.uint8)
    scales = np.empty((T, H, d // 32), np.uint8)
    _L().orc_quant_row(_p(xu), T, H, d, _p(codes), _p(scales))
    return codes, scales


def quant_key(x):
    """Per-key view: one scale per (token, head) over all d channels.
    x bf16 [T,H,d] -> (codes uint8 [T,H,d], scales uint8 [T,H])."""
    xu = _u16(x)
    T, H, d = xu.shape
    codes = np.empty((T, H, d), np.uint8)
    scales = np.empty((T, H), np.uint8)
    _L().orc_quant_key(_p(xu), T, H, d, _p(codes), _p(scales))
    return codes, scales


def dequant_key(codes, scales):
    """Decoded per-key view: E4M3 code values times 2^(byte - 127)."""
    tab = e4m3_table()
    e = scales.astype(np.int64) - 127
    return tab[codes] * np.exp2(e.astype(np.float64))[:, :, None]


def quant_tok(x, cu_seqlens=None):
    """Token view: per (doc, 32 doc-relative tokens, head, channel).
    -> (codes [T,H,d], scales logical [H, d, NB])."""
    xu = _u16(x)
    T, H, d = xu.shape
    cu, nd = _cu(cu_seqlens)
    NB = total_blocks(cu_seqlens, T)
    codes = np.zeros((T, H, d), np.uint8)
    scales = np.zeros((H, d, NB), np.uint8)
    _L().orc_quant_tok(_p(xu), T, H, d, _p(cu), nd, _p(codes), _p(scales))
    return codes, scales


def rmsnorm_f32(x, weight=None, eps=1e-6):
    """RMSNorm of every (token, head) vector in IEEE fp32 in the written order
    of orc_rmsnorm_f32.  x bf16 [T,H,d]; weight fp32 [d] or None.
    -> float32 [T,H,d]."""
    xu = _u16(x)
    T, H, d = xu.shape
    y = np.empty((T, H, d), np.float32)
    w = None if weight is None else np.ascontiguousarray(np.asarray(weight, dtype=np.float32))
    _L().orc_rmsnorm_f32(_p(xu), T, H, d, _p(w), float(eps), _p(y))
    return y


def quant_row_f32(y):
    """quant_row of fp32 values y [T,H,d]."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, H, d = y.shape
    codes = np.empty((T, H, d), np.uint8)
    scales = np.empty((T, H, d // 32), np.uint8)
    _L().orc_quant_row_f32(_p(y), T, H, d, _p(codes), _p(scales))
    return codes, scales


def quant_tok_f32(y, cu_seqlens=None):
    """quant_tok of fp32 values y [T,H,d]."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, H, d = y.shape
    cu, nd = _cu(cu_seqlens)
    NB = total_blocks(cu_seqlens, T)
    codes = np.zeros((T, H, d), np.uint8)
    scales = np.zeros((H, d, NB), np.uint8)
    _L().orc_quant_tok_f32(_p(y), T, H, d, _p(cu), nd, _p(codes), _p(scales))
    return codes, scales


def quant_tokblock_f32(y, cu_seqlens=None, hadamard=False):
    """quant_tokblock of fp32 values y [T,H,d]."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, H, d = y.shape
    if hadamard and d != 128:
        raise ValueError("hadamard rotation needs d == 128")
    cu, nd = _cu(cu_seqlens)
    NB = total_blocks(cu_seqlens, T)
    codes = np.zeros((T, H, d), np.uint8)
    scales = np.zeros((H, NB), np.uint8)
    _L().orc_quant_tokblock_f32(_p(y), T, H, d, _p(cu), nd, int(bool(hadamard)), _p(codes), _p(scales))
    return codes, scales


def quant_tokblock(x, cu_seqlens=None, hadamard=False):
    """Token-block view (FLAMIA sec. 3): one exponent per (doc, 32-token
    block, head).  -> (codes [T,H,d], scales logical [H, NB])."""
    xu = _u16(x)
    T, H, d = xu.shape
    if hadamard and d != 128:
        raise ValueError("hadamard rotation needs d == 128")
    cu, nd = _cu(cu_seqlens)
    NB = total_blocks(cu_seqlens, T)
    codes = np.zeros((T, H, d), np.uint8)
    scales = np.zeros((H, NB), np.uint8)
    _L().orc_quant_tokblock(_p(xu), T, H, d, _p(cu), nd, int(bool(hadamard)), _p(codes), _p(scales))
    return codes, scales


def hadamard128_f32(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (128,)
    out = np.empty(128, np.float32)
    _L().orc_hadamard128_f32(_p(v), _p(out))
    return out


def dequant_row(codes, scales):
    T, H, d = codes.shape
    out = np.empty((T, H, d), np.float64)
    _L().orc_dequant_row(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scales)), T, H, d, _p(out))
    return out


def dequant_tok(codes, scales, cu_seqlens=None):
    T, H, d = codes.shape
    cu, nd = _cu(cu_seqlens)
    out = np.zeros((T, H, d), np.float64)
    _L().orc_dequant_tok(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scales)), T, H, d, _p(cu), nd, _p(out))
    return out


def dequant_tokblock(codes, scales, cu_seqlens=None):
    T, H, d = codes.shape
    cu, nd = _cu(cu_seqlens)
    out = np.zeros((T, H, d), np.float64)
    _L().orc_dequant_tokblock(_p(np.ascontiguousarray(codes)), _p(np.ascontiguousarray(scales)), T, H, d, _p(cu), nd, _p(out))
    return out


# --------------------------------------------------------------------------
# attention (FLAMIA sec. 2)
# --------------------------------------------------------------------------

def attn_fwd(Q, K, V, cu_seqlens=None, causal=False, alpha=None, sel=None):
    """Direct softmax attention in fp64.  Q [T,Hq,d], K/V [T,Hkv,d] float64.
    sel: optional int array of (token, head) pairs; other rows stay NaN.
    Returns (O [T,Hq,d], LSE [Hq,T])."""
    Q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (Q, K, V))
    T, Hq, d = Q.shape
    Hkv = K.shape[1]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    O = np.full((T, Hq, d), np.nan)
    LSE = np.full((Hq, T), np.nan)
    if sel is not None:
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
    _L().orc_attn_fwd(_p(Q), _p(K), _p(V), T, Hq, Hkv, d, _p(cu), nd, int(bool(causal)), float(alpha),
                      _p(sel), -1 if sel is None else len(sel), _p(O), _p(LSE))
    return O, LSE


def attn_fwd_fold(Q, K, Vtok, Vkey, cu_seqlens=None, alpha=None):
    """Causal forward with the per-key fold on the diagonal tile (FLAMIA sec.
    4): key j's value row is Vkey_j when j is in query i's 128-token tile of
    the document, else Vtok_j.  Returns (O [T,Hq,d], LSE [Hq,T])."""
    Q, K, Vtok, Vkey = (np.ascontiguousarray(a, dtype=np.float64) for a in (Q, K, Vtok, Vkey))
    T, Hq, d = Q.shape
    Hkv = K.shape[1]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    O = np.full((T, Hq, d), np.nan)
    LSE = np.full((Hq, T), np.nan)
    _L().orc_attn_fwd_fold(_p(Q), _p(K), _p(Vtok), _p(Vkey), T, Hq, Hkv, d, _p(cu), nd, float(alpha), _p(O), _p(LSE))
    return O, LSE


def attn_bwd(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu_seqlens=None, causal=False, alpha=None, units=None):
    """Direct backward in fp64 (FLAMIA sec. 2).  See orc_attn_bwd for the role
    of each view.  units: optional (doc, kv-head) pairs.  Returns a dict with
    dQ, dK, dV, O, LSE, D (rows outside the units stay NaN)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt)]
    T, Hq, d = arrs[0].shape
    Hkv = arrs[1].shape[1]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    out = {
        "dQ": np.full((T, Hq, d), np.nan),
        "dK": np.full((T, Hkv, d), np.nan),
        "dV": np.full((T, Hkv, d), np.nan),
        "O": np.full((T, Hq, d), np.nan),
        "LSE": np.full((Hq, T), np.nan),
        "D": np.full((Hq, T), np.nan),
    }
    if units is not None:
        units = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    _L().orc_attn_bwd(*[_p(a) for a in arrs], T, Hq, Hkv, d, _p(cu), nd, int(bool(causal)), float(alpha),
                      _p(units), -1 if units is None else len(units),
                      *[_p(out[k]) for k in ("dQ", "dK", "dV", "O", "LSE", "D")])
    return out


def dq_row_boost(Gr, Vr, Kr, cu_seqlens=None, causal=False, alpha=None):
    """Per-row exponent beta of the strict FP16 dQ reduction (FLAMIA sec. 4,
    the accumulator scale): see orc_dq_row_boost.  Gr [T,Hq,d], Vr/Kr
    [T,Hkv,d] decoded ROW views; alpha is rounded to fp32 as the library's
    softmax scale is.  Returns int32 [Hq, T]."""
    Gr, Vr, Kr = (np.ascontiguousarray(a, dtype=np.float64) for a in (Gr, Vr, Kr))
    T, Hq, d = Gr.shape
    Hkv = Vr.shape[1]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    beta = np.zeros((Hq, T), dtype=np.int32)
    _L().orc_dq_row_boost(_p(Gr), _p(Vr), _p(Kr), T, Hq, Hkv, d, _p(cu), nd, int(bool(causal)), float(alpha),
                          _p(beta))
    return beta


def attn_bwd_fold(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, Vkey, Kkey, cu_seqlens=None, alpha=None):
    """Causal backward with the per-key folds on the diagonal tile (FLAMIA
    sec. 4): see orc_attn_bwd_fold.  Returns a dict with dQ, dK, dV, O, LSE,
    D."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, Vkey, Kkey)]
    T, Hq, d = arrs[0].shape
    Hkv = arrs[1].shape[1]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    out = {k: np.full(sh, np.nan) for k, sh in (("dQ", (T, Hq, d)), ("dK", (T, Hkv, d)), ("dV", (T, Hkv, d)),
                                                  ("O", (T, Hq, d)), ("LSE", (Hq, T)), ("D", (Hq, T)))}
    _L().orc_attn_bwd_fold(*[_p(a) for a in arrs], T, Hq, Hkv, d, _p(cu), nd, float(alpha),
                           *[_p(out[k]) for k in ("dQ", "dK", "dV", "O", "LSE", "D")])
    return out


def attn_fwd_x(Q, K, V, cu_q, cu_k, alpha=None):
    """Cross-attention forward in fp64 (no mask): the queries of document b
    (rows cu_q[b]..cu_q[b+1]) attend to its keys and values (rows
    cu_k[b]..cu_k[b+1]).  Q [Tq,Hq,d], K/V [Tk,Hkv,d].  Returns
    (O [Tq,Hq,d], LSE [Hq,Tq])."""
    Q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (Q, K, V))
    Tq, Hq, d = Q.shape
    Tk, Hkv = K.shape[:2]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cq, nd = _cu(cu_q)
    ck, ndk = _cu(cu_k)
    assert nd == ndk and cq[-1] == Tq and ck[-1] == Tk
    O = np.full((Tq, Hq, d), np.nan)
    LSE = np.full((Hq, Tq), np.nan)
    _L().orc_attn_fwd_x(_p(Q), _p(K), _p(V), Tq, Tk, Hq, Hkv, d, _p(cq), _p(ck), nd, float(alpha), _p(O), _p(LSE))
    return O, LSE


def attn_bwd_x(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu_q, cu_k, alpha=None):
    """Cross-attention backward in fp64 (no mask); views as in attn_bwd, with
    Ks, Vo, Vr, Kt over the key side's Tk rows.  Returns a dict with dQ, dK,
    dV, O, LSE, D."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt)]
    Tq, Hq, d = arrs[0].shape
    Tk, Hkv = arrs[1].shape[:2]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cq, nd = _cu(cu_q)
    ck, ndk = _cu(cu_k)
    assert nd == ndk and cq[-1] == Tq and ck[-1] == Tk
    out = {
        "dQ": np.full((Tq, Hq, d), np.nan),
        "dK": np.full((Tk, Hkv, d), np.nan),
        "dV": np.full((Tk, Hkv, d), np.nan),
        "O": np.full((Tq, Hq, d), np.nan),
        "LSE": np.full((Hq, Tq), np.nan),
        "D": np.full((Hq, Tq), np.nan),
    }
    _L().orc_attn_bwd_x(*[_p(a) for a in arrs], Tq, Tk, Hq, Hkv, d, _p(cq), _p(ck), nd, float(alpha),
                        *[_p(out[k]) for k in ("dQ", "dK", "dV", "O", "LSE", "D")])
    return out


# --------------------------------------------------------------------------
# Algorithm 1 (FLAMIA sec. 5): the forward and backward with the roundings
# its steps name
# --------------------------------------------------------------------------

RND_P = 1    # step 07: forward weights E4M3(2^4 p), p against the integer reference ceil(max)
RND_O = 2    # step 08: O saved in bf16
RND_P8 = 4   # step 15: dV's operand E4M3(2^8 P) 2^-8
RND_DS = 8   # step 14: U quantized per 32 x 32 block
RND_LSE = 16  # step 08: LSE saved in fp32, P rebuilt from it
RND_ALG1 = RND_P | RND_O | RND_P8 | RND_DS | RND_LSE
# key tile of the online reference schedule of step 07 (256 keys: the tile
# the attention kernels walk); 0 = one tile holding every visible key
REF_TILE = 256


def e4m3_round_array(y) -> np.ndarray:
    """Nearest E4M3 value of each element (ties to the even code, saturating
    to 448, sign kept), as float64."""
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64))
    out = np.empty(y.shape, np.float64)
    _L().orc_e4m3_round_array(_p(y), y.size, _p(out))
    return out


def round_bf16_array(x) -> np.ndarray:
    """Nearest bf16 value of each element (ties to even), as float64."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.float64)
    _L().orc_round_bf16_array(_p(x), x.size, _p(out))
    return out


def _opt(a, dtype):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=dtype))


def attn_fwd_alg1(Q, K, V, cu_seqlens=None, causal=False, alpha=None, rnd=RND_ALG1, cu_k=None, Vkey=None,
                  vkey_sf=None, sel=None, ref_tile=REF_TILE):
    """Algorithm 1's forward (steps 04-08) in fp64, direct: see
    orc_attn_fwd_alg1.  Q [Tq,Hq,d], K/V [Tk,Hkv,d] decoded views; cu_k:
    key-side offsets for cross-attention (None: self-attention); Vkey
    [Tk,Hkv,d] decoded per-key view of V with its UE8M0 bytes vkey_sf
    [Tk,Hkv] for the strict fold; rnd: the roundings (RND_* bits); ref_tile:
    the key tile of the lazy reference schedule.  Returns (O [Tq,Hq,d],
    LSE [Hq,Tq]); rows outside sel stay NaN."""
    Q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (Q, K, V))
    Tq, Hq, d = Q.shape
    Tk, Hkv = K.shape[:2]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    ck, ndk = _cu(cu_k)
    if ck is not None:
        assert cu is not None and ndk == nd and not causal
    Vkey, vkey_sf = _opt(Vkey, np.float64), _opt(vkey_sf, np.uint8)
    assert (Vkey is None) == (vkey_sf is None)
    O = np.full((Tq, Hq, d), np.nan)
    LSE = np.full((Hq, Tq), np.nan)
    if sel is not None:
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
    _L().orc_attn_fwd_alg1(_p(Q), _p(K), _p(V), _p(Vkey), _p(vkey_sf), Tq, Tk, Hq, Hkv, d, _p(cu), _p(ck), nd,
                           int(bool(causal)), float(alpha), int(rnd), int(ref_tile), _p(sel),
                           -1 if sel is None else len(sel), _p(O), _p(LSE))
    return O, LSE


def attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu_seqlens=None, causal=False, alpha=None, rnd=RND_ALG1,
                  cu_k=None, Vkey=None, vkey_sf=None, Kkey=None, kkey_sf=None, units=None, ref_tile=REF_TILE,
                  lse_ulps=0):
    """Algorithm 1's backward (steps 09-15) in fp64, direct: see
    orc_attn_bwd_alg1 for the role of each view.  Kkey/kkey_sf: the strict
    dQ operand (per-query dS scales, K fold).  lse_ulps: the saved fp32 LSE
    moved by that many ulps (RND_LSE).  units: optional (doc, kv-head)
    pairs.  Returns a dict with dQ, dK, dV, O, LSE, D (rows outside the units
    stay NaN)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt)]
    Tq, Hq, d = arrs[0].shape
    Tk, Hkv = arrs[1].shape[:2]
    if alpha is None:
        alpha = 1.0 / math.sqrt(d)
    cu, nd = _cu(cu_seqlens)
    ck, ndk = _cu(cu_k)
    if ck is not None:
        assert cu is not None and ndk == nd and not causal
    Vkey, vkey_sf = _opt(Vkey, np.float64), _opt(vkey_sf, np.uint8)
    Kkey, kkey_sf = _opt(Kkey, np.float64), _opt(kkey_sf, np.uint8)
    assert (Vkey is None) == (vkey_sf is None) and (Kkey is None) == (kkey_sf is None)
    out = {k: np.full(sh, np.nan) for k, sh in (("dQ", (Tq, Hq, d)), ("dK", (Tk, Hkv, d)), ("dV", (Tk, Hkv, d)),
                                                  ("O", (Tq, Hq, d)), ("LSE", (Hq, Tq)), ("D", (Hq, Tq)))}
    if units is not None:
        units = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    _L().orc_attn_bwd_alg1(*[_p(a) for a in arrs], _p(Vkey), _p(vkey_sf), _p(Kkey), _p(kkey_sf), Tq, Tk, Hq, Hkv,
                           d, _p(cu), _p(ck), nd, int(bool(causal)), float(alpha), int(rnd), int(ref_tile),
                           int(lse_ulps), _p(units),
                           -1 if units is None else len(units),
                           *[_p(out[k]) for k in ("dQ", "dK", "dV", "O", "LSE", "D")])
    return out


def num_threads() -> int:
    return int(_L().orc_num_threads())


# --------------------------------------------------------------------------
# small helpers that restate worked examples of the pages
# --------------------------------------------------------------------------

def shared_scale_prefix_output(a: float) -> float:
    """FLAMIA sec. 4 "两个数就够构造反例": an integer rounder with codes
    -2..2; values 1 and a share the scale s = max(1, |a|) / 2; query 1 sees
    only key 1, so its output is the reconstructed first value s*round(1/s)."""
    s = max(1.0, abs(a)) / 2.0
    q = max(-2.0, min(2.0, float(np.round(1.0 / s))))
    return s * q


def p_cap_reconstruction(c: int, tau: int, lag: float) -> float:
    """FLAMIA sec. 5 "概率上限由两个参数共同决定": a weight 2^lag (lag <= tau
    log2 units behind the true max) boosted by 2^c, encoded in E4M3 (which
    saturates at 448), then divided by 2^c."""
    return e4m3_decode(e4m3_encode(2.0 ** (c + lag))) / 2.0 ** c


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
