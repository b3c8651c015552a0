"""Thin ctypes binding of libmxa.so (include/mxa.h).

Argument marshalling only: every step of the attention path runs in the CUDA
library.  PyTorch supplies device memory (the output and workspace tensors
allocated here) and the current CUDA stream.  If the library is missing the
import of any entry point raises; there is no fallback.

The functions named like the C entry points (``mxa_quantize``, ``mxa_fwd``,
``mxa_bwd``, ...) take the same arguments (device tensors in place of raw
pointers).  ``quantize``, ``fwd`` and ``bwd`` are conveniences that allocate
the outputs with torch and call them.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmxa.so")

MXA_OK, MXA_ERR_ARG, MXA_ERR_ALIGN, MXA_ERR_UNSUPPORTED, MXA_ERR_WORKSPACE, MXA_ERR_CUDA, MXA_ERR_TIMEOUT = range(7)
MXA_SCALE_MX32, MXA_SCALE_TOKBLOCK32 = 0, 1
MXA_VIEW_ROW, MXA_VIEW_TOK = 1, 2
MXA_DQ_FP32, MXA_DQ_FP16_X512, MXA_DQ_FP16_ROW = 0, 1, 2
ATOM_BYTES = 512


class MxaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, status_str(status), status))
        self.status = status


class c_qview(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class c_shape(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64),
        ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int),
        ("cu_seqlens", ctypes.c_void_p),
        ("num_docs", ctypes.c_int),
        ("max_seqlen", ctypes.c_int),
        ("ntiles", ctypes.c_int64),
        ("causal", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("T_k", ctypes.c_int64),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("max_seqlen_k", ctypes.c_int),
        ("ntiles_k", ctypes.c_int64),
    ]


class c_fwd_params(ctypes.Structure):
    _fields_ = [
        ("shape", c_shape),
        ("q_row", c_qview),
        ("k_row", c_qview),
        ("v_tok", c_qview),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("v_key", c_qview),
    ]


class c_bwd_params(ctypes.Structure):
    _fields_ = [
        ("shape", c_shape),
        ("q_row", c_qview),
        ("k_row", c_qview),
        ("v_row", c_qview),
        ("g_row", c_qview),
        ("q_tok", c_qview),
        ("k_tok", c_qview),
        ("g_tok", c_qview),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p),
        ("dq_mode", ctypes.c_int),
        ("k_key", c_qview),
    ]


_lib = None

EXPORTS = [
    "mxa_abi_version", "mxa_status_str", "mxa_scale_tiles", "mxa_scale_tiles_bound", "mxa_scale_bytes",
    "mxa_quantize", "mxa_rmsnorm_quantize", "mxa_quantize_key", "mxa_key_scale_bytes", "mxa_fwd", "mxa_fwd_workspace_bytes", "mxa_bwd_workspace_bytes", "mxa_bwd_workspace_min_bytes", "mxa_bwd",
    "mxa_bwd_noalloc", "mxa_get_error",
]
# include/mxa_testing.h: the kernels' P and dS quantization run on caller data
EXPORTS_TESTING = ["mxa_test_e4m3", "mxa_test_ds_blocks", "mxa_test_wait_timeout", "mxa_test_mma_rate",
                   "mxa_test_ex2_rate", "mxa_test_tmem_max"]
MXA_BWD_NOALLOC_MAX_WORKSPACE = 32 * 1024 * 1024


def lib():
    """Load libmxa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmxa.so not built (%s); run block_scaled_mxfp8_gb300.build.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.mxa_abi_version.restype = i32
        L.mxa_abi_version.argtypes = []
        L.mxa_status_str.restype = ctypes.c_char_p
        L.mxa_status_str.argtypes = [i32]
        L.mxa_scale_tiles.restype = i64
        L.mxa_scale_tiles.argtypes = [i64, i32, P]
        L.mxa_scale_tiles_bound.restype = i64
        L.mxa_scale_tiles_bound.argtypes = [i64, i32]
        L.mxa_scale_bytes.restype = ctypes.c_size_t
        L.mxa_scale_bytes.argtypes = [i32, i64]
        L.mxa_quantize.restype = i32
        L.mxa_quantize.argtypes = [P, i64, i32, i32, P, i32, i32, i64, i32, i32, i32,
                                   ctypes.POINTER(c_qview), ctypes.POINTER(c_qview), P]
        L.mxa_rmsnorm_quantize.restype = i32
        L.mxa_rmsnorm_quantize.argtypes = [P, P, ctypes.c_float, i64, i32, i32, P, i32, i32, i64, i32, i32, i32,
                                           ctypes.POINTER(c_qview), ctypes.POINTER(c_qview), P]
        L.mxa_quantize_key.restype = i32
        L.mxa_quantize_key.argtypes = [P, i64, i32, i32, P, i32, i32, i64, ctypes.POINTER(c_qview), P]
        L.mxa_key_scale_bytes.restype = ctypes.c_size_t
        L.mxa_key_scale_bytes.argtypes = [i32, i64]
        L.mxa_fwd.restype = i32
        L.mxa_fwd.argtypes = [ctypes.POINTER(c_fwd_params), P]
        L.mxa_fwd_workspace_bytes.restype = ctypes.c_size_t
        L.mxa_fwd_workspace_bytes.argtypes = [ctypes.POINTER(c_fwd_params)]
        L.mxa_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.mxa_bwd_workspace_bytes.argtypes = [ctypes.POINTER(c_bwd_params)]
        L.mxa_bwd_workspace_min_bytes.restype = ctypes.c_size_t
        L.mxa_bwd_workspace_min_bytes.argtypes = [ctypes.POINTER(c_bwd_params)]
        L.mxa_bwd.restype = i32
        L.mxa_bwd.argtypes = [ctypes.POINTER(c_bwd_params), P, ctypes.c_size_t, P]
        L.mxa_bwd_noalloc.restype = i32
        L.mxa_bwd_noalloc.argtypes = [ctypes.POINTER(c_bwd_params), P]
        L.mxa_get_error.restype = i32
        L.mxa_get_error.argtypes = [P]
        L.mxa_test_e4m3.restype = i32
        L.mxa_test_e4m3.argtypes = [P, i64, P, P]
        L.mxa_test_ds_blocks.restype = i32
        L.mxa_test_ds_blocks.argtypes = [P, i32, i32, P, P, P]
        L.mxa_test_wait_timeout.restype = i32
        L.mxa_test_wait_timeout.argtypes = [ctypes.c_longlong, P]
        L.mxa_test_mma_rate.restype = i32
        L.mxa_test_mma_rate.argtypes = [i32, i32, P, P]
        L.mxa_test_ex2_rate.restype = i32
        L.mxa_test_ex2_rate.argtypes = [i32, i32, P, P]
        L.mxa_test_tmem_max.restype = i32
        L.mxa_test_tmem_max.argtypes = [P, P, P]
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != MXA_OK:
        raise MxaError(st, what)


# ----------------------------------------------------------------- C names

def mxa_abi_version() -> int:
    return lib().mxa_abi_version()


def status_str(st: int) -> str:
    return lib().mxa_status_str(int(st)).decode()


mxa_status_str = status_str


def mxa_scale_tiles(T: int, num_docs: int, cu_seqlens_host=None) -> int:
    if cu_seqlens_host is None:
        return int(lib().mxa_scale_tiles(T, num_docs, None))
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(v) for v in cu_seqlens_host])
    return int(lib().mxa_scale_tiles(T, num_docs, ctypes.cast(arr, ctypes.c_void_p)))


def mxa_scale_tiles_bound(T: int, num_docs: int) -> int:
    return int(lib().mxa_scale_tiles_bound(T, num_docs))


def mxa_scale_bytes(H: int, ntiles: int) -> int:
    return int(lib().mxa_scale_bytes(H, ntiles))


def mxa_quantize(x, T, H, d, cu_seqlens, num_docs, max_seqlen, ntiles, mode, views, hadamard, row, tok,
                 stream=None) -> int:
    """Raw call: row / tok are c_qview (or None)."""
    return lib().mxa_quantize(_ptr(x), T, H, d, _ptr(cu_seqlens), num_docs, max_seqlen, ntiles, mode, views,
                              int(bool(hadamard)), ctypes.byref(row) if row is not None else None,
                              ctypes.byref(tok) if tok is not None else None, _stream(stream))


def mxa_fwd(params: c_fwd_params, stream=None) -> int:
    return lib().mxa_fwd(ctypes.byref(params), _stream(stream))


def mxa_fwd_workspace_bytes(params: c_fwd_params) -> int:
    return int(lib().mxa_fwd_workspace_bytes(ctypes.byref(params)))


def mxa_bwd_workspace_bytes(params: c_bwd_params) -> int:
    return int(lib().mxa_bwd_workspace_bytes(ctypes.byref(params)))


def mxa_bwd_workspace_min_bytes(params: c_bwd_params) -> int:
    return int(lib().mxa_bwd_workspace_min_bytes(ctypes.byref(params)))


def mxa_bwd(params: c_bwd_params, workspace, ws_bytes: int, stream=None) -> int:
    return lib().mxa_bwd(ctypes.byref(params), _ptr(workspace), ws_bytes, _stream(stream))


def mxa_bwd_noalloc(params: c_bwd_params, stream=None) -> int:
    """Backward with the library-owned scratch array as workspace (for callers
    that cannot allocate device memory); see include/mxa.h."""
    return lib().mxa_bwd_noalloc(ctypes.byref(params), _stream(stream))


def mxa_test_e4m3(x: torch.Tensor, codes: torch.Tensor, stream=None) -> int:
    """include/mxa_testing.h: E4M3 codes of fp32 x through the kernels' packed conversion."""
    return lib().mxa_test_e4m3(_ptr(x), x.numel(), _ptr(codes), _stream(stream))


def mxa_test_ds_blocks(x: torch.Tensor, shift: int, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> int:
    """include/mxa_testing.h: the kernels' 32 x 32 dS block quantization of x [nblocks, 32, 32]."""
    return lib().mxa_test_ds_blocks(_ptr(x), x.shape[0], shift, _ptr(codes), _ptr(scales), _stream(stream))


def mxa_test_wait_timeout(budget_cycles: int, stream=None) -> int:
    """include/mxa_testing.h: the kernels' bounded wait, run out on purpose
    (a barrier nothing arrives on) with a short budget."""
    return lib().mxa_test_wait_timeout(int(budget_cycles), _stream(stream))


def mxa_test_mma_rate(iters: int, cycles: torch.Tensor, stream=None) -> int:
    """include/mxa_testing.h: block-scaled MMA rate probe, one CTA per
    element of cycles (int64, device)."""
    assert cycles.dtype == torch.int64 and cycles.is_cuda
    return lib().mxa_test_mma_rate(int(iters), cycles.numel(), _ptr(cycles), _stream(stream))


def mxa_test_ex2_rate(iters: int, cycles: torch.Tensor, stream=None) -> int:
    """include/mxa_testing.h: exponential-unit rate probe (ex2.approx.ftz.f32,
    512 threads x 8 chains per CTA), one CTA per element of cycles (int64,
    device)."""
    assert cycles.dtype == torch.int64 and cycles.is_cuda
    return lib().mxa_test_ex2_rate(int(iters), cycles.numel(), _ptr(cycles), _stream(stream))


def mxa_test_tmem_max(x: torch.Tensor, out: torch.Tensor, stream=None) -> int:
    """include/mxa_testing.h: TMEM round trip of x (fp32 [128, 64], device)
    with the load-with-maximum; out (fp32 [128, 3], device)."""
    assert x.dtype == torch.float32 and x.is_cuda and out.dtype == torch.float32 and out.is_cuda
    assert x.numel() == 128 * 64 and out.numel() == 128 * 3
    return lib().mxa_test_tmem_max(_ptr(x), _ptr(out), _stream(stream))


def mxa_get_error(stream=None) -> int:
    return lib().mxa_get_error(_stream(stream))


# ----------------------------------------------------------------- helpers

@dataclass
class QView:
    """E4M3 codes [T, H, d] (uint8) and UE8M0 scale atoms [H, NT, 512] (uint8)."""
    codes: torch.Tensor
    scales: torch.Tensor

    def c(self) -> c_qview:
        return c_qview(self.codes.data_ptr(), self.scales.data_ptr())


@dataclass
class Geometry:
    """Token layout of a call: T tokens in num_docs documents."""
    T: int
    num_docs: int
    max_seqlen: int
    ntiles: int
    cu_seqlens: Optional[torch.Tensor] = None  # device int32 [num_docs + 1] or None (equal documents)

    @staticmethod
    def batched(B: int, L: int) -> "Geometry":
        return Geometry(B * L, B, L, mxa_scale_tiles(B * L, B, None), None)

    @staticmethod
    def packed(lengths, device="cuda") -> "Geometry":
        import numpy as np

        cu = np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)
        T = int(cu[-1])
        return Geometry(T, len(lengths), int(max(lengths)), mxa_scale_tiles(T, len(lengths), cu.tolist()),
                        torch.from_numpy(cu).to(device))


def quantize(x: torch.Tensor, geo: Geometry, mode: int = MXA_SCALE_MX32, views: int = MXA_VIEW_ROW | MXA_VIEW_TOK,
             hadamard: bool = False, out=None, stream=None, rmsnorm=None):
    """x bf16 [T, H, d] on the GPU -> (row QView or None, tok QView or None).
    In token-block mode both views share one code tensor.  rmsnorm: None, or
    (weight fp32 [d] on the GPU or None, eps) to quantize the RMSNorm of x
    (mxa_rmsnorm_quantize)."""
    T, H, d = x.shape
    assert T == geo.T and x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    sb = mxa_scale_bytes(H, geo.ntiles)
    dev = x.device
    if out is not None:
        row, tok = out
    else:
        row = tok = None
        if views & MXA_VIEW_ROW or mode == MXA_SCALE_TOKBLOCK32:
            row = QView(torch.empty((T, H, d), dtype=torch.uint8, device=dev),
                        torch.empty((H, geo.ntiles, ATOM_BYTES), dtype=torch.uint8, device=dev))
        if views & MXA_VIEW_TOK or mode == MXA_SCALE_TOKBLOCK32:
            codes = row.codes if mode == MXA_SCALE_TOKBLOCK32 else torch.empty((T, H, d), dtype=torch.uint8, device=dev)
            tok = QView(codes, torch.empty((H, geo.ntiles, ATOM_BYTES), dtype=torch.uint8, device=dev))
    assert row is None or row.scales.numel() == sb
    if rmsnorm is None:
        st = mxa_quantize(x, T, H, d, geo.cu_seqlens, geo.num_docs, geo.max_seqlen, geo.ntiles, mode, views,
                          hadamard, row.c() if row is not None else None, tok.c() if tok is not None else None, stream)
        _check(st, "mxa_quantize")
    else:
        w, eps = rmsnorm
        assert w is None or (w.dtype == torch.float32 and w.is_cuda and w.numel() == d)
        st = lib().mxa_rmsnorm_quantize(_ptr(x), _ptr(w), float(eps), T, H, d, _ptr(geo.cu_seqlens), geo.num_docs,
                                        geo.max_seqlen, geo.ntiles, mode, views, int(bool(hadamard)),
                                        ctypes.byref(row.c()) if row is not None else None,
                                        ctypes.byref(tok.c()) if tok is not None else None, _stream(stream))
        _check(st, "mxa_rmsnorm_quantize")
    return row, tok


def quantize_key(x: torch.Tensor, geo: Geometry, out: Optional[QView] = None, stream=None) -> QView:
    """Per-key view of x bf16 [T, H, d] (mxa_quantize_key): codes [T, H, d],
    one UE8M0 exponent per (token, head) in scales [H, NT, 128]."""
    T, H, d = x.shape
    assert T == geo.T and x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    key = out if out is not None else QView(torch.empty((T, H, d), dtype=torch.uint8, device=x.device),
                                            torch.empty((H, geo.ntiles, 128), dtype=torch.uint8, device=x.device))
    assert key.scales.numel() == lib().mxa_key_scale_bytes(H, geo.ntiles)
    st = lib().mxa_quantize_key(_ptr(x), T, H, d, _ptr(geo.cu_seqlens), geo.num_docs, geo.max_seqlen, geo.ntiles,
                                ctypes.byref(key.c()), _stream(stream))
    _check(st, "mxa_quantize_key")
    return key


def _shape(geo: Geometry, Hq: int, Hkv: int, d: int, causal: bool, softmax_scale: float,
           kv_geo: Optional[Geometry] = None) -> c_shape:
    """kv_geo: the key/value documents of a cross-attention call (None: self-attention)."""
    sh = c_shape(geo.T, Hq, Hkv, d, geo.cu_seqlens.data_ptr() if geo.cu_seqlens is not None else None,
                 geo.num_docs, geo.max_seqlen, geo.ntiles, int(bool(causal)), float(softmax_scale))
    if kv_geo is not None:
        assert kv_geo.num_docs == geo.num_docs
        sh.T_k = kv_geo.T
        sh.cu_seqlens_k = kv_geo.cu_seqlens.data_ptr() if kv_geo.cu_seqlens is not None else None
        sh.max_seqlen_k = kv_geo.max_seqlen
        sh.ntiles_k = kv_geo.ntiles
    return sh


def fwd(q_row: QView, k_row: QView, v_tok: QView, geo: Geometry, causal: bool, softmax_scale: float = 0.0,
        out=None, stream=None, workspace=None, use_list: bool = True, kv_geo: Optional[Geometry] = None,
        v_key: Optional[QView] = None):
    """-> (O bf16 [T, Hq, d], LSE fp32 [Hq, T]).  With use_list (default) the
    CTAs are scheduled from the cost-sorted tile list, in `workspace` when it
    is large enough, else in a fresh device buffer.  v_key: the per-key view
    of V (quantize_key) for the strict causal fold on the diagonal tile."""
    T, Hq, d = q_row.codes.shape
    Hkv = k_row.codes.shape[1]
    if out is None:
        o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=q_row.codes.device)
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q_row.codes.device)
    else:
        o, lse = out
    p = c_fwd_params(_shape(geo, Hq, Hkv, d, causal, softmax_scale, kv_geo), q_row.c(), k_row.c(), v_tok.c(),
                     o.data_ptr(), lse.data_ptr(), None, 0)
    need = mxa_fwd_workspace_bytes(p) if use_list else 0
    if need:
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q_row.codes.device)
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel()
    if v_key is not None:
        p.v_key = v_key.c()
    _check(mxa_fwd(p, stream), "mxa_fwd")
    return o, lse


def bwd_params(views: dict, o, lse, dq, dk, dv, geo: Geometry, causal: bool, dq_mode: int = MXA_DQ_FP32,
               softmax_scale: float = 0.0, kv_geo: Optional[Geometry] = None,
               k_key: Optional[QView] = None) -> c_bwd_params:
    T, Hq, d = views["q_row"].codes.shape
    Hkv = views["k_row"].codes.shape[1]
    return c_bwd_params(_shape(geo, Hq, Hkv, d, causal, softmax_scale, kv_geo), views["q_row"].c(), views["k_row"].c(),
                        views["v_row"].c(), views["g_row"].c(), views["q_tok"].c(), views["k_tok"].c(),
                        views["g_tok"].c(), o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                        dv.data_ptr(), int(dq_mode), k_key.c() if k_key is not None else c_qview(None, None))


def bwd(views: dict, o, lse, geo: Geometry, causal: bool, dq_mode: int = MXA_DQ_FP32, softmax_scale: float = 0.0,
        workspace=None, out=None, stream=None, kv_geo: Optional[Geometry] = None, k_key: Optional[QView] = None):
    """views: dict with q_row, k_row, v_row, g_row, q_tok, k_tok, g_tok QViews
    (k_*, v_* over kv_geo's tokens for cross-attention).
    -> (dQ bf16 [T, Hq, d], dK, dV bf16 [Tk, Hkv, d])."""
    T, Hq, d = views["q_row"].codes.shape
    Tk, Hkv = views["k_row"].codes.shape[:2]
    dev = o.device
    if out is None:
        dq = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
        dk = torch.empty((Tk, Hkv, d), dtype=torch.bfloat16, device=dev)
        dv = torch.empty((Tk, Hkv, d), dtype=torch.bfloat16, device=dev)
    else:
        dq, dk, dv = out
    p = bwd_params(views, o, lse, dq, dk, dv, geo, causal, dq_mode, softmax_scale, kv_geo, k_key)
    need = mxa_bwd_workspace_bytes(p)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(mxa_bwd(p, workspace, workspace.numel(), stream), "mxa_bwd")
    return dq, dk, dv


def check_error(stream=None):
    _check(mxa_get_error(stream), "kernel")


# --------------------------------------------------- scale layout helpers

def atom_index(r: int, g: int) -> int:
    """Byte of (row r, group g) inside a 512-byte scale atom."""
    return (r % 32) * 16 + (r // 32) * 4 + g


def row_scales_logical(scales: torch.Tensor, lengths, d: int):
    """ROW-view atoms [H, NT, 512] -> logical [T, H, d/32] (numpy uint8)."""
    import numpy as np

    s = scales.cpu().numpy()
    H = s.shape[0]
    T = int(sum(lengths))
    out = np.zeros((T, H, d // 32), np.uint8)
    r = np.arange(128)
    idx = np.array([[atom_index(int(rr), g) for g in range(d // 32)] for rr in r])  # [128, G]
    t0 = tb = 0
    for n in lengths:
        for i in range((n + 127) // 128):
            rows = min(128, n - 128 * i)
            blk = s[:, tb + i, :][:, idx[:rows]]  # [H, rows, G]
            out[t0 + 128 * i: t0 + 128 * i + rows] = blk.transpose(1, 0, 2)
        t0 += n
        tb += (n + 127) // 128
    return out


def tok_scales_logical(scales: torch.Tensor, lengths, d: int):
    """TOK-view atoms [H, NT, 512] -> logical [H, d, NB] with NB = sum ceil(n/32)
    (document-relative 32-token groups, documents concatenated)."""
    import numpy as np

    s = scales.cpu().numpy()
    H = s.shape[0]
    NB = sum((n + 31) // 32 for n in lengths)
    out = np.zeros((H, d, NB), np.uint8)
    idx = np.array([[atom_index(c, g) for g in range(4)] for c in range(d)])  # [d, 4]
    tb = gb = 0
    for n in lengths:
        ng = (n + 31) // 32
        for q in range(ng):
            out[:, :, gb + q] = s[:, tb + q // 4, :][:, idx[:, q % 4]]
        tb += (n + 127) // 128
        gb += ng
    return out
