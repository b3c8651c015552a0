"""Host-side checks of the C ABI (no GPU work): the library builds, loads and
exports every entry point include/mxa.h declares; pure host helpers compute
the documented layouts; invalid arguments return a status without launching."""
import ctypes
import os
import re

import pytest

from block_scaled_mxfp8_gb300 import build as mbuild
from block_scaled_mxfp8_gb300 import mxa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mxa.lib()


def declared_functions(header="mxa.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mxa_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mxa_quantize" in names and "mxa_fwd" in names and "mxa_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(mxa.EXPORTS) | set(names)
    assert mxa.mxa_abi_version() == 4


def test_exports_testing_hooks(lib):
    names = [n for n in declared_functions("mxa_testing.h") if n.startswith("mxa_test_")]
    assert names == sorted(mxa.EXPORTS_TESTING)
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layouts_match_header():
    # sizes of the C structs on this platform (x86-64 / aarch64 LP64)
    assert ctypes.sizeof(mxa.c_qview) == 16
    assert ctypes.sizeof(mxa.c_shape) == 88
    assert ctypes.sizeof(mxa.c_fwd_params) == 184  # + v_key
    assert ctypes.sizeof(mxa.c_bwd_params) == 264  # + k_key


def test_scale_tile_helpers(lib):
    assert mxa.mxa_scale_tiles(32768, 8) == 8 * 32
    assert mxa.mxa_scale_tiles(300, 3, [0, 100, 250, 300]) == 1 + 2 + 1
    assert mxa.mxa_scale_tiles(300, 3, [0, 100, 250, 299]) == -1  # last offset must be T
    assert mxa.mxa_scale_tiles(10, 3) == -1  # T not divisible
    assert mxa.mxa_scale_tiles_bound(300, 3) == 3 + 3
    assert mxa.mxa_scale_bytes(4, 10) == 4 * 10 * 512
    assert [mxa.atom_index(r, 0) for r in (0, 1, 31, 32, 127)] == [0, 16, 496, 4, 508]


def test_status_strings(lib):
    for s in range(7):
        assert isinstance(mxa.status_str(s), str) and mxa.status_str(s)


def _qv(p=256):
    return mxa.c_qview(p, p)


def test_quantize_rejects_bad_arguments_without_launch(lib):
    L = lib
    q = _qv()
    P = ctypes.c_void_p
    call = lambda *a: L.mxa_quantize(*a)
    ok_args = [P(256), 256, 2, 128, None, 1, 256, 2, 0, 3, 0, ctypes.byref(q), ctypes.byref(q), None]
    a = list(ok_args)
    a[0] = None
    assert call(*a) == mxa.MXA_ERR_ARG
    a = list(ok_args)
    a[3] = 96
    assert call(*a) == mxa.MXA_ERR_UNSUPPORTED
    a = list(ok_args)
    a[5] = 3  # 256 % 3 != 0 with cu_seqlens NULL
    assert call(*a) == mxa.MXA_ERR_ARG
    a = list(ok_args)
    a[8] = 7  # bad mode
    assert call(*a) == mxa.MXA_ERR_ARG
    a = list(ok_args)
    a[10] = 1  # hadamard needs token-block mode
    assert call(*a) == mxa.MXA_ERR_UNSUPPORTED
    a = list(ok_args)
    a[0] = P(257)  # misaligned input
    assert call(*a) == mxa.MXA_ERR_ALIGN
    a = list(ok_args)
    q2 = mxa.c_qview(264, 256)  # codes not 16-byte aligned
    a[11] = ctypes.byref(q2)
    assert call(*a) == mxa.MXA_ERR_ALIGN
    a = list(ok_args)
    a[8], a[10] = 1, 1
    a[3] = 64  # hadamard with d != 128
    assert call(*a) == mxa.MXA_ERR_UNSUPPORTED
    a = list(ok_args)
    a[9] = 0  # no view
    assert call(*a) == mxa.MXA_ERR_ARG


def _fwd(T=256, Hq=2, Hkv=2, d=128, nd=1, maxlen=256, nt=2):
    sh = mxa.c_shape(T, Hq, Hkv, d, None, nd, maxlen, nt, 0, 0.0)
    return mxa.c_fwd_params(sh, _qv(), _qv(), _qv(), 256, 256, None, 0)


def test_fwd_bwd_reject_bad_arguments_without_launch(lib):
    L = lib
    assert L.mxa_fwd(None, None) == mxa.MXA_ERR_ARG
    p = _fwd(Hq=3, Hkv=2)
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_UNSUPPORTED  # Hq % Hkv
    p = _fwd(d=96)
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_UNSUPPORTED
    p = _fwd()
    p.o = 0
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    p = _fwd()
    p.q_row = mxa.c_qview(0, 256)
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    p = _fwd(maxlen=100)  # documents longer than max_seqlen
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    p = _fwd()
    p.shape.softmax_scale = -1.0
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    # the tile work list: nothing to do for equal documents (masked or not);
    # packed documents take 256 bytes of header, 16 bytes per query tile and
    # 2 x 4 per document, rounded up to 256
    p = _fwd()
    assert L.mxa_fwd_workspace_bytes(ctypes.byref(p)) == 0
    p.shape.causal = 1
    assert L.mxa_fwd_workspace_bytes(ctypes.byref(p)) == 0
    pj = _fwd(T=1000, nd=3, maxlen=600, nt=10)
    pj.shape.cu_seqlens = 4096  # never read: sizing needs no device data
    assert L.mxa_fwd_workspace_bytes(ctypes.byref(pj)) == 512  # 256 + 10 * 16 + 2 * 3 * 4 = 440
    pj.workspace, pj.workspace_bytes = 8, 768  # used, but not 256-byte aligned
    assert L.mxa_fwd(ctypes.byref(pj), None) == mxa.MXA_ERR_ALIGN
    sh = mxa.c_shape(256, 2, 2, 128, None, 1, 256, 2, 1, 0.0)
    bp = mxa.c_bwd_params(sh, *[_qv()] * 7, 256, 256, 256, 256, 256, 0)
    need = L.mxa_bwd_workspace_bytes(ctypes.byref(bp))
    need_min = L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp))
    # padded D and LSE rows [Hq, NT, 128] fp32; fp32 mode adds the emitted dS:
    # one 16 KB code tile + 16 block scales per (head, key tile, query-tile
    # slot) pair
    assert need_min == 2 * 2 * 2 * 128 * 4 + 2 * 512  # + the query and key tile lists
    assert need == need_min + 2 * 2 * 2 * (16384 + 16)
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), need_min - 1, None) == mxa.MXA_ERR_WORKSPACE
    assert L.mxa_bwd(ctypes.byref(bp), None, need, None) == mxa.MXA_ERR_WORKSPACE
    bp.dq_mode = 5
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), need, None) == mxa.MXA_ERR_ARG
    bp.dq_mode = 1
    # FP16 x 2^9 mode: the emitted dS as in FP32 mode, or at least the fused
    # kernel's fp16 dQ accumulator (whichever is smaller)
    assert L.mxa_bwd_workspace_bytes(ctypes.byref(bp)) == need
    assert L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp)) == need_min + min(256 * 2 * 128 * 2, 2 * 2 * 2 * 16400)
    # FP16 per-row boost: boost rows fp32 [Hq, T], key bounds int32 [T, Hkv]
    # and tile maxima int32 [Hkv, NT] after the D and LSE rows; the dQ GEMM
    # path only (min == full)
    bp.dq_mode = mxa.MXA_DQ_FP16_ROW
    full2 = need + 256 * 2 * 4 + 256 * 2 * 4 + 256
    assert L.mxa_bwd_workspace_bytes(ctypes.byref(bp)) == full2
    assert L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp)) == full2
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), full2 - 1, None) == mxa.MXA_ERR_WORKSPACE
    bp.dq_mode = 3
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), full2, None) == mxa.MXA_ERR_ARG


def test_noalloc_gives_mxa_bwd_status_codes_without_launch(lib):
    """mxa_bwd_noalloc returns the status mxa_bwd gives the same arguments
    (its argument checks run first, before any device call), and
    MXA_ERR_WORKSPACE for a valid call too large for its scratch array."""
    L = lib
    big = mxa.c_shape(1 << 16, 8, 8, 128, None, 1, 1 << 16, (1 << 16) // 128, 1, 0.0)
    small = mxa.c_shape(256, 2, 2, 128, None, 1, 256, 2, 1, 0.0)
    for sh in (big, small):
        bp = mxa.c_bwd_params(sh, *[_qv()] * 7, 256, 256, 256, 256, 256, 0)
        bp.dq = None
        assert L.mxa_bwd_noalloc(ctypes.byref(bp), None) == mxa.MXA_ERR_ARG
        bp.dq = 256
        bp.dq_mode = 7
        assert L.mxa_bwd_noalloc(ctypes.byref(bp), None) == mxa.MXA_ERR_ARG
        bp.dq_mode = 0
        bp.o = 8
        assert L.mxa_bwd_noalloc(ctypes.byref(bp), None) == mxa.MXA_ERR_ALIGN
    bad_d = mxa.c_shape(256, 2, 2, 96, None, 1, 256, 2, 1, 0.0)
    bp = mxa.c_bwd_params(bad_d, *[_qv()] * 7, 256, 256, 256, 256, 256, 0)
    assert L.mxa_bwd_noalloc(ctypes.byref(bp), None) == mxa.MXA_ERR_UNSUPPORTED
    assert L.mxa_bwd_noalloc(None, None) == mxa.MXA_ERR_ARG
    bp = mxa.c_bwd_params(big, *[_qv()] * 7, 256, 256, 256, 256, 256, mxa.MXA_DQ_FP16_X512)
    assert L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp)) > mxa.MXA_BWD_NOALLOC_MAX_WORKSPACE
    assert L.mxa_bwd_noalloc(ctypes.byref(bp), None) == mxa.MXA_ERR_WORKSPACE


def test_cross_attention_shape_checks(lib):
    """Cross-attention (T_k > 0): no causal mask, FP32 dQ only, equal key
    documents must divide T_k; the list sizes follow each side's NT."""
    L = lib
    p = _fwd(T=1024, nd=2, maxlen=512, nt=8)
    p.shape.T_k, p.shape.max_seqlen_k, p.shape.ntiles_k = 4096, 2048, 32
    # equal documents on both sides but Lq != Lk: a work list (8 query tiles)
    assert L.mxa_fwd_workspace_bytes(ctypes.byref(p)) == 512  # 256 + 8 * 16 + 2 * 2 * 4 = 400
    p.shape.causal = 1
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_UNSUPPORTED
    p.shape.causal = 0
    p.shape.T_k = 4095  # not divisible by the 2 documents
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    p.shape.T_k, p.shape.max_seqlen_k = 4096, 1000  # documents longer than max_seqlen_k
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ARG
    sh = mxa.c_shape(1024, 2, 2, 128, None, 2, 512, 8, 0, 0.0)
    sh.T_k, sh.max_seqlen_k, sh.ntiles_k = 4096, 2048, 32
    bp = mxa.c_bwd_params(sh, *[_qv()] * 7, 256, 256, 256, 256, 256, 0)
    need_min = L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp))
    # rows [Hq, NT_q, 128] x 2 fp32, then the query list (8 tiles) and the key list (32 tiles)
    assert need_min == 2 * 2 * 8 * 128 * 4 + 512 + 1024  # 256 + 32 * 16 + 16 = 784 -> 1024
    # the emitted dS: Hq x NT_k x mt(query tiles of the longest document) pairs
    assert L.mxa_bwd_workspace_bytes(ctypes.byref(bp)) == need_min + 2 * 32 * 4 * (16384 + 16)
    for mode in (mxa.MXA_DQ_FP16_X512, mxa.MXA_DQ_FP16_ROW):
        bp.dq_mode = mode
        assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), 1 << 30, None) == mxa.MXA_ERR_UNSUPPORTED


def test_rmsnorm_quantize_rejects_bad_eps_without_launch(lib):
    L = lib
    qv = mxa.c_qview(256, 256)
    for eps in (-1.0, float("inf"), float("nan")):
        st = L.mxa_rmsnorm_quantize(256, None, eps, 256, 1, 128, None, 1, 256, 2, 0, 1, 0, qv, None, None)
        assert st == mxa.MXA_ERR_ARG
    st = L.mxa_rmsnorm_quantize(256, 258, 1e-6, 256, 1, 128, None, 1, 256, 2, 0, 1, 0, qv, None, None)
    assert st == mxa.MXA_ERR_ALIGN


def test_key_view_and_fold_reject_bad_arguments_without_launch(lib):
    L = lib
    P = ctypes.c_void_p
    key = _qv()
    ok = [P(256), 256, 2, 128, None, 1, 256, 2, ctypes.byref(key), None]
    assert L.mxa_key_scale_bytes(2, 2) == 2 * 2 * 128
    for i, bad, st in ((0, None, mxa.MXA_ERR_ARG), (8, None, mxa.MXA_ERR_ARG), (3, 96, mxa.MXA_ERR_UNSUPPORTED),
                       (0, P(8), mxa.MXA_ERR_ALIGN), (1, 300, mxa.MXA_ERR_ARG)):  # T above max_seqlen
        a = list(ok)
        a[i] = bad
        assert L.mxa_quantize_key(*a) == st, (i, bad)
    misaligned = mxa.c_qview(264, 256 + 4)
    a = list(ok)
    a[8] = ctypes.byref(misaligned)
    assert L.mxa_quantize_key(*a) == mxa.MXA_ERR_ALIGN
    # the fold needs self-attention: a per-key view with a key side is refused
    p = _fwd(T=1024, nd=2, maxlen=512, nt=8)
    p.shape.T_k, p.shape.max_seqlen_k, p.shape.ntiles_k = 4096, 2048, 32
    p.v_key = _qv()
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_UNSUPPORTED
    p = _fwd()
    p.v_key = mxa.c_qview(256, 8)
    assert L.mxa_fwd(ctypes.byref(p), None) == mxa.MXA_ERR_ALIGN


def test_strict_backward_workspace_and_refusals(lib):
    L = lib
    sh = mxa.c_shape(256, 2, 2, 128, None, 1, 256, 2, 1, 0.0)
    bp = mxa.c_bwd_params(sh, *[_qv()] * 7, 256, 256, 256, 256, 256, 0)
    plain = L.mxa_bwd_workspace_bytes(ctypes.byref(bp))
    bp.k_key = _qv()
    # one 512-byte scale atom per pair instead of 16 block scales; min == full
    full = L.mxa_bwd_workspace_bytes(ctypes.byref(bp))
    assert full == plain + 2 * 2 * 2 * (512 - 16)
    assert L.mxa_bwd_workspace_min_bytes(ctypes.byref(bp)) == full
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), full - 1, None) == mxa.MXA_ERR_WORKSPACE
    bp.k_key = mxa.c_qview(256, 8)
    assert L.mxa_bwd(ctypes.byref(bp), ctypes.c_void_p(256), 1 << 30, None) == mxa.MXA_ERR_ALIGN
