"""Pins of the oracle's per-row boost of the strict FP16 dQ reduction (FLAMIA
reading notes, sec. 4, "the last channel is in the accumulator": dQ partial
sums boosted by a power of two chosen from the magnitudes of G, V and K; the
strict option takes each row's own G with the maxima of V and K over the
visible keys only).

CPU only.  Checked against: hand-computed exponents where every term of the
bound is nonzero and distinct (so a dropped term or a flipped sign changes the
result), the special cases (all-zero rows, E4M3 subnormals, long documents),
causality (a future spike changes no earlier row), and the property the boost
exists for: 2^beta_i * max_c |dQ_ic| stays below 2^15 on the exact backward
of quantized operands, including gradients large enough that the fixed 2^9
boost would overflow fp16.
"""
import math

import numpy as np
import torch

from oracle import oracle as orc


def test_closed_form_every_term_distinct():
    # g = cl2(4) = 2, V = cl2(5) = 3, K = cl2(0.5) = -1, cl2(alpha = 2^-3.5) = -3,
    # log2 d = 7, n = 300 -> s = 1:  beta = 15 - (4 - 3 + 7 + 1 + 2 + 3 - 1) = 2
    T, d = 300, 128
    G = np.full((T, 2, d), 4.0)
    V = np.zeros((T, 1, d))
    V[7, 0, 3] = -5.0
    K = np.zeros((T, 1, d))
    K[:, 0, 0] = 0.5
    b = orc.dq_row_boost(G, V, K, None, False)
    assert b.shape == (2, T) and (b == 2).all()
    # causal: rows 0..6 see only zero V rows (bound 0 -> the clamp, 100)
    bc = orc.dq_row_boost(G, V, K, None, True)
    assert (bc[:, :7] == 100).all() and (bc[:, 7:] == 2).all()
    # a G row scaled by 2^5 (and one of V's keys by 2^2) moves beta by exactly that
    G2 = G.copy()
    G2[11, 1] *= 32.0
    b2 = orc.dq_row_boost(G2, V, K, None, False)
    assert b2[1, 11] == -3 and b2[0, 11] == 2
    V2 = V.copy()
    V2[200, 0, 0] = 20.0  # cl2(20) = 5
    assert (orc.dq_row_boost(G, V2, K, None, False) == 0).all()


def test_alpha_headdim_and_long_document_terms():
    # d = 64: log2 d = 6; alpha = 1 -> cl2 = 0; g = V = K = 0 (max |x| = 1)
    T, d = 40, 64
    ones = np.ones((T, 1, d))
    assert (orc.dq_row_boost(ones, ones, ones, None, False, alpha=1.0) == 15 - (4 + 0 + 6 + 1)).all()
    # n visible keys > 2^14: s(n) = 1 + cl2(n) - 14
    T = 20000
    G = np.ones((T, 1, 128))
    b = orc.dq_row_boost(G, G, G, None, True, alpha=1.0)[0]
    n = np.arange(1, T + 1)
    s = 1 + np.maximum(0, np.ceil(np.log2(n)).astype(int) - 14)
    assert (b == 15 - (4 + 7) - s).all()
    assert b[16383] == 3 and b[16384] == 2 and b[19999] == 2  # n = 16384, 16385, 20000


def test_subnormal_and_zero_rows():
    T, d = 8, 128
    G = np.zeros((T, 1, d))
    G[1, 0, 5] = 3 * 2.0 ** -9  # an E4M3 subnormal (scale 1): cl2 = -7
    G[2, 0, 5] = 2.0 ** -9      # the smallest one: cl2 = -9
    V = np.ones((T, 1, d))
    b = orc.dq_row_boost(G, V, V, None, False, alpha=1.0)[0]
    base = 15 - (4 + 7 + 1)
    assert b[0] == 100 and b[1] == base + 7 and b[2] == base + 9


def test_future_spike_changes_no_earlier_row():
    rng = np.random.default_rng(5)
    lens = [200, 130]
    T = sum(lens)
    cu = np.array([0, 200, 330], np.int32)
    G, V, K = (rng.standard_normal((T, h, 64)) for h in (4, 2, 2))
    base = orc.dq_row_boost(G, V, K, cu, True)
    for p, which in ((120, "V"), (57, "K"), (250, "V")):
        V2, K2 = V.copy(), K.copy()
        (V2 if which == "V" else K2)[p, 1, 3] = 1.0e6
        got = orc.dq_row_boost(G, V2, K2, cu, True)
        doc_start = 0 if p < 200 else 200
        doc_end = 200 if p < 200 else 330
        # kv head 1 serves query heads 2 and 3
        assert np.array_equal(got[:, :p], base[:, :p])
        assert np.array_equal(got[:2], base[:2])
        assert (got[2:, p:doc_end] < base[2:, p:doc_end]).all()
        assert np.array_equal(got[:, doc_end:], base[:, doc_end:])
        assert doc_start <= p


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _row(x):
    c, s = orc.quant_row(_bf16(x))
    return orc.dequant_row(c, s)


def _tok(x, cu):
    c, s = orc.quant_tok(_bf16(x), cu)
    return orc.dequant_tok(c, s, cu)


def test_boost_bounds_the_exact_dq_of_quantized_operands():
    """2^beta_i * |dQ_i| <= 2^15 on the exact backward (fp64) of MX views,
    with G large enough that the fixed 2^9 boost would overflow fp16."""
    rng = np.random.default_rng(9)
    lens = [150, 77, 40]
    T = sum(lens)
    cu = np.array(np.concatenate([[0], np.cumsum(lens)]), np.int32)
    Hq, Hkv, d = 4, 2, 128
    for causal in (False, True):
        Q = rng.standard_normal((T, Hq, d)) * 3
        K = rng.standard_normal((T, Hkv, d)) * 2
        V = rng.standard_normal((T, Hkv, d)) * rng.choice([1.0, 50.0], size=(T, Hkv, 1))
        G = rng.standard_normal((T, Hq, d)) * 2.0 ** 12
        Qr, Kr, Vr, Gr = _row(Q), _row(K), _row(V), _row(G)
        Qt, Kt, Vt, Gt = _tok(Q, cu), _tok(K, cu), _tok(V, cu), _tok(G, cu)
        r = orc.attn_bwd(Qr, Kr, Vt, Vr, Gr, Qt, Kt, Gt, cu, causal)
        beta = orc.dq_row_boost(Gr, Vr, Kr, cu, causal)
        dqmax = np.abs(r["dQ"]).max(axis=2).T  # [Hq, T]
        boosted = dqmax * np.exp2(beta.astype(np.float64))
        assert (boosted <= 2.0 ** 15).all()
        assert (dqmax * 512 > 65504).any(), "the case must overflow the fixed 2^9 boost"
        # not vacuous: the bound is loose by a bounded factor -- d, the
        # margins, and the cancellation in sum_j P_ij (dP_ij - D_i) K_j that a
        # bound cannot count on (random rows sit ~18 binades below it; fp16
        # keeps full relative precision down to 2^-14, 29 binades below 2^15)
        med = np.median(np.log2(boosted[boosted > 0]))
        assert 15 - 24 < med < 15 - 8, med
