"""Pins of the oracle's Algorithm 1 variant (FLAMIA reading notes, sec. 5,
"算法 1。低精度前向与一致的反向重算"): the forward with its weights quantized
as E4M3(2^4 p) (step 07) and O saved in bf16 (step 08), the backward with
U = P (E - D) quantized per 32 x 32 block (step 14) and dV's operand
E4M3(2^8 P) (step 15), the strict dQ operand (per-query dS scales and the K
fold, sec. 4).

CPU only.  What fixes each part, other than the oracle itself:
  * the fast E4M3 rounding against the pinned encoder, bf16 rounding against
    torch's cast;
  * with every rounding off, the direct oracle (itself pinned to torch SDPA +
    autograd) for self-, cross- and folded attention;
  * hand-worked rows (tests/golden/alg1_examples.json);
  * exact special cases: the first causal query, equal scores, power-of-two
    scaling of V and G;
  * brute force on tiny inputs: one-hot value and gradient views read the
    quantized weight, dV operand and U matrices out of O, dV, dQ and dK, which
    are compared element by element with the block rule applied here;
  * the view routing: each output depends on exactly the views its formula
    names, linearly where the formula is linear;
  * which rows a perturbation may move: documents are isolated, O is causal,
    dQ of rows in earlier 32-query blocks keeps its bits, and with the strict
    dQ operand every earlier row keeps its bits.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "alg1_examples.json")))
LN2 = math.log(2.0)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return scale * torch.randn(*shape, generator=g, dtype=torch.float64).numpy()


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _views(T, Hq, Hkv, d, seed):
    """Eight distinct random views: Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt."""
    shapes = [(T, Hq, d), (T, Hkv, d), (T, Hkv, d), (T, Hkv, d), (T, Hq, d), (T, Hq, d), (T, Hkv, d), (T, Hq, d)]
    return [_rand(s, seed + i) for i, s in enumerate(shapes)]


# ---------------------------------------------------------------- codecs

def test_e4m3_round_is_the_pinned_encoder():
    """orc_e4m3_round (binary search) equals decode(encode(y)) of the pinned
    scan encoder on every bf16 pattern at several scales, and on every tie
    between neighbouring codes and one fp64 ulp either side of it."""
    pats = np.arange(65536, dtype=np.uint32) << 16
    vals = pats.view(np.float32).astype(np.float64)
    vals = vals[np.isfinite(vals)]
    tab = orc.e4m3_table()
    for e in (-12, -4, 0, 3):
        y = np.ldexp(vals, e)
        got = orc.e4m3_round_array(y)
        want = tab[orc.e4m3_encode_array(y)]
        assert np.array_equal(got, want, equal_nan=True), e
    pos = tab[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    y = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), -mids, [448.0, 449.0, 1e30, 0.0]])
    assert np.array_equal(orc.e4m3_round_array(y), tab[orc.e4m3_encode_array(y)])


def test_round_bf16_matches_torch_cast():
    """fp32 values (random, plus exact ties at several binades) round to the
    bf16 value torch's RNE cast gives."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(200000, generator=g, dtype=torch.float32) * torch.exp2(torch.randint(-30, 30, (200000,),
                                                                                       generator=g).float())
    ties = torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -3.0 * (1 + 2.0 ** -8), 2.0 ** -100 * (1 + 2.0 ** -8)],
                        dtype=torch.float32)
    x = torch.cat([x, ties])
    want = x.to(torch.bfloat16).double().numpy()
    got = orc.round_bf16_array(x.double().numpy())
    assert np.array_equal(got, want)


# ------------------------------------------------- reduction to the direct oracle

@pytest.mark.parametrize("causal", [False, True])
def test_rounding_off_is_the_direct_oracle(causal):
    lens, Hq, Hkv, d = [37, 1, 140, 64], 4, 2, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 100)
    O0, L0 = orc.attn_fwd(Qs, Ks, Vo, cu, causal)
    O1, L1 = orc.attn_fwd_alg1(Qs, Ks, Vo, cu, causal, rnd=0)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-13)
    r0 = orc.attn_bwd(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, causal)
    r1 = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, causal, rnd=0)
    for k in ("dQ", "dK", "dV", "O", "LSE", "D"):
        np.testing.assert_allclose(r1[k], r0[k], rtol=0, atol=1e-12, err_msg=k)


def test_rounding_off_is_the_direct_cross_oracle():
    lq, lk, Hq, Hkv, d = [20, 0, 70], [90, 33, 5], 2, 1, 32
    cq, ck = _cu(lq), _cu(lk)
    Tq, Tk = sum(lq), sum(lk)
    Qs, Gr, Qt, Gt = (_rand((Tq, Hq, d), s) for s in (1, 2, 3, 4))
    Ks, Vo, Vr, Kt = (_rand((Tk, Hkv, d), s) for s in (5, 6, 7, 8))
    O0, L0 = orc.attn_fwd_x(Qs, Ks, Vo, cq, ck)
    O1, L1 = orc.attn_fwd_alg1(Qs, Ks, Vo, cq, False, rnd=0, cu_k=ck)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-13)
    r0 = orc.attn_bwd_x(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cq, ck)
    r1 = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cq, False, rnd=0, cu_k=ck)
    for k in ("dQ", "dK", "dV", "O", "LSE", "D"):
        np.testing.assert_allclose(r1[k], r0[k], rtol=0, atol=1e-12, err_msg=k)


def test_rounding_off_is_the_direct_fold_oracle():
    lens, Hq, Hkv, d = [300, 45], 2, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 200)
    vsf = (127 + np.random.default_rng(1).integers(-3, 4, (T, Hkv))).astype(np.uint8)
    ksf = (127 + np.random.default_rng(2).integers(-3, 4, (T, Hkv))).astype(np.uint8)
    Vkey, Kkey = _rand((T, Hkv, d), 300), _rand((T, Hkv, d), 301)
    O0, L0 = orc.attn_fwd_fold(Qs, Ks, Vo, Vkey, cu)
    O1, L1 = orc.attn_fwd_alg1(Qs, Ks, Vo, cu, True, rnd=0, Vkey=Vkey, vkey_sf=vsf)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-13)
    r0 = orc.attn_bwd_fold(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, Vkey, Kkey, cu)
    r1 = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, True, rnd=0, Vkey=Vkey, vkey_sf=vsf, Kkey=Kkey,
                           kkey_sf=ksf)
    for k in ("dQ", "dK", "dV", "O", "LSE", "D"):
        np.testing.assert_allclose(r1[k], r0[k], rtol=0, atol=1e-12, err_msg=k)


# ------------------------------------------------------- hand-worked examples

def test_two_key_row_hand_worked():
    ex = GOLD["two_key_row"]
    Q = np.array([[[1.0]], [[0.0]]])
    K = np.array([[[0.4 * LN2]], [[-0.7 * LN2]]])
    V = np.array([[[1.0]], [[-2.0]]])
    O, LSE = orc.attn_fwd_alg1(Q, K, V, None, False, alpha=1.0)
    assert O[0, 0, 0] == ex["O"]
    assert abs(LSE[0, 0] - ex["LSE"]) < 1e-14
    O0, _ = orc.attn_fwd_alg1(Q, K, V, None, False, alpha=1.0, rnd=0)
    assert abs(O0[0, 0, 0] - ex["O_unrounded"]) < 1e-14
    # the reading of the reference (integer ceil of the max) is what decides
    # the value: the exact maximum would give a different one
    assert O[0, 0, 0] != ex["O_if_reference_were_the_exact_max"]


def test_dv_operand_boost_hand_worked():
    ex = GOLD["dv_operand_boost"]
    r = ex["r"]
    a = math.log(r / (1 - r))
    Q = np.array([[[0.5]], [[1.0]]])
    K = np.array([[[a]], [[0.0]]])
    V = np.array([[[1.0]], [[3.0]]])
    G = np.array([[[1.0]], [[1.0]]])
    cu = _cu([2])
    rnd = orc.RND_ALG1 & ~orc.RND_LSE  # P from the exact LSE
    out = orc.attn_bwd_alg1(Q, K, V, V, G, Q, K, G, cu, True, alpha=1.0, rnd=rnd)
    assert out["dV"][0, 0, 0] == ex["dV0"]
    assert out["dV"][1, 0, 0] == ex["dV1"]
    un = orc.attn_bwd_alg1(Q, K, V, V, G, Q, K, G, cu, True, alpha=1.0, rnd=rnd & ~orc.RND_P8)
    assert abs(un["dV"][0, 0, 0] - ex["dV0_unrounded"]) < 1e-15


def test_lazy_reference_row_hand_worked():
    """Step 07's reference schedule with one key per tile: the reference
    rises only when a tile's maximum passes it by more than tau = 4, and the
    one weight in E4M3's subnormal range depends on it."""
    ex = GOLD["lazy_reference_row"]
    x = [-5.3, 2.5, 5.7]
    Q = np.array([[[1.0]], [[0.0]], [[0.0]]])
    K = np.array([[[v * LN2]] for v in x])
    V = np.array([[[1000.0]], [[2.0]], [[-1.0]]])
    O, _ = orc.attn_fwd_alg1(Q, K, V, None, False, alpha=1.0, rnd=orc.RND_P, ref_tile=1)
    assert abs(O[0, 0, 0] - ex["O"]) < 1e-15
    Od, _ = orc.attn_fwd_alg1(Q, K, V, None, False, alpha=1.0, rnd=orc.RND_P, ref_tile=0)
    assert abs(Od[0, 0, 0] - ex["O_direct_reference"]) < 1e-15
    assert ex["weights"][0] != ex["direct_weights"][0]


def test_reference_schedule_properties():
    """One tile covering every key is the direct reference; with scores
    spread over a few binades every weight stays in E4M3's normal range and
    any tile size gives the same bits; dV never depends on the schedule (its
    operand is P = exp(S - LSE))."""
    lens, Hq, Hkv, d = [300, 513], 2, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 1400)
    for causal in (False, True):
        a = orc.attn_fwd_alg1(Qs, Ks, Vo, cu, causal, ref_tile=0)
        b = orc.attn_fwd_alg1(Qs, Ks, Vo, cu, causal, ref_tile=1024)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        small = [0.05 * v for v in (Qs, Ks)]
        outs = [orc.attn_fwd_alg1(small[0], small[1], Vo, cu, causal, ref_tile=r)[0] for r in (0, 1, 7, 256)]
        assert all(np.array_equal(o, outs[0]) for o in outs[1:])
        big = [3.0 * v for v in (Qs, Ks)]
        r0 = orc.attn_bwd_alg1(big[0], big[1], Vo, Vr, Gr, Qt, Kt, Gt, cu, causal, ref_tile=0)
        r1 = orc.attn_bwd_alg1(big[0], big[1], Vo, Vr, Gr, Qt, Kt, Gt, cu, causal, ref_tile=16)
        assert np.array_equal(r0["dV"], r1["dV"]) and np.array_equal(r0["LSE"], r1["LSE"])
        assert not np.array_equal(r0["O"], r1["O"])  # wide scores: subnormal weights follow the schedule


def test_saved_lse_is_fp32_and_moves_by_ulps():
    """Step 08 saves the LSE in fp32 and step 12 rebuilds P from it: the LSE
    output is the fp32 rounding of the exact one (lse_ulps moves it by whole
    fp32 ulps), and with one-hot Gt, dV reads P = exp(S - LSE_saved)."""
    lens, H, d = [40, 25], 1, 65
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks = _rand((T, H, d), 1500, 3.0), _rand((T, H, d), 1501, 3.0)
    Vo, Vr, Gr = _rand((T, H, d), 1502), _rand((T, H, d), 1503), _rand((T, H, d), 1504)
    eye = np.eye(T).reshape(T, 1, T)
    rnd = orc.RND_LSE
    exact = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, True, rnd=0)
    for k in (-1, 0, 2):
        r = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, True, rnd=rnd, lse_ulps=k)
        want = exact["LSE"].astype(np.float32)
        for _ in range(abs(k)):
            want = np.nextafter(want, np.float32(np.inf if k > 0 else -np.inf))
        assert np.array_equal(r["LSE"], want.astype(np.float64)), k
        for b in range(len(lens)):
            s_, e = cu[b], cu[b + 1]
            S = Qs[s_:e, 0] @ Ks[s_:e, 0].T / math.sqrt(d)
            P = np.tril(np.exp(S - r["LSE"][0, s_:e, None]))
            np.testing.assert_allclose(r["dV"][s_:e, 0, s_:e].T, P, rtol=1e-13, atol=0)


def test_p_cap_keeps_algorithm1_weights_in_range():
    """The (c, tau) = (4, 4) choice of the P-cap passage: with the reference
    at most tau = 4 behind, 2^(c + tau) = 256 <= 448, so no boosted weight
    saturates; the direct definition (reference = ceil(max)) keeps every
    boosted weight at or below 2^4."""
    cap = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))["p_cap"]
    c0 = cap["cases"][0]
    assert 2.0 ** (c0["c"] + c0["tau"]) == c0["max_boosted"] <= 448
    x = np.linspace(-30, 0, 100001)
    assert orc.e4m3_round_array(16 * np.exp2(x)).max() <= 16.0


# ------------------------------------------------------------ exact special cases

def test_first_causal_query_and_equal_scores():
    lens, Hq, Hkv, d = [5, 40, 1], 2, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 400)
    Vq = orc.e4m3_round_array(Vo)  # values with 4 significant bits, like decoded codes
    O, _ = orc.attn_fwd_alg1(Qs, Ks, Vq, cu, True)
    for s in cu[:-1]:
        for h in range(Hq):
            assert np.array_equal(O[s, h], Vq[s, h // 2])
    # equal scores: p = 1 for every key, so O is the mean of the values,
    # rounded to bf16
    Oe, _ = orc.attn_fwd_alg1(np.zeros_like(Qs), Ks, Vq, cu, False)
    for b in range(len(lens)):
        s, e = cu[b], cu[b + 1]
        want = orc.round_bf16_array(Vq[s:e].sum(0) / (e - s))
        np.testing.assert_allclose(Oe[s:e, 0], np.broadcast_to(want[0], (e - s, d)), rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_power_of_two_scaling_is_exact(causal):
    """E4M3 after the MX rule commutes with powers of two, and the forward
    weights do not depend on V or G: V -> 2^5 V scales O (and D, U, dQ, dK)
    by 2^5 exactly, G -> 2^-7 G scales D, dQ, dK and dV by 2^-7 exactly."""
    lens, Hq, Hkv, d = [70, 33], 2, 2, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 500)
    r = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, causal)
    rv = orc.attn_bwd_alg1(Qs, Ks, 32 * Vo, 32 * Vr, Gr, Qt, Kt, Gt, cu, causal)
    for k in ("O", "D", "dQ", "dK"):
        assert np.array_equal(rv[k], 32 * r[k]), k
    assert np.array_equal(rv["dV"], r["dV"])
    assert np.array_equal(rv["LSE"], r["LSE"])
    rg = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr / 128, Qt, Kt, Gt / 128, cu, causal)
    for k in ("D", "dQ", "dK", "dV"):
        assert np.array_equal(rg[k], r[k] / 128), k
    assert np.array_equal(rg["O"], r["O"])


# ------------------------------------------------- brute force with one-hot views

def _scores(Qs, Ks, lo, hi, klo, khi, h, hk, alpha):
    return alpha * Qs[lo:hi, h] @ Ks[klo:khi, hk].T


def _boosted_weights(raw, alpha, tile=256):
    """The forward's boosted weights 2^4 p of one row from its visible raw
    scores q.k, as the oracle defines them: the reference schedule over key
    tiles (ceil of an fp32 tile maximum times fp32 alpha log2 e, raised when
    it passes the reference by more than 4) and the exponent argument
    fma32(fl32(q.k), fl32(alpha log2 e), 4 - m), whose power of two is
    rounded to fp32.  Returns (2^4 p, the reference of each key)."""
    sl2 = np.float32(np.float32(alpha) * np.float32(1.4426950408889634))
    r32 = raw.astype(np.float32)
    m = np.empty(len(raw))
    mref = None
    for t0 in range(0, len(raw), tile):
        ts = np.float32(r32[t0:t0 + tile].max() * sl2)
        if mref is None or ts > mref + 4:
            mref = float(np.ceil(ts))
        m[t0:t0 + tile] = mref
    # the product of two fp32 values is exact in fp64; one rounding to fp32
    # then gives the fused multiply-add
    x32 = (r32.astype(np.float64) * np.float64(sl2) + (4.0 - m)).astype(np.float32)
    return np.exp2(x32.astype(np.float64)).astype(np.float32).astype(np.float64), m


def test_one_hot_views_read_out_the_quantized_matrices():
    """With Kt_j = e_j (and Qt_i, Gt_i = e_i) the gradients are the quantized
    matrices themselves: dQ_i[j] = alpha U~_ij, dK_j[i] = alpha U~_ij,
    dV_j[i] = E4M3(2^8 P_ij) 2^-8.  U is read the same way with the dS
    rounding off, and U~ must be its 32 x 32 blocks, counted from each
    document's first token, rounded by the MX rule.  With V_j = e_j the
    forward's O_i[j] W_i reads the weights E4M3(2^4 p_ij) 2^-4 against the
    integer reference ceil(max_j x_ij)."""
    lens = [7, 73]
    T, H, d = sum(lens), 1, sum(lens)
    cu = _cu(lens)
    alpha = 0.125
    Qs, Ks = _rand((T, H, d), 600, 0.6), _rand((T, H, d), 601, 0.6)
    Vo, Vr, Gr = _rand((T, H, d), 602), _rand((T, H, d), 603), _rand((T, H, d), 604)
    eye = np.eye(T).reshape(T, 1, T)
    for causal in (False, True):
        rnd_u = orc.RND_P | orc.RND_O
        ru = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, causal, alpha, rnd=rnd_u)
        rq = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, causal, alpha)
        for b in range(len(lens)):
            s, e = cu[b], cu[b + 1]
            U = ru["dQ"][s:e, 0, s:e] / alpha
            Uq = rq["dQ"][s:e, 0, s:e] / alpha
            want = np.zeros_like(U)
            n = e - s
            for qb in range(0, n, 32):
                for kb in range(0, n, 32):
                    blk = U[qb:qb + 32, kb:kb + 32]
                    ex = orc.mx_exponent(float(np.abs(blk).max()))
                    want[qb:qb + 32, kb:kb + 32] = np.ldexp(orc.e4m3_round_array(np.ldexp(blk, -ex)), ex)
            assert np.array_equal(Uq, want), (causal, b)
            assert np.array_equal(rq["dK"][s:e, 0, s:e].T / alpha, want), (causal, b)
            # dV operand
            S = _scores(Qs, Ks, s, e, s, e, 0, 0, alpha)
            P = np.exp(S - rq["LSE"][0, s:e, None])
            if causal:
                P = np.tril(P)
            assert np.array_equal(rq["dV"][s:e, 0, s:e].T, orc.e4m3_round_array(256 * P) / 256), (causal, b)
        # forward weights
        O, _ = orc.attn_fwd_alg1(Qs, Ks, eye, cu, causal, alpha, rnd=orc.RND_P)
        for b in range(len(lens)):
            s, e = cu[b], cu[b + 1]
            raw = Qs[s:e, 0] @ Ks[s:e, 0].T
            for i in range(e - s):
                kend = i + 1 if causal else e - s
                y, _ = _boosted_weights(raw[i, :kend], alpha)
                w = orc.e4m3_round_array(y) / 16
                np.testing.assert_allclose(O[s + i, 0, s:s + kend], w / w.sum(), rtol=1e-15, atol=0)


def test_one_hot_strict_dq_operand():
    """The strict dQ operand: dQ_i[j] (Kt_j = e_j, Kkey_j = 2^ek_j e_j)
    reads U_ij 2^ek_j on query i's own 128-token tile and U_ij before it,
    rounded per (query i, 32 keys from the document start) by the MX rule;
    dK keeps the 32 x 32 blocks."""
    lens = [7, 293]
    T, H, d = sum(lens), 1, sum(lens)
    cu = _cu(lens)
    alpha = 0.125
    Qs, Ks = _rand((T, H, d), 700, 0.6), _rand((T, H, d), 701, 0.6)
    Vo, Vr, Gr = _rand((T, H, d), 702), _rand((T, H, d), 703), _rand((T, H, d), 704)
    ek = np.random.default_rng(5).integers(-4, 5, (T, H))
    eye = np.eye(T).reshape(T, 1, T)
    kkey = eye * np.exp2(ek)[:, :, None]
    ksf = (ek + 127).astype(np.uint8)
    ru = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, True, alpha, rnd=orc.RND_P | orc.RND_O)
    rs = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, True, alpha, Kkey=kkey, kkey_sf=ksf)
    rb = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, eye, eye, eye, cu, True, alpha)
    assert np.array_equal(rs["dK"], rb["dK"])
    for b in range(len(lens)):
        s, e = cu[b], cu[b + 1]
        n = e - s
        U = ru["dQ"][s:e, 0, s:e] / alpha
        want = np.zeros_like(U)
        for i in range(n):
            y = U[i, :i + 1].copy()
            t0 = (i // 128) * 128
            y[t0:] *= np.exp2(ek[s + t0:s + i + 1, 0])
            for g in range(0, i + 1, 32):
                blk = y[g:g + 32]
                ex = orc.mx_exponent(float(np.abs(blk).max()))
                y[g:g + 32] = np.ldexp(orc.e4m3_round_array(np.ldexp(blk, -ex)), ex)
            want[i, :i + 1] = y
        assert np.array_equal(rs["dQ"][s:e, 0, s:e] / alpha, want), b


def test_one_hot_fold_weights():
    """The forward's per-key fold (FLAMIA sec. 4): with V_j = e_j and the
    per-key view Vkey_j = 2^ev_j e_j, O_i[j] reads the weight on key j's
    codes over the row's total weight W_i: E4M3(2^4 p_ij) 2^-4 before query
    i's own 128-token tile; on it, y_j = 2^4 p_ij 2^ev_j rounded per 32 keys
    from the document start by the MX rule, weight y_j 2^-4 on the codes and
    y_j 2^-4 2^-ev_j in W_i."""
    lens = [5, 290]
    T, H, d = sum(lens), 1, sum(lens)
    cu = _cu(lens)
    alpha = 0.125
    Qs, Ks = _rand((T, H, d), 750, 0.6), _rand((T, H, d), 751, 0.6)
    ev = np.random.default_rng(6).integers(-4, 5, (T, H))
    eye = np.eye(T).reshape(T, 1, T)
    vkey = eye * np.exp2(ev)[:, :, None]
    O, _ = orc.attn_fwd_alg1(Qs, Ks, eye, cu, True, alpha, rnd=orc.RND_P, Vkey=vkey,
                             vkey_sf=(ev + 127).astype(np.uint8))
    for b in range(len(lens)):
        s, e = cu[b], cu[b + 1]
        raw = Qs[s:e, 0] @ Ks[s:e, 0].T
        for i in range(e - s):
            p16, m = _boosted_weights(raw[i, :i + 1], alpha)
            p16 = p16 * np.exp2(m - m[-1])  # the frame of the last reference
            t0 = (i // 128) * 128
            w = orc.e4m3_round_array(p16[:t0] / np.exp2(m[:t0] - m[-1])) * np.exp2(m[:t0] - m[-1]) / 16
            y = p16[t0:] * np.exp2(ev[s + t0:s + i + 1, 0])
            for g in range(0, len(y), 32):
                ex = orc.mx_exponent(float(np.abs(y[g:g + 32]).max()))
                y[g:g + 32] = np.ldexp(orc.e4m3_round_array(np.ldexp(y[g:g + 32], -ex)), ex)
            wc = y / 16
            W = w.sum() + (wc * np.exp2(-ev[s + t0:s + i + 1, 0])).sum()
            want = np.concatenate([w, wc]) / W
            np.testing.assert_allclose(O[s + i, 0, s:s + i + 1], want, rtol=1e-15, atol=0, err_msg=str((b, i)))


# ------------------------------------------------------------------ view routing

DEPENDS = {  # output -> the views it may depend on (beyond the score views Qs, Ks)
    "O": {"Vo"},
    "D": {"Vo", "Gr"},
    "dV": {"Gt"},
    "dK": {"Vo", "Vr", "Gr", "Qt"},
    "dQ": {"Vo", "Vr", "Gr", "Kt"},
}
LINEAR = {"dV": "Gt", "dK": "Qt", "dQ": "Kt", "O": "Vo"}
NAMES = ["Qs", "Ks", "Vo", "Vr", "Gr", "Qt", "Kt", "Gt"]


@pytest.mark.parametrize("fn", ["direct", "alg1"])
def test_each_output_reads_exactly_its_views(fn):
    """dV = P^T Gt, dK = alpha U^T Qt, dQ = alpha U Kt, U = P (Gr Vr^T - D),
    D = Gr . O, O = P Vo: replacing any other view leaves an output's bits
    unchanged; replacing a view it names moves it; doubling the linear
    factor doubles it exactly.  A swapped operand in any product fails."""
    lens, Hq, Hkv, d = [50, 21], 2, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    views = dict(zip(NAMES, _views(T, Hq, Hkv, d, 800)))

    def run(**kw):
        v = dict(views, **kw)
        a = [v[k] for k in NAMES]
        if fn == "direct":
            return orc.attn_bwd(*a, cu, True)
        return orc.attn_bwd_alg1(*a, cu, True)

    base = run()
    for i, nm in enumerate(NAMES[2:]):
        alt = run(**{nm: _rand(views[nm].shape, 900 + i)})
        for out, deps in DEPENDS.items():
            same = np.array_equal(alt[out], base[out])
            assert same == (nm not in deps), (out, nm)
    for out, nm in LINEAR.items():
        dbl = run(**{nm: 2 * views[nm]})
        assert np.array_equal(dbl[out], 2 * base[out]), (out, nm)


def test_direct_routing_matches_torch_with_distinct_views():
    """The direct backward with eight distinct views against the same
    products formed with torch matmuls (no shared code with the oracle)."""
    lens, Hq, Hkv, d = [40, 23], 2, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 1000)
    alpha = 1 / math.sqrt(d)
    r = orc.attn_bwd(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, False, alpha)
    t = lambda a: torch.from_numpy(a)
    dK = torch.zeros(T, Hkv, d, dtype=torch.float64)
    dV = torch.zeros_like(dK)
    for b in range(len(lens)):
        s, e = int(cu[b]), int(cu[b + 1])
        for h in range(Hq):
            P = torch.softmax(alpha * t(Qs[s:e, h]) @ t(Ks[s:e, 0]).T, -1)
            O = P @ t(Vo[s:e, 0])
            D = (t(Gr[s:e, h]) * O).sum(-1, keepdim=True)
            U = P * (t(Gr[s:e, h]) @ t(Vr[s:e, 0]).T - D)
            np.testing.assert_allclose(r["O"][s:e, h], O.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["dQ"][s:e, h], (alpha * U @ t(Kt[s:e, 0])).numpy(), rtol=0, atol=1e-12)
            dK[s:e, 0] += alpha * U.T @ t(Qt[s:e, h])
            dV[s:e, 0] += P.T @ t(Gt[s:e, h])
    np.testing.assert_allclose(r["dK"], dK.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dV"], dV.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------- which rows a change moves

def test_documents_isolated_and_forward_causal():
    lens, Hq, Hkv, d = [60, 90], 2, 2, 32
    T = sum(lens)
    cu = _cu(lens)
    views = _views(T, Hq, Hkv, d, 1100)
    base = orc.attn_bwd_alg1(*views, cu, True)
    p = 60 + 50
    pert = [v.copy() for v in views]
    for v in pert:
        v[p] += 3.0
    alt = orc.attn_bwd_alg1(*pert, cu, True)
    for k in ("O", "dQ"):
        assert np.array_equal(alt[k][:60], base[k][:60]), k  # the other document
    assert np.array_equal(alt["dK"][:60], base["dK"][:60]) and np.array_equal(alt["dV"][:60], base["dV"][:60])
    assert np.array_equal(alt["O"][:p], base["O"][:p])  # earlier rows of the same document
    assert np.array_equal(alt["LSE"][:, :p], base["LSE"][:, :p])


def test_dq_prefix_blocks_and_the_strict_operand():
    """Changing query p's incoming gradient (and its score and value views
    after p) leaves dQ of every row in the 32-query blocks before p's block
    bit-identical.  Rows of p's own block before p can move through the block
    scale (the residual the FLAMIA notes concede in sec. 4); with the strict
    operand (per-query scales) none of the rows before p moves."""
    lens, Hq, Hkv, d = [9, 200], 1, 1, 32
    T = sum(lens)
    cu = _cu(lens)
    Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt = _views(T, Hq, Hkv, d, 1200)
    ksf = (127 + np.random.default_rng(3).integers(-3, 4, (T, Hkv))).astype(np.uint8)
    Kkey = _rand((T, Hkv, d), 1300)
    p = 9 + 32 * 3 + 20  # row 20 of the document's fourth 32-query block
    Gr2, Gt2 = Gr.copy(), Gt.copy()
    Gr2[p] *= 4096.0
    Gt2[p] *= 4096.0
    for strict in (False, True):
        kw = dict(Kkey=Kkey, kkey_sf=ksf) if strict else {}
        a = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt, cu, True, **kw)
        b = orc.attn_bwd_alg1(Qs, Ks, Vo, Vr, Gr2, Qt, Kt, Gt2, cu, True, **kw)
        blk0 = 9 + 32 * 3
        assert np.array_equal(a["dQ"][:blk0], b["dQ"][:blk0]), strict
        same_in_block = np.array_equal(a["dQ"][blk0:p], b["dQ"][blk0:p])
        assert same_in_block == strict, strict
