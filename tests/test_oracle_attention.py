"""Pins of the oracle's attention forward/backward (FLAMIA reading notes, sec. 2).

CPU only.  The oracle's direct attention is checked against: torch's fp64
scaled_dot_product_attention + autograd (a library routine), an online
(tiled) softmax written here from the merge equations, and the identities
the pages state: sum_j P_ij = 1, D = G . O, sum_t U_t = 0, the causal first
query seeing one key.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64).numpy()


def _torch_ref(Q, K, V, G, lens, causal, alpha):
    """fp64 SDPA + autograd per document (GQA via repeat_interleave)."""
    Hq, Hkv = Q.shape[1], K.shape[1]
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    outs, lses = [], []
    s = 0
    for n in lens:
        qq = q[s:s + n].permute(1, 0, 2)
        kk = k[s:s + n].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vv = v[s:s + n].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        outs.append(F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=alpha).permute(1, 0, 2))
        sc = alpha * qq @ kk.transpose(1, 2)
        if causal:
            sc = sc.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
        lses.append(torch.logsumexp(sc, -1))
        s += n
    O = torch.cat(outs, 0)
    (O * torch.tensor(G)).sum().backward()
    return O.detach().numpy(), torch.cat(lses, 1).detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", ["tiny", "jagged_gqa"])
def test_fwd_bwd_match_torch_sdpa_autograd(case, causal):
    if case == "tiny":
        lens, Hq, Hkv, d = [256], 2, 2, 64
    else:
        lens, Hq, Hkv, d = [17, 1, 64, 45], 4, 2, 32
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Q, K, V, G = _rand((T, Hq, d), 1), _rand((T, Hkv, d), 2), _rand((T, Hkv, d), 3), _rand((T, Hq, d), 4)
    alpha = 1.0 / math.sqrt(d)
    O, LSE = orc.attn_fwd(Q, K, V, cu, causal, alpha)
    r = orc.attn_bwd(Q, K, V, V, G, Q, K, G, cu, causal, alpha)
    O_t, L_t, dq_t, dk_t, dv_t = _torch_ref(Q, K, V, G, lens, causal, alpha)
    np.testing.assert_allclose(O, O_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, L_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["O"], O_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dQ"], dq_t, rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dK"], dk_t, rtol=0, atol=1e-11)
    np.testing.assert_allclose(r["dV"], dv_t, rtol=0, atol=1e-11)


def _online_softmax(Q, K, V, alpha, tile, rng):
    """FlashAttention merge (FLAMIA sec. 2 'FlashAttention 留哪些中间量'):
    per row keep m, l, a; on each tile m' = max(m, max S), scale the old
    state by exp(m - m'), add the tile.  Tile boundaries are random."""
    n, d = Q.shape[0], Q.shape[1]
    O = np.zeros_like(Q)
    LSE = np.zeros(n)
    for i in range(n):
        m, l, a = -np.inf, 0.0, np.zeros(d)
        j = 0
        while j < K.shape[0]:
            w = int(rng.integers(1, tile + 1))
            S = alpha * K[j:j + w] @ Q[i]
            m2 = max(m, S.max())
            l = math.exp(m - m2) * l + np.exp(S - m2).sum()
            a = math.exp(m - m2) * a + np.exp(S - m2) @ V[j:j + w]
            m = m2
            j += w
        O[i] = a / l
        LSE[i] = m + math.log(l)
    return O, LSE


def test_online_merge_equals_direct_softmax():
    rng = np.random.default_rng(11)
    Q, K, V = _rand((40, 1, 32), 5), _rand((300, 1, 32), 6) * 3, _rand((300, 1, 32), 7)
    # cross-shaped test: 40 queries over 300 keys, one document each side via sel
    O, LSE = orc.attn_fwd(np.concatenate([Q, np.zeros((260, 1, 32))]), K, V, None, False, 0.2,
                          sel=[[i, 0] for i in range(40)])
    O2, L2 = _online_softmax(Q[:, 0], K[:, 0], V[:, 0], 0.2, 50, rng)
    np.testing.assert_allclose(O[:40, 0], O2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(LSE[0, :40], L2, rtol=1e-13, atol=1e-13)


def test_probabilities_sum_to_one_and_D_is_G_dot_O():
    """sum_j exp(S_ij - LSE_i) = 1; D_i = sum_j P_ij E_ij = G_i . O_i."""
    T, H, d = 96, 1, 32
    Q, K, V, G = _rand((T, H, d), 8), _rand((T, H, d), 9), _rand((T, H, d), 10), _rand((T, H, d), 11)
    for causal in (False, True):
        r = orc.attn_bwd(Q, K, V, V, G, Q, K, G, None, causal, 0.3)
        S = 0.3 * Q[:, 0] @ K[:, 0].T
        if causal:
            S = np.where(np.tril(np.ones((T, T))) > 0, S, -np.inf)
        P = np.exp(S - r["LSE"][0][:, None])
        np.testing.assert_allclose(P.sum(1), 1.0, rtol=0, atol=1e-13)
        E = G[:, 0] @ V[:, 0].T
        np.testing.assert_allclose((P * E).sum(1), r["D"][0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose((G[:, 0] * r["O"][:, 0]).sum(1), r["D"][0], rtol=1e-12, atol=1e-12)


def test_softmax_gradient_rows_sum_to_zero():
    """sum_t U_t = 0 (FLAMIA sec. 2): dQ is unchanged when every key of the dQ
    view is shifted by one vector, and the dK of a document sums to zero."""
    lens = [50, 30]
    cu = np.array([0, 50, 80], np.int32)
    T, H, d = 80, 2, 32
    Q, K, V, G = _rand((T, H, d), 12), _rand((T, H, d), 13), _rand((T, H, d), 14), _rand((T, H, d), 15)
    for causal in (False, True):
        r0 = orc.attn_bwd(Q, K, V, V, G, Q, K, G, cu, causal, 0.25)
        shift = _rand((1, H, d), 16) * 5
        r1 = orc.attn_bwd(Q, K, V, V, G, Q, K + shift, G, cu, causal, 0.25)
        np.testing.assert_allclose(r1["dQ"], r0["dQ"], rtol=0, atol=1e-11)
        s = 0
        for n in lens:
            np.testing.assert_allclose(r0["dK"][s:s + n].sum(0), 0.0, atol=1e-11)
            s += n


def test_causal_first_query_sees_one_key():
    lens = [7, 33, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, d = sum(lens), 32
    Q, K, V = _rand((T, 2, d), 17), _rand((T, 2, d), 18), _rand((T, 2, d), 19)
    O, LSE = orc.attn_fwd(Q, K, V, cu, True, 0.5)
    for s in cu[:-1]:
        np.testing.assert_array_equal(O[s], V[s])
        for h in range(2):
            assert LSE[h, s] == pytest.approx(0.5 * Q[s, h] @ K[s, h], abs=1e-14)


def test_documents_are_isolated():
    """Changing every token of one document leaves the others' outputs and
    gradients bit-identical (packed rows, FLAMIA sec. 6)."""
    lens = [20, 40, 12]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, d = sum(lens), 1, 32
    A = [_rand((T, H, d), s) for s in (20, 21, 22, 23)]
    B = [a.copy() for a in A]
    for b in B:
        b[20:60] = _rand((40, H, d), 99)
    ra = orc.attn_bwd(A[0], A[1], A[2], A[2], A[3], A[0], A[1], A[3], cu, True, 0.3)
    rb = orc.attn_bwd(B[0], B[1], B[2], B[2], B[3], B[0], B[1], B[3], cu, True, 0.3)
    for key in ("O", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(ra[key][:20], rb[key][:20])
        np.testing.assert_array_equal(ra[key][60:], rb[key][60:])


def test_prefix_invariance_of_O_and_dQ_not_dK():
    """FLAMIA sec. 4 (end): with G fixed, O and dQ of earlier queries do not
    depend on later tokens; dK/dV of a key legitimately do."""
    T, H, d = 64, 1, 32
    Q, K, V, G = (_rand((T, H, d), s) for s in (30, 31, 32, 33))
    K2, V2, Q2 = K.copy(), V.copy(), Q.copy()
    K2[40:] += 3.0
    V2[40:] -= 2.0
    Q2[40:] *= 2.0
    r1 = orc.attn_bwd(Q, K, V, V, G, Q, K, G, None, True, 0.3)
    r2 = orc.attn_bwd(Q2, K2, V2, V2, G, Q2, K2, G, None, True, 0.3)
    np.testing.assert_array_equal(r1["O"][:40], r2["O"][:40])
    np.testing.assert_array_equal(r1["dQ"][:40], r2["dQ"][:40])
    assert not np.allclose(r1["dK"][:40], r2["dK"][:40])


def _torch_cross_ref(Q, K, V, G, lq, lk, alpha):
    """fp64 SDPA + autograd per document with Lq != Lk (no mask)."""
    Hq, Hkv = Q.shape[1], K.shape[1]
    q = torch.tensor(Q, requires_grad=True)
    k = torch.tensor(K, requires_grad=True)
    v = torch.tensor(V, requires_grad=True)
    outs, lses = [], []
    sq = sk = 0
    for nq, nk in zip(lq, lk):
        qq = q[sq:sq + nq].permute(1, 0, 2)
        kk = k[sk:sk + nk].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vv = v[sk:sk + nk].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        outs.append(F.scaled_dot_product_attention(qq, kk, vv, scale=alpha).permute(1, 0, 2))
        lses.append(torch.logsumexp(alpha * qq @ kk.transpose(1, 2), -1))
        sq, sk = sq + nq, sk + nk
    O = torch.cat(outs, 0)
    O.backward(torch.tensor(G))
    return O.detach().numpy(), torch.cat(lses, 1).detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def test_cross_attention_matches_torch_sdpa_autograd():
    """Cross-attention oracle (queries and keys of a document have their own
    lengths) against torch's fp64 SDPA + autograd, GQA 4/2, d = 16."""
    lq, lk = [5, 1, 12, 7], [9, 30, 1, 16]
    Tq, Tk, Hq, Hkv, d = sum(lq), sum(lk), 4, 2, 16
    Q, G = _rand((Tq, Hq, d), 71), _rand((Tq, Hq, d), 72)
    K, V = _rand((Tk, Hkv, d), 73), _rand((Tk, Hkv, d), 74)
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    alpha = 1.0 / math.sqrt(d)
    O, LSE = orc.attn_fwd_x(Q, K, V, cq, ck, alpha)
    r = orc.attn_bwd_x(Q, K, V, V, G, Q, K, G, cq, ck, alpha)
    Ot, Lt, dQt, dKt, dVt = _torch_cross_ref(Q, K, V, G, lq, lk, alpha)
    for name, a, b in (("O", O, Ot), ("LSE", LSE, Lt), ("bwd O", r["O"], Ot), ("bwd LSE", r["LSE"], Lt),
                       ("dQ", r["dQ"], dQt), ("dK", r["dK"], dKt), ("dV", r["dV"], dVt)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12, err_msg=name)


def test_cross_attention_reduces_to_self_attention_and_one_key():
    """With the key side equal to the query side the cross oracle is the
    self-attention oracle; a document with a single key gives O = V of that
    key for every query and LSE = alpha q . k."""
    lens = [6, 11]
    T, Hq, Hkv, d = sum(lens), 2, 1, 8
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Q, K, V = _rand((T, Hq, d), 81), _rand((T, Hkv, d), 82), _rand((T, Hkv, d), 83)
    O1, L1 = orc.attn_fwd_x(Q, K, V, cu, cu)
    O2, L2 = orc.attn_fwd(Q, K, V, cu, False)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    ck = np.array([0, 1, 2], np.int32)
    K1, V1 = K[:2], V[:2]
    O, LSE = orc.attn_fwd_x(Q, K1, V1, cu, ck, 0.5)
    for b in range(2):
        for i in range(cu[b], cu[b + 1]):
            for h in range(Hq):
                np.testing.assert_allclose(O[i, h], V1[b, 0], rtol=1e-15)
                np.testing.assert_allclose(LSE[h, i], 0.5 * Q[i, h] @ K1[b, 0], rtol=1e-13)
