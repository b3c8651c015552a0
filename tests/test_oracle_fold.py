"""Pins of the oracle's per-key view and folded causal forward (FLAMIA
reading notes sec. 4, moving the scale across the boundary: on the diagonal
tile each key's value row carries its own power-of-two scale).

CPU only.  The per-key view is checked against two other pinned quantizers
it must reduce to -- the row view when d = 32 (one group per token) and the
token-block view on one-token documents (one block per token) -- and against
the scale-doubling property of E4M3 (FLAMIA sec. 4); the folded forward
against the plain causal forward when both value views coincide, against a
per-row evaluation that names each key's value row directly, and for the
property it exists for: rows keep their output when later keys of their own
32-token block change.
"""
import math

import numpy as np
import torch

from oracle import oracle as orc


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)


def test_key_view_is_the_row_view_at_d32():
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((50, 3, 32)) * np.exp(rng.uniform(-8, 8, (50, 3, 1))))
    kc, ks = orc.quant_key(x)
    rc, rs = orc.quant_row(x)
    assert np.array_equal(kc, rc) and np.array_equal(ks, rs[:, :, 0])


def test_key_view_is_the_token_block_view_of_one_token_documents():
    rng = np.random.default_rng(2)
    T, H, d = 40, 2, 128
    x = _bf16(rng.standard_normal((T, H, d)) * np.exp(rng.uniform(-6, 6, (T, H, 1))))
    x[5] = 0  # all-zero vectors: scale byte 127 (exponent 0), codes 0
    cu = np.arange(T + 1, dtype=np.int32)
    bc, bs = orc.quant_tokblock(x, cu)
    kc, ks = orc.quant_key(x)
    assert np.array_equal(kc, bc)
    # the block layout's one scale per (head, block) -- [H, NB], NB = T here --
    # is the per-token scale
    assert bs.shape == (H, T) and np.array_equal(ks, bs.T)
    assert (ks[5] == 127).all() and (kc[5] == 0).all()


def test_key_view_scale_doubling():
    # FLAMIA sec. 4: doubling a normal-range vector raises its exponent by one
    # and leaves the codes unchanged
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 2, 64))
    c1, s1 = orc.quant_key(_bf16(x))
    c2, s2 = orc.quant_key(_bf16(2 * x))
    assert np.array_equal(c1, c2) and np.array_equal(s2.astype(int), s1.astype(int) + 1)
    v = orc.dequant_key(c1, s1)
    assert np.abs(v - _bf16(x).double().numpy()).max() <= np.abs(x).max() / 16


def test_fold_with_equal_views_is_the_causal_forward():
    rng = np.random.default_rng(4)
    lens = [300, 17, 129]
    T = sum(lens)
    cu = np.array(np.concatenate([[0], np.cumsum(lens)]), np.int32)
    Q, K, V = rng.standard_normal((T, 4, 64)), rng.standard_normal((T, 2, 64)), rng.standard_normal((T, 2, 64))
    O1, L1 = orc.attn_fwd_fold(Q, K, V, V, cu)
    O2, L2 = orc.attn_fwd(Q, K, V, cu, True)
    assert np.abs(O1 - O2).max() < 1e-12 and np.abs(L1 - L2).max() < 1e-12


def test_fold_uses_the_key_view_exactly_on_the_diagonal_tile():
    # one document of 300 tokens: query i's diagonal tile starts at 128 (i // 128)
    rng = np.random.default_rng(5)
    T, d = 300, 32
    Q, K = rng.standard_normal((T, 1, d)), rng.standard_normal((T, 1, d))
    Vt, Vk = rng.standard_normal((T, 1, d)), rng.standard_normal((T, 1, d))
    O, L = orc.attn_fwd_fold(Q, K, Vt, Vk, None)
    alpha = 1.0 / math.sqrt(d)
    for i in (0, 1, 127, 128, 129, 255, 256, 299):
        s = alpha * (K[: i + 1, 0] @ Q[i, 0])
        p = np.exp(s - s.max())
        t0 = (i // 128) * 128
        V = np.concatenate([Vt[:t0, 0], Vk[t0: i + 1, 0]])
        assert np.abs(O[i, 0] - (p @ V) / p.sum()).max() < 1e-12
        assert abs(L[0, i] - (s.max() + math.log(p.sum()))) < 1e-12


def test_fold_rows_ignore_later_keys_of_their_block():
    """With the per-key view on the diagonal tile, changing keys and values
    after position p (inside p's 32-token block) leaves rows <= p unchanged;
    the token view alone would not (its scale groups straddle p)."""
    rng = np.random.default_rng(6)
    T, H, d = 160, 1, 64
    x = {k: rng.standard_normal((T, H, d)) for k in "qkv"}
    cu = np.array([0, T], np.int32)
    p = 140  # block [128, 160)
    x2 = {k: v.copy() for k, v in x.items()}
    for k in "kv":
        x2[k][p + 1:] *= 300.0

    def run(xx, fold):
        q = orc.dequant_row(*orc.quant_row(_bf16(xx["q"])))
        k = orc.dequant_row(*orc.quant_row(_bf16(xx["k"])))
        vt = orc.dequant_tok(*orc.quant_tok(_bf16(xx["v"]), cu), cu)
        vk = orc.dequant_key(*orc.quant_key(_bf16(xx["v"]))) if fold else vt
        return orc.attn_fwd_fold(q, k, vt, vk, cu)[0]

    a, b = run(x, True), run(x2, True)
    assert np.array_equal(a[: p + 1], b[: p + 1])
    a, b = run(x, False), run(x2, False)
    assert not np.array_equal(a[128: p + 1], b[128: p + 1])
    assert np.array_equal(a[:128], b[:128])


def test_backward_fold_with_equal_views_is_the_causal_backward():
    rng = np.random.default_rng(7)
    lens = [260, 40, 130]
    T = sum(lens)
    cu = np.array(np.concatenate([[0], np.cumsum(lens)]), np.int32)
    Q, G = rng.standard_normal((T, 4, 32)), rng.standard_normal((T, 4, 32))
    K, V = rng.standard_normal((T, 2, 32)), rng.standard_normal((T, 2, 32))
    a = orc.attn_bwd_fold(Q, K, V, V, G, Q, K, G, V, K, cu)
    b = orc.attn_bwd(Q, K, V, V, G, Q, K, G, cu, True)
    for k in ("dQ", "dK", "dV", "O", "LSE", "D"):
        assert np.abs(a[k] - b[k]).max() < 1e-10, k


def test_backward_fold_uses_the_key_views_exactly_on_the_diagonal_tile():
    # dQ_i = alpha sum_j U_ij Khat_j with Khat_j = Kkey_j on i's own 128-token
    # tile and Kt_j before it; O_i takes Vkey the same way, and D = G . O
    rng = np.random.default_rng(8)
    T, d = 300, 32
    Q, K, G = (rng.standard_normal((T, 1, d)) for _ in range(3))
    Vt, Vk, Vr, Kt, Kk = (rng.standard_normal((T, 1, d)) for _ in range(5))
    r = orc.attn_bwd_fold(Q, K, Vt, Vr, G, Q, Kt, G, Vk, Kk, None)
    alpha = 1.0 / math.sqrt(d)
    for i in (0, 5, 127, 128, 200, 255, 256, 299):
        s = alpha * (K[: i + 1, 0] @ Q[i, 0])
        p = np.exp(s - s.max())
        P = p / p.sum()
        t0 = (i // 128) * 128
        V = np.concatenate([Vt[:t0, 0], Vk[t0: i + 1, 0]])
        O = P @ V
        Di = G[i, 0] @ O
        U = P * (Vr[: i + 1, 0] @ G[i, 0] - Di)
        Kh = np.concatenate([Kt[:t0, 0], Kk[t0: i + 1, 0]])
        assert np.abs(r["O"][i, 0] - O).max() < 1e-12
        assert abs(r["D"][0, i] - Di) < 1e-12
        assert np.abs(r["dQ"][i, 0] - alpha * U @ Kh).max() < 1e-12
