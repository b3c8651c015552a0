"""Pins of the oracle's formats and quantizers against what the pages fix.

CPU only.  Every check compares the oracle with something other than itself:
values the pages print (tests/golden/pages_examples.json), hand-worked codes,
torch's own float8_e4m3fn cast (a library routine), an fp64 log2 restatement
of the scale rule, a matrix Hadamard, and invariants stated on the pages.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def test_e4m3_hand_values():
    for y, code in GOLD["e4m3_hand_values"]["cases"]:
        assert orc.e4m3_encode(y) == code, (y, hex(orc.e4m3_encode(y)), hex(code))


def test_e4m3_decode_table_structure():
    t = orc.e4m3_table()
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6
    fin = t[:0x7F]
    assert np.all(np.diff(fin) > 0), "positive codes must be strictly increasing"
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F]), "sign bit only flips the sign"


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = orc.e4m3_table()
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~fin)
    assert np.array_equal(ours[fin], ref[fin])


def test_e4m3_encode_exhaustive_bf16_vs_torch():
    """All 65,536 bf16 patterns times 2^-e for e in [-20, 20], against torch's
    RNE float8_e4m3fn cast wherever |y| <= 448 (torch does not saturate)."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    base = bits.to(torch.float64)
    ys = []
    for e in range(-20, 21):
        ys.append(base * 2.0 ** (-e))
    y = torch.cat(ys)
    ok = torch.isfinite(y) & (y.abs() <= 448.0)
    y = y[ok]
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = orc.e4m3_encode_array(y.numpy())
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(y[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_saturates_above_448():
    for y in (448.5, 460.0, 464.0, 480.0, 1e6):
        assert orc.e4m3_encode(y) == 0x7E
        assert orc.e4m3_encode(-y) == 0xFE


def test_scale_exponent_hand_values():
    for amax, e in GOLD["scale_exponents"]["cases"]:
        assert orc.mx_exponent(amax) == e, (amax, orc.mx_exponent(amax), e)


def test_scale_rule_480_example():
    g = GOLD["scale_rule_480"]
    e = orc.mx_exponent(g["amax"])
    assert e == g["exponent"]
    c = orc.e4m3_encode(g["amax"] / 2.0 ** e)
    assert c == g["code_of_480"]
    assert orc.e4m3_decode(c) * 2.0 ** e == g["decoded"]
    # the floor rule of the pages' counter-argument saturates instead
    ef = math.floor(math.log2(g["amax"] / 448.0))
    assert ef == g["floor_rule_exponent"]
    assert orc.e4m3_decode(orc.e4m3_encode(g["amax"] / 2.0 ** ef)) * 2.0 ** ef == g["floor_rule_decoded"]


def test_scale_exponent_vs_float_log2_rule():
    """ceil(log2(amax/448)) in fp64 (the pages' formula, and the demo quantizer's)
    agrees with the oracle's exact search away from exact powers of two."""
    rng = np.random.default_rng(0)
    amax = np.abs(rng.standard_normal(20000)) * 2.0 ** rng.integers(-30, 30, 20000)
    for a in amax:
        if a == 0:
            continue
        want = math.ceil(math.log2(a / 448.0))
        assert orc.mx_exponent(a) == want, a
    # and exactly at the boundary 448 * 2^k
    for k in range(-20, 21):
        assert orc.mx_exponent(448.0 * 2.0 ** k) == k
        assert orc.mx_exponent(np.nextafter(448.0 * 2.0 ** k, np.inf)) == k + 1


def test_scale_never_saturates_group_max():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        a = float(np.abs(rng.standard_normal()) * 2.0 ** rng.integers(-40, 40))
        e = orc.mx_exponent(a)
        assert a / 2.0 ** e <= 448.0 and a / 2.0 ** (e - 1) > 448.0


def test_scale_doubling_invariance_normal_range():
    """FLAMIA sec. 4: in the normal range the reconstruction is unchanged when
    the scale doubles; it fails at the smallest subnormal 2^-9."""
    rng = np.random.default_rng(2)
    for _ in range(5000):
        s = 2.0 ** int(rng.integers(-10, 10))
        r = float(2.0 ** rng.uniform(-5, math.log2(448.0)))
        y = r * s * (1 if rng.random() < 0.5 else -1)
        a = orc.e4m3_decode(orc.e4m3_encode(y / s)) * s
        b = orc.e4m3_decode(orc.e4m3_encode(y / (2 * s))) * 2 * s
        assert a == b, (y, s)
    ms = GOLD["subnormal_doubling"]["min_subnormal"]
    s = 1.0
    a = orc.e4m3_decode(orc.e4m3_encode(ms)) * s
    b = orc.e4m3_decode(orc.e4m3_encode(ms / 2)) * 2 * s
    assert a == ms and b == 0.0


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def test_quant_row_matches_definition():
    """Row view against the definition restated with torch ops: e from the
    fp64 log2 rule, codes from torch's fp8 cast (values here stay <= 448)."""
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(37, 3, 64, generator=g) * 3).to(torch.bfloat16)
    x[5, 1, 0:32] = 0.0  # all-zero group
    codes, scales = orc.quant_row(x)
    xd = x.to(torch.float64).view(37, 3, 2, 32)
    amax = xd.abs().amax(-1)
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / 448.0)), torch.zeros_like(amax))
    assert np.array_equal(scales.astype(np.int64) - 127, e.numpy().astype(np.int64))
    y = (xd / torch.pow(2.0, e)[..., None]).reshape(37, 3, 64)
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    assert scales[5, 1, 0] == 127


def test_quant_tok_groups_are_doc_relative():
    g = torch.Generator().manual_seed(4)
    lens = [5, 40, 64, 1, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    x = torch.randn(T, 2, 32, generator=g).to(torch.bfloat16)
    codes, scales = orc.quant_tok(x, cu)
    assert scales.shape == (2, 32, sum((n + 31) // 32 for n in lens))
    xd = x.to(torch.float64)
    for b, n in enumerate(lens):
        s = int(cu[b])
        off = orc.block_offset(cu, T, b)
        for kb in range((n + 31) // 32):
            t0, t1 = s + 32 * kb, min(s + 32 * kb + 32, s + n)
            amax = xd[t0:t1].abs().amax(0)  # [H, d]
            e = torch.ceil(torch.log2(amax / 448.0))
            assert np.array_equal(scales[:, :, off + kb].astype(np.int64) - 127, e.numpy().astype(np.int64))
            ref = (xd[t0:t1] / torch.pow(2.0, e)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(codes[t0:t1], ref)


def test_dequant_is_exact_product():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(64, 2, 64, generator=g).to(torch.bfloat16)
    codes, scales = orc.quant_row(x)
    dq = orc.dequant_row(codes, scales)
    t = orc.e4m3_table()
    want = t[codes] * np.repeat(2.0 ** (scales.astype(np.float64) - 127), 32, axis=-1)
    assert np.array_equal(dq, want)
    # relative error of a normal-range code is at most 2^-4
    xd = x.to(torch.float64).numpy()
    big = np.abs(xd) > np.repeat(np.abs(xd).reshape(64, 2, 2, 32).max(-1), 32, -1) * 2.0 ** -6
    assert np.all(np.abs(dq - xd)[big] <= np.abs(xd)[big] * 2.0 ** -4 + 1e-300)


def test_hadamard_fp32_vs_matrix_definition():
    """The fp32 butterfly equals the normalized Sylvester matrix product
    within fp32 rounding, and leaves dot products unchanged (FLAMIA sec. 3)."""
    from scipy.linalg import hadamard

    Hm = hadamard(128).astype(np.float64) / math.sqrt(128.0)
    assert np.allclose(Hm @ Hm.T, np.eye(128), atol=1e-12)
    rng = np.random.default_rng(6)
    q = rng.standard_normal(128).astype(np.float32)
    k = rng.standard_normal(128).astype(np.float32)
    hq, hk = orc.hadamard128_f32(q), orc.hadamard128_f32(k)
    want = Hm @ q.astype(np.float64)  # Sylvester H is symmetric, so x H = H x
    assert np.allclose(hq, want, rtol=0, atol=1e-5 * np.abs(q).sum())
    assert abs(float(hq.astype(np.float64) @ hk) - float(q.astype(np.float64) @ k)) < 1e-4 * np.linalg.norm(q) * np.linalg.norm(k)
    # exact (QH)(KH)^T = QK^T with the fp64 matrix
    Q = rng.standard_normal((8, 128))
    K = rng.standard_normal((9, 128))
    assert np.allclose((Q @ Hm) @ (K @ Hm).T, Q @ K.T, atol=1e-12)


def test_tokblock_shares_one_exponent_per_block():
    g = torch.Generator().manual_seed(7)
    lens = [70, 3, 32]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = torch.randn(int(cu[-1]), 2, 128, generator=g).to(torch.bfloat16)
    for had in (False, True):
        codes, scales = orc.quant_tokblock(x, cu, hadamard=had)
        assert scales.shape == (2, 3 + 1 + 1)
        y = x.to(torch.float32).numpy()
        if had:
            y = np.stack([[orc.hadamard128_f32(y[t, h]) for h in range(2)] for t in range(y.shape[0])])
        for b, n in enumerate(lens):
            s = int(cu[b])
            off = orc.block_offset(cu, int(cu[-1]), b)
            for kb in range((n + 31) // 32):
                t0, t1 = s + 32 * kb, min(s + 32 * kb + 32, s + n)
                for h in range(2):
                    amax = float(np.abs(y[t0:t1, h].astype(np.float64)).max())
                    e = math.ceil(math.log2(amax / 448.0))
                    assert int(scales[h, off + kb]) - 127 == e
                    ref = torch.from_numpy(y[t0:t1, h].astype(np.float64) / 2.0 ** e).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    assert np.array_equal(codes[t0:t1, h], ref)


def test_two_value_counterexample():
    for a, out in GOLD["two_value_counterexample"]["cases"]:
        assert orc.shared_scale_prefix_output(a) == out


def test_future_value_leaks_through_shared_group_scale():
    """MXFP8 analogue of the two-value counterexample: in the token view a
    later token in the same 32-token group raises the group's exponent and
    changes the code of token 0, so the causal output of query 0 (which sees
    only key 0) changes; a change in a later group does not."""
    g = torch.Generator().manual_seed(8)
    T, d = 64, 32
    q = torch.randn(T, 1, d, generator=g).to(torch.bfloat16)
    k = torch.randn(T, 1, d, generator=g).to(torch.bfloat16)
    v = torch.randn(T, 1, d, generator=g).to(torch.bfloat16)

    def out0(vv, mode):
        if mode == "tok":
            c, s = orc.quant_tok(vv)
            Vd = orc.dequant_tok(c, s)
        else:
            c, s = orc.quant_tokblock(vv)
            Vd = orc.dequant_tokblock(c, s)
        Qd = q.to(torch.float64).numpy()
        Kd = k.to(torch.float64).numpy()
        O, _ = orc.attn_fwd(Qd, Kd, Vd, causal=True, sel=[[0, 0]])
        return O[0, 0]

    base_tok, base_blk = out0(v, "tok"), out0(v, "blk")
    v2 = v.clone()
    v2[5, 0, :] = 1000.0  # same 32-token group as token 0
    assert not np.array_equal(out0(v2, "tok"), base_tok)
    assert not np.array_equal(out0(v2, "blk"), base_blk)
    v3 = v.clone()
    v3[40, 0, :] = 1000.0  # next group
    assert np.array_equal(out0(v3, "tok"), base_tok)
    assert np.array_equal(out0(v3, "blk"), base_blk)


def test_p_cap_examples():
    g = GOLD["p_cap"]
    assert math.log2(448) == pytest.approx(g["log2_448"], abs=0.005)
    c0, c1 = g["cases"]
    assert orc.p_cap_reconstruction(c0["c"], c0["tau"], c0["tau"]) == c0["reconstructed"]
    assert orc.p_cap_reconstruction(c1["c"], c1["tau"], c1["tau"]) == c1["reconstructed"]
    assert c1["true"] == 2.0 ** c1["tau"]


def test_cosine_hides_small_entries():
    g = GOLD["cosine_small_entries"]
    a = np.concatenate([[1.0], np.full(100, 0.001)])
    b = np.concatenate([[1.0], np.zeros(100)])
    assert orc.cosine(a, b) == pytest.approx(g["cosine"], abs=5e-6)
    assert np.linalg.norm(a - b) / np.linalg.norm(a) == pytest.approx(g["rel_l2"], rel=0.01)


def test_visible_pairs_examples():
    for case in GOLD["visible_pairs"]["cases"]:
        lens = []
        for n, cnt in case["lengths"]:
            lens += [n] * cnt
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        assert orc.visible_pairs(cu, int(cu[-1])) == case["pairs"]
