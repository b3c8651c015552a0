"""The quantizers inside the attention kernels, run through the test hooks of
include/mxa_testing.h and compared bit for bit with the oracle codec.

P is rounded to E4M3 with saturation at 448 (FLAMIA notes sec. 5: a P value
above the cap 2^(c+tau) saturates silently); dS takes one UE8M0 scale per
32 x 32 block from the block max-abs, e = ceil(log2(amax / 448)) (the MX rule
of "Что такое MXFP8"), over the register layout of one warp (FA4 write-up,
"Квантование dS без транспонирования").  The boosted form (values carrying
2^8, as in the dK/dV kernel) must give the scale of the unboosted block."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _e4m3_gpu(x: np.ndarray) -> np.ndarray:
    from block_scaled_mxfp8_gb300 import mxa

    xs = np.ascontiguousarray(x, dtype=np.float32)
    pad = (-xs.size) % 4
    xs = np.concatenate([xs, np.zeros(pad, np.float32)])
    xd = torch.from_numpy(xs).cuda()
    cd = torch.empty(xs.size, dtype=torch.uint8, device="cuda")
    st = mxa.mxa_test_e4m3(xd, cd)
    assert st == mxa.MXA_OK, mxa.status_str(st)
    torch.cuda.synchronize()
    return cd.cpu().numpy()[: x.size]


def _codec_inputs() -> np.ndarray:
    tab = orc.e4m3_table()
    finite = np.array([tab[c] for c in range(256) if not np.isnan(tab[c])], np.float64)
    pos = np.unique(np.abs(finite))
    mids = (pos[1:] + pos[:-1]) / 2  # exact ties: round to the even code
    vals = [finite, mids, -mids]
    for m in mids:  # one fp32 ulp either side of every tie
        f = np.float32(m)
        vals.append(np.array([np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(1e9))], np.float64))
    # saturation: 448 < |x|, including the P cap case 2^(8+2) = 1024 -> 448
    vals.append(np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1024.0, 3.0e38, -1024.0, -500.0]))
    # zeros and underflow: below half the smallest subnormal 2^-9 rounds to zero
    vals.append(np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -10 * 1.0001, 1e-30, -1e-30, 1e-45]))
    rng = np.random.default_rng(21)
    r = rng.standard_normal(1 << 18) * np.exp2(rng.uniform(-14, 10, 1 << 18))
    vals.append(r)
    return np.concatenate(vals).astype(np.float32).astype(np.float64)


def test_p_codec_bit_exact():
    x = _codec_inputs()
    got = _e4m3_gpu(x)
    want = orc.e4m3_encode_array(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(x[i], int(got[i]), int(want[i])) for i in bad[:10]]


def test_p_cap_saturates_to_448():
    # (c, tau) = (8, 2): P reaches 2^10 and is stored as 448, i.e. 1.75 after
    # the 2^-8 unboost (the pages' worked example of an over-large cap)
    got = _e4m3_gpu(np.array([1024.0, 256.0, 448.0]))
    assert [orc.e4m3_decode(int(c)) for c in got] == [448.0, 256.0, 448.0]
    assert orc.p_cap_reconstruction(8, 2, 2.0) == 1.75


def _ds_blocks(rng, shift: int) -> np.ndarray:
    blocks = []
    for k in range(-20, 12, 3):  # amax exactly at the boundary 448 * 2^k (e = k)
        b = rng.uniform(-1, 1, (32, 32)) * 448.0 * 2.0 ** k
        b[rng.integers(32), rng.integers(32)] = 448.0 * 2.0 ** k
        blocks.append(b)
        c = b.copy()  # one fp32 ulp above the boundary (e = k + 1)
        c[0, 0] = -float(np.nextafter(np.float32(448.0 * 2.0 ** k), np.float32(np.inf)))
        blocks.append(c)
    for m in (-3, 0, 5):  # fraction exactly 1.75 and just above
        b = rng.uniform(-1, 1, (32, 32)) * 2.0 ** m
        b[5, 7] = 1.75 * 2.0 ** m
        blocks.append(b)
        c = b.copy()
        c[5, 7] = float(np.nextafter(np.float32(1.75 * 2.0 ** m), np.float32(np.inf)))
        blocks.append(c)
    blocks.append(np.zeros((32, 32)))
    one = np.zeros((32, 32))
    one[31, 31] = -3.0
    blocks.append(one)
    blocks.append(rng.standard_normal((32, 32)) * 1e-40)  # fp32 subnormals: e floors at -127
    blocks.append(rng.standard_normal((32, 32)) * 1e-36)
    for _ in range(200):  # dS-like heavy-tailed blocks over a wide range
        b = rng.standard_normal((32, 32)) * rng.exponential(1.0, (32, 1)) * 2.0 ** rng.uniform(-25, 8)
        blocks.append(b)
    x = np.stack(blocks).astype(np.float32)
    return x * np.float32(2.0 ** shift)


def _ds_oracle(x: np.ndarray, shift: int):
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[0], np.uint8)
    for i, b in enumerate(x.astype(np.float64)):
        e = orc.mx_exponent(float(np.abs(b).max()) / 2.0 ** shift)
        scales[i] = e + 127
        codes[i] = orc.e4m3_encode_array(b / 2.0 ** (e + shift))
    return codes, scales


@pytest.mark.parametrize("shift", [0, 8])
def test_ds_block_quant_bit_exact(shift):
    from block_scaled_mxfp8_gb300 import mxa

    x = _ds_blocks(np.random.default_rng(30 + shift), shift)
    xd = torch.from_numpy(x).cuda()
    cd = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    sd = torch.empty(x.shape[0], dtype=torch.uint8, device="cuda")
    st = mxa.mxa_test_ds_blocks(xd, shift, cd, sd)
    assert st == mxa.MXA_OK, mxa.status_str(st)
    torch.cuda.synchronize()
    want_c, want_s = _ds_oracle(x, shift)
    got_s = sd.cpu().numpy()
    bad = np.nonzero(got_s != want_s)[0]
    assert bad.size == 0, [(i, int(got_s[i]), int(want_s[i])) for i in bad[:10]]
    got_c = cd.cpu().numpy()
    assert np.array_equal(got_c, want_c), int((got_c != want_c).sum())


def test_hooks_reject_bad_arguments():
    from block_scaled_mxfp8_gb300 import mxa

    x = torch.zeros(8, device="cuda")
    c = torch.zeros(8, dtype=torch.uint8, device="cuda")
    assert mxa.lib().mxa_test_e4m3(mxa._ptr(x), 6, mxa._ptr(c), None) == mxa.MXA_ERR_ARG
    assert mxa.lib().mxa_test_e4m3(mxa._ptr(x[1:]), 4, mxa._ptr(c), None) == mxa.MXA_ERR_ALIGN
    s = torch.zeros(1, dtype=torch.uint8, device="cuda")
    assert mxa.lib().mxa_test_ds_blocks(mxa._ptr(x), 1, 17, mxa._ptr(c), mxa._ptr(s), None) == mxa.MXA_ERR_ARG
