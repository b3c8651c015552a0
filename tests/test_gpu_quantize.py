"""GPU quantizer vs the oracle: codes and scales bit-exact (every view)."""
import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import gpu_views, oracle_views

pytestmark = pytest.mark.gpu

CASES = [
    inp.workload("tiny"),
    inp.make_custom("ragged_d128", lengths=[1, 31, 32, 33, 127, 128, 129, 300], Hq=3, Hkv=3, d=128, seed=11,
                    outlier_channels=2, outlier_gain=50.0),
    inp.make_custom("ragged_d64", lengths=[17, 200, 64, 5], Hq=2, Hkv=2, d=64, seed=12),
    inp.make_custom("tokblock_had", lengths=[70, 3, 300, 32], Hq=4, Hkv=4, d=128, mode="tokblock", hadamard=True,
                    seed=13, outlier_channels=2, outlier_gain=50.0),
    inp.make_custom("tokblock_d64", lengths=[40, 90], Hq=2, Hkv=2, d=64, mode="tokblock", seed=14),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_quantize_bit_exact(w):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=False)
    geo, gv = gpu_views(w, t, names=("q",))
    torch.cuda.synchronize()
    mxa.check_error()
    ov, _ = oracle_views(w, t, names=("q",))
    row, tok = gv["q"]
    lens = w.doc_lengths
    if w.mode == "tokblock":
        c, s = ov["q"]["blk"]
        assert np.array_equal(row.codes.cpu().numpy(), c)
        assert tok.codes.data_ptr() == row.codes.data_ptr()
        # both layouts carry the block exponent
        rs = mxa.row_scales_logical(row.scales, lens, w.d)  # [T, H, G]
        ts = mxa.tok_scales_logical(tok.scales, lens, w.d)  # [H, d, NB]
        nb = np.concatenate([orc.block_offset(w.cu_seqlens.numpy(), w.T, b) + np.arange(n) // 32
                             for b, n in enumerate(lens)])  # global 32-token block of every token
        assert np.array_equal(rs, np.broadcast_to(s.T[nb][:, :, None], rs.shape))
        assert np.array_equal(ts, np.broadcast_to(s[:, None, :], ts.shape))
    else:
        rc, rsl = ov["q"]["row"]
        tc, tsl = ov["q"]["tok"]
        assert np.array_equal(row.codes.cpu().numpy(), rc)
        assert np.array_equal(mxa.row_scales_logical(row.scales, lens, w.d), rsl)
        assert np.array_equal(tok.codes.cpu().numpy(), tc)
        assert np.array_equal(mxa.tok_scales_logical(tok.scales, lens, w.d), tsl)


def test_quantize_padding_and_edge_values():
    """Exact powers of two at the 448 boundary, zeros, tiny values, negatives:
    the device scale rule and RNE/satfinite conversion match the oracle."""
    from block_scaled_mxfp8_gb300 import mxa

    T, H, d = 128, 1, 128
    vals = torch.tensor([448.0, 450.0, 480.0, 1.0, 1.75, 1.7578125, -2.0 ** -9, 2.0 ** -126, 3e38, -3e38, 0.0,
                         -0.0, 2.0 ** -133, 1e-30, 65504.0, 0.1], dtype=torch.float32)
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(T, H, d, generator=g) * 3).to(torch.bfloat16)
    x[0, 0, :16] = vals.to(torch.bfloat16)
    x[1, 0, :32] = 0.0                      # all-zero row group -> exponent 0
    x[2, 0, :] = 2.0 ** -130                # subnormal bf16 everywhere
    x[3:35, 0, 5] = 0.0                     # all-zero token group of channel 5
    x[40, 0, 7] = 448.0 * 2 ** 20           # huge outlier
    geo = mxa.Geometry.batched(1, T)
    row, tok = mxa.quantize(x.cuda(), geo)
    torch.cuda.synchronize()
    rc, rs = orc.quant_row(x)
    tc, ts = orc.quant_tok(x)
    assert np.array_equal(row.codes.cpu().numpy(), rc)
    assert np.array_equal(mxa.row_scales_logical(row.scales, [T], d), rs)
    assert np.array_equal(tok.codes.cpu().numpy(), tc)
    assert np.array_equal(mxa.tok_scales_logical(tok.scales, [T], d), ts)
    # unused atom bytes hold 0x7F (d=128 uses all 4 groups; pad rows beyond T do not exist here)
    assert int(row.scales.cpu()[0, 0, mxa.atom_index(1, 0)]) == 127


def _atom_images(rs, ts, lens, H, d, NT):
    """The full [H, NT, 512] scale layouts expected from the logical scales:
    every byte 0x7F except the (row, group) cells the layout documents
    (include/mxa.h: row r, group g at (r % 32) * 16 + (r / 32) * 4 + g)."""
    from block_scaled_mxfp8_gb300 import mxa

    row = np.full((H, NT, 512), 0x7F, np.uint8)
    tok = np.full((H, NT, 512), 0x7F, np.uint8)
    t0 = tb = nb = 0
    for n in lens:
        for t in range(n):
            for g in range(d // 32):
                row[:, tb + t // 128, mxa.atom_index(t % 128, g)] = rs[t0 + t, :, g]
        for blk in range((n + 31) // 32):
            for c in range(d):
                tok[:, tb + blk // 4, mxa.atom_index(c, blk % 4)] = ts[:, c, nb + blk]
        t0 += n
        tb += (n + 127) // 128
        nb += (n + 31) // 32
    return row, tok


@pytest.mark.parametrize("case", [("batched_d64", None, 2, 200, 64), ("batched_d128", None, 3, 130, 128),
                                  ("packed_d64", [1, 129, 40], 0, 0, 64)], ids=lambda c: c[0])
def test_every_scale_byte_is_written(case):
    """Scale buffers pre-filled with two different patterns come out
    identical and equal, byte for byte, to the documented atom image (logical
    scales from the oracle, 0x7F in every unused byte): the call writes every
    byte of both layouts, whether its kernel fills the padding itself (equal
    documents) or the layouts are filled first (packed documents)."""
    from block_scaled_mxfp8_gb300 import mxa

    name, lens, B, L, d = case
    H = 3
    w = (inp.make_custom(name, lengths=lens, Hq=H, Hkv=H, d=d, seed=15) if lens
         else inp.make_custom(name, B=B, L=L, Hq=H, Hkv=H, d=d, seed=15))
    t = inp.tensors(w, with_grad=False)
    geo, _ = gpu_views(w, t, names=())
    x = t["q"].cuda().contiguous()
    outs = []
    for fill in (0x00, 0xAB):
        mk = lambda: mxa.QView(torch.zeros((w.T, H, d), dtype=torch.uint8, device="cuda"),
                               torch.full((H, geo.ntiles, 512), fill, dtype=torch.uint8, device="cuda"))
        row, tok = mxa.quantize(x, geo, out=(mk(), mk()))
        torch.cuda.synchronize()
        outs.append((row.scales.cpu().numpy(), tok.scales.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    cu = w.cu_seqlens.numpy()
    _, rs = orc.quant_row(t["q"])
    _, ts = orc.quant_tok(t["q"], cu)
    want_row, want_tok = _atom_images(rs, ts, w.doc_lengths, H, d, geo.ntiles)
    assert np.array_equal(outs[0][0], want_row)
    assert np.array_equal(outs[0][1], want_tok)
