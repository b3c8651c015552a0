"""GPU fused RMSNorm + quantize vs the oracle (fp32 RMSNorm in the same
written order, then the quantizers on the fp32 values): codes and scales
bit-exact in every view (FA4 write-up, "Fused RMSNorm+Quantize")."""
import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

CASES = [
    # name, workload, weighted, eps
    ("batched_d128", inp.make_custom("rms_b", B=2, L=256, Hq=3, Hkv=3, d=128, seed=31, outlier_channels=2,
                                     outlier_gain=50.0), True, 1e-6),
    ("ragged_d64", inp.make_custom("rms_r", lengths=[17, 200, 64, 5], Hq=2, Hkv=2, d=64, seed=32), False, 1e-5),
    ("tokblock_had", inp.make_custom("rms_t", lengths=[70, 3, 300, 32], Hq=4, Hkv=4, d=128, mode="tokblock",
                                     hadamard=True, seed=33), True, 1e-6),
    ("eps0_zero_rows", inp.make_custom("rms_z", lengths=[40, 90], Hq=2, Hkv=2, d=128, seed=34), True, 0.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rmsnorm_quantize_bit_exact(case):
    from block_scaled_mxfp8_gb300 import mxa

    name, w, weighted, eps = case
    x = inp.tensors(w, with_grad=False)["q"]
    if name == "eps0_zero_rows":
        x[3] = 0.0          # all-zero vectors: y = 0 by the reading
        x[50, 1] = 0.0
    d = w.d
    wt = torch.from_numpy(np.random.default_rng(35).uniform(0.5, 1.5, d).astype(np.float32)) if weighted else None
    geo = mxa.Geometry.batched(w.B, w.L) if w.lengths is None else mxa.Geometry.packed(w.lengths)
    mode = mxa.MXA_SCALE_TOKBLOCK32 if w.mode == "tokblock" else mxa.MXA_SCALE_MX32
    row, tok = mxa.quantize(x.cuda(), geo, mode=mode, hadamard=w.hadamard,
                            rmsnorm=(wt.cuda() if wt is not None else None, eps))
    torch.cuda.synchronize()
    mxa.check_error()
    y = orc.rmsnorm_f32(x, None if wt is None else wt.numpy(), eps)
    cu = w.cu_seqlens.numpy()
    lens = w.doc_lengths
    if w.mode == "tokblock":
        c, s = orc.quant_tokblock_f32(y, cu, hadamard=w.hadamard)
        assert np.array_equal(row.codes.cpu().numpy(), c)
        ts = mxa.tok_scales_logical(tok.scales, lens, d)
        assert np.array_equal(ts, np.broadcast_to(s[:, None, :], ts.shape))
    else:
        rc, rs = orc.quant_row_f32(y)
        tc, ts = orc.quant_tok_f32(y, cu)
        assert np.array_equal(row.codes.cpu().numpy(), rc)
        assert np.array_equal(mxa.row_scales_logical(row.scales, lens, d), rs)
        assert np.array_equal(tok.codes.cpu().numpy(), tc)
        assert np.array_equal(mxa.tok_scales_logical(tok.scales, lens, d), ts)
    if name == "eps0_zero_rows":
        assert not row.codes.cpu().numpy()[3].any()
