"""GPU forward vs the oracle on the same quantized operands (O, LSE)."""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import assert_close, gpu_views, metrics, oracle_views, to_np

pytestmark = pytest.mark.gpu

CASES = [
    inp.workload("tiny", causal=False),
    inp.workload("tiny", causal=True),
    inp.make_custom("d128_ragged_causal", lengths=[1, 129, 300, 64, 7], Hq=4, Hkv=2, d=128, causal=True, seed=21),
    inp.make_custom("d128_ragged", lengths=[250, 33, 513], Hq=2, Hkv=1, d=128, causal=False, seed=22,
                    outlier_channels=2, outlier_gain=50.0),
    inp.make_custom("d64_batched_causal", B=2, L=384, Hq=2, Hkv=2, d=64, causal=True, seed=23),
    inp.make_custom("tokblock_gqa", lengths=[100, 400, 37], Hq=4, Hkv=2, d=128, causal=True, mode="tokblock",
                    hadamard=True, seed=24),
]


def run_fwd(w):
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=False)
    geo, gv = gpu_views(w, t, names=("q", "k", "v"))
    o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
    torch.cuda.synchronize()
    mxa.check_error()
    _, dq = oracle_views(w, t, names=("q", "k", "v"))
    cu = w.cu_seqlens.numpy()
    O, LSE = orc.attn_fwd(dq["q"]["row"], dq["k"]["row"], dq["v"]["tok"], cu, w.causal, 1.0 / math.sqrt(w.d))
    return t, o, lse, O, LSE


@pytest.mark.parametrize("w", CASES, ids=[c.name + ("_causal" if c.causal else "") for c in CASES])
def test_fwd_matches_oracle(w):
    t, o, lse, O, LSE = run_fwd(w)
    cu = w.cu_seqlens.numpy()
    Or, _ = orc.attn_fwd(to_np(t["q"]), to_np(t["k"]), to_np(t["v"]), cu, w.causal, 1.0 / math.sqrt(w.d))
    lse_err = float(np.abs(lse.cpu().numpy() - LSE).max())
    print(w.name, "O vs oracle", metrics(to_np(o), O), "vs unquantised", metrics(to_np(o), Or), "LSE maxerr", lse_err)
    assert_close("O", to_np(o), O)
    assert lse_err <= 1e-3 * max(1.0, float(np.abs(LSE).max())), lse_err


def test_fwd_first_causal_query_is_exact():
    """The first query of every causal document sees only its own key: P = 1
    is exact in E4M3 after the 2^4 boost, so O equals bf16(V~_start)."""
    w = inp.make_custom("first_query", lengths=[5, 200, 1, 130], Hq=2, Hkv=2, d=128, causal=True, seed=25)
    t, o, lse, O, LSE = run_fwd(w)
    on = o.float().cpu().numpy()
    for s in w.cu_seqlens.numpy()[:-1]:
        want = torch.from_numpy(O[s]).to(torch.bfloat16).float().numpy()
        assert np.array_equal(on[s], want), s
