"""GPU forward vs the Algorithm 1 oracle on the same quantized operands (O,
LSE), with the direct oracle's and the unquantized inputs' errors reported."""
import math

import numpy as np
import pytest
import torch

from block_scaled_mxfp8_gb300 import inputs as inp
from oracle import oracle as orc

from ._common import check_outputs, gpu_views, metrics, oracle_views, to_np

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
    inp.make_custom("d64_ragged_gqa4_causal", lengths=[300, 1, 129, 640], Hq=8, Hkv=2, d=64, causal=True, seed=34),
    # more items than SMs: persistent CTAs take two items each (zig-zag
    # rounds of 152), so the per-item barrier phases and the Q / O hand-over
    # between items are exercised element by element
    inp.make_custom("persist_batched_causal_gqa", B=3, L=1100, Hq=8, Hkv=4, d=128, causal=True, seed=29),
    inp.make_custom("persist_batched_d64", B=2, L=700, Hq=16, Hkv=16, d=64, causal=False, seed=30),
    inp.make_custom("persist_list_causal", lengths=[900, 5, 1000, 260, 700], Hq=8, Hkv=8, d=128, causal=True,
                    seed=31),
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
    O, LSE = orc.attn_fwd_alg1(dq["q"]["row"], dq["k"]["row"], dq["v"]["tok"], cu, w.causal, 1.0 / math.sqrt(w.d))
    return t, o, lse, O, LSE


@pytest.mark.parametrize("w", CASES, ids=[c.name + ("_causal" if c.causal else "") for c in CASES])
def test_fwd_matches_oracle(w):
    t, o, lse, O, LSE = run_fwd(w)
    cu = w.cu_seqlens.numpy()
    _, dq = oracle_views(w, t, names=("q", "k", "v"))
    alpha = 1.0 / math.sqrt(w.d)
    Od, _ = orc.attn_fwd(dq["q"]["row"], dq["k"]["row"], dq["v"]["tok"], cu, w.causal, alpha)
    Or, _ = orc.attn_fwd(to_np(t["q"]), to_np(t["k"]), to_np(t["v"]), cu, w.causal, alpha)
    print(w.name, "O vs unquantised inputs", metrics(to_np(o), Or))
    check_outputs(w.name, {"O": to_np(o), "LSE": lse.cpu().numpy()}, {"O": O, "LSE": LSE}, {"O": Od})


def test_fwd_first_causal_query_is_exact():
    """The first query of every causal document sees only its own key: its
    one quantized weight cancels in O = w V / w, so O equals bf16(V~_start)."""
    w = inp.make_custom("first_query", lengths=[5, 200, 1, 130], Hq=2, Hkv=2, d=128, causal=True, seed=25)
    t, o, lse, O, LSE = run_fwd(w)
    on = o.float().cpu().numpy()
    for s in w.cu_seqlens.numpy()[:-1]:
        want = torch.from_numpy(O[s]).to(torch.bfloat16).float().numpy()
        assert np.array_equal(on[s], want), s


SCHED_CASES = [
    inp.make_custom("sched_ragged_causal", lengths=[300, 0, 129, 1, 700, 128], Hq=4, Hkv=2, d=128, causal=True,
                    seed=26),
    inp.make_custom("sched_ragged", lengths=[513, 64, 0, 250], Hq=2, Hkv=1, d=128, causal=False, seed=27),
    inp.make_custom("sched_batched_causal", B=3, L=640, Hq=2, Hkv=2, d=64, causal=True, seed=28),
]


@pytest.mark.parametrize("w", SCHED_CASES, ids=[c.name for c in SCHED_CASES])
def test_fwd_work_list_schedule(w):
    """The cost-sorted work list (FLAMIA notes, Algorithm 2) only changes
    which CTA computes which tile: O and LSE are bit-identical to the
    max_seqlen grid.  The list holds every (document, query tile) pair once,
    the items that visit the most key tiles first."""
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=False)
    geo, gv = gpu_views(w, t, names=("q", "k", "v"))
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    o1, l1 = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal, workspace=ws)
    o0, l0 = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal, use_list=False)
    torch.cuda.synchronize()
    mxa.check_error()
    assert torch.equal(o1.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l0.view(torch.int32))

    lengths = np.diff(w.cu_seqlens.numpy())
    tiles = [(int(n) + 127) // 128 for n in lengths]
    pairs = sorted((b, t_) for b, n in enumerate(tiles) for t_ in range(n))
    if geo.cu_seqlens is None:  # equal documents: the grid itself, no list
        return
    raw = ws.cpu().numpy()
    count = int(raw[:4].view(np.int32)[0])
    assert count == len(pairs)
    nt = geo.ntiles
    it = raw[256:256 + nt * 16].view(np.int32).reshape(nt, 4)[:count]
    base = np.concatenate([[0], np.cumsum(tiles)])[:-1]
    # the forward's query list: every (document, tile) once, with the first
    # scale tile of its document on both sides (the same for self-attention),
    # ordered by the key tiles each query tile visits, most first
    assert sorted(map(tuple, it[:, :2].tolist())) == pairs
    assert all(it[i, 2] == base[it[i, 0]] and it[i, 3] == base[it[i, 0]] for i in range(count))
    cost = [it[i, 1] + 1 if w.causal else tiles[it[i, 0]] for i in range(count)]
    assert all(cost[i] >= cost[i + 1] for i in range(count - 1))


REPEAT_CASES = [
    inp.make_custom("repeat_batched_causal", B=2, L=2048, Hq=16, Hkv=8, d=128, causal=True, seed=32),
    inp.make_custom("repeat_batched", B=2, L=2048, Hq=16, Hkv=16, d=128, causal=False, seed=33),
    inp.make_custom("repeat_list_causal", lengths=[1500, 3, 900, 2000, 130, 700], Hq=8, Hkv=2, d=128, causal=True,
                    seed=34),
]


@pytest.mark.parametrize("w", REPEAT_CASES, ids=[c.name for c in REPEAT_CASES])
def test_fwd_repeat_is_bit_identical(w):
    """With more items than SMs the CTAs take over items dynamically, so which
    CTA computes which query tile changes from run to run; every item is
    computed the same way on any CTA, so O and LSE repeat bit for bit."""
    from block_scaled_mxfp8_gb300 import mxa

    t = inp.tensors(w, with_grad=False)
    geo, gv = gpu_views(w, t, names=("q", "k", "v"))
    outs = []
    for _ in range(3):
        o, lse = mxa.fwd(gv["q"][0], gv["k"][0], gv["v"][1], geo, w.causal)
        torch.cuda.synchronize()
        mxa.check_error()
        outs.append((o.view(torch.int16).clone(), lse.view(torch.int32).clone()))
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
