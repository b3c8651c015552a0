"""Seeded synthetic inputs shaped like the attention workloads of the pages.

Shared by the tests, the benchmark and the oracle side; holds none of the
method's arithmetic (no quantisation, no attention) -- only random draws and
document-length recipes.

Workloads (the pages' "LLM shapes" and packed-document runs):
  * tiny:    B1 H2 L256 d64, Q/K/V/dO ~ N(0,1).
  * llm:     B8 H32 L4096 d128, N(0,1) with two channels per (tensor, head)
             scaled x50 for every token (activation outliers).
  * train:   B4 H16 L8192 d128 causal, 0.5 * N(0,1).
  * jagged:  256 packed documents, lengths ~ lognormal with mean 512 and
             sigma 1.0 (mu = ln 512 - sigma^2/2), rounded, clipped to
             [16, 4096]; H4 d128 causal, N(0,1).
  * tokblock: one packed row of T = 8192 tokens cut into documents of
             uniform length in [64, 2048] (the last one truncated to fit);
             32 query heads, 8 kv heads, d128.
Draws use torch's CPU generator (``manual_seed``), fp32 ``randn`` rounded to
bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    B: int            # batch (documents of equal length) when cu_seqlens is None
    L: int            # per-document length for batched inputs; max length otherwise
    Hq: int
    Hkv: int
    d: int
    causal: bool
    lengths: Optional[list] = None   # packed document lengths (jagged)
    mode: str = "mx32"               # "mx32" (1-D groups of 32) or "tokblock"
    hadamard: bool = False
    std: float = 1.0
    outlier_channels: int = 0
    outlier_gain: float = 1.0
    seed: int = 1001
    extra: dict = field(default_factory=dict)
    lengths_k: Optional[list] = None  # cross-attention: key/value tokens of each document

    @property
    def T_k(self) -> int:
        return int(sum(self.lengths_k)) if self.lengths_k is not None else self.T

    @property
    def cu_seqlens_k(self) -> torch.Tensor:
        if self.lengths_k is None:
            return self.cu_seqlens
        return torch.tensor(np.concatenate([[0], np.cumsum(self.lengths_k)]), dtype=torch.int32)

    @property
    def T(self) -> int:
        return int(sum(self.lengths)) if self.lengths is not None else self.B * self.L

    @property
    def cu_seqlens(self) -> torch.Tensor:
        if self.lengths is not None:
            lens = self.lengths
        else:
            lens = [self.L] * self.B
        return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)

    @property
    def doc_lengths(self) -> list:
        return list(self.lengths) if self.lengths is not None else [self.L] * self.B

    @property
    def max_seqlen(self) -> int:
        return int(max(self.doc_lengths))


def lognormal_lengths(n_docs: int, mean: float, sigma: float, lo: int, hi: int, seed: int) -> list:
    rng = np.random.default_rng(seed)
    mu = math.log(mean) - sigma * sigma / 2.0
    x = rng.lognormal(mu, sigma, size=n_docs)
    return [int(v) for v in np.clip(np.rint(x), lo, hi)]


def uniform_packed_lengths(total: int, lo: int, hi: int, seed: int) -> list:
    rng = np.random.default_rng(seed)
    out, acc = [], 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def workload(name: str, causal: Optional[bool] = None) -> Workload:
    if name == "tiny":
        w = Workload("tiny", B=1, L=256, Hq=2, Hkv=2, d=64, causal=False, seed=1001)
    elif name == "llm":
        w = Workload("llm", B=8, L=4096, Hq=32, Hkv=32, d=128, causal=False,
                     outlier_channels=2, outlier_gain=50.0, seed=1002)
    elif name == "train":
        w = Workload("train", B=4, L=8192, Hq=16, Hkv=16, d=128, causal=True, std=0.5, seed=1003)
    elif name == "jagged":
        lens = lognormal_lengths(256, 512.0, 1.0, 16, 4096, seed=1004)
        w = Workload("jagged", B=len(lens), L=max(lens), Hq=4, Hkv=4, d=128, causal=True,
                     lengths=lens, seed=1004)
    elif name == "cross":
        # cross-attention module: 768 sequences of 512 query tokens against
        # jagged key/value sets of up to 16384 tokens (uniform, mean ~8192),
        # model width 384 = 3 heads of 128
        _, lk = cross_lengths(768, 512, 16384, seed=1006)
        w = Workload("cross", B=768, L=512, Hq=3, Hkv=3, d=128, causal=False, seed=1006, lengths_k=lk)
    elif name == "tokblock":
        lens = uniform_packed_lengths(8192, 64, 2048, seed=1005)
        w = Workload("tokblock", B=len(lens), L=max(lens), Hq=32, Hkv=8, d=128, causal=True,
                     lengths=lens, mode="tokblock", hadamard=True, seed=1005)
    else:
        raise KeyError(name)
    if causal is not None:
        w.causal = causal
    return w


def make_custom(name, lengths=None, B=1, L=256, Hq=2, Hkv=2, d=64, causal=False, mode="mx32",
                hadamard=False, std=1.0, seed=7, outlier_channels=0, outlier_gain=1.0) -> Workload:
    return Workload(name, B=B if lengths is None else len(lengths), L=L if lengths is None else max(lengths),
                    Hq=Hq, Hkv=Hkv, d=d, causal=causal, lengths=lengths, mode=mode, hadamard=hadamard,
                    std=std, seed=seed, outlier_channels=outlier_channels, outlier_gain=outlier_gain)


def _randn_bf16(gen: torch.Generator, shape, std: float, outlier_channels: int, gain: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_channels:
        T, H, d = shape
        for h in range(H):
            ch = torch.randperm(d, generator=gen)[:outlier_channels]
            x[:, h, ch] *= gain
    return x.to(torch.bfloat16)


def tensors(w: Workload, with_grad: bool = True) -> dict:
    """bf16 CPU tensors q [T,Hq,d], k/v [T,Hkv,d] (T_k rows for
    cross-attention) and (with_grad) do [T,Hq,d]."""
    if w.lengths_k is not None:
        out = cross_tensors(w.doc_lengths, w.lengths_k, w.Hq, w.Hkv, w.d, w.seed, w.std)
        if not with_grad:
            del out["do"]
        return out
    gen = torch.Generator().manual_seed(w.seed)
    T = w.T
    out = {
        "q": _randn_bf16(gen, (T, w.Hq, w.d), w.std, w.outlier_channels, w.outlier_gain),
        "k": _randn_bf16(gen, (T, w.Hkv, w.d), w.std, w.outlier_channels, w.outlier_gain),
        "v": _randn_bf16(gen, (T, w.Hkv, w.d), w.std, w.outlier_channels, w.outlier_gain),
    }
    if with_grad:
        out["do"] = _randn_bf16(gen, (T, w.Hq, w.d), w.std, 0, 1.0)
    return out


def cross_lengths(n_docs: int, lq: int, max_k: int, seed: int) -> tuple:
    """Cross-attention document lengths: every document has lq query tokens
    and a jagged key/value length drawn uniformly from [1, max_k] (mean about
    max_k / 2: the "sparsity 0.5" of the production shapes)."""
    g = torch.Generator().manual_seed(seed)
    lk = torch.randint(1, max_k + 1, (n_docs,), generator=g).tolist()
    return [lq] * n_docs, [int(x) for x in lk]


def cross_tensors(lq: list, lk: list, Hq: int, Hkv: int, d: int, seed: int, std: float = 1.0) -> dict:
    """bf16 CPU tensors of a cross-attention call: q, do [sum lq, Hq, d] and
    k, v [sum lk, Hkv, d], N(0, std^2) from one seeded generator."""
    gen = torch.Generator().manual_seed(seed)
    Tq, Tk = int(sum(lq)), int(sum(lk))
    return {
        "q": _randn_bf16(gen, (Tq, Hq, d), std, 0, 1.0),
        "k": _randn_bf16(gen, (Tk, Hkv, d), std, 0, 1.0),
        "v": _randn_bf16(gen, (Tk, Hkv, d), std, 0, 1.0),
        "do": _randn_bf16(gen, (Tq, Hq, d), std, 0, 1.0),
    }
