#!/usr/bin/env python
"""Benchmark: MXFP8 attention forward + backward on one GB300.

One step is the whole hot path over one batch of seeded synthetic inputs
already resident in HBM: quantize Q, K, V (row + token views), forward,
quantize dO, backward (D prep, main kernel, dQ convert).  Workload: B8 H32
L4096 d128 (the pages' LLM shape), non-causal by default, N(0,1) inputs with
two x50 outlier channels per head.

FLOP convention (the pages' / FLAMIA's): forward 4 B H L^2 d (halved when
causal), backward 2.5 x forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--causal] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
replica of the workload (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP8 attention fwd/bwd PFLOP/s and % of dense MXFP8 peak, B8 H32 L4096 d128"
UNIT = "PFLOP/s"
# Dense MXFP8 tensor peak: MEASURED_PEAKS.json's bf16 figure x the nominal
# fp8/bf16 ratio (4.5 / 2.25 = 2); fallback 1.9 PFLOP/s bf16 burst.
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
# tcgen05 kind::mxf8f6f4 block-scaled MMA (M=128, N=256, K=32) issued back
# to back on every SM (mxa_test_mma_rate, run by every bench): FLOP per SM
# clock, scaled by the SM count and the clock sampled during the timed region,
# gives the microbenchmark peak.  This value (measured on a GB300 at 2070 MHz)
# is used only if the probe cannot run.
MXFP8_MMA_FLOP_PER_SM_CLK = 16374.0
PROBE_FLOP_PER_ITER = 4 * 2 * 128 * 256 * 32
GB300_SMS = 152
DQ_MODE_NAMES = {0: "FP32", 1: "FP16x2^9", 2: "FP16 per-row boost"}


def bind_gpu_local_cpus(dev_index):
    """Run this process on the CPUs the GPU's PCI function lists as local, so
    that the pinned host buffers it fills (first touch) sit in the memory
    attached to that GPU's host socket.  Returns the CPU list as written in
    sysfs, or None when the topology is not available (the binding is then
    left as it was)."""
    import torch

    try:
        pr = torch.cuda.get_device_properties(dev_index)
        bus = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return spec
    except (AttributeError, OSError, RuntimeError, ValueError):
        return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            bf16 = d.get("bf16_tflops") or d.get("bf16_tflops_burst")
            bf16s = d.get("bf16_tflops_sustained", bf16)
            hbm = d.get("hbm_gbs")
            if bf16 and hbm:
                return {"mxfp8_tflops": 2.0 * float(bf16), "mxfp8_tflops_sustained": 2.0 * float(bf16s),
                        "hbm_gbs": float(hbm), "source": "measured (MEASURED_PEAKS.json bf16 x nominal fp8/bf16 ratio 2)"}
        except Exception:
            pass
    return {"mxfp8_tflops": 2.0 * FALLBACK_BF16_TFLOPS, "mxfp8_tflops_sustained": 2.0 * 1700.0,
            "hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback (1.9 PFLOP/s bf16 burst x nominal fp8/bf16 ratio 2)"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.times = []  # host arrival time of each line (time.monotonic)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.times.append(time.monotonic())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock, its maximum and the throttle reasons seen, over
        the samples that arrived in [t0, t1] (all samples by default)."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln, t in zip(self.lines, self.times):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# dram__bytes_read.sum + dram__bytes_write.sum of attn_bwd_dkdv_kernel and
# attn_dq_gemm_kernel at B2 H32 L4096 d128 (one ncu --set full capture)
BWD_DRAM_BYTES_B2 = (0.267507 + 1.156908 + 1.114415 + 0.062640) * 1e9


def flops(B, H, L, d, causal, lengths=None, lengths_k=None):
    """FLOP convention of the pages: forward 4 * H * d * sum_b n_b^2 (B * L^2 for
    equal lengths; sum_b nq_b * nk_b for cross-attention), halved when causal;
    backward 2.5 x forward."""
    if lengths_k is not None:
        lq = lengths if lengths is not None else [L] * B
        sq = float(sum(int(a) * int(b) for a, b in zip(lq, lengths_k)))
    else:
        sq = float(sum(int(n) * int(n) for n in lengths)) if lengths is not None else float(B) * L * L
    f = 4.0 * H * sq * d
    if causal:
        f *= 0.5
    return f, 2.5 * f


def job_time_ms(ms_local, dist=None, device="cpu"):
    """Whole-job time of a replica run: the slowest rank's timed region (the
    replicas share no data; this max is the only exchange)."""
    if dist is None:
        return float(ms_local)
    import torch

    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample(L=4096, H=1, d=128, causal=False, seed=1002):
    """The oracle, as it stands, on a bounded sample of the workload: one
    document of L tokens, H heads, same value recipe (two x50 outlier
    channels per head).  Returns (seconds, flop, threads)."""
    from block_scaled_mxfp8_gb300 import inputs as inp
    from oracle import oracle as orc

    w = inp.make_custom("cpu_sample", B=1, L=L, Hq=H, Hkv=H, d=d, causal=causal, seed=seed,
                        outlier_channels=2, outlier_gain=50.0)
    t = inp.tensors(w)
    orc.build()
    t0 = time.perf_counter()
    v = {}
    for k in ("q", "k", "v", "do"):
        rc, rs = orc.quant_row(t[k])
        tc, ts = orc.quant_tok(t[k])
        v[k] = (orc.dequant_row(rc, rs), orc.dequant_tok(tc, ts))
    alpha = 1.0 / math.sqrt(d)
    orc.attn_fwd_alg1(v["q"][0], v["k"][0], v["v"][1], None, causal, alpha)
    orc.attn_bwd_alg1(v["q"][0], v["k"][0], v["v"][1], v["v"][0], v["do"][0], v["q"][1], v["k"][1], v["do"][1],
                      None, causal, alpha)
    dt = time.perf_counter() - t0
    ff, fb = flops(1, H, L, d, causal)
    return dt, ff + fb, orc.num_threads()


def oracle_sample_cross(Lq=512, Lk=8192, H=1, d=128, seed=1006):
    """The oracle on one cross-attention document: Lq queries against Lk keys
    and values, H heads.  Returns (seconds, flop, threads)."""
    from block_scaled_mxfp8_gb300 import inputs as inp
    from oracle import oracle as orc

    t = inp.cross_tensors([Lq], [Lk], H, H, d, seed)
    cq = np.array([0, Lq], np.int32)
    ck = np.array([0, Lk], np.int32)
    orc.build()
    t0 = time.perf_counter()
    v = {}
    for k, cu in (("q", cq), ("do", cq), ("k", ck), ("v", ck)):
        rc, rs = orc.quant_row(t[k])
        tc, ts = orc.quant_tok(t[k], cu)
        v[k] = (orc.dequant_row(rc, rs), orc.dequant_tok(tc, ts, cu))
    alpha = 1.0 / math.sqrt(d)
    orc.attn_fwd_alg1(v["q"][0], v["k"][0], v["v"][1], cq, False, alpha, cu_k=ck)
    orc.attn_bwd_alg1(v["q"][0], v["k"][0], v["v"][1], v["v"][0], v["do"][0], v["q"][1], v["k"][1], v["do"][1],
                      cq, False, alpha, cu_k=ck)
    dt = time.perf_counter() - t0
    ff, fb = flops(1, H, Lq, d, False, [Lq], [Lk])
    return dt, ff + fb, orc.num_threads()


# ------------------------------------------------------------------ GPU leg

def run_gpu(args):
    import torch

    from block_scaled_mxfp8_gb300 import build as mbuild
    from block_scaled_mxfp8_gb300 import inputs as inp
    from block_scaled_mxfp8_gb300 import mxa

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    mbuild.build()

    w = inp.workload(args.workload, causal=True if args.causal else None)
    if args.batch:  # smaller batch of the same per-document shape (profiler captures)
        if w.lengths is not None:
            raise SystemExit("--batch applies to batched workloads only")
        w.B = args.batch
    B, L, Hq, Hkv, d = w.B, w.L, w.Hq, w.Hkv, w.d
    T = w.T
    t = inp.tensors(w)
    dev = torch.device("cuda", local)
    x = {k: v.to(dev) for k, v in t.items()}
    geo = mxa.Geometry.batched(B, L) if w.lengths is None else mxa.Geometry.packed(w.lengths, dev)
    cross = w.lengths_k is not None
    gk = mxa.Geometry.packed(w.lengths_k, dev) if cross else geo  # key/value documents
    kv_geo = gk if cross else None
    Tk = gk.T

    def alloc_views(H, g):
        mk = lambda: mxa.QView(torch.empty((g.T, H, d), dtype=torch.uint8, device=dev),
                               torch.empty((H, g.ntiles, mxa.ATOM_BYTES), dtype=torch.uint8, device=dev))
        return mk(), mk()

    qv = {k: alloc_views(Hq, geo) for k in ("q", "do")}
    qv.update({k: alloc_views(Hkv, gk) for k in ("k", "v")})
    o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    dq = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((Tk, Hkv, d), dtype=torch.bfloat16, device=dev)
    dv = torch.empty((Tk, Hkv, d), dtype=torch.bfloat16, device=dev)
    views = {"q_row": qv["q"][0], "k_row": qv["k"][0], "v_row": qv["v"][0], "g_row": qv["do"][0],
             "q_tok": qv["q"][1], "k_tok": qv["k"][1], "g_tok": qv["do"][1]}
    bp0 = mxa.bwd_params(views, o, lse, dq, dk, dv, geo, w.causal, args.dq_mode, kv_geo=kv_geo)
    fws = torch.empty(max(1, mxa.mxa_fwd_workspace_bytes(mxa.c_fwd_params(bp0.shape))), dtype=torch.uint8, device=dev)
    # strict causal forward: the per-key view of V, folded in on the diagonal tile
    if args.fold and (cross or not w.causal):
        raise SystemExit("--fold applies to causal self-attention workloads")
    mk_key = lambda: mxa.QView(torch.empty((T, Hkv, d), dtype=torch.uint8, device=dev),
                               torch.empty((Hkv, geo.ntiles, 128), dtype=torch.uint8, device=dev))
    vkey = mk_key() if args.fold else None
    kkey = mk_key() if args.fold else None  # strict dQ: per-key view of K
    bp = mxa.bwd_params(views, o, lse, dq, dk, dv, geo, w.causal, args.dq_mode, kv_geo=kv_geo, k_key=kkey)
    # this library's kernels per step: 4 quantizers (+2 per-key views), the
    # forward (+ its tile list), the backward's prep, dK/dV and dQ kernels
    # (+ two tile lists, + the two key-bound passes of the per-row FP16 mode)
    lists = fws.numel() > 1
    launches_per_step = (4 + (2 if args.fold else 0) + 1 + (1 if lists else 0) + 3 + (2 if lists else 0) +
                         (2 if args.dq_mode == 2 else 0))
    ws = torch.empty(mxa.mxa_bwd_workspace_bytes(bp), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(src, rec=None, outs=None, wait=None, fwd_done=None):
        # wait: per-input events (each quantize waits only for its own
        # tensor's upload); fwd_done: recorded once O is final
        o_, lse_, dq_, dk_, dv_ = outs if outs is not None else (o, lse, dq, dk, dv)
        e = [ev() for _ in range(4)] if rec is not None else None
        if e: e[0].record(stream)
        if wait: stream.wait_event(wait["q"])
        mxa.quantize(src["q"], geo, out=qv["q"])
        for k in ("k", "v"):
            if wait: stream.wait_event(wait[k])
            mxa.quantize(src[k], gk, out=qv[k])
        if vkey is not None:
            mxa.quantize_key(src["v"], geo, out=vkey)
            mxa.quantize_key(src["k"], geo, out=kkey)
        if e: e[1].record(stream)
        mxa.fwd(qv["q"][0], qv["k"][0], qv["v"][1], geo, w.causal, out=(o_, lse_), workspace=fws, kv_geo=kv_geo,
                v_key=vkey)
        if e: e[2].record(stream)
        if fwd_done is not None: fwd_done.record(stream)
        if wait: stream.wait_event(wait["do"])
        mxa.quantize(src["do"], geo, out=qv["do"])
        mxa.bwd(views, o_, lse_, geo, w.causal, dq_mode=args.dq_mode, workspace=ws, out=(dq_, dk_, dv_),
                kv_geo=kv_geo, k_key=kkey)
        if e:
            e[3].record(stream)
            rec.append(e)

    # the block-scaled MMA and exponential rates of this GPU, measured before
    # the timed region
    probe = mma_probe(dev)
    eprobe = ex2_probe(dev)

    for _ in range(args.warmup):
        step(x)
    torch.cuda.synchronize()
    mxa.check_error()

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    recs = []
    with ClockSampler(local) as clk:
        t_start, t_end = ev(), ev()
        t_start.record(stream)
        for _ in range(args.steps):
            step(x, recs)
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    mxa.check_error()
    ms_total = job_time_ms(t_start.elapsed_time(t_end), dist, dev)
    ms_step = ms_total / args.steps
    ms_quant = statistics.mean(r[0].elapsed_time(r[1]) for r in recs)
    ms_fwd = statistics.mean(r[1].elapsed_time(r[2]) for r in recs)
    ms_bwd = statistics.mean(r[2].elapsed_time(r[3]) for r in recs)  # includes the dO quantize

    ffwd, fbwd = flops(B, Hq, L, d, w.causal, w.lengths, w.lengths_k)
    step_flop = ffwd + fbwd
    value = world * step_flop / (ms_step * 1e-3) / 1e15

    # bwd alone (prep + main + dq convert), timed separately after the loop
    bw_ev = []
    for _ in range(max(3, min(args.steps, 10))):
        a_, b_ = ev(), ev()
        a_.record(stream)
        mxa.bwd(views, o, lse, geo, w.causal, dq_mode=args.dq_mode, workspace=ws, out=(dq, dk, dv), kv_geo=kv_geo,
                k_key=kkey)
        b_.record(stream)
        bw_ev.append((a_, b_))
    torch.cuda.synchronize()
    ms_bwd_only = statistics.mean(a_.elapsed_time(b_) for a_, b_ in bw_ev)

    # fused RMSNorm + quantize of Q into both views (one pass over x) against
    # torch's RMSNorm followed by the quantizer (the normalization as a pass of
    # its own); effective bandwidth = algorithmic bytes (x read once, codes and
    # scales of both views written) / time
    rms = None
    try:
        import torch.nn.functional as F

        wq = (torch.rand(d, generator=torch.Generator().manual_seed(7)) + 0.5).to(dev)
        wq16 = wq.to(torch.bfloat16)
        xq = x["q"]

        def fused():
            mxa.quantize(xq, geo, out=qv["q"], rmsnorm=(wq, 1e-6))

        def unfused():
            mxa.quantize(F.rms_norm(xq, (d,), weight=wq16, eps=1e-6), geo, out=qv["q"])

        res = {}
        for nm, fn in (("fused", fused), ("unfused", unfused)):
            for _ in range(3):
                fn()
            a_, b_ = ev(), ev()
            a_.record(stream)
            for _ in range(10):
                fn()
            b_.record(stream)
            torch.cuda.synchronize()
            res[nm] = a_.elapsed_time(b_) / 10
        nbytes = T * Hq * d * 2 + 2 * (T * Hq * d + T * Hq * d // 32)
        rms = {"tensor": "q [T, Hq, d] bf16, both views", "fused_ms": round(res["fused"], 4),
               "unfused_ms": round(res["unfused"], 4), "fused_tbps": round(nbytes / res["fused"] / 1e9, 3),
               "unfused_tbps": round(nbytes / res["unfused"] / 1e9, 3),
               "speedup": round(res["unfused"] / res["fused"], 2)}
        mxa.check_error()
    except (AttributeError, RuntimeError) as exc:  # torch without rms_norm
        rms = {"unavailable": str(exc)[:200]}

    pk = peaks()
    fwd_pf = ffwd / (ms_fwd * 1e-3) / 1e15
    bwd_pf = fbwd / (ms_bwd_only * 1e-3) / 1e15
    # dominant kernel: the backward (2.5x the forward's flops)
    dom = {"kernel": ("mxa_bwd call: bwd_prep_kernel + attn_bwd_dkdv_kernel + attn_dq_gemm_kernel "
                      "(%s dQ; the dK/dV kernel takes ~80%% of the call)" % DQ_MODE_NAMES[args.dq_mode]),
           "pflops": bwd_pf}
    peak_pf = pk["mxfp8_tflops"] / 1e3
    sm_mhz = clk.summary().get("sm_mhz") or 2070.0
    probe_rate = probe["flop_per_sm_clk"] if probe else MXFP8_MMA_FLOP_PER_SM_CLK
    micro_tflops = probe_rate * (probe["sms"] if probe else GB300_SMS) * sm_mhz * 1e6 / 1e12
    # DRAM bytes of the backward call's dK/dV and dQ kernels from one ncu
    # capture at B2 (the --set full capture of the attention kernels),
    # scaled by the tile pairs (B / 2); only for the workload it was taken on
    traffic = None
    if w.name == "llm" and not w.causal and not args.dq_mode and w.lengths is None:
        traffic = round(BWD_DRAM_BYTES_B2 * B / 2)
    roofline = {"bound": "tensor", "achieved": round(dom["pflops"] * 1e3, 1), "peak": round(pk["mxfp8_tflops"], 1),
                "unit": "TFLOP/s", "frac": round(dom["pflops"] / peak_pf, 4), "traffic": traffic,
                "kernel": dom["kernel"], "peak_source": pk["source"],
                "fwd": {"achieved": round(fwd_pf * 1e3, 1), "frac": round(fwd_pf / peak_pf, 4)},
                "bwd": {"achieved": round(bwd_pf * 1e3, 1), "frac": round(bwd_pf / peak_pf, 4)},
                # dense block-scaled MXFP8 rate of a back-to-back tcgen05.mma
                # microbenchmark at the sampled SM clock
                "mxfp8_microbench_tflops": round(micro_tflops, 1),
                "mma_probe": probe if probe else "not run (the measured constant %.0f FLOP/SM/clk is used)" %
                MXFP8_MMA_FLOP_PER_SM_CLK,
                "frac_of_microbench": {"fwd": round(fwd_pf * 1e3 / micro_tflops, 4),
                                       "bwd": round(bwd_pf * 1e3 / micro_tflops, 4)}}
    # the co-bound: exponentials, one per visible (query, key) pair and head
    # in the forward and again in the backward's P rebuild (forward FLOP / 4d)
    n_exp = ffwd / (4.0 * w.d)
    exp_unit = None
    if eprobe:
        exp_rate = eprobe["ex2_per_sm_clk"] * eprobe["sms"] * sm_mhz * 1e6  # per second at the sampled clock
        exp_unit = {"exps_per_pass": n_exp, "peak_per_s": round(exp_rate, 1),
                    "fwd_frac": round(n_exp / (ms_fwd * 1e-3) / exp_rate, 4),
                    "bwd_frac": round(n_exp / (ms_bwd_only * 1e-3) / exp_rate, 4), "probe": eprobe}

    # e2e through the C ABI with host buffers: H2D of q, k, v, dO and D2H of o, dq, dk, dv inside the timed region
    host_cpus = bind_gpu_local_cpus(local)  # pinned buffers in the memory next to this GPU
    host_in = {k: v.pin_memory() for k, v in t.items()}
    host_out = {k: torch.empty(s, dtype=torch.bfloat16).pin_memory()
                for k, s in (("o", o.shape), ("dq", dq.shape), ("dk", dk.shape), ("dv", dv.shape))}
    dev_in = {k: torch.empty_like(v) for k, v in x.items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    # Pipelined like a training loop: step i+1's inputs go up on one stream and
    # step i's outputs come down on another while the next step computes;
    # inputs and outputs are double-buffered on the device.  Each quantize
    # waits only for its own input, and O comes down once the forward is
    # done.  Every byte of every step crosses the host link inside the timed
    # region.  (One stream per tensor and direction was slower: the copies
    # contend for the link.)
    dev_in2 = [dev_in, {k: torch.empty_like(v) for k, v in x.items()}]
    outs2 = [(o, lse, dq, dk, dv), tuple(torch.empty_like(tn) for tn in (o, lse, dq, dk, dv))]
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def upload(b):
        """The inputs of buffer b on the upload stream, one event per tensor."""
        evs = {}
        with torch.cuda.stream(s_h2d):
            for k in dev_in2[b]:
                dev_in2[b][k].copy_(host_in[k], non_blocking=True)
                evs[k] = ev()
                evs[k].record(s_h2d)
        return evs

    def e2e_run(n):
        start, end = ev(), ev()
        start.record(stream)
        done = [None, None]
        out_free = [None, None]
        s_h2d.wait_event(start)
        in_ready = [upload(0), None]
        for i in range(n):
            bb = i % 2
            if out_free[bb] is not None:
                stream.wait_event(out_free[bb])
            fwd_done = ev()
            step(dev_in2[bb], outs=outs2[bb], wait=in_ready[bb], fwd_done=fwd_done)
            done[bb] = ev()
            done[bb].record(stream)
            if i + 1 < n:  # the next inputs, once the step that last read that buffer is done
                nb = (i + 1) % 2
                if done[nb] is not None:
                    s_h2d.wait_event(done[nb])
                in_ready[nb] = upload(nb)
            # O comes down as soon as the forward has written it, the
            # gradients once the step is done
            s_d2h.wait_event(fwd_done)
            with torch.cuda.stream(s_d2h):
                host_out["o"].copy_(outs2[bb][0], non_blocking=True)
            s_d2h.wait_event(done[bb])
            with torch.cuda.stream(s_d2h):
                for k, tn in zip(("dq", "dk", "dv"), (outs2[bb][2], outs2[bb][3], outs2[bb][4])):
                    host_out[k].copy_(tn, non_blocking=True)
            out_free[bb] = ev()
            out_free[bb].record(s_d2h)
        stream.wait_stream(s_d2h)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    e2e_run(2)
    # the host link is shared with other users of the machine: the median of
    # five passes, with their spread.  A pass runs the timed step count (at
    # most 30): its first upload and last download are not overlapped with
    # compute, and a training loop runs long enough for the steady state
    # The SM clock of each pass comes from one sampler over all five: they
    # run for about a second in all, long enough for the GPU to reach its
    # power cap, unlike the 0.2 s timed region above
    n_e2e = max(3, min(args.steps, 30))
    passes, windows = [], []
    with ClockSampler(local) as eclk:
        for _ in range(5):
            t0 = time.monotonic()
            passes.append(e2e_run(n_e2e) / n_e2e)
            windows.append((t0, time.monotonic()))
    ms_e2e = sorted(passes)[len(passes) // 2]
    pass_clk = [eclk.summary(t0, t1) for t0, t1 in windows]
    e2e = {"value": round(world * step_flop / (ms_e2e * 1e-3) / 1e15, 4), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 3),
           "ms_per_step_passes": [round(x, 3) for x in passes], "steps_per_pass": n_e2e,
           "sm_mhz_passes": [c["sm_mhz"] for c in pass_clk],
           "clock_reasons": sorted(set(r for c in pass_clk for r in c["reasons"])), "host_cpus": host_cpus}

    # the quantizer of Q, K and V (both views) against HBM: 2 B read and
    # (1 + 1/32) B written per element per view (padding scale bytes excluded)
    q_elems = T * Hq * d + 2 * Tk * Hkv * d
    q_bytes = q_elems * (2.0 + 2 * (1.0 + 1.0 / 32))
    q_gbs = q_bytes / (ms_quant * 1e-3) / 1e9
    quant_line = {"ms": round(ms_quant, 4), "bytes": int(q_bytes), "gbs": round(q_gbs, 1),
                  "peak_gbs": pk["hbm_gbs"], "frac_hbm": round(q_gbs / pk["hbm_gbs"], 4),
                  "what": "Q, K, V quantized, ROW and TOK views each, bf16 in"}

    out = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8 (e4m3 codes, ue8m0 scales, fp32 accumulate)", "data": "synthetic",
        "config": {"workload": ("%s: B%d H%d L%d d%d %s, fwd+bwd, dQ %s" % (
            w.name, B, Hq, L, d, "causal" + (" strict (per-key folds)" if args.fold else "") if w.causal
            else "non-causal", DQ_MODE_NAMES[args.dq_mode].lower()))
            if not cross else ("%s: B%d Lq%d x jagged Lk U[1,%d] (T_k %d) H%d d%d, fwd+bwd, dQ fp32" % (
                w.name, B, L, max(w.lengths_k), Tk, Hq, d)),
            "global_batch": B * world, "seq_len": L, "heads": Hq, "head_dim": d, "causal": w.causal,
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "l2": "inputs larger than L2 (each bf16 tensor %.0f MB)" % (T * Hq * d * 2 / 1e6),
            "flop_per_step": step_flop},
        "pct_of_peak": round(100.0 * value / world / peak_pf, 2),
        "fwd_pflops": round(fwd_pf, 4), "bwd_pflops": round(bwd_pf, 4),
        "ms": {"quantize_qkv": round(ms_quant, 3), "fwd": round(ms_fwd, 3), "quantize_do_plus_bwd": round(ms_bwd, 3),
               "bwd": round(ms_bwd_only, 3)},
        "roofline": roofline,
        "exp_unit": exp_unit if exp_unit else "probe did not run",
        "quantize": quant_line,
        "rmsnorm_quantize": rms,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # one (document, head) at a time until about 12 s of oracle work
        dt = fl = 0.0
        heads = 0
        while dt < 12.0 and heads < 32:
            if cross:
                t_, f_, thr = oracle_sample_cross(Lq=L, Lk=8192, H=1, d=d, seed=1006 + heads)
            else:
                t_, f_, thr = oracle_sample(L=min(L, 4096), H=1, d=d, causal=w.causal, seed=1002 + heads)
            dt, fl, heads = dt + t_, fl + f_, heads + 1
        what = ("(document, head) pairs of %d x 8192 tokens" % L) if cross else \
            ("(document, head) pairs of %d tokens" % min(L, 4096))
        out["cpu_baseline"] = {"value": fl / dt / 1e15, "unit": UNIT, "cores": thr, "kind": "oracle",
                               "sample": "%d %s, d%d (oracle quantize + fwd + bwd), %.1f s" % (heads, what, d, dt)}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def run_reference(args):
    """The oracle on the host cores, per step a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from block_scaled_mxfp8_gb300 import inputs as inp

    w = inp.workload(args.workload, causal=True if args.causal else None)
    cross = w.lengths_k is not None
    L = min(w.L, 2048)
    total, fl_total, thr = 0.0, 0.0, 1
    for i in range(args.warmup + args.steps):
        if cross:
            dt, fl, thr = oracle_sample_cross(Lq=w.L, Lk=2048, H=1, d=w.d, seed=1006 + i)
        else:
            dt, fl, thr = oracle_sample(L=L, H=1, d=w.d, causal=w.causal, seed=1002 + i)
        if i >= args.warmup:
            total += dt
            fl_total += fl
    v = fl_total / total / 1e15
    sample = "per step one document of %d tokens, 1 head, d%d of the %s workload (oracle quantize + fwd + bwd)" % (
        L, w.d, w.name) if not cross else (
        "per step one document of %d queries x 2048 keys, 1 head, d%d of the %s workload (oracle quantize + fwd + bwd)"
        % (w.L, w.d, w.name))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "%s: B%d H%d L%d d%d %s, fwd+bwd" % (w.name, w.B, w.Hq, w.L, w.d,
                                                                    "causal" if w.causal else "non-causal")},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def mma_probe(dev, iters=20000):
    """Block-scaled MMA rate on every SM (include/mxa_testing.h): one warm-up
    launch, then one timed launch with CUDA events.  Returns a dict with the
    FLOP per SM clock (median over the CTAs' own clock counts) and the
    PFLOP/s over the whole GPU (events)."""
    import torch
    from block_scaled_mxfp8_gb300 import mxa

    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    if mxa.mxa_test_mma_rate(200, cyc, stream) != mxa.MXA_OK:
        return None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st = mxa.mxa_test_mma_rate(iters, cyc, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    c = cyc.cpu().tolist()
    if st != mxa.MXA_OK or mxa.mxa_get_error() != mxa.MXA_OK or min(c) <= 0:
        return None
    ms = e0.elapsed_time(e1)
    fl = float(PROBE_FLOP_PER_ITER) * iters
    return {"flop_per_sm_clk": round(fl / statistics.median(c), 1), "sms": n_sm, "iters": iters,
            "pflops": round(fl * n_sm / (ms * 1e-3) / 1e15, 4), "ms": round(ms, 4),
            "what": "tcgen05.mma kind::mxf8f6f4 block_scale, M128 N256 K32, E4M3, SS operands, one issuing "
                    "thread per SM, back to back"}


def run_mma_probe(args):
    import torch

    from block_scaled_mxfp8_gb300 import build as mbuild

    mbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    with ClockSampler(0) as clk:
        r = mma_probe(dev)
    if r is None:
        raise SystemExit("mma probe failed")
    r["clocks"] = clk.summary()
    print(json.dumps({"mma_probe": r}))


def ex2_probe(dev, iters=4096):
    """Exponential-unit rate on every SM (include/mxa_testing.h): one warm-up
    launch, then one timed launch.  Returns the ex2 per SM clock (median over
    the CTAs' own clock counts)."""
    import torch
    from block_scaled_mxfp8_gb300 import mxa

    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    if mxa.mxa_test_ex2_rate(64, cyc, stream) != mxa.MXA_OK:
        return None
    st = mxa.mxa_test_ex2_rate(iters, cyc, stream)
    torch.cuda.synchronize(dev)
    c = cyc.cpu().tolist()
    if st != mxa.MXA_OK or mxa.mxa_get_error() != mxa.MXA_OK or min(c) <= 0:
        return None
    n = float(iters) * 8 * 512
    return {"ex2_per_sm_clk": round(n / statistics.median(c), 2), "sms": n_sm, "iters": iters,
            "what": "ex2.approx.ftz.f32, 512 threads x 8 independent chains per SM"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mxa", choices=["mxa", "reference"])
    ap.add_argument("--workload", default="llm")
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--dq-mode", type=int, default=0, choices=[0, 1, 2],
                    help="0 = fp32 dQ accumulation, 1 = fp16 x 2^9, 2 = fp16 with a per-row boost")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fold", action="store_true",
                    help="strict causal attention: per-key V and K scales folded on the diagonal tile, "
                         "per-query dS scales for dQ")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling only)")
    ap.add_argument("--mma-probe", action="store_true",
                    help="only measure the block-scaled MMA rate (one GPU) and print it")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.mma_probe:
        run_mma_probe(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
