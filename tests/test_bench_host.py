"""Host logic of bench.py that needs no GPU: binding the process to the CPUs
local to the GPU before the end-to-end loop pins its host buffers."""
import io
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Props:
    pci_domain_id = 0
    pci_bus_id = 0x1B
    pci_device_id = 0


def test_binds_to_the_listed_cpus_it_may_run_on(monkeypatch):
    seen = {}
    allowed = set(os.sched_getaffinity(0))
    listed = sorted(allowed)[:3]
    spec = ",".join(str(c) for c in listed) + ",%d-%d" % (10000, 10002)  # CPUs this process may not use
    real_open = open

    def fake_open(path, *a, **k):
        if str(path).startswith("/sys/bus/pci/devices/"):
            seen["path"] = path
            return io.StringIO(spec + "\n")
        return real_open(path, *a, **k)

    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda i: _Props())
    monkeypatch.setattr("builtins.open", fake_open)
    monkeypatch.setattr(os, "sched_setaffinity", lambda pid, cpus: seen.setdefault("cpus", sorted(cpus)))
    assert bench.bind_gpu_local_cpus(0) == spec
    assert seen["path"] == "/sys/bus/pci/devices/0000:1b:00.0/local_cpulist"
    assert seen["cpus"] == listed


def test_leaves_the_binding_alone_without_topology(monkeypatch):
    called = []
    monkeypatch.setattr(os, "sched_setaffinity", lambda pid, cpus: called.append(cpus))
    # no GPU here: the device query raises, nothing is bound
    if not torch.cuda.is_available():
        assert bench.bind_gpu_local_cpus(0) is None
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda i: _Props())
    monkeypatch.setattr("builtins.open", lambda *a, **k: (_ for _ in ()).throw(OSError("no sysfs")))
    assert bench.bind_gpu_local_cpus(0) is None
    assert called == []


def test_bench_names_resolve():
    """Every global name a function of bench.py reads exists in the module or
    the builtins.  Most of bench.py runs on a GPU only, so this catches a
    missing import or a misspelt helper on the CPU first."""
    import builtins
    import symtable

    src = open(os.path.join(ROOT, "bench.py")).read()
    known = set(dir(bench)) | set(dir(builtins))

    def unresolved(t):
        bad = [(t.get_name(), s.get_name()) for s in t.get_symbols()
               if s.is_global() and s.is_referenced() and not s.is_assigned() and s.get_name() not in known]
        for ch in t.get_children():
            bad += unresolved(ch)
        return bad

    assert unresolved(symtable.symtable(src, "bench.py", "exec")) == []


def test_clock_summary_by_time_window():
    """The clock record of each end-to-end pass: the samples that arrived
    inside the pass's window, their median SM clock and the throttle reasons
    they show (nvidia-smi csv, noheader, nounits)."""
    c = bench.ClockSampler(0)
    rows = [  # index, sm, max sm, power, active, hw, hw thermal, sw thermal, sw power cap
        (1.0, "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (1.1, "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (2.0, "0, 1500, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (2.1, "0, 1480, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (2.2, "0, 1490, 2070, 1399.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (2.3, "garbled line"),
    ]
    for t, ln in rows:
        c.times.append(t)
        c.lines.append(ln)
    first = c.summary(0.9, 1.5)
    assert first == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 2}
    late = c.summary(1.9, 3.0)
    assert late["sm_mhz"] == 1490.0 and late["reasons"] == ["sw_power_cap"] and late["samples"] == 3
    assert c.summary()["samples"] == 5
    assert c.summary(5.0, 6.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
