"""Host-side pieces of bench.py on CPU: the workload options, the oracle baseline's
single-thread figure on the small workloads, and when the recorded DRAM traffic applies."""
import dataclasses
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _args(**kw):
    a = dict(workload="ling3", heads=0, max_segs=0)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_workload_options():
    wl = bench.bench_workload(_args())
    assert wl == synth.WORKLOADS["ling3"]
    h4 = bench.bench_workload(_args(heads=4))
    assert (h4.H, h4.B, h4.T, h4.max_segs) == (4, wl.B, wl.T, wl.max_segs)
    m = bench.bench_workload(_args(max_segs=4096))
    assert m.max_segs == 4096 and m.H == wl.H
    assert "max_segs=4096" in bench.workload_label(m)


def test_traffic_only_for_the_captured_workload():
    # the recorded traffic belongs to the full ling3 launch; any other shape reports null
    assert bench.chunk_traffic(synth.WORKLOADS["b2"]) is None
    assert bench.chunk_traffic(dataclasses.replace(synth.WORKLOADS["ling3"], H=4)) is None
    assert bench.chunk_traffic(dataclasses.replace(synth.WORKLOADS["ling3"], max_segs=4096)) is None


def test_cpu_baseline_small_workload_has_single_thread_figure():
    r = bench.cpu_baseline(synth.WORKLOADS["tiny"], seconds=0.2)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] >= 1
    st = r["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["unit"] == r["unit"]
