"""GPU parity: kda_segids_to_cu_seqlens must match the oracle bit for bit."""
import os

import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth

pytestmark = pytest.mark.gpu


def _gpu(seg_np, max_segs):
    seg = torch.from_numpy(np.ascontiguousarray(seg_np, dtype=np.int32)).cuda()
    cu, n = kda.kda_segids_to_cu_seqlens(seg, max_segs)
    torch.cuda.synchronize()
    return cu.cpu().numpy(), int(n.item())


def _compare(seg_np, max_segs):
    cu_ref, n_ref = oracle.cu_seqlens(seg_np, max_segs)
    cu, n = _gpu(seg_np, max_segs)
    assert n == n_ref
    assert cu.tolist() == cu_ref.tolist(), (seg_np, max_segs)


def test_worked_examples(golden_dir):
    path = os.path.join(golden_dir, "cu_seqlens_examples.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        seg, ms, exp = (p.strip() for p in line.split(";"))
        cu, _ = _gpu(np.array([[int(x) for x in seg.split(",")]]), int(ms))
        assert cu.tolist() == [int(x) for x in exp.split(",")]


@pytest.mark.parametrize("name", ["tiny", "b2", "ling3", "short", "long"])
def test_workloads(name):
    wl = synth.WORKLOADS[name]
    seg, _ = synth.make_segment_ids(wl, synth.default_seed(name))
    _compare(seg, wl.max_segs)
    # results for smaller max_segs (overflow) and larger ones
    _compare(seg, 1)
    _compare(seg, max(1, wl.max_segs // 7))
    _compare(seg, wl.max_segs * 3 + 1)
    _compare(seg, 4096)                       # the no-inflation sweep's size


def test_random_sweep():
    rng = np.random.default_rng(123)
    for trial in range(300):
        B = int(rng.integers(1, 5))
        T = int(rng.integers(1, 300))
        seg = synth.random_segment_ids(rng, B, T, max_len=int(rng.integers(1, 40)),
                                       pad_prob=float(rng.choice([0.0, 0.2, 0.5])),
                                       ids=str(rng.choice(["increasing", "arbitrary"])))
        _compare(seg, int(rng.integers(1, 50)))


def test_multi_tile_and_edges():
    rng = np.random.default_rng(5)
    # several 16384-token tiles and a ragged tail, starts at tile edges
    T = 16384 * 3 + 77
    seg = synth.random_segment_ids(rng, 1, T, max_len=3000, pad_prob=0.1)
    _compare(seg, 64)
    seg2 = np.ones((2, 16384), np.int32)      # row start exactly at a tile edge
    _compare(seg2, 4)
    _compare(np.zeros((3, 100), np.int32), 5)     # all padding
    _compare(np.ones((1, 1), np.int32), 1)        # one token
    _compare(np.arange(1, 5001, dtype=np.int32)[None], 4096)   # every token a segment
