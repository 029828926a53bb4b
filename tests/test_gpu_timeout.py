"""The failure detection behind KDA_DEV_TIMEOUT, made to fire without a fault.

Every in-kernel wait of the chunk kernels is bounded by wall time: a warp that gives up
makes the kernel OR KDA_DEV_TIMEOUT into the caller's status word and leave, with the context
intact. kda_selftest_wait_timeout runs that bounded wait on a barrier that nothing arrives on
(a short limit, no trap, no fault). The test checks that the kernel returns after about the
limit, that the bit is set, and that the context still runs a forward that matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import kda_segids_cu_gb300 as kda
import oracle
import synth
from tests.parity import check_kda_output

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kda.kda_selftest_wait_timeout(0.05, status)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) & kda.KDA_DEV_TIMEOUT
    assert 0.04 <= dt < 5.0, f"the wait took {dt:.3f} s"
    # the context is usable: a forward after it runs clean and matches the oracle
    rng = np.random.default_rng(3)
    seg = torch.from_numpy(synth.random_segment_ids(rng, 2, 300, max_len=120, pad_prob=0.05))
    gen = torch.Generator().manual_seed(3)
    N, H, D = 600, 2, 128
    q = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn(N, H, D, generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn(N, H, D, generator=gen).to(torch.bfloat16)
    g = (-torch.exp(torch.randn(N, H, D, generator=gen) * 0.5 - 2.0)).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).to(torch.bfloat16)
    o = kda.kda_chunk_fwd_varlen(*(t.cuda() for t in (q, k, v, g, beta)), seg.cuda())
    check_kda_output(o, oracle.kda_fwd(q, k, v, g, beta, seg, 2, 300), seg, torch.bfloat16,
                     label="after the timeout")
