"""Failure detection on the device without a GPU fault: every mbarrier wait in the library is
bounded in wall time, and a wait that runs out sets DG_ST_TIMEOUT and lets its kernel return.
The self-test kernel waits on a barrier nothing ever arrives on."""
import time

import pytest
import torch


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    assert torch.cuda.is_available()
    m.lib()
    return m


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_stays_usable(dg, orc):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dg.dg_selftest_wait_timeout(st)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(st[0]) & dg.ST_TIMEOUT
    assert 1.5 <= waited < 30.0, waited      # the bound is about 2 s of wall time
    # the same context runs a pass normally right after
    from test_gpu_parity import _run_step
    from parity import TOL, check_stats
    g, o, _ = _run_step(dg, orc, 1, 256, 1000, 128, "bf16", K=32, seed=3, pass_=0)
    assert int(g["status"][0]) == 0
    check_stats(g, o, TOL["bf16"])
