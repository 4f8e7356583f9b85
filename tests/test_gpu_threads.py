"""Several host threads driving the library at once, each on its own stream and workspace: the
per-device caches (launch attributes, device facts, the host-entry copy sessions) are shared
under locks, and every result is bit-identical to the same call made alone."""
import threading

import numpy as np
import pytest
import torch

from parity import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    import uniform_state_denoising_vocab_b300 as m
    m.lib()
    return m


def _case(seed, B, S, V, d):
    rng = np.random.default_rng(seed)
    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    h = bits(rng.standard_normal(B * S * d).astype(np.float32))
    w = bits((rng.standard_normal(V * d) / np.sqrt(d)).astype(np.float32))
    c = rng.integers(0, V, B * S).astype(np.int32)
    return dev_bf16(h, (B * S, d)), dev_bf16(w, (V, d)), dev(c)


def _passes(dg, h, w, c, B, S, stream, n=4):
    outs = []
    with torch.cuda.stream(stream):
        canvas = c.clone()
        for p in range(n):
            r = dg.dg_canvas_step(h, w, canvas, 32, 99, p, B=B, S=S, stream=stream)
            canvas = r["canvas"]
            outs.append(r)
    return outs


def test_two_threads_two_streams_match_sequential_runs(dg):
    shapes = [(1, 256, 5000, 256), (2, 150, 3000, 512)]
    cases = [_case(11 + i, *sh) for i, sh in enumerate(shapes)]
    # each workload alone
    ref = []
    for (h, w, c), (B, S, V, d) in zip(cases, shapes):
        st = torch.cuda.Stream()
        ref.append(_passes(dg, h, w, c, B, S, st))
        st.synchronize()
    # both at once from two host threads
    got, errors = [None, None], []

    def run(i):
        try:
            (h, w, c), (B, S, V, d) = cases[i], shapes[i]
            st = torch.cuda.Stream()
            got[i] = _passes(dg, h, w, c, B, S, st)
            st.synchronize()
        except Exception as e:   # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for g_run, r_run in zip(got, ref):
        for g, r in zip(g_run, r_run):
            assert int(g["status"][0]) == 0
            for k in ("canvas", "argmax", "conf", "entropy", "kept", "mean_entropy"):
                assert torch.equal(g[k], r[k]), k
