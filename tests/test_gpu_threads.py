"""Several host threads calling the library at once, each on its own CUDA stream
with its own buffers and workspace: every call's outputs are bit-identical to the
same call made alone. The library's per-device state (the side stream and its
fork / join events of the two-kernel gradient phase, the device attributes, the
profiling records) is shared between the threads behind mutexes."""
import threading

import pytest
import torch

from lce_synth import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


CASES = [(1500, 1024, 20000, 512, False), (900, 512, 9000, 256, True), (2100, 2048, 12000, 1024, False),
         (700, 1536, 16411, 384, True)]


def _inputs(i):
    N, D, V, chunk, frozen = CASES[i]
    H, W, y = make_inputs(N, D, V, seed=100 + i, n_ignored=N // 30, w_std=0.05)
    return H.to(DEV), W.to(DEV), y.to(DEV), chunk, frozen


def test_concurrent_calls_from_threads(lce):
    inputs = [_inputs(i) for i in range(len(CASES))]
    # each case alone, on the default stream
    alone = []
    for H, W, y, chunk, frozen in inputs:
        out = lce.lce_fwd_bwd(H, W, y, chunk=chunk, compute_dW=not frozen)
        torch.cuda.synchronize()
        alone.append([None if t is None else t.clone() for t in out])

    results = [None] * len(CASES)
    errors = []
    start = threading.Barrier(len(CASES))

    def worker(i):
        try:
            H, W, y, chunk, frozen = inputs[i]
            s = torch.cuda.Stream(DEV)
            with torch.cuda.stream(s):
                start.wait()
                outs = []
                for _ in range(3):
                    o = lce.lce_fwd_bwd(H, W, y, chunk=chunk, compute_dW=not frozen, stream=s)
                    outs.append(o)
                s.synchronize()
            results[i] = outs
        except Exception as e:  # reported below, in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    for i, outs in enumerate(results):
        for o in outs:
            for a, b in zip(alone[i], o):
                if a is None:
                    assert b is None
                else:
                    assert torch.equal(a, b), f"case {i} differs when run concurrently"
