"""lce_forward_noalloc: the forward for callers that cannot allocate device
memory (no allocator inside a host runtime, no cudaMalloc allowed on their hot
path, or a device-memory budget fixed at start-up). It runs on a scratch array
built into the library instead of a caller workspace. Every case is checked
against the fp64 oracle and against lce_forward with a workspace. This file
sorts last so a run that stops at the first failure has run every other test
before it."""
import ctypes

import numpy as np
import pytest
import torch

from lce_synth import WORKLOADS, make_inputs, workload_inputs
from oracle import lce_oracle as O
from tests.gpu_util import LOSS_REL, LSE_ABS, check_loss, check_lse

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LCE_ERR_WORKSPACE = 3
LCE_ERR_LABEL_RANGE = 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as lce
    lce.build()
    L = lce.lib()
    f = L.lce_forward_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp]
    f.restype = ctypes.c_int
    L.lce_noalloc_read_status.argtypes = [vp]
    L.lce_noalloc_read_status.restype = ctypes.c_int
    return L


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(L, H, W, y, chunk, loss, lse):
    N, D = H.shape
    V = W.shape[0]
    return L.lce_forward_noalloc(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                 ctypes.c_void_p(y.data_ptr()), N, D, V, -100, chunk,
                                 ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                 _stream())


def _run_and_check(L, H, W, y, chunk):
    """One no-alloc call against lce_forward (with a workspace) and the oracle."""
    import linear_cross_entropy_chunked_gb300 as lce
    N = H.shape[0]
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    ref_loss, ref_lse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    loss = torch.full((1,), float("nan"), device=DEV)
    lse = torch.full((N,), float("nan"), device=DEV)
    assert _call(L, Hd, Wd, yd, chunk, loss, lse) == 0
    assert L.lce_noalloc_read_status(_stream()) == 0
    rl = ref_loss.item()
    assert abs(loss.item() - rl) <= LOSS_REL * abs(rl)
    got_lse = lse.cpu().double().numpy()
    assert np.abs(got_lse - ref_lse.cpu().double().numpy()).max() <= LSE_ABS
    o_loss, o_lse, _, _ = O.forward(H, W, y)
    check_loss(loss.item(), o_loss)
    check_lse(got_lse, o_lse)


def test_forward_noalloc_two_calls_in_a_row(lib):
    N, D, V, chunk = 2048, 1024, 32000, 256
    for seed in (31, 32):       # two calls in a row, on different inputs
        H, W, y = make_inputs(N, D, V, seed=seed, n_ignored=40)
        _run_and_check(lib, H, W, y, chunk)


def test_forward_noalloc_larger_then_smaller(lib):
    """A call that fills more of the array followed by a smaller one: contents the
    first call left beyond what the second clears must not leak into it."""
    H, W, y = make_inputs(3000, 512, 50000, seed=41, n_ignored=70)
    _run_and_check(lib, H, W, y, 1024)
    H, W, y = make_inputs(300, 264, 1000, seed=42, n_ignored=9)
    _run_and_check(lib, H, W, y, 128)


def test_forward_noalloc_llama2_head(lib):
    """The Llama-2-shaped head (N = 4096, D = 4096, V = 32000) at chunk 1024: its
    forward workspace (~2.1 MB) fits the 64 MiB array."""
    H, W, y = workload_inputs(WORKLOADS["llama2-7b"])
    _run_and_check(lib, H, W, y, 1024)


def test_forward_noalloc_allocates_nothing(lib):
    """After a first call (which looks up the array's address), further calls
    leave the device's free memory unchanged."""
    H, W, y = make_inputs(1024, 512, 20000, seed=43, n_ignored=10)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(1024, device=DEV)
    assert _call(lib, Hd, Wd, yd, 256, loss, lse) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(lib, Hd, Wd, yd, 256, loss, lse) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    check_loss(loss.item(), O.forward(H, W, y)[0])


def test_forward_noalloc_reports_device_status(lib):
    """A label outside [0, V) is flagged in the array's header and read back by
    lce_noalloc_read_status (then cleared); the row counts as ignored."""
    H, W, y = make_inputs(200, 128, 700, seed=44)
    y[7] = 700
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(200, device=DEV)
    assert _call(lib, Hd, Wd, yd, 64, loss, lse) == 0
    assert lib.lce_noalloc_read_status(_stream()) == LCE_ERR_LABEL_RANGE
    assert lib.lce_noalloc_read_status(_stream()) == 0
    o_loss, o_lse, _, n_bad = O.forward(H, W, y)
    assert n_bad == 1
    check_loss(loss.item(), o_loss)
    check_lse(lse.cpu().double().numpy(), o_lse)


def test_forward_noalloc_rejects_sizes_beyond_its_scratch(lib):
    H = torch.zeros(8, 8, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(8, dtype=torch.int64, device=DEV)
    loss = torch.zeros(1, device=DEV)
    # Llama-3-sized head in one chunk of 16384 rows: the slab partials alone take
    # 16384 x 1002 x 8 B = 131 MB, beyond the 64 MiB array; the size check returns
    # before any pointer is used or anything is enqueued.
    st = lib.lce_forward_noalloc(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(H.data_ptr()),
                                 ctypes.c_void_p(y.data_ptr()), 16384, 4096, 128256, -100, 16384,
                                 ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                 _stream())
    assert st == LCE_ERR_WORKSPACE
