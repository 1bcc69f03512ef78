"""lce_forward_noalloc: the forward for callers that cannot allocate device
memory (no allocator inside a host runtime, no cudaMalloc allowed on their hot
path, or a device-memory budget fixed at start-up). It runs on a scratch array
built into the library instead of a caller workspace. This file sorts last so a
run that stops at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from lce_synth import make_inputs
from tests.gpu_util import LOSS_REL, LSE_ABS

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LCE_ERR_WORKSPACE = 3


def _noalloc_fn(lib):
    f = lib.lce_forward_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _call(f, H, W, y, chunk, loss, lse):
    N, D = H.shape
    V = W.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(W.data_ptr()),
             ctypes.c_void_p(y.data_ptr()), N, D, V, -100, chunk,
             ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)


def test_forward_noalloc_matches_forward():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as lce
    lce.build()
    f = _noalloc_fn(lce.lib())
    N, D, V, chunk = 2048, 1024, 32000, 256
    # two calls in a row, on different inputs, each against lce_forward
    for seed in (31, 32):
        H, W, y = make_inputs(N, D, V, seed=seed, n_ignored=40)
        Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
        ref_loss, ref_lse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
        loss = torch.full((1,), float("nan"), device=DEV)
        lse = torch.full((N,), float("nan"), device=DEV)
        assert _call(f, Hd, Wd, yd, chunk, loss, lse) == 0
        torch.cuda.synchronize()
        rl = ref_loss.item()
        assert abs(loss.item() - rl) <= LOSS_REL * abs(rl)
        assert np.abs(lse.cpu().double().numpy() - ref_lse.cpu().double().numpy()).max() <= LSE_ABS


def test_forward_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as lce
    lce.build()
    f = _noalloc_fn(lce.lib())
    H = torch.zeros(8, 8, dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(8, dtype=torch.int64, device=DEV)
    loss = torch.zeros(1, device=DEV)
    # Llama-3-sized head: the workspace (~271 MB at chunk 1024) exceeds the 64 MiB array;
    # the size check returns before any pointer is used or anything is enqueued.
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = f(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(H.data_ptr()),
           ctypes.c_void_p(y.data_ptr()), 16384, 4096, 128256, -100, 1024,
           ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(loss.data_ptr()), stream)
    assert st == LCE_ERR_WORKSPACE
