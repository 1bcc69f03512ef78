"""Frozen LM head (LCE_FROZEN_W, compute_dW=False): the gradient phase is the dH
contraction alone and dW is neither computed nor written. Against the fp64
oracle's loss, lse and dH on ragged shapes and on shapes whose dH tiles are split
in 2 or 4 vocabulary parts (with W frozen the split fills one wave of the GPU's
CTA pairs: 32 tiles of a 1024-row chunk at D 4096 -> 2 parts); dW memory is left
as it was; accumulation into dH, fp16 inputs and the autograd wrapper (a W that
does not require grad) take the same path."""
import ctypes

import numpy as np
import pytest
import torch

from lce_synth import make_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FROZEN_W = 8


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


def _inputs(N, D, V, dtype="bf16"):
    return make_inputs(N, D, V, seed=N + 2 * D + V, labels="uniform", n_ignored=N // 25,
                       w_std=0.05, dtype=dtype)


@pytest.mark.parametrize("N,D,V,chunk", [
    (300, 264, 1000, 128),       # ragged, one part
    (1000, 1024, 8229, 256),     # 4 parts
    (777, 1536, 16411, 384),     # 4 parts, a pair's second tile past the rows
    (4096, 4096, 32000, 1024),   # Llama-2 head: 2 parts
])
def test_frozen_w_matches_oracle(lce, N, D, V, chunk):
    H, W, y = _inputs(N, D, V)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = torch.tensor([0.8], device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, compute_dW=False)
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, dloss=dl, chunk=chunk, compute_dW=False)
    torch.cuda.synchronize()
    assert dW is None and bdW is None
    ref = O.forward_backward(H, W, y, dloss=0.8)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dH (backward)", to64(bdH), ref["dH"])


def test_frozen_w_leaves_dw_memory_alone(lce):
    """Through the C ABI with a canary-filled dW buffer: not one byte changes."""
    N, D, V, chunk = 1000, 1024, 8229, 256
    H, W, y = _inputs(N, D, V)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    L = lce.lib()
    ws = lce.alloc_workspace(N, D, V, chunk, DEV, FROZEN_W)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(N, device=DEV)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.full((V * D * 4,), 0x5A, dtype=torch.uint8, device=DEV).view(torch.float32)
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.lce_fwd_bwd_opt(vp(Hd), vp(Wd), vp(yd), None, N, D, V, -100, chunk, 0, FROZEN_W,
                           vp(loss), vp(lse), vp(dH), vp(dW), vp(ws), ws.numel(),
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert bool((dW.view(torch.uint8) == 0x5A).all().item())
    ref = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, compute_dW=False)
    torch.cuda.synchronize()
    assert torch.equal(dH, ref[2]) and torch.equal(loss, ref[0])


def test_frozen_w_equals_full_dh_and_is_reproducible(lce):
    """dH with W frozen agrees with dH of the full call (the parts differ, so within
    rounding) and repeats bit for bit."""
    N, D, V, chunk = 2048, 2048, 16000, 1024
    H, W, y = _inputs(N, D, V)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    a = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, compute_dW=False)
    b = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, compute_dW=False)
    full = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2]) and torch.equal(a[0], b[0])
    assert torch.equal(a[0], full[0]) and torch.equal(a[1], full[1])
    assert np.abs(to64(a[2]) - to64(full[2])).max() <= 2.0 ** -7 * np.abs(to64(full[2])).max()


def test_frozen_w_accumulate_dh_and_fp16(lce):
    N, D, V, chunk = 777, 1536, 16411, 384
    H, W, y = _inputs(N, D, V)
    dH0 = (torch.randn(N, D, generator=torch.Generator().manual_seed(2)) * 1e-4).to(torch.bfloat16)
    loss, lse, dH, dW = lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=chunk,
                                        dH=dH0.to(DEV), accumulate=("dH",), compute_dW=False)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    check_grad("dH (accumulated)", to64(dH), ref["dH"] + to64(dH0))
    with pytest.raises(ValueError):
        lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=chunk, dW=torch.zeros(V, D, device=DEV),
                        accumulate=("dW",), compute_dW=False)
    H16, W16, y16 = _inputs(1000, 1024, 8229, dtype="fp16")
    loss, lse, dH, dW = lce.lce_fwd_bwd(H16.to(DEV), W16.to(DEV), y16.to(DEV), chunk=256,
                                        compute_dW=False)
    torch.cuda.synchronize()
    assert dH.dtype == torch.float16
    ref = O.forward_backward(H16, W16, y16)
    check_loss(loss.item(), ref["loss"])
    check_grad("dH (fp16)", to64(dH), ref["dH"])


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("train_w", [True, False])
def test_autograd_schedules(lce, reduction, train_w):
    """The autograd wrapper: fused (gradients formed in the forward, mean / sum)
    and recompute (none, or fused=False) against the oracle; a W without
    requires_grad gets no gradient and takes the frozen path."""
    N, D, V, chunk = 700, 512, 9001, 256
    H, W, y = _inputs(N, D, V)
    g = torch.linspace(-1, 1, N) if reduction == "none" else torch.tensor(1.7)
    ref = O.forward_backward(H, W, y, dloss=g.double().numpy() if reduction == "none" else 1.7,
                             reduction=reduction)
    for fused in (True, False):
        Hd = H.to(DEV).requires_grad_(True)
        Wd = W.to(DEV).requires_grad_(train_w)
        out = lce.linear_cross_entropy(Hd, Wd, y.to(DEV), chunk=chunk, reduction=reduction,
                                       fused=fused)
        (out * g.to(DEV)).sum().backward()
        torch.cuda.synchronize()
        if reduction == "none":
            assert np.abs(to64(out) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
        else:
            check_loss(out.item(), ref["loss"])
        check_grad(f"dH (fused={fused})", to64(Hd.grad), ref["dH"])
        if train_w:
            check_grad(f"dW (fused={fused})", to64(Wd.grad), ref["dW"])
        else:
            assert Wd.grad is None
