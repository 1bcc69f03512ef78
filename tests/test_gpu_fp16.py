"""fp16 inputs (LCE_INPUT_FP16) through the C ABI against the fp64 oracle on
the same fp16-rounded values: forward, separate backward and fused paths,
ragged shapes, reductions mean / sum, accumulation into dH, the autograd
wrapper; reduction none is refused for fp16."""
import numpy as np
import pytest
import torch

from lce_synth import make_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


@pytest.mark.parametrize("reduction", ["mean", "sum"])
@pytest.mark.parametrize("N,D,V,chunk,n_ign", [(300, 264, 1000, 128, 17), (129, 64, 257, 64, 5),
                                               (1000, 520, 3000, 384, 40)])
def test_fp16_all_paths_match_oracle(lce, N, D, V, chunk, n_ign, reduction):
    H, W, y = make_inputs(N, D, V, seed=N + D, n_ignored=n_ign, w_std=0.05, dtype="fp16")
    assert H.dtype == torch.float16
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = torch.tensor([0.7], device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, reduction=reduction)
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk, reduction=reduction)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, dloss=dl, chunk=chunk, reduction=reduction)
    torch.cuda.synchronize()
    assert dH.dtype == torch.float16 and bdH.dtype == torch.float16
    ref = O.forward_backward(H, W, y, dloss=0.7, reduction=reduction)
    check_loss(loss.item(), ref["loss"])
    check_loss(floss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_lse(to64(flse), ref["lse"])
    for name, got, exp in (("dH", dH, ref["dH"]), ("dW", dW, ref["dW"]),
                           ("dH (backward)", bdH, ref["dH"]), ("dW (backward)", bdW, ref["dW"])):
        check_grad(name, to64(got), exp)


def test_fp16_mid_size_full_oracle(lce):
    """The Llama-2 LM-head shape in fp16 (N 4096, D 4096, V 32000, chunk 1024)."""
    H, W, y = make_inputs(4096, 4096, 32000, seed=1, n_ignored=205, dtype="fp16")
    loss, lse, dH, dW = lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=1024)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dW", to64(dW), ref["dW"])


def test_fp16_accumulate_dh(lce):
    N, D, V = 500, 256, 2000
    H, W, y = make_inputs(N, D, V, seed=41, n_ignored=10, w_std=0.05, dtype="fp16")
    dH0 = (torch.randn(N, D, generator=torch.Generator().manual_seed(2)) * 1e-3).half().to(DEV)
    dH = dH0.clone()
    lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=128, dH=dH, accumulate=("dH",))
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    check_grad("dH accumulated", to64(dH), ref["dH"] + to64(dH0))


def test_fp16_reduction_none_refused(lce):
    H, W, y = make_inputs(64, 64, 300, seed=43, dtype="fp16")
    with pytest.raises(lce.LCEError):
        lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=64, reduction="none")
    torch.cuda.synchronize()


def test_fp16_autograd_wrapper(lce):
    H, W, y = make_inputs(300, 128, 900, seed=45, n_ignored=10, dtype="fp16")
    Hd = H.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    loss = lce.linear_cross_entropy(Hd, Wd, y.to(DEV), chunk=128)
    (loss * 3.0).backward()
    ref = O.forward_backward(H, W, y, dloss=3.0)
    check_loss(loss.item(), ref["loss"])
    check_grad("dH", to64(Hd.grad), ref["dH"])
    check_grad("dW", to64(Wd.grad), ref["dW"])


def test_fp16_mixed_dtypes_refused(lce):
    H, W, y = make_inputs(64, 64, 300, seed=47)
    with pytest.raises(TypeError):
        lce.lce_fwd_bwd(H.to(DEV).half(), W.to(DEV), y.to(DEV), chunk=64)
