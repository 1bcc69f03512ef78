"""Cross-entropy over precomputed logits (the streaming row kernel) through the
C ABI against the fp64 oracle on the same logit values."""
import numpy as np
import pytest
import torch

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


def _logits(N, V, ld, dtype, seed, scale=3.0):
    """(host copy [N, V], device view [N, V] with row stride ld) of the same values."""
    g = torch.Generator().manual_seed(seed)
    Zfull = (torch.randn(N, ld, generator=g) * scale).to(dtype)
    return Zfull[:, :V].contiguous(), Zfull.to(DEV)[:, :V]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("N,V,ld", [(300, 1003, 1008), (64, 32000, 32000), (5, 7, 8)])
def test_ce_logits_matches_oracle(lce, dtype, reduction, N, V, ld):
    Z, Zd = _logits(N, V, ld, dtype, seed=N + V)
    assert Zd.stride(0) == ld
    rng = np.random.default_rng(V)
    y = torch.from_numpy(rng.integers(0, V, size=N))
    y[::7] = -100
    dl = torch.from_numpy(rng.standard_normal(N)).float() if reduction == "none" else torch.tensor([0.8])
    loss, lse, dZ = lce.ce_logits(Zd, y.to(DEV), dloss=dl.to(DEV), reduction=reduction)
    torch.cuda.synchronize()
    ref = O.ce_from_logits(Z.double().numpy(), y.numpy(),
                           dloss=dl.double().numpy() if reduction == "none" else 0.8,
                           reduction=reduction)
    check_lse(to64(lse), ref["lse"])
    if reduction == "none":
        assert np.abs(to64(loss) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    else:
        check_loss(loss.item(), ref["loss"])
    check_grad("dZ", to64(dZ), ref["dZ"])


def test_ce_logits_in_place_and_forward_only(lce):
    N, V = 200, 5000
    Z, Zd = _logits(N, V, V, torch.bfloat16, seed=3)
    y = torch.randint(0, V, (N,))
    ref = O.ce_from_logits(Z.double().numpy(), y.numpy())
    loss_f, lse_f, none = lce.ce_logits(Zd, y.to(DEV), grad=False)
    assert none is None
    loss, lse, dZ = lce.ce_logits(Zd, y.to(DEV), inplace=True)
    torch.cuda.synchronize()
    assert dZ.data_ptr() == Zd.data_ptr()
    check_loss(loss_f.item(), ref["loss"])
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dZ in place", to64(Zd), ref["dZ"])


def test_ce_logits_large_logits(lce):
    N, V = 64, 4096
    Z, Zd = _logits(N, V, V, torch.float32, seed=5, scale=300.0)
    y = torch.randint(0, V, (N,))
    loss, lse, dZ = lce.ce_logits(Zd, y.to(DEV), reduction="sum")
    torch.cuda.synchronize()
    ref = O.ce_from_logits(Z.double().numpy(), y.numpy(), reduction="sum")
    assert torch.isfinite(dZ).all() and torch.isfinite(lse).all()
    check_lse(to64(lse), ref["lse"])
    check_loss(loss.item(), ref["loss"])
    check_grad("dZ", to64(dZ), ref["dZ"])
