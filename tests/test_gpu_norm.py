"""GPU parity of the final-RMSNorm path through the C ABI against the fp64 oracle:
the standalone RMSNorm forward / backward kernels and the fused
RMSNorm + LM head + cross-entropy call (lce_norm_fwd_bwd), element by element at
sizes the oracle finishes in seconds (ragged N, D not a multiple of the CTA's
vector count, several chunks), plus edge cases, determinism and agreement with
the same computation composed from the separate entry points."""
import numpy as np
import pytest
import torch

from lce_synth import IGNORE_INDEX, make_norm_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EPS = 1e-6


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


def _xg(N, D, seed):
    X, g, _, _ = make_norm_inputs(N, D, 16, seed)
    return X, g


# H is bf16: each element within half a bf16 ulp of the fp64 value (2^-9 relative),
# checked as 2^-8 of the row's largest |h| to stay clear of values near a rounding tie
def check_h(got, ref):
    got = to64(got)
    err = np.abs(got - ref).max(axis=1)
    bound = 2.0 ** -8 * np.abs(ref).max(axis=1) + 1e-30
    assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.parametrize("N,D", [(1, 8), (300, 264), (1000, 4096), (77, 8192), (513, 2056)])
def test_rmsnorm_forward_matches_oracle(lce, N, D):
    X, g = _xg(N, D, seed=N + D)
    H, rstd = lce.rmsnorm_forward(X.to(DEV), g.to(DEV), eps=EPS, want_rstd=True)
    torch.cuda.synchronize()
    H_ref, rstd_ref = O.rmsnorm_forward(X, g, EPS)
    check_h(H, H_ref)
    assert np.abs(to64(rstd) - rstd_ref).max() <= 1e-5 * np.abs(rstd_ref).max()


@pytest.mark.parametrize("dh_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N,D", [(1, 8), (300, 264), (1000, 4096), (77, 8192), (513, 2056)])
def test_rmsnorm_backward_matches_oracle(lce, N, D, dh_dtype):
    X, g = _xg(N, D, seed=3 * N + D)
    gen = torch.Generator().manual_seed(N)
    dH = (torch.randn(N, D, generator=gen) * 0.01).to(dh_dtype)
    dX, dgamma = lce.rmsnorm_backward(X.to(DEV), g.to(DEV), dH.to(DEV), eps=EPS)
    torch.cuda.synchronize()
    dX_ref, dg_ref = O.rmsnorm_backward(X, g, EPS, dH)
    check_grad("dX", to64(dX), dX_ref)
    check_grad("dgamma", to64(dgamma), dg_ref)


def test_rmsnorm_backward_deterministic(lce):
    X, g = _xg(700, 4096, seed=9)
    dH = torch.randn(700, 4096).to(DEV)
    a = lce.rmsnorm_backward(X.to(DEV), g.to(DEV), dH, eps=EPS)
    b = lce.rmsnorm_backward(X.to(DEV), g.to(DEV), dH, eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _norm_case(N, D, V, seed, n_ign):
    return make_norm_inputs(N, D, V, seed, labels="uniform", n_ignored=n_ign, w_std=0.05)


def _run_norm(lce, X, g, W, y, chunk, dloss_host, reduction):
    dl = None if dloss_host is None else torch.tensor(np.atleast_1d(dloss_host), dtype=torch.float32,
                                                      device=DEV)
    out = lce.norm_fwd_bwd(X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV), eps=EPS, dloss=dl,
                           chunk=chunk, reduction=reduction)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("N,D,V,chunk", [(300, 264, 1000, 128), (1000, 520, 3000, 384),
                                         (77, 128, 100, 1024), (1024, 4096, 8000, 256)])
def test_norm_fwd_bwd_matches_oracle(lce, N, D, V, chunk, reduction):
    X, g, W, y = _norm_case(N, D, V, seed=N + V, n_ign=N // 20)
    rng = np.random.default_rng(N)
    dl = rng.standard_normal(N) if reduction == "none" else 0.9
    loss, lse, dX, dgamma, dW = _run_norm(lce, X, g, W, y, chunk, dl, reduction)
    ref = O.norm_forward_backward(X, g, EPS, W, y, dloss=dl, reduction=reduction)
    if reduction == "none":
        assert np.abs(to64(loss) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    else:
        check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dX", to64(dX), ref["dX"])
    check_grad("dgamma", to64(dgamma), ref["dgamma"])
    check_grad("dW", to64(dW), ref["dW"])


def test_norm_fwd_bwd_llama2_shape(lce):
    """The Llama-2 LM-head shape (N 4096, D 4096, V 32000, chunk 1024) against the
    full fp64 oracle."""
    X, g, W, y = make_norm_inputs(4096, 4096, 32000, seed=1, n_ignored=205)
    loss, lse, dX, dgamma, dW = _run_norm(lce, X, g, W, y, 1024, None, "mean")
    ref = O.norm_forward_backward(X, g, EPS, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dX", to64(dX), ref["dX"])
    check_grad("dgamma", to64(dgamma), ref["dgamma"])
    check_grad("dW", to64(dW), ref["dW"])


@pytest.mark.parametrize("low_memory", [False, True])
def test_norm_fused_equals_composed_calls(lce, low_memory):
    """lce_norm_fwd_bwd against rmsnorm_forward -> lce_fwd_bwd -> rmsnorm_backward
    on the GPU, both with the same schedule (chunk pairs with one dW contraction
    each, or with low_memory one buffer and one dW contraction per chunk): the same
    H, so loss, lse and dW are bit-identical; dX differs only by the bf16 rounding
    of dH in the composed path."""
    N, D, V, chunk = 1500, 1024, 5000, 512
    X, g, W, y = _norm_case(N, D, V, seed=17, n_ign=40)
    Xd, gd, Wd, yd = X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dX, dgamma, dW = lce.norm_fwd_bwd(Xd, gd, Wd, yd, eps=EPS, chunk=chunk,
                                                 low_memory=low_memory)
    H = lce.rmsnorm_forward(Xd, gd, eps=EPS)
    loss2, lse2, dH2, dW2 = lce.lce_fwd_bwd(H, Wd, yd, chunk=chunk, low_memory=low_memory)
    dX2, dgamma2 = lce.rmsnorm_backward(Xd, gd, dH2, eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(loss, loss2) and torch.equal(lse, lse2) and torch.equal(dW, dW2)
    check_grad("dX (composed)", to64(dX2), to64(dX))
    check_grad("dgamma (composed)", to64(dgamma2), to64(dgamma))


@pytest.mark.parametrize("N,D,V,chunk", [(1000, 520, 3000, 384), (1024, 4096, 8000, 256)])
def test_norm_one_buffer_matches_oracle(lce, N, D, V, chunk):
    """The RMSNorm path with one chunk buffer (LCE_LOW_MEMORY) against the oracle."""
    X, g, W, y = _norm_case(N, D, V, seed=N + V + 3, n_ign=N // 20)
    loss, lse, dX, dgamma, dW = lce.norm_fwd_bwd(X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV),
                                                 eps=EPS, chunk=chunk, low_memory=True)
    torch.cuda.synchronize()
    ref = O.norm_forward_backward(X, g, EPS, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dX", to64(dX), ref["dX"])
    check_grad("dgamma", to64(dgamma), ref["dgamma"])
    check_grad("dW", to64(dW), ref["dW"])


def test_norm_fwd_bwd_deterministic(lce):
    X, g, W, y = _norm_case(600, 512, 3000, seed=21, n_ign=10)
    a = _run_norm(lce, X, g, W, y, 256, None, "mean")
    b = _run_norm(lce, X, g, W, y, 256, None, "mean")
    for p, q in zip(a, b):
        assert torch.equal(p, q)


def test_norm_all_ignored_and_empty(lce):
    X, g, W, y = _norm_case(130, 64, 300, seed=4, n_ign=0)
    y[:] = IGNORE_INDEX
    loss, lse, dX, dgamma, dW = _run_norm(lce, X, g, W, y, 64, None, "mean")
    assert loss.item() == 0.0
    assert dX.abs().max().item() == 0.0 and dgamma.abs().max().item() == 0.0
    assert dW.abs().max().item() == 0.0
    check_lse(to64(lse), O.norm_forward_backward(X, g, EPS, W, y)["lse"])
    X0 = torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV)
    y0 = torch.zeros(0, dtype=torch.int64, device=DEV)
    loss, lse, dX, dgamma, dW = lce.norm_fwd_bwd(X0, g.to(DEV), W.to(DEV), y0, chunk=64)
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and dgamma.abs().max().item() == 0.0 and dW.abs().max().item() == 0.0


def test_norm_autograd_wrapper(lce):
    X, g, W, y = _norm_case(260, 128, 700, seed=23, n_ign=9)
    Xd = X.to(DEV).requires_grad_(True)
    gd = g.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    loss = lce.norm_linear_cross_entropy(Xd, gd, Wd, y.to(DEV), eps=EPS, chunk=128)
    (loss * 2.0).backward()
    ref = O.norm_forward_backward(X, g, EPS, W, y, dloss=2.0)
    check_loss(loss.item(), ref["loss"])
    check_grad("dX", to64(Xd.grad), ref["dX"])
    check_grad("dgamma", to64(gd.grad), ref["dgamma"])
    check_grad("dW", to64(Wd.grad), ref["dW"])


@pytest.mark.parametrize("N,D,V,chunk", [(300, 264, 1000, 128), (1100, 2048, 16411, 512)])
def test_norm_frozen_w(lce, N, D, V, chunk):
    """W frozen (LCE_FROZEN_W): loss, lse, dX and dgamma as with W trained, no dW;
    the second shape splits its dH tiles in vocabulary parts that the RMSNorm
    backward adds as it reads them."""
    X, g, W, y = _norm_case(N, D, V, seed=N + 3, n_ign=N // 20)
    loss, lse, dX, dgamma, dW = lce.norm_fwd_bwd(X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV),
                                                 eps=EPS, chunk=chunk, compute_dW=False)
    torch.cuda.synchronize()
    assert dW is None
    ref = O.norm_forward_backward(X, g, EPS, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dX", to64(dX), ref["dX"])
    check_grad("dgamma", to64(dgamma), ref["dgamma"])
    Xd = X.to(DEV).requires_grad_(True)
    gd = g.to(DEV).requires_grad_(True)
    Wd = W.to(DEV)
    out = lce.norm_linear_cross_entropy(Xd, gd, Wd, y.to(DEV), eps=EPS, chunk=chunk)
    (out * 0.5).backward()
    torch.cuda.synchronize()
    check_grad("dX (autograd, W frozen)", to64(Xd.grad), 0.5 * ref["dX"])
    check_grad("dgamma (autograd, W frozen)", to64(gd.grad), 0.5 * ref["dgamma"])
