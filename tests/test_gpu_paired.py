"""The paired-chunk schedule (two chunk buffers: chunks go in pairs, each chunk's
logits and dH computed by itself, one dW contraction over both chunks of a pair)
against the fp64 oracle, beside the one-buffer schedule (LCE_LOW_MEMORY: one dW
contraction per chunk). The two differ only in the rounding order of dW and of
split dH contractions, so each is checked against the oracle and for
determinism; lse and the loss come out of the same arithmetic in both and must be
the same bits."""
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


CASES = [
    # N, D, V, chunk, ignored
    (1000, 520, 3000, 384, 40),      # one pair and a ragged last chunk by itself
    (900, 264, 4000, 256, 30),       # two pairs, the second chunk of the last pair ragged
    (2500, 1024, 9000, 512, 60),     # vocabulary-split dH tiles (the first chunk of a pair alone)
    (1536, 256, 40000, 256, 30),     # three full pairs, wide vocabulary
    (129, 64, 257, 64, 5),           # a pair and a last chunk of one row
    (500, 64, 1000, 100, 9),         # chunk not a multiple of 8: one buffer, no pairs
    (40, 8, 300, 8, 3),              # chunks of 8 rows (the second chunk's H^T from column 8), D = 8
    (100, 64, 513, 16, 5),           # chunks of 16: a pair's dW contraction in one k block
    (4096, 1024, 32000, 1024, 100),  # four full chunks, two pairs, no ignored-row edge
]


def _check(out, ref):
    check_loss(out[0].item(), ref["loss"])
    check_lse(to64(out[1]), ref["lse"])
    check_grad("dH", to64(out[2]), ref["dH"])
    check_grad("dW", to64(out[3]), ref["dW"])


@pytest.mark.parametrize("N,D,V,chunk,n_ign", CASES)
def test_fused_pairs_match_oracle(lce, N, D, V, chunk, n_ign):
    H, W, y = make_inputs(N, D, V, seed=N + V, n_ignored=n_ign, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = torch.tensor([0.8], dtype=torch.float32, device=DEV)
    a = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk)
    a2 = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk)
    b = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, low_memory=True)
    torch.cuda.synchronize()
    for x, z in zip(a, a2):
        assert torch.equal(x, z)                    # deterministic
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])   # loss and lse: same arithmetic
    ref = O.forward_backward(H, W, y, dloss=0.8)
    _check(a, ref)
    _check(b, ref)


@pytest.mark.parametrize("N,D,V,chunk,n_ign", CASES[:3])
def test_backward_pairs_match_oracle(lce, N, D, V, chunk, n_ign):
    H, W, y = make_inputs(N, D, V, seed=N + V + 1, n_ignored=n_ign, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    a = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk)
    a2 = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk)
    b = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, low_memory=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], a2[0]) and torch.equal(a[1], a2[1])
    ref = O.forward_backward(H, W, y)
    for got in (a, b):
        check_grad("dH", to64(got[0]), ref["dH"])
        check_grad("dW", to64(got[1]), ref["dW"])


@pytest.mark.parametrize("reduction", ["sum", "none"])
def test_pairs_reductions_and_accumulation(lce, reduction):
    N, D, V, chunk = 1100, 392, 5000, 256
    H, W, y = make_inputs(N, D, V, seed=77, n_ignored=25, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    rng = np.random.default_rng(3)
    dl_host = rng.standard_normal(N) if reduction == "none" else 0.6
    dl = torch.tensor(np.atleast_1d(dl_host), dtype=torch.float32, device=DEV)
    gen = torch.Generator().manual_seed(9)
    dH0 = (torch.randn(N, D, generator=gen) * 1e-4).to(torch.bfloat16).to(DEV)
    dW0 = (torch.randn(V, D, generator=gen) * 1e-4).to(DEV)
    ref = O.forward_backward(H, W, y, dloss=dl_host, reduction=reduction)
    for low in (False, True):
        dH, dW = dH0.clone(), dW0.clone()
        out = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, dH=dH, dW=dW,
                              reduction=reduction, accumulate=("dW", "dH"), low_memory=low)
        torch.cuda.synchronize()
        check_grad("dH", to64(out[2]), ref["dH"] + to64(dH0))
        check_grad("dW", to64(out[3]), ref["dW"] + to64(dW0))


def test_pairs_fp16(lce):
    N, D, V, chunk = 900, 264, 4000, 256
    H, W, y = make_inputs(N, D, V, seed=78, n_ignored=20, w_std=0.05, dtype="fp16")
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    ref = O.forward_backward(H, W, y)
    for low in (False, True):
        out = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, low_memory=low)
        torch.cuda.synchronize()
        check_loss(out[0].item(), ref["loss"])
        check_grad("dH", to64(out[2]), ref["dH"])
        check_grad("dW", to64(out[3]), ref["dW"])
