"""dH tiles split along the vocabulary. A chunk whose dH tiles (256 rows x 512
columns on a CTA pair) are too few to run beside the dW tiles has each of them
split in 2 to 4 vocabulary parts; every part leaves fp32 partial sums that a
combining kernel (or the RMSNorm backward) adds in a fixed order.

The shapes below reach (tiles = row pairs x 512-column blocks of a full chunk;
parts = ceil(28 / tiles), at most 4, over the 64-column k blocks of V):

    N 1000, D 1024, V 8229,  chunk 256   1 x 2 tiles -> 4 parts (33,33,33,30 k blocks)
    N 1100, D 3584, V 9000,  chunk 512   2 x 7 tiles -> 2 parts (71,70)
    N  600, D 2560, V 8500,  chunk 512   2 x 5 tiles -> 3 parts (45,45,43)
    N  777, D 1536, V 16411, chunk 384   2 x 3 tiles -> 4 parts (65,65,65,62); 3 row
                                         blocks per chunk (a pair's second tile past
                                         the rows), a last chunk of 9 rows

each against the fp64 oracle through every entry point that produces dH."""
import numpy as np
import pytest
import torch

from lce_synth import make_inputs, make_norm_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [(1000, 1024, 8229, 256), (1100, 3584, 9000, 512), (600, 2560, 8500, 512),
         (777, 1536, 16411, 384)]


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


def _inputs(N, D, V, dtype="bf16"):
    return make_inputs(N, D, V, seed=N + D + V, labels="uniform", n_ignored=N // 25, w_std=0.05,
                       dtype=dtype)


@pytest.mark.parametrize("N,D,V,chunk", CASES)
def test_split_dh_all_paths_match_oracle(lce, N, D, V, chunk):
    H, W, y = _inputs(N, D, V)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = torch.tensor([1.7], device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk)
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, dloss=dl, chunk=chunk)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y, dloss=1.7)
    check_loss(loss.item(), ref["loss"])
    check_loss(floss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    for name, got, exp in (("dH", dH, ref["dH"]), ("dW", dW, ref["dW"]),
                           ("dH (backward)", bdH, ref["dH"]), ("dW (backward)", bdW, ref["dW"])):
        check_grad(name, to64(got), exp)
    # ignored rows: exactly zero, whatever the parts hold
    ign = (y == -100).numpy()
    assert not np.any(to64(dH)[ign]) and not np.any(to64(bdH)[ign])


@pytest.mark.parametrize("N,D,V,chunk", [CASES[0], CASES[2]])
def test_split_dh_reduction_none(lce, N, D, V, chunk):
    H, W, y = _inputs(N, D, V)
    dl_host = np.random.default_rng(N).standard_normal(N)
    dl = torch.tensor(dl_host, dtype=torch.float32, device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), dloss=dl, chunk=chunk,
                                        reduction="none")
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y, dloss=dl_host, reduction="none")
    assert np.abs(to64(loss) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dW", to64(dW), ref["dW"])


@pytest.mark.parametrize("acc", [("dH",), ("dW", "dH")])
@pytest.mark.parametrize("N,D,V,chunk", [CASES[1], CASES[3]])
def test_split_dh_accumulate(lce, N, D, V, chunk, acc):
    H, W, y = _inputs(N, D, V)
    gen = torch.Generator().manual_seed(3)
    dH0 = (torch.randn(N, D, generator=gen) * 1e-4).to(torch.bfloat16).to(DEV)
    dW0 = (torch.randn(V, D, generator=gen) * 1e-4).to(DEV)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, dH=dH0.clone(), dW=dW0.clone(),
                                        accumulate=acc)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, dH=dH0.clone(), dW=dW0.clone(),
                                accumulate=acc)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    exp_dH = ref["dH"] + to64(dH0)
    exp_dW = ref["dW"] + (to64(dW0) if "dW" in acc else 0.0)
    for name, got, exp in (("dH", dH, exp_dH), ("dW", dW, exp_dW), ("dH (backward)", bdH, exp_dH),
                           ("dW (backward)", bdW, exp_dW)):
        check_grad(name, to64(got), exp)


@pytest.mark.parametrize("N,D,V,chunk", [CASES[0], CASES[3]])
def test_split_dh_fp16(lce, N, D, V, chunk):
    H, W, y = _inputs(N, D, V, dtype="fp16")
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    assert dH.dtype == torch.float16
    ref = O.forward_backward(H, W, y)
    check_loss(loss.item(), ref["loss"])
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dW", to64(dW), ref["dW"])


@pytest.mark.parametrize("N,D,V,chunk", [CASES[1], CASES[2]])
def test_split_dh_norm_path(lce, N, D, V, chunk):
    """The RMSNorm backward reads the chunk's dH as the sum of the parts."""
    X, g, W, y = make_norm_inputs(N, D, V, seed=N + V, n_ignored=N // 25, w_std=0.05)
    loss, lse, dX, dgamma, dW = lce.norm_fwd_bwd(X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV),
                                                 eps=1e-6, chunk=chunk)
    torch.cuda.synchronize()
    ref = O.norm_forward_backward(X, g, 1e-6, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dX", to64(dX), ref["dX"])
    check_grad("dgamma", to64(dgamma), ref["dgamma"])
    check_grad("dW", to64(dW), ref["dW"])


def test_split_dh_bit_reproducible_and_close_to_unsplit(lce, monkeypatch):
    """The parts are added in a fixed order: two runs agree bit for bit. The
    one-CTA-per-tile variant does not split; its dH agrees within rounding."""
    N, D, V, chunk = CASES[3]
    H, W, y = _inputs(N, D, V)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    a = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    b = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    for x, z in zip(a, b):
        assert torch.equal(x, z)
    monkeypatch.setenv("LCE_GEMM_CLUSTER", "1")
    c = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    check_grad("dH (split vs one part)", to64(a[2]), to64(c[2]))
    assert np.abs(to64(a[2]) - to64(c[2])).max() <= 2.0 ** -7 * np.abs(to64(c[2])).max()
