"""Cross-entropy over precomputed logits through the C ABI against the fp64
oracle on the same logit values.

The library picks one of two kernels by row size. Rows that fit in the
registers of a cluster of at most 8 CTAs (512 threads x 16 vectors of 16 bytes
each: V up to 524288 bf16 / 262144 fp32) go to the cluster kernel, with the
smallest cluster that holds the row, the fewest vectors per thread (4, 8 or 16)
that hold a segment, and as many copy buffers (up to 3) as fit in 227 KB of
shared memory; larger rows go to the streaming kernel. The shapes below reach:

    bf16 V = 7, 1003, 5000            cluster 1, 4 vectors/thread, 3 buffers (ragged tails)
    bf16 V = 32000                    cluster 1, 8 vectors/thread
    fp32 V = 32000                    cluster 1, 16 vectors/thread, 1 buffer
    bf16 V = 65537, fp32 V = 32769    cluster 2, one-element tail
    bf16 V = 100003 (ld 100008)       cluster 2, 2 buffers, 3-element tail
    bf16 V = 128256                   cluster 2, 1 buffer
    bf16 V = 152064                   cluster 3
    fp32 V = 128256                   cluster 4
    fp32 V = 152064                   cluster 5
    bf16 V = 500000                   cluster 8
    bf16 V = 600000, fp32 V = 300000  streaming kernel
    fp16 logits take the bf16 shapes (same element size).
"""
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


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
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


def _labels_and_dloss(N, V, reduction, seed):
    rng = np.random.default_rng(seed)
    y = torch.from_numpy(rng.integers(0, V, size=N))
    y[::7] = -100
    dl = torch.from_numpy(rng.standard_normal(N)).float() if reduction == "none" else torch.tensor([1.3])
    return y, dl


def _check_against_oracle(Z, y, dl, reduction, loss, lse, dZ):
    ref = O.ce_from_logits(Z.double().numpy(), y.numpy(),
                           dloss=dl.double().numpy() if reduction == "none" else 1.3,
                           reduction=reduction)
    check_lse(to64(lse), ref["lse"])
    if reduction == "none":
        assert np.abs(to64(loss) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    else:
        check_loss(loss.item(), ref["loss"])
    check_grad("dZ", to64(dZ), ref["dZ"])


@pytest.mark.parametrize("N,V,ld,dtype,reduction", [
    (300, 128256, 128256, torch.bfloat16, "mean"),    # cluster 2; ~4 rows per cluster
    (200, 100003, 100008, torch.bfloat16, "none"),    # cluster 2, 2 buffers, 3-element tail
    (160, 152064, 152064, torch.bfloat16, "sum"),     # cluster 3
    (100, 128256, 128256, torch.float32, "mean"),     # cluster 4
    (64, 152064, 152064, torch.float32, "none"),      # cluster 5
    (300, 32000, 32000, torch.float32, "sum"),        # cluster 1, 16 vectors per thread
    (90, 65537, 65544, torch.bfloat16, "mean"),       # cluster 2, one-element tail
    (70, 32769, 32772, torch.float32, "mean"),        # cluster 2, one-element tail
    (16, 500000, 500000, torch.bfloat16, "mean"),     # cluster 8
    (8, 600000, 600000, torch.bfloat16, "sum"),       # streaming kernel
    (200, 128256, 128256, torch.float16, "mean"),     # fp16, cluster 2
    (6, 600000, 600008, torch.float16, "none"),       # fp16, streaming kernel
    (12, 300000, 300000, torch.float32, "none"),      # streaming kernel
])
def test_ce_logits_cluster_shapes(lce, N, V, ld, dtype, reduction):
    Z, Zd = _logits(N, V, ld, dtype, seed=V + N)
    y, dl = _labels_and_dloss(N, V, reduction, seed=N)
    loss, lse, dZ = lce.ce_logits(Zd, y.to(DEV), dloss=dl.to(DEV), reduction=reduction)
    torch.cuda.synchronize()
    _check_against_oracle(Z, y, dl, reduction, loss, lse, dZ)


def test_ce_logits_labels_on_segment_edges_in_place(lce):
    """Labels on both sides of every segment boundary and in the last segment's
    ragged tail (read from global memory, not shared memory), gradient in place.
    bf16 V = 100003 runs as a 2-CTA cluster with 50008-element segments; the tail
    is elements 100000..100002."""
    V, ld = 100003, 100008
    edges = [0, 1, 50006, 50007, 50008, 50009, 99999, 100000, 100001, 100002]
    N = 3 * len(edges)
    Z, Zd = _logits(N, V, ld, torch.bfloat16, seed=11)
    y = torch.tensor(edges * 3, dtype=torch.int64)
    y[len(edges)] = -100
    ref = O.ce_from_logits(Z.double().numpy(), y.numpy())
    loss, lse, dZ = lce.ce_logits(Zd, y.to(DEV), inplace=True)
    torch.cuda.synchronize()
    assert dZ.data_ptr() == Zd.data_ptr()
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dZ in place", to64(Zd), ref["dZ"])
    # the target column carries (p - 1) * scale < 0
    dz = to64(Zd)
    for i, yi in enumerate(y.tolist()):
        if yi >= 0:
            assert dz[i, yi] < 0


def test_ce_logits_cluster_deterministic(lce):
    N, V = 96, 128256
    _, Zd = _logits(N, V, V, torch.bfloat16, seed=13)
    y = torch.randint(0, V, (N,)).to(DEV)
    a = lce.ce_logits(Zd, y)
    b = lce.ce_logits(Zd, y)
    torch.cuda.synchronize()
    for x, z in zip(a, b):
        assert torch.equal(x, z)


def test_ce_logits_bench_workload(lce):
    """The benchmark's CE-over-logits workload in its launch configuration: the
    Llama-3 logits N = 16384 x V = 128256 bf16 (4.2 GB), drawn as bench.py draws
    them, 5 % of the rows ignored, forward and the gradient written in place.
    The oracle, on a copy of the logits taken before the call, 512 rows at a
    time: every row's lse, the loss over all rows, dZ of sampled rows (the first
    and the last rows, an ignored row, random rows)."""
    N, V, n_ign = 16384, 128256, 819
    g = torch.Generator(device=DEV).manual_seed(3)
    Z = torch.randn(N, V, device=DEV, generator=g).mul_(1.3).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), device=DEV, generator=g)
    y[torch.randperm(N, device=DEV, generator=g)[:n_ign]] = -100
    Z0 = Z.clone()
    loss, lse, dZ = lce.ce_logits(Z, y, inplace=True)
    torch.cuda.synchronize()
    assert dZ.data_ptr() == Z.data_ptr()
    y_h = y.cpu()
    valid = (y_h != -100).numpy()
    n_valid = int(valid.sum())
    assert n_valid == N - n_ign
    lse_o = np.empty(N)
    loss_sum = 0.0
    for r in range(0, N, 512):
        ref = O.ce_from_logits(Z0[r:r + 512].cpu(), y_h[r:r + 512], reduction="sum")
        lse_o[r:r + 512] = ref["lse"]
        loss_sum += ref["loss"]
    check_lse(to64(lse), lse_o)
    check_loss(loss.item(), loss_sum / n_valid)
    rng = np.random.default_rng(16384)
    rows = sorted({0, 1, N - 2, N - 1, int(np.nonzero(~valid)[0][0])} |
                  {int(r) for r in rng.choice(N, 59, replace=False)})
    ref = O.ce_from_logits(Z0[rows].cpu(), y_h[rows], dloss=1.0 / n_valid, reduction="sum")
    check_grad("dZ rows", to64(dZ[rows]), ref["dZ"])
    assert dZ[torch.from_numpy(~valid).to(DEV)].abs().max().item() == 0.0
