"""The token-sharded call on the GPU through a one-rank NCCL group (the
exchange logic with two ranks is tested over gloo on the CPU): with every row
on one rank it must match the fp64 oracle on the whole batch, and give the
single-GPU fused call's loss, lse, dH and dW."""
import os
import socket

import numpy as np
import pytest
import torch

from lce_synth import make_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


@pytest.fixture(scope="module")
def group():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import torch.distributed as dist
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1)
    yield dist.group.WORLD
    dist.destroy_process_group()


@pytest.mark.parametrize("compute_dW", [True, False])
def test_one_rank_sharded_equals_fused(group, compute_dW):
    import linear_cross_entropy_chunked_gb300 as lce
    H, W, y = make_inputs(1500, 1024, 9000, seed=12, n_ignored=60, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.sharded_fwd_bwd(Hd, Wd, yd, group=group, chunk=512,
                                            compute_dW=compute_dW)
    rl, rlse, rdH, rdW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=512, compute_dW=compute_dW)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    check_loss(loss.item(), ref["loss"])
    check_lse(to64(lse), ref["lse"])
    check_grad("dH vs oracle", to64(dH), ref["dH"])
    if compute_dW:
        check_grad("dW vs oracle", to64(dW), ref["dW"])
    assert abs(loss.item() - rl.item()) <= 1e-6 * abs(rl.item())
    assert torch.equal(lse, rlse)
    check_grad("dH", to64(dH), to64(rdH))
    if compute_dW:
        check_grad("dW", to64(dW), to64(rdW))
    else:
        assert dW is None


def test_count_valid_matches_the_oracle():
    """lce_count_valid counts the labels in [0, V) other than ignore_index (the
    oracle's reading: out-of-range labels count as ignored)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as lce
    lce.build()
    for N, V, seed in ((7, 10, 1), (5000, 300, 2), (70000, 32000, 3), (0, 10, 4)):
        rng = np.random.default_rng(seed)
        y = rng.integers(-5, V + 5, size=N).astype(np.int64)
        y[rng.random(N) < 0.1] = -100
        yt = torch.from_numpy(y)
        got = lce.count_valid(yt.to(DEV), V).item()
        valid, _ = O.valid_rows(y, V)
        assert got == int(valid.sum())


@pytest.mark.parametrize("factor", [1, 3])
def test_sharded_normaliser_matches_the_oracle(factor):
    """lce_fwd_bwd_sharded with a given total count N_total: the loss is this
    call's loss sum / N_total and G carries 1 / N_total (oracle: reduction sum with
    dloss = 1 / N_total)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as lce
    lce.build()
    H, W, y = make_inputs(900, 264, 3000, seed=13, n_ignored=31, w_std=0.05)
    y[4] = 3000                            # out of range: ignored, as in every call
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    n_local = lce.count_valid(yd, 3000)
    n_total = n_local * factor
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=256, n_valid_total=n_total)
    torch.cuda.synchronize()
    nt = int(n_total.item())
    ref = O.forward_backward(H, W, y, dloss=1.0 / nt, reduction="sum")
    check_loss(loss.item(), ref["loss"] / nt)
    check_lse(to64(lse), ref["lse"])
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dW", to64(dW), ref["dW"])
