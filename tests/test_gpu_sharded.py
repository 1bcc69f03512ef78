"""The token-sharded call on the GPU through a one-rank NCCL group (the
exchange logic with two ranks is tested over gloo on the CPU): with every row
on one rank it must give the single-GPU fused call's loss, lse, dH and dW (up to
the rounding of 1 / N_valid, formed on the host side of the call here and inside
the kernels there)."""
import os
import socket

import pytest
import torch

from lce_synth import make_inputs
from tests.gpu_util import check_grad, to64

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
    assert abs(loss.item() - rl.item()) <= 1e-6 * abs(rl.item())
    assert torch.equal(lse, rlse)
    check_grad("dH", to64(dH), to64(rdH))
    if compute_dW:
        check_grad("dW", to64(dW), to64(rdW))
    else:
        assert dW is None
