"""Token-sharded data parallelism for the fused loss: each rank holds its own rows
(H, y) and the whole W; the loss is the mean over the valid rows of all ranks.

The rows are independent except for three global quantities, so the exchange is
three all-reduces (sums): the valid-row count before G is formed (8 bytes), the
loss sum, and dW (V x D fp32). dH stays on its rank. Each rank runs the
library's fused call with reduction "sum" and dloss = 1 / N_valid(global), which
makes its G rows exactly those of the global mean
(G_ij = (p_ij - 1[j = y_i]) / N_valid); the sum of the ranks' dW is then the
global dW, and the sum of their loss sums over N_valid the global loss.
Labels outside [0, V) that are not ignore_index count as ignored, as in the
single-GPU call."""
from __future__ import annotations

import torch

from . import _binding


def count_valid(y: torch.Tensor, V: int, ignore_index: int = _binding.IGNORE_INDEX) -> torch.Tensor:
    """Rows of y with a label in [0, V) (int64, 1 element, on y's device)."""
    ok = (y != ignore_index) & (y >= 0) & (y < V)
    return ok.sum().reshape(1).to(torch.int64)


def sharded_fwd_bwd(H, W, y, group=None, chunk: int = 1024,
                    ignore_index: int = _binding.IGNORE_INDEX, compute_dW: bool = True,
                    fwd_bwd=None):
    """(loss, lse, dH, dW) of this rank's rows for the global mean loss over all
    ranks of `group`: loss and dW are the global ones (identical on every rank),
    lse and dH this rank's rows. compute_dW=False: W frozen, no dW exchange.
    fwd_bwd: the per-rank fused call (default: the library's lce_fwd_bwd)."""
    import torch.distributed as dist

    fwd_bwd = fwd_bwd or _binding.lce_fwd_bwd
    V = W.shape[0]
    n_valid = count_valid(y, V, ignore_index)
    dist.all_reduce(n_valid, group=group)
    # 1 / N_valid on the device (0 when no row of any rank is valid): no host sync
    n = n_valid.to(torch.float64)
    inv_n = torch.where(n > 0, 1.0 / n.clamp(min=1.0), torch.zeros_like(n))
    dloss = inv_n.to(torch.float32).contiguous()
    loss_sum, lse, dH, dW = fwd_bwd(H, W, y, dloss=dloss, chunk=chunk, ignore_index=ignore_index,
                                    reduction="sum", compute_dW=compute_dW)
    loss = loss_sum.reshape(1).to(torch.float64)
    dist.all_reduce(loss, group=group)
    loss = (loss * inv_n).to(torch.float32).reshape(())
    if dW is not None:
        dist.all_reduce(dW, group=group)
    return loss, lse, dH, dW
