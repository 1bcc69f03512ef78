"""Token-sharded data parallelism for the fused loss: each rank holds its own rows
(H, y) and the whole W; the loss is the mean over the valid rows of all ranks.

The rows are independent except for three global quantities, so the exchange is
three all-reduces (sums): the valid-row count before G is formed (8 bytes), the
loss, and dW (V x D fp32). dH stays on its rank. Every step of the method runs
in the library: the rank's count (lce_count_valid) and its fused call with the
all-reduced count as the normaliser of the mean (lce_fwd_bwd_sharded), whose G
rows are then exactly those of the global mean, G_ij = (p_ij - 1[j = y_i]) /
N_valid(global), and whose loss is the rank's share of the global mean. This
module only moves those results between the ranks. Labels outside [0, V) that
are not ignore_index count as ignored, as in the single-GPU call."""
from __future__ import annotations

from . import _binding


def sharded_fwd_bwd(H, W, y, group=None, chunk: int = 1024,
                    ignore_index: int = _binding.IGNORE_INDEX, compute_dW: bool = True,
                    fwd_bwd=None, count=None):
    """(loss, lse, dH, dW) of this rank's rows for the global mean loss over all
    ranks of `group`: loss and dW are the global ones (identical on every rank),
    lse and dH this rank's rows. compute_dW=False: W frozen, no dW exchange.
    fwd_bwd / count: the per-rank fused call and valid-row count (default: the
    library's lce_fwd_bwd with n_valid_total, and lce_count_valid)."""
    import torch.distributed as dist

    fwd_bwd = fwd_bwd or _binding.lce_fwd_bwd
    count = count or _binding.count_valid
    n_valid = count(y, W.shape[0], ignore_index)
    dist.all_reduce(n_valid, group=group)
    loss, lse, dH, dW = fwd_bwd(H, W, y, chunk=chunk, ignore_index=ignore_index,
                                compute_dW=compute_dW, n_valid_total=n_valid)
    dist.all_reduce(loss, group=group)
    if dW is not None:
        dist.all_reduce(dW, group=group)
    return loss.reshape(()), lse, dH, dW
