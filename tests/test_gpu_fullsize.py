"""Parity at full size: the Llama-3-8B and Qwen-2.5-7B LM-head workloads, run
through the C ABI in the launch configuration the benchmark times (fused
forward + backward, chunk from the workload), checked on outputs the fp64 oracle
computes one by one and on properties that hold at any size:

  * lse of sampled rows (oracle: that row's full logit vector);
  * dH of sampled rows (oracle: that row's softmax - onehot times W);
  * dW of sampled vocabulary rows (oracle: the column of G over all N rows, with
    every row's lse taken from the GPU; those lse are checked on the samples);
  * loss = mean over valid rows of (lse_i - z_{i,y_i}), with z_{i,y_i} = h_i . w_{y_i}
    from the oracle for every row and lse_i from the GPU;
  * sum over the vocabulary of dW is 0 (rows of softmax - onehot sum to 0);
  * dH rows of ignored labels are exactly 0.
"""
import math

import numpy as np
import pytest
import torch

from lce_synth import IGNORE_INDEX, WORKLOADS, workload_inputs
from oracle import lce_oracle as O
from tests.gpu_util import GRAD_REL, LOSS_REL, LSE_ABS, check_grad, check_lse

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
W_STD = 0.02      # the workloads' W ~ N(0, 0.02^2)


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


def _cases():
    out = []
    for name in ("llama3-8b", "qwen2.5-7b"):
        for chunk in WORKLOADS[name].chunks:
            out.append((name, chunk))
    return out


_inputs_cache = {}


def _inputs(name):
    if name not in _inputs_cache:
        _inputs_cache.clear()
        _inputs_cache[name] = workload_inputs(name)
    return _inputs_cache[name]


@pytest.mark.parametrize("name,chunk", _cases())
def test_fullsize_sampled_parity(lce, name, chunk):
    wl = WORKLOADS[name]
    H, W, y = _inputs(name)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    lse_g = lse.double().cpu().numpy()
    y_np = y.numpy()
    valid = y_np != IGNORE_INDEX
    n_valid = int(valid.sum())
    assert n_valid == wl.N - wl.n_ignored

    rng = np.random.default_rng(1234 + chunk)
    # sampled rows: first / last row of a chunk, ragged positions, an ignored row
    rows = sorted(set([0, chunk - 1, chunk, wl.N - 1, int(np.nonzero(~valid)[0][0])] +
                      rng.choice(wl.N, 11, replace=False).tolist()))
    lse_o, zy_o = O.rows_lse_and_target(H, W, y, rows)
    check_lse(lse_g[rows], lse_o)

    dH_o = O.rows_dH(H, W, y, rows, n_valid)
    dH_g = dH[rows].float().double().cpu().numpy()
    check_grad("dH rows", dH_g, dH_o)

    vrows = sorted(set([0, wl.V - 1] + rng.choice(wl.V, 6, replace=False).tolist() +
                       [int(y_np[valid][0])]))
    dW_o = O.cols_dW(H, W, y, vrows, lse_g, n_valid)
    dW_g = dW[vrows].double().cpu().numpy()
    check_grad("dW rows", dW_g, dW_o)

    # loss against every row's target logit (oracle) and the GPU lse
    Hf = H.double().numpy()
    Wf = W.double().numpy()
    idx = np.nonzero(valid)[0]
    zy_all = np.einsum("ij,ij->i", Hf[idx], Wf[y_np[idx]])
    loss_ref = float(np.sum(lse_g[idx] - zy_all) / n_valid)
    assert abs(loss.item() - loss_ref) <= LOSS_REL * abs(loss_ref)
    # level at initialisation, independent of any implementation: a row's logits are
    # Gaussian with variance |h|^2 sigma_w^2 (E = D sigma_w^2), so E[lse] = log V +
    # D sigma_w^2 / 2 up to O(1/V), and E[z_y] = 0 (W is drawn independently of the
    # labels); the mean over ~15k rows has a spread of ~0.01
    expected = math.log(wl.V) + wl.D * W_STD ** 2 / 2
    assert abs(loss.item() - expected) < 0.05, (loss.item(), expected)

    # invariants on the whole GPU output. Rows of softmax - onehot sum to 0, so
    # sum_v dW[v, d] = sum_i H_id * sum_v (G~_iv - G_iv), where G~ is G rounded to
    # bf16 (at most 2 ulp = 2^-8 relative, P' and then G being rounded), and
    # sum_v |G_iv| <= 2 * dloss / N_valid: |sum_v dW[v, d]| <= 2^-7 / N_valid * sum_i |H_id|.
    colsum = dW.sum(dim=0).abs().double().cpu().numpy()
    bound = 2.0 ** -7 / n_valid * np.abs(Hf[idx]).sum(axis=0)
    assert np.all(colsum <= bound), float(np.max(colsum / bound))
    ign = torch.from_numpy(~valid).to(DEV)
    assert dH[ign].abs().max().item() == 0.0


def test_fullsize_chunk_sweep_agrees(lce):
    """The Qwen workload at chunk 512, 1024 and 2048 gives the same results."""
    H, W, y = _inputs("qwen2.5-7b")
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    ref = None
    for chunk in (512, 1024, 2048):
        loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
        torch.cuda.synchronize()
        cur = (loss.item(), lse.clone(), dH[:512].float().clone(), dW[:2048].clone())
        if ref is None:
            ref = cur
            continue
        assert abs(cur[0] - ref[0]) <= 1e-5 * abs(ref[0])
        assert (cur[1] - ref[1]).abs().max().item() <= 1e-5
        assert (cur[2] - ref[2]).abs().max().item() <= GRAD_REL * ref[2].abs().max().item()
        assert (cur[3] - ref[3]).abs().max().item() <= GRAD_REL * ref[3].abs().max().item()
        del loss, lse, dH, dW
    _inputs_cache.clear()
