"""Parity at full size: the Llama-3-8B and Qwen-2.5-7B LM-head workloads, run
through the C ABI in the launch configuration the benchmark times (fused
forward + backward, chunk from the workload), and on the Llama-3 head the
separate forward + backward (the recompute path), the fused call's other
schedules (one chunk buffer; W frozen), fp16 inputs and the RMSNorm path. Every expected value comes
from the fp64 oracle alone; no GPU output enters a reference:

  * lse of all N rows and the loss: the oracle's forward over every row (the
    logits materialised in row blocks on the host, one run per workload, shared
    by the cases of that workload);
  * dH of sampled rows (>= 64: the first and the last row of every chunk, an
    ignored row, random rows), from that row's softmax - onehot times W;
  * dW of sampled vocabulary rows (>= 32: ids 0..7, which are the most frequent
    ids of a Zipf workload, ids of the last 128-column slab, a label that occurs,
    random ids), from the column of G over all N rows with the oracle's lse;
  * properties that hold at any size: sum over the vocabulary of dW is 0 (rows of
    softmax - onehot sum to 0), dH rows of ignored labels are exactly 0, and the
    loss sits at its level at initialisation.
"""
import math

import numpy as np
import pytest
import torch

from lce_synth import IGNORE_INDEX, WORKLOADS, workload_inputs
from oracle import lce_oracle as O
from tests.gpu_util import GRAD_REL, check_grad, check_loss, check_lse

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
_oracle_cache = {}


def _inputs(name):
    if name not in _inputs_cache:
        _inputs_cache.clear()
        _inputs_cache[name] = workload_inputs(name)
    return _inputs_cache[name]


def _oracle_forward(name):
    """The oracle's loss and lse over every row of the workload (fp64)."""
    if name not in _oracle_cache:
        H, W, y = _inputs(name)
        loss, lse, n_valid, n_bad = O.forward(H, W, y)
        assert n_bad == 0
        _oracle_cache[name] = (loss, lse, n_valid)
    return _oracle_cache[name]


def _sample_rows(wl, chunk, valid, rng):
    """The first and the last row of every chunk, the first ignored row, and
    random rows up to at least 64 in all."""
    rows = set()
    for r0 in range(0, wl.N, chunk):
        rows.add(r0)
        rows.add(min(r0 + chunk, wl.N) - 1)
    rows.add(int(np.nonzero(~valid)[0][0]))
    want = max(64, len(rows) + 8)
    for r in rng.permutation(wl.N):
        if len(rows) >= want:
            break
        rows.add(int(r))
    return sorted(rows)


def _sample_vocab(wl, y_np, valid, rng):
    """Vocabulary rows of dW to check: ids 0..7 (the most frequent ids of a Zipf
    workload, where rank k is id k), ids across the last 128-column slab, a label
    that occurs, and random ids up to at least 32 in all."""
    last0 = 128 * ((wl.V - 1) // 128)       # first id of the last 128-column slab
    ids = set(range(8)) | {last0, (last0 + wl.V) // 2, wl.V - 2, wl.V - 1,
                           int(y_np[valid][0])}
    for v in rng.permutation(wl.V):
        if len(ids) >= 34:
            break
        ids.add(int(v))
    return sorted(ids)


def _check_against_oracle(name, chunk, H, W, y, loss, lse, dH, dW, rng, oracle=None):
    wl = WORKLOADS[name]
    loss_o, lse_o, n_valid = oracle if oracle is not None else _oracle_forward(name)
    y_np = y.numpy()
    valid = y_np != IGNORE_INDEX
    assert n_valid == wl.N - wl.n_ignored

    # every row's lse, and the loss, against the oracle's forward
    check_lse(lse.double().cpu().numpy(), lse_o)
    check_loss(loss.item(), loss_o)

    rows = _sample_rows(wl, chunk, valid, rng)
    assert len(rows) >= 64
    dH_o = O.rows_dH(H, W, y, rows, n_valid)
    check_grad("dH rows", dH[rows].float().double().cpu().numpy(), dH_o)

    ign = torch.from_numpy(~valid).to(DEV)
    assert dH[ign].abs().max().item() == 0.0

    # level at initialisation, independent of any implementation: a row's logits are
    # Gaussian with variance |h|^2 sigma_w^2 (E = D sigma_w^2), so E[lse] = log V +
    # D sigma_w^2 / 2 up to O(1/V), and E[z_y] = 0 (W is drawn independently of the
    # labels); the mean over ~15k rows has a spread of ~0.01
    expected = math.log(wl.V) + wl.D * W_STD ** 2 / 2
    assert abs(loss.item() - expected) < 0.05, (loss.item(), expected)

    if dW is None:      # W frozen: no dW computed
        return
    vrows = _sample_vocab(wl, y_np, valid, rng)
    assert len(vrows) >= 32
    dW_o = O.cols_dW(H, W, y, vrows, lse_o, n_valid)
    check_grad("dW rows", dW[vrows].double().cpu().numpy(), dW_o)

    # invariants on the whole GPU output. Rows of softmax - onehot sum to 0, so
    # sum_v dW[v, d] = sum_i H_id * sum_v (G~_iv - G_iv), where G~ is G rounded to
    # bf16 (at most 2 ulp = 2^-8 relative, P' and then G being rounded), and
    # sum_v |G_iv| <= 2 * dloss / N_valid: |sum_v dW[v, d]| <= 2^-7 / N_valid * sum_i |H_id|.
    Hf = H.double().numpy()
    colsum = dW.sum(dim=0).abs().double().cpu().numpy()
    bound = 2.0 ** -7 / n_valid * np.abs(Hf[valid]).sum(axis=0)
    assert np.all(colsum <= bound), float(np.max(colsum / bound))


def test_fullsize_separate_path_matches_oracle(lce):
    """lce_forward, then lce_backward from the saved lse (the logits recomputed
    with the gradient epilogue), on the Llama-3 head at the benchmark's chunk."""
    name = "llama3-8b"
    chunk = WORKLOADS[name].chunks[0]
    H, W, y = _inputs(name)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    dH, dW = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk)
    torch.cuda.synchronize()
    del Hd, Wd, yd
    _check_against_oracle(name, chunk, H, W, y, loss, lse, dH, dW, np.random.default_rng(77))


@pytest.mark.parametrize("variant", ["low_memory", "frozen_w"])
def test_fullsize_other_schedules_match_oracle(lce, variant):
    """The fused call's other schedules on the Llama-3 head at the benchmark's
    chunk: one chunk buffer (LCE_LOW_MEMORY: one dW contraction per chunk), and W
    frozen (no dW; each chunk's dH with the next chunk's logits beside it)."""
    name = "llama3-8b"
    chunk = WORKLOADS[name].chunks[0]
    H, W, y = _inputs(name)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    if variant == "low_memory":
        loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, low_memory=True)
    else:
        loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, compute_dW=False)
        assert dW is None
    torch.cuda.synchronize()
    del Hd, Wd, yd
    _check_against_oracle(name, chunk, H, W, y, loss, lse, dH, dW,
                          np.random.default_rng(4321 if variant == "low_memory" else 8765))


def test_fullsize_fp16_matches_oracle(lce):
    """fp16 H and W (LCE_INPUT_FP16: fp16 MMAs, G stored as (p - onehot) * 2^14)
    on the Llama-3 head at the benchmark's chunk, drawn as the benchmark's fp16
    run draws them; the oracle on the same fp16 values."""
    from lce_synth import make_inputs
    name = "llama3-8b"
    wl = WORKLOADS[name]
    chunk = wl.chunks[0]
    H, W, y = make_inputs(wl.N, wl.D, wl.V, wl.seed, wl.labels, wl.n_ignored, dtype="fp16")
    assert H.dtype == torch.float16 and W.dtype == torch.float16
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    del Hd, Wd, yd
    assert dH.dtype == torch.float16
    loss_o, lse_o, n_valid, n_bad = O.forward(H, W, y)
    assert n_bad == 0
    _check_against_oracle(name, chunk, H, W, y, loss, lse, dH, dW, np.random.default_rng(1616),
                          oracle=(loss_o, lse_o, n_valid))


@pytest.mark.parametrize("name,chunk", _cases())
def test_fullsize_fused_matches_oracle(lce, name, chunk):
    H, W, y = _inputs(name)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk)
    torch.cuda.synchronize()
    del Hd, Wd, yd
    _check_against_oracle(name, chunk, H, W, y, loss, lse, dH, dW,
                          np.random.default_rng(1234 + chunk))


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
    _oracle_cache.clear()


def test_fullsize_norm_path_matches_oracle(lce):
    """Final RMSNorm + LM head + cross-entropy (lce_norm_fwd_bwd) on the Llama-3
    head at the benchmark's chunk, with the inputs the benchmark's norm path
    draws. Expected values from the oracle alone: H = RMSNorm(X) rounded to bf16,
    then the oracle's forward over every row (lse, loss), dX of sampled rows
    (that row's dH through the RMSNorm backward), dW of sampled vocabulary rows.
    dgamma sums over every row's dH and is checked against the full oracle at
    the Llama-2 shape (tests/test_gpu_norm.py)."""
    from lce_synth import workload_norm_inputs
    name = "llama3-8b"
    wl = WORKLOADS[name]
    chunk = wl.chunks[0]
    eps = 1e-6
    X, g, W, y = workload_norm_inputs(name)
    out = lce.norm_fwd_bwd(X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV), eps=eps, chunk=chunk)
    torch.cuda.synchronize()
    loss, lse, dX, dgamma, dW = out
    assert torch.isfinite(dgamma).all()

    H_o = O.round_bf16(O.rmsnorm_forward(X, g, eps)[0])
    loss_o, lse_o, n_valid, n_bad = O.forward(H_o, W, y)
    assert n_bad == 0 and n_valid == wl.N - wl.n_ignored
    check_lse(lse.double().cpu().numpy(), lse_o)
    check_loss(loss.item(), loss_o)

    y_np = y.numpy()
    valid = y_np != IGNORE_INDEX
    rng = np.random.default_rng(2468)
    rows = _sample_rows(wl, chunk, valid, rng)
    dH_rows = O.rows_dH(H_o, W, y, rows, n_valid)
    dX_o, _ = O.rmsnorm_backward(X[rows], g, eps, dH_rows)
    check_grad("dX rows", dX[rows].double().cpu().numpy(), dX_o)

    vrows = _sample_vocab(wl, y_np, valid, rng)
    dW_o = O.cols_dW(H_o, W, y, vrows, lse_o, n_valid)
    check_grad("dW rows", dW[vrows].double().cpu().numpy(), dW_o)
