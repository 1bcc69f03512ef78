"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on
the same seeded inputs, element by element at sizes the oracle finishes in
seconds, plus edge cases and invariants."""
import numpy as np
import pytest
import torch

from lce_synth import IGNORE_INDEX, WORKLOADS, make_inputs, workload_inputs
from oracle import lce_oracle as O
from tests.gpu_util import check_grad, check_loss, check_lse, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


DEV = "cuda:0"


def run_all_paths(lce, H, W, y, chunk, dloss=1.0):
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = torch.tensor([dloss], dtype=torch.float32, device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk)
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, dloss=dl, chunk=chunk)
    torch.cuda.synchronize()
    return dict(loss=loss.item(), lse=to64(lse), dH=to64(dH), dW=to64(dW),
                floss=floss.item(), flse=to64(flse), bdH=to64(bdH), bdW=to64(bdW))


def compare(r, ref):
    check_loss(r["loss"], ref["loss"])
    check_lse(r["lse"], ref["lse"])
    check_grad("dH", r["dH"], ref["dH"])
    check_grad("dW", r["dW"], ref["dW"])
    check_loss(r["floss"], ref["loss"])
    check_lse(r["flse"], ref["lse"])
    check_grad("dH (backward)", r["bdH"], ref["dH"])
    check_grad("dW (backward)", r["bdW"], ref["dW"])


def test_tiny_workload(lce):
    H, W, y = workload_inputs("tiny")
    r = run_all_paths(lce, H, W, y, chunk=1024)
    compare(r, O.forward_backward(H, W, y))


@pytest.mark.parametrize("N,D,V,chunk,n_ign,dloss", [
    (300, 264, 1000, 128, 17, 0.7),      # ragged in every dimension, several chunks
    (129, 64, 257, 64, 5, 1.0),          # one row past a tile, V one past a tile
    (1000, 520, 3000, 384, 40, 2.5),     # chunk not a multiple of the tile
    (77, 128, 100, 1024, 3, 1.0),        # N < chunk, V < one tile
    (256, 8, 513, 256, 0, 1.0),          # tiny D (one partial K block)
    (5000, 64, 3000, 64, 200, 1.0),      # 79 chunks: one tile counter per launch in the header
    (1, 64, 1000, 1024, 0, 1.0),         # a single row
    (2, 72, 9000, 1, 0, 0.5),            # chunk 1: every row its own chunk
])
def test_ragged_shapes(lce, N, D, V, chunk, n_ign, dloss):
    H, W, y = make_inputs(N, D, V, seed=N + D + V, labels="uniform", n_ignored=n_ign, w_std=0.05)
    r = run_all_paths(lce, H, W, y, chunk=chunk, dloss=dloss)
    compare(r, O.forward_backward(H, W, y, dloss=dloss))


@pytest.mark.parametrize("N,D,V,chunk", [
    (600, 8192, 20000, 256),     # a 70B-class hidden size: 128 k blocks per logits tile,
                                 # 16 wide dH column tiles, 32 dW column tiles
    (300, 16384, 5000, 128),     # 256 k blocks, 32 dH / 64 dW column tiles, 256 transpose columns
    (520, 12288, 9000, 192),     # D a multiple of 512 but not of 1024; chunk not of 128
    (257, 6152, 4099, 128),      # D a multiple of 8 only: ragged last k block and column tile
])
def test_large_hidden_sizes(lce, N, D, V, chunk):
    """Hidden sizes beyond the workloads' (up to 16384) through every path, against
    the full oracle."""
    H, W, y = make_inputs(N, D, V, seed=D + N, labels="uniform", n_ignored=N // 25, w_std=0.01)
    r = run_all_paths(lce, H, W, y, chunk=chunk, dloss=0.8)
    compare(r, O.forward_backward(H, W, y, dloss=0.8))


def test_two_word_vocabulary(lce):
    """V = 2: the loss is the logistic loss of the logit difference (pinned in the
    oracle's tests); every path against the full oracle."""
    H, W, y = make_inputs(300, 72, 2, seed=2, labels="uniform", n_ignored=9, w_std=0.1)
    r = run_all_paths(lce, H, W, y, chunk=128, dloss=1.0)
    compare(r, O.forward_backward(H, W, y))


def test_one_word_vocabulary(lce):
    """V = 1: softmax of one logit is 1 and the label is that word, so the loss and
    both gradients are 0 and lse is the logit itself. On the GPU lse - z and G come
    out as rounding residues of the log2(e) scaling (|.| ~ 1e-7 relative), so they
    are checked against bounds rather than for exact zeros."""
    H, W, y = make_inputs(200, 64, 1, seed=1, labels="uniform", n_ignored=7, w_std=0.1)
    r = run_all_paths(lce, H, W, y, chunk=64, dloss=1.0)
    ref = O.forward_backward(H, W, y)
    assert ref["loss"] == 0.0 and np.all(ref["dH"] == 0.0) and np.all(ref["dW"] == 0.0)
    for k in ("lse", "flse"):
        check_lse(r[k], ref["lse"])
    for k in ("loss", "floss"):
        assert abs(r[k]) <= 1e-6, (k, r[k])
    for k in ("dH", "dW", "bdH", "bdW"):
        assert np.abs(r[k]).max() <= 1e-6, (k, float(np.abs(r[k]).max()))


def test_labels_at_vocab_ends(lce):
    N, D, V = 200, 128, 777
    H, W, y = make_inputs(N, D, V, seed=3)
    y[::2] = 0
    y[1::2] = V - 1
    r = run_all_paths(lce, H, W, y, chunk=128)
    compare(r, O.forward_backward(H, W, y))


def test_all_rows_ignored(lce):
    N, D, V = 130, 64, 300
    H, W, y = make_inputs(N, D, V, seed=4)
    y[:] = IGNORE_INDEX
    r = run_all_paths(lce, H, W, y, chunk=64)
    assert r["loss"] == 0.0 and r["floss"] == 0.0
    for k in ("dH", "dW", "bdH", "bdW"):
        assert not np.any(r[k]), k
    check_lse(r["lse"], O.forward(H, W, y)[1])


def test_empty_batch(lce):
    D, V = 64, 300
    H = torch.zeros(0, D, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(V, D, device=DEV).to(torch.bfloat16)
    y = torch.zeros(0, dtype=torch.int64, device=DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(H, W, y, chunk=128)
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and dW.abs().max().item() == 0.0


def test_label_out_of_range_reports_status(lce):
    N, D, V = 140, 64, 500
    H, W, y = make_inputs(N, D, V, seed=5)
    y[3] = V
    y[9] = -7
    ws = lce.alloc_workspace(N, D, V, 64, DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(H.to(DEV), W.to(DEV), y.to(DEV), chunk=64, ws=ws)
    assert lce.read_status(ws) == 4          # LCE_ERR_LABEL_RANGE
    assert lce.read_status(ws) == 0          # cleared
    ref = O.forward_backward(H, W, y)
    assert ref["n_bad"] == 2
    check_loss(loss.item(), ref["loss"])
    check_grad("dH", to64(dH), ref["dH"])
    check_grad("dW", to64(dW), ref["dW"])


@pytest.mark.parametrize("ign", [7, 0, -1])
def test_custom_ignore_index(lce, ign):
    """An ignore_index other than -100: a vocabulary id (7, or 0, the first column;
    rows whose label is that id take no part even though it is in range) or -1.
    A label of -100 is then out of range: flagged, and its row counts as ignored.
    Fused, forward and backward paths and CE over the same logits, against the
    oracle called with the same ignore_index."""
    N, D, V, chunk = 400, 136, 3000, 128
    H, W, y = make_inputs(N, D, V, seed=40 + ign, w_std=0.05)
    y[::9] = ign
    y[5] = -100
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    ws = lce.alloc_workspace(N, D, V, chunk, DEV)
    ref = O.forward_backward(H, W, y, ignore_index=ign)
    assert ref["n_bad"] == 1 and ref["n_valid"] == N - int((y == ign).sum()) - 1
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, ignore_index=ign, ws=ws)
    assert lce.read_status(ws) == 4          # LCE_ERR_LABEL_RANGE: the -100 label
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk, ignore_index=ign, ws=ws)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, chunk=chunk, ignore_index=ign, ws=ws)
    lce.read_status(ws)
    for got_loss, got_lse in ((loss, lse), (floss, flse)):
        check_loss(got_loss.item(), ref["loss"])
        check_lse(to64(got_lse), ref["lse"])
    for name, got, exp in (("dH", dH, ref["dH"]), ("dW", dW, ref["dW"]),
                           ("dH (backward)", bdH, ref["dH"]), ("dW (backward)", bdW, ref["dW"])):
        check_grad(name, to64(got), exp)
    Z = (H.double() @ W.double().T).float()
    cl, clse, cdZ = lce.ce_logits(Z.to(DEV), yd, ignore_index=ign)
    cref = O.ce_from_logits(Z.double().numpy(), y.numpy(), ignore_index=ign)
    check_loss(cl.item(), cref["loss"])
    check_lse(to64(clse), cref["lse"])
    check_grad("dZ", to64(cdZ), cref["dZ"])


def test_deterministic_bits(lce):
    H, W, y = make_inputs(520, 256, 4000, seed=6, n_ignored=20)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    a = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=256)
    b = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=256)
    torch.cuda.synchronize()
    for x, z in zip(a, b):
        assert torch.equal(x, z)


def test_chunk_invariance(lce):
    H, W, y = make_inputs(1024, 512, 5000, seed=8, n_ignored=30)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    outs = [lce.lce_fwd_bwd(Hd, Wd, yd, chunk=c) for c in (128, 512, 1024)]
    torch.cuda.synchronize()
    base = outs[0]
    for o in outs[1:]:
        assert abs(o[0].item() - base[0].item()) <= 1e-5 * abs(base[0].item())
        assert (o[1] - base[1]).abs().max().item() <= 1e-5
        check_grad("dH", to64(o[2]), to64(base[2]))
        check_grad("dW", to64(o[3]), to64(base[3]))


def test_autograd_wrapper(lce):
    H, W, y = make_inputs(300, 128, 900, seed=9, n_ignored=10)
    Hd = H.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    loss = lce.linear_cross_entropy(Hd, Wd, y.to(DEV), chunk=128)
    (loss * 3.0).backward()
    ref = O.forward_backward(H, W, y, dloss=3.0)
    check_loss(loss.item(), ref["loss"])
    check_grad("dH", to64(Hd.grad), ref["dH"])
    check_grad("dW", to64(Wd.grad), ref["dW"])


@pytest.mark.parametrize("name", ["llama2-7b", "mistral-7b"])
def test_workload_full_oracle(lce, name):
    """Whole-output comparison on the two mid-size workloads (oracle in fp64),
    for the fused call and for the separate forward + backward (the backward
    recomputes each chunk's logits from the saved lse)."""
    wl = WORKLOADS[name]
    H, W, y = workload_inputs(wl)
    r = run_all_paths(lce, H, W, y, chunk=wl.chunks[0])
    compare(r, O.forward_backward(H, W, y))


def test_autograd_per_row_losses_llama2(lce):
    """The autograd wrapper with reduction "none" (per-row incoming gradients:
    it keeps lse and runs the separate backward) on the Llama-2 workload."""
    wl = WORKLOADS["llama2-7b"]
    H, W, y = workload_inputs(wl)
    Hd = H.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    rows = lce.linear_cross_entropy(Hd, Wd, y.to(DEV), chunk=wl.chunks[0], reduction="none")
    g = torch.from_numpy(np.random.default_rng(5).standard_normal(wl.N)).float().to(DEV)
    (rows * g).sum().backward()
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y, dloss=g.double().cpu().numpy(), reduction="none")
    assert np.abs(to64(rows) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    check_grad("dH", to64(Hd.grad), ref["dH"])
    check_grad("dW", to64(Wd.grad), ref["dW"])


@pytest.mark.parametrize("N,D,V,chunk", [(300, 264, 1000, 128), (1000, 520, 3000, 384),
                                         (4096, 1024, 32000, 1024)])
def test_single_cta_tiles_match_oracle(lce, monkeypatch, N, D, V, chunk):
    """The one-CTA-per-tile GEMM variant (the default runs CTA pairs with
    cta_group::2; odd row-block counts there give a pair whose second tile lies
    past the output, covered by the other tests)."""
    monkeypatch.setenv("LCE_GEMM_CLUSTER", "1")
    H, W, y = make_inputs(N, D, V, seed=N + 7, labels="uniform", n_ignored=N // 20, w_std=0.05)
    r = run_all_paths(lce, H, W, y, chunk=chunk, dloss=1.3)
    compare(r, O.forward_backward(H, W, y, dloss=1.3))


@pytest.mark.parametrize("reduction", ["sum", "none"])
@pytest.mark.parametrize("N,D,V,chunk", [(300, 264, 1000, 128), (1000, 520, 3000, 384)])
def test_reduction_variants(lce, reduction, N, D, V, chunk):
    """reduction sum / none through the three paths; 'none' with a per-row dloss."""
    H, W, y = make_inputs(N, D, V, seed=N + 11, labels="uniform", n_ignored=N // 25, w_std=0.05)
    rng = np.random.default_rng(N)
    dl_host = rng.standard_normal(N) if reduction == "none" else 0.37
    dl = torch.tensor(np.atleast_1d(dl_host), dtype=torch.float32, device=DEV)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, reduction=reduction)
    floss, flse = lce.lce_forward(Hd, Wd, yd, chunk=chunk, reduction=reduction)
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, flse, dloss=dl, chunk=chunk, reduction=reduction)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y, dloss=np.float64(dl_host) if reduction == "sum" else dl_host,
                             reduction=reduction)
    if reduction == "sum":
        check_loss(loss.item(), ref["loss"])
        check_loss(floss.item(), ref["loss"])
    else:
        assert loss.shape == (N,)
        for got in (loss, floss):
            err = np.abs(to64(got) - ref["loss"]).max()
            assert err <= 1e-3 * np.abs(ref["loss"]).max(), err
    check_lse(to64(lse), ref["lse"])
    for name, got, exp in (("dH", dH, ref["dH"]), ("dW", dW, ref["dW"]),
                           ("dH (backward)", bdH, ref["dH"]), ("dW (backward)", bdW, ref["dW"])):
        check_grad(name, to64(got), exp)


def test_autograd_per_row_losses(lce):
    H, W, y = make_inputs(260, 128, 700, seed=21, n_ignored=9)
    Hd = H.to(DEV).requires_grad_(True)
    Wd = W.to(DEV).requires_grad_(True)
    rows = lce.linear_cross_entropy(Hd, Wd, y.to(DEV), chunk=128, reduction="none")
    g = torch.linspace(-1, 1, 260, device=DEV)
    (rows * g).sum().backward()
    ref = O.forward_backward(H, W, y, dloss=g.double().cpu().numpy(), reduction="none")
    assert np.abs(to64(rows) - ref["loss"]).max() <= 1e-3 * np.abs(ref["loss"]).max()
    check_grad("dH", to64(Hd.grad), ref["dH"])
    check_grad("dW", to64(Wd.grad), ref["dW"])


@pytest.mark.parametrize("acc", [("dW",), ("dH",), ("dW", "dH")])
def test_accumulate_into_existing_gradients(lce, acc):
    """accumulate=... adds this call's dW / dH to what the tensors hold."""
    N, D, V, chunk = 700, 264, 3000, 256
    H, W, y = make_inputs(N, D, V, seed=31, n_ignored=20, w_std=0.05)
    gen = torch.Generator().manual_seed(7)
    dH0 = (torch.randn(N, D, generator=gen) * 1e-4).to(torch.bfloat16).to(DEV)
    dW0 = (torch.randn(V, D, generator=gen) * 1e-4).to(DEV)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dH, dW = dH0.clone(), dW0.clone()
    loss, lse, dH, dW = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, dH=dH, dW=dW, accumulate=acc)
    bdH, bdW = dH0.clone(), dW0.clone()
    bdH, bdW = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, dH=bdH, dW=bdW, accumulate=acc)
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y)
    exp_dH = ref["dH"] + (to64(dH0) if "dH" in acc else 0.0)
    exp_dW = ref["dW"] + (to64(dW0) if "dW" in acc else 0.0)
    for name, got, exp in (("dH", dH, exp_dH), ("dW", dW, exp_dW), ("dH (backward)", bdH, exp_dH),
                           ("dW (backward)", bdW, exp_dW)):
        check_grad(name, to64(got), exp)


def test_accumulate_dw_over_micro_batches(lce):
    """dW summed over two micro-batches (reduction sum) equals the oracle's dW of
    the whole batch."""
    N, D, V = 1000, 256, 2000
    H, W, y = make_inputs(N, D, V, seed=33, n_ignored=30, w_std=0.05)
    Wd = W.to(DEV)
    dW = torch.empty(V, D, dtype=torch.float32, device=DEV)
    half = N // 2
    lce.lce_fwd_bwd(H[:half].to(DEV), Wd, y[:half].to(DEV), chunk=128, dW=dW, reduction="sum")
    lce.lce_fwd_bwd(H[half:].to(DEV), Wd, y[half:].to(DEV), chunk=128, dW=dW, reduction="sum",
                    accumulate=("dW",))
    torch.cuda.synchronize()
    ref = O.forward_backward(H, W, y, reduction="sum")
    check_grad("dW (two micro-batches)", to64(dW), ref["dW"])


def test_bounded_wait_times_out_and_context_survives(lce):
    """A wait that nothing ends gives up after its limit, reports LCE_ERR_TIMEOUT
    through the workspace, and the device keeps working."""
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    lce.selftest_wait_timeout(ws, limit_us=20000)
    assert lce.read_status(ws) == 5          # LCE_ERR_TIMEOUT
    assert lce.read_status(ws) == 0          # cleared
    H, W, y = make_inputs(200, 64, 500, seed=35)
    loss, lse = lce.lce_forward(H.to(DEV), W.to(DEV), y.to(DEV), chunk=64)
    torch.cuda.synchronize()
    check_loss(loss.item(), O.forward_backward(H, W, y)["loss"])


def test_large_vocabulary(lce):
    """A vocabulary of a million (ragged: 1,000,003), two chunks, dH tiles in four
    vocabulary parts; labels at both ends of the vocabulary."""
    N, D, V, chunk = 160, 64, 1_000_003, 128
    H, W, y = make_inputs(N, D, V, seed=41, n_ignored=8, w_std=0.3)
    y[0] = V - 1
    y[1] = 0
    r = run_all_paths(lce, H, W, y, chunk=chunk, dloss=1.0)
    compare(r, O.forward_backward(H, W, y))
