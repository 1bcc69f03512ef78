"""CUDA-graph capture of the library's calls. Every call enqueues only stream
work (a memset, kernel launches, the event fork / join of the two-kernel
gradient phase with the library's side stream); the host-side work (tensor-map
encoding, the first call's device set-up) happens at capture. A captured call
replayed on new input contents (written into the same buffers) gives outputs
bit-identical to the same call made eagerly."""
import pytest
import torch

from lce_synth import make_inputs, make_norm_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


def _eager(fn, *args):
    out = fn(*args)
    torch.cuda.synchronize()
    return [None if t is None else t.clone() for t in out]


@pytest.mark.parametrize("frozen", [False, True])
def test_fwd_bwd_graph_replay(lce, frozen):
    N, D, V, chunk = 2048, 1024, 16000, 512
    inputs = [make_inputs(N, D, V, seed=s, n_ignored=50, w_std=0.05) for s in (1, 2)]
    H, W, y = (t.to(DEV) for t in inputs[0])
    flags = lce.FROZEN_W if frozen else 0
    ws = lce.alloc_workspace(N, D, V, chunk, DEV, flags)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(N, device=DEV)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = None if frozen else torch.empty(V, D, device=DEV)

    def call():
        return lce.lce_fwd_bwd(H, W, y, chunk=chunk, loss=loss, lse=lse, dH=dH, dW=dW, ws=ws,
                               compute_dW=not frozen)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for Hh, Wh, yh in inputs:
        H.copy_(Hh)
        W.copy_(Wh)
        y.copy_(yh)
        g.replay()
        torch.cuda.synchronize()
        got = [loss.clone(), lse.clone(), dH.clone(), None if dW is None else dW.clone()]
        ref = _eager(lambda: lce.lce_fwd_bwd(Hh.to(DEV), Wh.to(DEV), yh.to(DEV), chunk=chunk,
                                             compute_dW=not frozen))
        for a, b in zip(got, ref):
            assert (a is None and b is None) or torch.equal(a, b)
        assert lce.read_status(ws) == 0


def test_ce_logits_and_norm_graph_replay(lce):
    N, V = 512, 128256
    Z = (torch.randn(N, V, generator=torch.Generator().manual_seed(3)) * 3).to(torch.bfloat16).to(DEV)
    y = torch.randint(0, V, (N,), generator=torch.Generator().manual_seed(4)).to(DEV)
    X, g, W, yn = make_norm_inputs(700, 1024, 9000, seed=5, n_ignored=20, w_std=0.05)
    Xd, gd, Wd, ynd = X.to(DEV), g.to(DEV), W.to(DEV), yn.to(DEV)
    nws = torch.empty(lce.norm_workspace_size(700, 1024, 9000, 256), dtype=torch.uint8, device=DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    nloss, nlse = torch.empty(1, device=DEV), torch.empty(700, device=DEV)
    import ctypes
    cws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    nbytes = ctypes.c_size_t(0)
    lce.lib().lce_ce_logits_workspace_size(N, ctypes.byref(nbytes))
    assert nbytes.value <= cws.numel()
    out = {}

    def calls():
        out["ce"] = lce.ce_logits(Z, y, loss=loss, lse=lse, ws=cws)
        out["norm"] = lce.norm_fwd_bwd(Xd, gd, Wd, ynd, chunk=256, ws=nws, loss=nloss, lse=nlse)

    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        calls()
    ce_out, norm_out = out["ce"], out["norm"]
    gr.replay()
    torch.cuda.synchronize()
    ref_ce = _eager(lambda: lce.ce_logits(Z, y))
    ref_norm = _eager(lambda: lce.norm_fwd_bwd(Xd, gd, Wd, ynd, chunk=256))
    for a, b in zip(ce_out, ref_ce):
        assert torch.equal(a, b)
    for a, b in zip(norm_out, ref_norm):
        assert torch.equal(a, b)
