"""Memory behaviour of every entry point on the GPU, without a sanitizer:

  * guard canaries: each output buffer and the workspace are carved out of a
    larger allocation with GUARD bytes of a fixed pattern on both sides; after
    the call the pattern must be intact (no write before or past any buffer,
    the workspace used only up to the size the library asked for), the padding
    columns of a strided logits matrix are untouched, and the inputs are
    bit-identical to before the call;
  * no hidden allocations: with every buffer passed in, a call changes neither
    the device's free memory (driver view) nor the PyTorch allocator's peak, so
    the extra memory of the method is exactly the workspace the caller passed,
    whose size is checked against the chunk x V bound of the chunked design.

Results computed in guarded buffers must equal, bit for bit, those of the same
call on plainly allocated buffers (the position of a buffer changes nothing)."""
import ctypes

import numpy as np
import pytest
import torch

from lce_synth import make_inputs, make_norm_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module")
def lce():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_cross_entropy_chunked_gb300 as pkg
    pkg.build()
    return pkg


class Guarded:
    """A device tensor of the given shape and dtype inside an allocation that has
    GUARD canary bytes before and after it."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8,
                              device=DEV)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == CANARY).all().item()) and bool((tail == CANARY).all().item())


def _check_all(bufs):
    torch.cuda.synchronize()
    bad = [name for name, b in bufs.items() if not b.intact()]
    assert not bad, f"canary overwritten around: {bad}"


def _snapshot(*ts):
    return [t.clone() for t in ts]


def _unchanged(before, *ts):
    for a, b in zip(before, ts):
        assert torch.equal(a, b), "an input was modified"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("reduction", ["mean", "none"])
@pytest.mark.parametrize("N,D,V,chunk", [(1000, 520, 3001, 384), (77, 128, 100, 1024),
                                         (2300, 1024, 9000, 1024)])
def test_fwd_bwd_writes_only_its_buffers(lce, N, D, V, chunk, reduction, dtype):
    if dtype == torch.float16 and reduction == "none":
        pytest.skip("fp16 inputs take reductions mean and sum")
    H, W, y = make_inputs(N, D, V, seed=N + V, n_ignored=N // 30, w_std=0.05,
                          dtype="fp16" if dtype == torch.float16 else "bf16")
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    dl = (torch.linspace(-1, 1, N) if reduction == "none" else torch.tensor([0.7])).to(DEV)
    before = _snapshot(Hd, Wd, yd, dl)
    flags = lce.INPUT_FP16 if dtype == torch.float16 else 0
    nl = N if reduction == "none" else 1
    b = dict(loss=Guarded((nl,), torch.float32), lse=Guarded((N,), torch.float32),
             dH=Guarded((N, D), dtype), dW=Guarded((V, D), torch.float32),
             ws=Guarded((lce.workspace_size_opt(N, D, V, chunk, flags),), torch.uint8))
    out = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, reduction=reduction,
                          loss=b["loss"].t, lse=b["lse"].t, dH=b["dH"].t, dW=b["dW"].t,
                          ws=b["ws"].t)
    _check_all(b)
    _unchanged(before, Hd, Wd, yd, dl)
    ref = lce.lce_fwd_bwd(Hd, Wd, yd, dloss=dl, chunk=chunk, reduction=reduction)
    torch.cuda.synchronize()
    for x, z in zip(out, ref):
        assert torch.equal(x, z)


def test_forward_and_backward_write_only_their_buffers(lce):
    N, D, V, chunk = 1500, 264, 4097, 512
    H, W, y = make_inputs(N, D, V, seed=11, n_ignored=40, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    before = _snapshot(Hd, Wd, yd)
    ws_n = lce.workspace_size(N, D, V, chunk)
    # the forward gets exactly its own share of the workspace (no chunk buffer)
    f = dict(loss=Guarded((1,), torch.float32), lse=Guarded((N,), torch.float32),
             ws=Guarded((lce.forward_workspace_size(N, D, V, chunk),), torch.uint8))
    loss, lse = lce.lce_forward(Hd, Wd, yd, chunk=chunk, loss=f["loss"].t, lse=f["lse"].t,
                                ws=f["ws"].t)
    _check_all(f)
    lse_saved = lse.clone()
    bk = dict(dH=Guarded((N, D), torch.bfloat16), dW=Guarded((V, D), torch.float32),
              ws=Guarded((ws_n,), torch.uint8))
    dH, dW = lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, dH=bk["dH"].t, dW=bk["dW"].t,
                              ws=bk["ws"].t)
    _check_all(bk)
    _unchanged(before + [lse_saved], Hd, Wd, yd, lse)
    loss2, lse2 = lce.lce_forward(Hd, Wd, yd, chunk=chunk)
    dH2, dW2 = lce.lce_backward(Hd, Wd, yd, lse2, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(loss, loss2) and torch.equal(lse, lse2)
    assert torch.equal(dH, dH2) and torch.equal(dW, dW2)


@pytest.mark.parametrize("acc", [("dW",), ("dH",), ("dW", "dH")])
def test_accumulate_writes_only_its_buffers(lce, acc):
    N, D, V, chunk = 900, 256, 2500, 256
    H, W, y = make_inputs(N, D, V, seed=13, n_ignored=20, w_std=0.05)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    gen = torch.Generator().manual_seed(5)
    dH0 = (torch.randn(N, D, generator=gen) * 1e-3).to(torch.bfloat16).to(DEV)
    dW0 = (torch.randn(V, D, generator=gen) * 1e-3).to(DEV)
    flags = sum(lce.ACCUMULATE[a] for a in acc)
    b = dict(loss=Guarded((1,), torch.float32), lse=Guarded((N,), torch.float32),
             dH=Guarded((N, D), torch.bfloat16, fill=dH0), dW=Guarded((V, D), torch.float32, fill=dW0),
             ws=Guarded((lce.workspace_size_opt(N, D, V, chunk, flags),), torch.uint8))
    out = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, loss=b["loss"].t, lse=b["lse"].t,
                          dH=b["dH"].t, dW=b["dW"].t, ws=b["ws"].t, accumulate=acc)
    _check_all(b)
    ref = lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, dH=dH0.clone(), dW=dW0.clone(), accumulate=acc)
    torch.cuda.synchronize()
    for x, z in zip(out, ref):
        assert torch.equal(x, z)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("N,V,ld", [(300, 1003, 1008), (40, 128256, 128264), (9, 300000, 300008)])
def test_ce_logits_leaves_padding_and_guards(lce, N, V, ld, dtype):
    """In-place gradient over a strided logits matrix: the columns between V and
    the row stride keep the canary, and so do the bytes around every buffer."""
    g = torch.Generator().manual_seed(V)
    Zfull = Guarded((N, ld), dtype, fill=(torch.randn(N, ld, generator=g) * 3).to(dtype))
    pad_canary = torch.full((N, ld - V), 0.0, dtype=dtype)
    pad_canary.view(torch.uint8).fill_(CANARY)
    Zfull.t[:, V:].copy_(pad_canary.to(DEV))
    Z0 = Zfull.t[:, :V].clone()
    y = torch.from_numpy(np.random.default_rng(N).integers(0, V, size=N)).to(DEV)
    y[::5] = -100
    nbytes = ctypes.c_size_t(0)
    lce.lib().lce_ce_logits_workspace_size(N, ctypes.byref(nbytes))
    b = dict(Z=Zfull, loss=Guarded((1,), torch.float32), lse=Guarded((N,), torch.float32),
             ws=Guarded((nbytes.value,), torch.uint8))
    loss, lse, dZ = lce.ce_logits(Zfull.t[:, :V], y, inplace=True, loss=b["loss"].t,
                                  lse=b["lse"].t, ws=b["ws"].t)
    _check_all(b)
    pad = Zfull.t[:, V:].contiguous().view(torch.uint8)
    assert bool((pad == CANARY).all().item()), "padding columns were written"
    Zref = torch.empty(N, ld, dtype=dtype, device=DEV)
    Zref[:, :V].copy_(Z0)
    ref_loss, ref_lse, ref_dZ = lce.ce_logits(Zref[:, :V], y)
    torch.cuda.synchronize()
    assert torch.equal(loss, ref_loss) and torch.equal(lse, ref_lse)
    assert torch.equal(dZ, ref_dZ)


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("N,D", [(300, 264), (1000, 4096), (77, 8192)])
def test_rmsnorm_kernels_write_only_their_buffers(lce, N, D):
    X, g, _, _ = make_norm_inputs(N, D, 16, seed=D)
    Xd, gd = X.to(DEV), g.to(DEV)
    dH = (torch.randn(N, D, generator=torch.Generator().manual_seed(N)) * 0.01).to(DEV)
    before = _snapshot(Xd, gd, dH)
    L = lce.lib()
    f = dict(H=Guarded((N, D), torch.bfloat16), rstd=Guarded((N,), torch.float32))
    assert L.lce_rmsnorm_forward(_vp(Xd), _vp(gd), N, D, 1e-6, _vp(f["H"].t), _vp(f["rstd"].t),
                                 _stream()) == 0
    _check_all(f)
    nbytes = ctypes.c_size_t(0)
    L.lce_rmsnorm_backward_workspace_size(D, ctypes.byref(nbytes))
    bk = dict(dX=Guarded((N, D), torch.bfloat16), dg=Guarded((D,), torch.float32),
              ws=Guarded((nbytes.value,), torch.uint8))
    assert L.lce_rmsnorm_backward(_vp(Xd), _vp(gd), _vp(dH), 1, N, D, 1e-6, _vp(bk["dX"].t),
                                  _vp(bk["dg"].t), _vp(bk["ws"].t), nbytes.value, _stream()) == 0
    _check_all(bk)
    _unchanged(before, Xd, gd, dH)
    H2, r2 = lce.rmsnorm_forward(Xd, gd, eps=1e-6, want_rstd=True)
    dX2, dg2 = lce.rmsnorm_backward(Xd, gd, dH, eps=1e-6)
    torch.cuda.synchronize()
    assert torch.equal(f["H"].t, H2) and torch.equal(f["rstd"].t, r2)
    assert torch.equal(bk["dX"].t, dX2) and torch.equal(bk["dg"].t, dg2)


def test_norm_fwd_bwd_writes_only_its_buffers(lce):
    N, D, V, chunk = 1300, 1024, 5000, 512
    X, g, W, y = make_norm_inputs(N, D, V, seed=3, n_ignored=30, w_std=0.05)
    Xd, gd, Wd, yd = X.to(DEV), g.to(DEV), W.to(DEV), y.to(DEV)
    before = _snapshot(Xd, gd, Wd, yd)
    ws_n = lce.norm_workspace_size(N, D, V, chunk)
    b = dict(loss=Guarded((1,), torch.float32), lse=Guarded((N,), torch.float32),
             dX=Guarded((N, D), torch.bfloat16), dg=Guarded((D,), torch.float32),
             dW=Guarded((V, D), torch.float32), ws=Guarded((ws_n,), torch.uint8))
    st = lce.lib().lce_norm_fwd_bwd(_vp(Xd), _vp(gd), 1e-6, _vp(Wd), _vp(yd), None, N, D, V, -100,
                                    chunk, 0, _vp(b["loss"].t), _vp(b["lse"].t), _vp(b["dX"].t),
                                    _vp(b["dg"].t), _vp(b["dW"].t), _vp(b["ws"].t), ws_n,
                                    _stream())
    assert st == 0
    _check_all(b)
    _unchanged(before, Xd, gd, Wd, yd)
    ref = lce.norm_fwd_bwd(Xd, gd, Wd, yd, eps=1e-6, chunk=chunk)
    torch.cuda.synchronize()
    for name, r in zip(("loss", "lse", "dX", "dg", "dW"), ref):
        assert torch.equal(b[name].t, r), name


def _quiet_delta(fn):
    """(change of the device's free bytes, PyTorch allocator peak above the
    allocated bytes) across fn(), after a warm-up call."""
    fn()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    alloc0 = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    fn()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    return free0 - free1, torch.cuda.max_memory_allocated() - alloc0


def test_calls_allocate_nothing(lce):
    """With every buffer passed in, no entry point allocates device memory, through
    the driver or through PyTorch: the workspace is the method's whole extra
    memory, and it is a small multiple of chunk x V."""
    N, D, V, chunk = 4096, 2048, 32000, 1024
    H, W, y = make_inputs(N, D, V, seed=2, n_ignored=100)
    Hd, Wd, yd = H.to(DEV), W.to(DEV), y.to(DEV)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(N, device=DEV)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(V, D, device=DEV)
    ws = lce.alloc_workspace(N, D, V, chunk, DEV)
    # two bf16 chunk buffers (the G of a pair of chunks), the pair's H^T, the dH
    # parts of the pair's first chunk and per-row statistics: a few bytes per logit
    # of one chunk
    assert ws.numel() <= 6 * chunk * V
    assert ws.numel() < 0.5 * N * V * 4    # well below the fp32 logits of the batch (4 chunks)
    deltas = {
        "fwd_bwd": _quiet_delta(lambda: lce.lce_fwd_bwd(Hd, Wd, yd, chunk=chunk, loss=loss, lse=lse,
                                                        dH=dH, dW=dW, ws=ws)),
        "forward": _quiet_delta(lambda: lce.lce_forward(Hd, Wd, yd, chunk=chunk, loss=loss,
                                                        lse=lse, ws=ws)),
        "backward": _quiet_delta(lambda: lce.lce_backward(Hd, Wd, yd, lse, chunk=chunk, dH=dH,
                                                          dW=dW, ws=ws)),
    }
    Z = torch.randn(N, V, device=DEV).to(torch.bfloat16)
    nbytes = ctypes.c_size_t(0)
    lce.lib().lce_ce_logits_workspace_size(N, ctypes.byref(nbytes))
    cws = torch.empty(nbytes.value, dtype=torch.uint8, device=DEV)
    deltas["ce_logits"] = _quiet_delta(lambda: lce.ce_logits(Z, yd, inplace=True, loss=loss,
                                                             lse=lse, ws=cws))
    for name, (driver, peak) in deltas.items():
        assert driver == 0, f"{name}: device free memory changed by {driver} bytes"
        assert peak == 0, f"{name}: PyTorch allocator peak rose by {peak} bytes"
