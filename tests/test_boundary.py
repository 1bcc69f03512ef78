"""Host-side tests of the C ABI (no GPU needed): the library loads, exports every
function include/lce.h declares, sizes its workspace as documented, and returns
argument errors before touching the device. Pointer arguments below are fake
addresses that the library must reject or never dereference."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lce.h")

OK, INVALID, ALIGN, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    import linear_cross_entropy_chunked_gb300 as pkg
    try:
        pkg.build()
    except RuntimeError as e:  # no nvcc here
        pytest.skip(str(e))
    return pkg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:lce_status|const\s+char|int|void)[\s*]+(lce_\w+)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ("lce_forward", "lce_backward", "lce_fwd_bwd", "lce_workspace_size",
              "lce_read_status", "lce_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    import linear_cross_entropy_chunked_gb300 as pkg
    names = set(declared_functions()) - {"lce_forward_noalloc"}
    assert names <= set(pkg.EXPORTED), names - set(pkg.EXPORTED)


def ws_size(L, N, D, V, chunk):
    out = ctypes.c_size_t(0)
    st = L.lce_workspace_size(N, D, V, chunk, ctypes.byref(out))
    return st, out.value


def test_workspace_size_is_order_chunk_times_V(L):
    st, b1 = ws_size(L, 16384, 4096, 128256, 1024)
    assert st == OK
    st, b2 = ws_size(L, 16384, 4096, 128256, 2048)
    assert st == OK
    # the bf16 chunk buffer (P', then G) dominates: ~2 bytes per chunk row per vocab id
    assert 2 * 1024 * 128256 <= b1 <= 2 * 1024 * 128256 * 1.15
    assert 1.8 < b2 / b1 < 2.05
    # it does not grow with N beyond O(N) bytes
    st, b3 = ws_size(L, 4 * 16384, 4096, 128256, 1024)
    assert b3 - b1 < 64 * 16384 * 4
    # far below the full logit tensor the fused loss avoids (N*V*2 bytes in bf16):
    # the chunk buffer is chunk/N of it
    assert b1 < 0.075 * 16384 * 128256 * 2


@pytest.mark.parametrize("N,D,V,chunk", [(-1, 64, 100, 64), (8, 0, 100, 64), (8, 12, 100, 64),
                                         (8, 64, 0, 64), (8, 64, 100, 0), (8, 64, 100, -5)])
def test_workspace_size_rejects_bad_sizes(L, N, D, V, chunk):
    assert ws_size(L, N, D, V, chunk)[0] == INVALID


def test_workspace_size_null_out(L):
    assert L.lce_workspace_size(8, 64, 100, 64, None) == INVALID


FAKE = 0x10000000  # 256 MB-aligned fake device address: never dereferenced below


def fwd(L, H=FAKE, W=FAKE, y=FAKE, N=128, D=64, V=1000, chunk=64, loss=FAKE, lse=FAKE,
        ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = ws_size(L, N, D, V, chunk)[1]
    vp = ctypes.c_void_p
    return L.lce_forward(vp(H), vp(W), vp(y), N, D, V, -100, chunk, vp(loss), vp(lse), vp(ws),
                         ws_bytes, None)


def test_forward_argument_errors_return_before_launch(L):
    assert fwd(L, D=12) == INVALID             # D % 8 != 0
    assert fwd(L, chunk=0) == INVALID
    assert fwd(L, H=0) == INVALID              # null H with N > 0
    assert fwd(L, W=0) == INVALID
    assert fwd(L, loss=0) == INVALID
    assert fwd(L, ws=0) == INVALID
    assert fwd(L, H=FAKE + 2) == ALIGN
    assert fwd(L, ws=FAKE + 8) == ALIGN
    assert fwd(L, lse=FAKE + 4) == ALIGN
    need = ws_size(L, 128, 64, 1000, 64)[1]
    assert fwd(L, ws_bytes=need - 1) == WORKSPACE


def test_backward_and_fused_argument_errors(L):
    vp = ctypes.c_void_p
    N, D, V, chunk = 128, 64, 1000, 64
    need = ws_size(L, N, D, V, chunk)[1]
    # lce_backward: null dW, misaligned dH, small workspace
    assert L.lce_backward(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), None, N, D, V,
                          -100, chunk, vp(FAKE), need, None) == INVALID
    assert L.lce_backward(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE + 2), vp(FAKE),
                          N, D, V, -100, chunk, vp(FAKE), need, None) == ALIGN
    assert L.lce_backward(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE), N, D,
                          V, -100, chunk, vp(FAKE), need - 1024, None) == WORKSPACE
    # lce_fwd_bwd: null loss, bad sizes
    assert L.lce_fwd_bwd(vp(FAKE), vp(FAKE), vp(FAKE), None, N, D, V, -100, chunk, None,
                         vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), need, None) == INVALID
    assert L.lce_fwd_bwd(vp(FAKE), vp(FAKE), vp(FAKE), None, N, 20, V, -100, chunk, vp(FAKE),
                         vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), need, None) == INVALID


def test_status_strings_and_version(L):
    for code in range(8):
        s = L.lce_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.lce_status_string(99) == b"unknown status"
    assert L.lce_version() >= 100
    assert L.lce_read_status(None, None) == INVALID


def test_profile_api_without_gpu(L):
    L.lce_profile_reset()
    assert L.lce_profile_enable(1) == OK
    ms = ctypes.c_double(-1)
    n = ctypes.c_int64(-1)
    assert L.lce_profile_read(0, ctypes.byref(ms), ctypes.byref(n)) == OK
    assert ms.value == 0.0 and n.value == 0
    assert L.lce_profile_read(7, ctypes.byref(ms), ctypes.byref(n)) == INVALID
    assert L.lce_profile_enable(0) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    import linear_cross_entropy_chunked_gb300 as pkg
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(16, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        pkg.lce_forward(H, W, y)


# ---------------------------------------------------------------- final RMSNorm

def test_norm_workspace_sizes(L):
    N, D, V, chunk = 16384, 4096, 128256, 1024
    base = ws_size(L, N, D, V, chunk)[1]
    out = ctypes.c_size_t(0)
    assert L.lce_norm_workspace_size(N, D, V, chunk, ctypes.byref(out)) == OK
    # the loss path's workspace + the chunk's H (bf16) and dH (fp32) + 256 dgamma partial rows
    assert out.value == base + 2 * chunk * D + 4 * chunk * D + 4 * 256 * D
    assert L.lce_norm_workspace_size(N, 8200, V, chunk, ctypes.byref(out)) == INVALID  # D > 8192
    assert L.lce_rmsnorm_backward_workspace_size(D, ctypes.byref(out)) == OK
    assert out.value == 4 * 256 * D
    assert L.lce_rmsnorm_backward_workspace_size(12, ctypes.byref(out)) == INVALID
    assert L.lce_rmsnorm_backward_workspace_size(D, None) == INVALID


def test_rmsnorm_argument_errors_return_before_launch(L):
    vp = ctypes.c_void_p
    f = L.lce_rmsnorm_forward
    assert f(vp(FAKE), vp(FAKE), 8, 12, 1e-6, vp(FAKE), None, None) == INVALID      # D % 8
    assert f(vp(FAKE), vp(FAKE), 8, 8200, 1e-6, vp(FAKE), None, None) == INVALID    # D > 8192
    assert f(vp(FAKE), vp(FAKE), 8, 64, -1.0, vp(FAKE), None, None) == INVALID      # eps < 0
    assert f(vp(FAKE), vp(FAKE), 8, 64, 1e-6, None, None, None) == INVALID          # null H
    assert f(vp(FAKE + 2), vp(FAKE), 8, 64, 1e-6, vp(FAKE), None, None) == ALIGN
    b = L.lce_rmsnorm_backward
    need = 4 * 256 * 64
    assert b(vp(FAKE), vp(FAKE), vp(FAKE), 0, 8, 64, 1e-6, vp(FAKE), None, vp(FAKE), need,
             None) == INVALID                                                        # null dgamma
    assert b(vp(FAKE), vp(FAKE), vp(FAKE), 1, 8, 64, 1e-6, vp(FAKE), vp(FAKE), vp(FAKE), need - 4,
             None) == WORKSPACE
    assert b(vp(FAKE), vp(FAKE), vp(FAKE + 8), 1, 8, 64, 1e-6, vp(FAKE), vp(FAKE), vp(FAKE), need,
             None) == ALIGN


def test_norm_fwd_bwd_argument_errors(L):
    vp = ctypes.c_void_p
    N, D, V, chunk = 128, 64, 1000, 64
    out = ctypes.c_size_t(0)
    assert L.lce_norm_workspace_size(N, D, V, chunk, ctypes.byref(out)) == OK
    need = out.value

    def call(dgamma=FAKE, ws_bytes=need, D_=D, X=FAKE):
        return L.lce_norm_fwd_bwd(vp(X), vp(FAKE), 1e-6, vp(FAKE), vp(FAKE), None, N, D_, V, -100,
                                  chunk, 0, vp(FAKE), vp(FAKE), vp(FAKE), vp(dgamma), vp(FAKE),
                                  vp(FAKE), ws_bytes, None)
    assert call(dgamma=0) == INVALID
    assert call(D_=12) == INVALID
    assert call(ws_bytes=need - 1) == WORKSPACE
    assert call(X=FAKE + 2) == ALIGN


def test_accumulate_workspace_and_flags(L):
    N, D, V, chunk = 16384, 4096, 128256, 1024
    base = ws_size(L, N, D, V, chunk)[1]
    out = ctypes.c_size_t(0)
    assert L.lce_workspace_size_opt(N, D, V, chunk, 1, ctypes.byref(out)) == OK
    assert out.value == base                                   # dW accumulation needs nothing
    assert L.lce_workspace_size_opt(N, D, V, chunk, 3, ctypes.byref(out)) == OK
    assert out.value == base + 4 * chunk * D                   # the chunk's dH in fp32
    assert L.lce_workspace_size_opt(N, D, V, chunk, 8, ctypes.byref(out)) == INVALID
    vp = ctypes.c_void_p
    # dH accumulation with only the plain workspace: refused before anything runs
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, 128, 64, 1000, -100, 64, 0, 2,
                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                             ws_size(L, 128, 64, 1000, 64)[1], None) == WORKSPACE
    assert L.lce_backward_opt(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE), 128,
                              64, 1000, -100, 64, 0, 8, vp(FAKE), 1 << 30, None) == INVALID
    # fp16 inputs with per-row losses: refused
    UNSUPPORTED = 7
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, 128, 64, 1000, -100, 64, 2, 4,
                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1 << 30,
                             None) == UNSUPPORTED
    assert L.lce_forward_opt(vp(FAKE), vp(FAKE), vp(FAKE), 128, 64, 1000, -100, 64, 0, 1, vp(FAKE),
                             vp(FAKE), vp(FAKE), 1 << 30, None) == INVALID      # no accumulate in fwd
