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
    names = set(declared_functions())
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
    # the two bf16 chunk buffers (P', then G, of the two chunks of a pair) dominate:
    # ~4 bytes per chunk row per vocab id; next come the pair's H^T (bf16), the fp32
    # dH parts of the first chunk's dH tiles (split in two when they run alone) and
    # the (max, sum) partials
    assert 2 * 2 * 1024 * 128256 <= b1 <= 2 * 2 * 1024 * 128256 * 1.15
    assert 1.7 < b2 / b1 < 2.05
    # LCE_LOW_MEMORY keeps one chunk buffer and one chunk's H^T, and no dH parts at
    # chunk 1024 (32 dH tiles beside the dW tiles): about half
    low = ctypes.c_size_t(0)
    assert L.lce_workspace_size_opt(16384, 4096, 128256, 1024, 16, ctypes.byref(low)) == OK
    assert 2 * 1024 * 128256 <= low.value <= 2 * 1024 * 128256 * 1.2
    ldg = -(-128256 // 256) * 256
    assert b1 - low.value == 2 * 1024 * ldg + 2 * 4096 * 1024 + 2 * 4 * 1024 * 4096
    # it does not grow with N beyond O(N) bytes
    st, b3 = ws_size(L, 4 * 16384, 4096, 128256, 1024)
    assert b3 - b1 < 64 * 16384 * 4
    # far below the full logit tensor the fused loss avoids (N*V*2 bytes in bf16):
    # each chunk buffer is chunk/N of it
    assert b1 < 0.14 * 16384 * 128256 * 2


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
    # the forward needs only its own share of the workspace (no chunk buffer)
    need = ctypes.c_size_t(0)
    assert L.lce_forward_workspace_size(128, 64, 1000, 64, ctypes.byref(need)) == OK
    assert fwd(L, ws_bytes=need.value - 1) == WORKSPACE


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

def ws_size_low(L, N, D, V, chunk):
    out = ctypes.c_size_t(0)
    assert L.lce_workspace_size_opt(N, D, V, chunk, 16, ctypes.byref(out)) == OK   # LCE_LOW_MEMORY
    return out.value


def test_norm_workspace_sizes(L):
    N, D, V, chunk = 16384, 4096, 128256, 1024
    out = ctypes.c_size_t(0)
    # two chunk buffers (chunk pairs, as on the loss path): the loss path's workspace
    # (whose dH parts hold the chunk's fp32 dH) + the pair's normalised rows H (bf16)
    # + 256 dgamma partial rows
    assert L.lce_norm_workspace_size(N, D, V, chunk, ctypes.byref(out)) == OK
    assert out.value == ws_size(L, N, D, V, chunk)[1] + 2 * 2 * chunk * D + 4 * 256 * D
    # one chunk buffer (LCE_LOW_MEMORY): the loss path's + the chunk's dH (fp32) and H
    base = ws_size_low(L, N, D, V, chunk)
    assert L.lce_norm_workspace_size_opt(N, D, V, chunk, 16, ctypes.byref(out)) == OK
    assert out.value == base + 4 * chunk * D + 2 * chunk * D + 4 * 256 * D
    # two vocabulary parts (chunk 512): the loss path's partial arrays hold dH
    base2 = ws_size_low(L, N, D, V, 512)
    assert L.lce_norm_workspace_size_opt(N, D, V, 512, 16, ctypes.byref(out)) == OK
    assert out.value == base2 + 2 * 512 * D + 4 * 256 * D
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
    assert out.value == base   # the dH parts of a pair's first chunk serve
    low = ws_size_low(L, N, D, V, chunk)
    assert L.lce_workspace_size_opt(N, D, V, chunk, 3 | 16, ctypes.byref(out)) == OK
    assert out.value == low + 4 * chunk * D    # one buffer: the chunk's dH in fp32
    base2 = ws_size(L, N, D, V, 512)[1]        # two vocabulary parts: their arrays serve
    assert L.lce_workspace_size_opt(N, D, V, 512, 2, ctypes.byref(out)) == OK
    assert out.value == base2
    assert L.lce_workspace_size_opt(N, D, V, chunk, 32, ctypes.byref(out)) == INVALID   # unknown flag
    vp = ctypes.c_void_p
    # dH accumulation with only the plain workspace: refused before anything runs
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, 128, 64, 1000, -100, 64, 0, 2,
                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                             ws_size(L, 128, 64, 1000, 64)[1], None) == WORKSPACE
    assert L.lce_backward_opt(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE), 128,
                              64, 1000, -100, 64, 0, 32, vp(FAKE), 1 << 30, None) == INVALID
    # fp16 inputs with per-row losses: refused
    UNSUPPORTED = 7
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, 128, 64, 1000, -100, 64, 2, 4,
                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1 << 30,
                             None) == UNSUPPORTED
    assert L.lce_forward_opt(vp(FAKE), vp(FAKE), vp(FAKE), 128, 64, 1000, -100, 64, 0, 1, vp(FAKE),
                             vp(FAKE), vp(FAKE), 1 << 30, None) == INVALID      # no accumulate in fwd


def test_library_source_allocates_no_device_memory():
    """The library takes all device memory from its caller (outputs and a workspace
    sized by the *_workspace_size calls) or from its own static scratch array: no
    allocation or free call appears in its code, outside comments."""
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "linear_cross_entropy_chunked_gb300", "csrc")
    pat = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|cudaHostAlloc|"
                     r"cuMemCreate|cudaMallocAsync)\s*\(")
    hits = []
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h", ".cpp")):
            continue
        text = open(os.path.join(csrc, name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for i, line in enumerate(text.splitlines(), 1):
            code = line.split("//", 1)[0]
            if pat.search(code):
                hits.append(f"{name}:{i}: {code.strip()}")
    assert not hits, hits


def test_dh_vocabulary_split_workspace(L):
    """The dH tiles of a chunk (256 rows x 512 columns each) are split along the
    vocabulary until there are at least 28 of them, in at most 4 parts, for
    vocabularies of at least 8192; each part needs one fp32 [chunk rows rounded up
    to 128] x D array in the workspace. (Sizes with one chunk buffer,
    LCE_LOW_MEMORY: the parts are the same either way.)"""
    N, D, chunk = 4096, 1024, 1024
    small = ws_size_low(L, N, D, 8191, chunk)
    big = ws_size_low(L, N, D, 8192, chunk)     # same G row stride (both round to 8192)
    # 4 row pairs x 2 column blocks = 8 tiles -> 4 parts
    assert big - small == 4 * 4 * 1024 * D
    # 1000 rows round up to 1024 per part; 4 x 2 tiles again
    assert ws_size_low(L, N, D, 8192, 1000) - ws_size_low(L, N, D, 8191, 1000) == 4 * 4 * 1024 * D
    stats = lambda c, V: 8 * c * (-(-V // 128))     # per-row (max, sum) of each 128-column slab
    # Llama-3-8B head: at chunk 512, 2 x 8 = 16 tiles -> 2 parts; at chunk 1024,
    # 4 x 8 = 32 tiles -> one part, no partial arrays
    b0 = ws_size_low(L, 16384, 4096, 128256, 512)
    g0 = 2 * 512 * 128256 + 2 * 4096 * 512          # G (bf16) and H^T (bf16)
    assert b0 - g0 >= 2 * 4 * 512 * 4096 + stats(512, 128256)
    assert b0 - g0 < 2 * 4 * 512 * 4096 + stats(512, 128256) + (1 << 20)
    b1 = ws_size_low(L, 16384, 4096, 128256, 1024)
    assert b1 - (2 * 1024 * 128256 + 2 * 4096 * 1024) < stats(1024, 128256) + (1 << 20)
    # Qwen-2.5-7B head (D 3584: 7 column blocks): chunk 1024 -> 28 tiles, one part;
    # chunk 512 -> 14 tiles, 2 parts
    q1 = ws_size_low(L, 16384, 3584, 152064, 1024)
    assert q1 - (2 * 1024 * 152064 + 2 * 3584 * 1024) < stats(1024, 152064) + (1 << 20)
    q0 = ws_size_low(L, 16384, 3584, 152064, 512)
    assert q0 - (2 * 512 * 152064 + 2 * 3584 * 512) >= 2 * 4 * 512 * 3584


def test_frozen_w_flag(L):
    """LCE_FROZEN_W (8): no dW contraction. Its workspace drops the H chunk^T and
    splits the dH tiles for the whole GPU (one wave of 76 CTA pairs: 32 tiles of
    a Llama-3 chunk -> 2 vocabulary parts), and keeps two chunk buffers (the next
    chunk's logits beside a chunk's dH; one with LCE_LOW_MEMORY); dW may be NULL;
    it does not combine with accumulating into dW."""
    N, D, V, chunk = 16384, 4096, 128256, 1024
    base = ws_size_low(L, N, D, V, chunk)    # one chunk buffer, H^T, no dH parts
    gbuf = 2 * chunk * (-(-V // 256) * 256)
    out = ctypes.c_size_t(0)
    assert L.lce_workspace_size_opt(N, D, V, chunk, 8, ctypes.byref(out)) == OK
    assert out.value == base - 2 * D * chunk + 2 * 4 * chunk * D + gbuf
    assert L.lce_workspace_size_opt(N, D, V, chunk, 8 | 2, ctypes.byref(out)) == OK
    assert out.value == base - 2 * D * chunk + 2 * 4 * chunk * D + gbuf   # the parts serve dH += too
    assert L.lce_workspace_size_opt(N, D, V, chunk, 8 | 16, ctypes.byref(out)) == OK
    assert out.value == base - 2 * D * chunk + 2 * 4 * chunk * D
    vp = ctypes.c_void_p
    n, d, v, c = 128, 64, 1000, 64
    assert L.lce_workspace_size_opt(n, d, v, c, 8, ctypes.byref(out)) == OK
    need = out.value
    # frozen W with accumulation into dW: refused before anything runs
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, n, d, v, -100, c, 0, 8 | 1,
                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), need,
                             None) == INVALID
    assert L.lce_backward_opt(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE),
                              n, d, v, -100, c, 0, 8 | 1, vp(FAKE), need, None) == INVALID
    # without the flag a NULL dW is an argument error; with it, the argument checks pass
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, n, d, v, -100, c, 0, 0,
                             vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), need,
                             None) == INVALID
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, n, d, v, -100, c, 0, 8,
                             vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), need,
                             None) not in (OK, INVALID, ALIGN, WORKSPACE)
    # a frozen-W call given the plain workspace size may be short of its parts
    assert L.lce_fwd_bwd_opt(vp(FAKE), vp(FAKE), vp(FAKE), None, N, D, V, -100, chunk, 0, 8,
                             vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), base,
                             None) == WORKSPACE


def test_norm_opt_flags(L):
    """lce_norm_*_opt take 0 or LCE_FROZEN_W; the flag-less calls equal flags = 0."""
    N, D, V, chunk = 16384, 4096, 128256, 1024
    out = ctypes.c_size_t(0)
    plain = ctypes.c_size_t(0)
    assert L.lce_norm_workspace_size(N, D, V, chunk, ctypes.byref(plain)) == OK
    assert L.lce_norm_workspace_size_opt(N, D, V, chunk, 0, ctypes.byref(out)) == OK
    assert out.value == plain.value
    for bad in (1, 2, 4, 32):
        assert L.lce_norm_workspace_size_opt(N, D, V, chunk, bad, ctypes.byref(out)) == INVALID
    assert L.lce_norm_workspace_size_opt(N, D, V, chunk, 8, ctypes.byref(out)) == OK
    # frozen W: no H chunk^T; the two dH parts of the frozen split hold the chunk's dH
    assert out.value == (ws_size_low(L, N, D, V, chunk) - 2 * D * chunk + 2 * 4 * chunk * D
                         + 2 * chunk * D + 4 * 256 * D)
    vp = ctypes.c_void_p
    n, d, v, c = 128, 64, 1000, 64
    assert L.lce_norm_workspace_size_opt(n, d, v, c, 8, ctypes.byref(out)) == OK
    need = out.value

    def call(flags, dW):
        return L.lce_norm_fwd_bwd_opt(vp(FAKE), vp(FAKE), 1e-6, vp(FAKE), vp(FAKE), None, n, d, v,
                                      -100, c, 0, flags, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                      dW, vp(FAKE), need, None)
    assert call(0, None) == INVALID                 # dW needed without the flag
    assert call(1, vp(FAKE)) == INVALID             # accumulation flags are not taken here
    assert call(8, vp(FAKE + 4)) == ALIGN           # a given dW is still checked
    assert call(8, None) not in (OK, INVALID, ALIGN, WORKSPACE)   # argument checks pass
    # without flags, the size lce_norm_workspace_size gives passes the checks too
    assert L.lce_norm_workspace_size(n, d, v, c, ctypes.byref(out)) == OK
    assert L.lce_norm_fwd_bwd_opt(vp(FAKE), vp(FAKE), 1e-6, vp(FAKE), vp(FAKE), None, n, d, v,
                                  -100, c, 0, 0, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                  vp(FAKE), out.value, None) not in (OK, INVALID, ALIGN, WORKSPACE)


def test_binding_constants_match_the_header():
    """Status codes, reductions, flags and profiling kinds: the binding's copies
    equal the values include/lce.h declares."""
    import linear_cross_entropy_chunked_gb300._binding as B
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    consts = {k: int(v) for k, v in re.findall(r"\b(LCE_[A-Z0-9_]+)\s*=\s*(\d+)", src)}
    for code, name in B.STATUS_NAMES.items():
        assert consts[name] == code, name
    for name, v in B.REDUCTIONS.items():
        assert consts[f"LCE_REDUCTION_{name.upper()}"] == v
    assert consts["LCE_ACCUMULATE_DW"] == B.ACCUMULATE["dW"]
    assert consts["LCE_ACCUMULATE_DH"] == B.ACCUMULATE["dH"]
    assert consts["LCE_INPUT_FP16"] == B.INPUT_FP16
    assert consts["LCE_FROZEN_W"] == B.FROZEN_W
    assert consts["LCE_LOW_MEMORY"] == B.LOW_MEMORY
    assert consts["LCE_FLAGS_ALL"] == (B.ACCUMULATE["dW"] | B.ACCUMULATE["dH"] | B.INPUT_FP16 |
                                       B.FROZEN_W | B.LOW_MEMORY)
    for name, v in B.KERNEL_KINDS.items():
        assert consts[f"LCE_KERNEL_{name.upper()}"] == v
    assert consts["LCE_KERNEL_KINDS"] == len(B.KERNEL_KINDS)


def test_binding_flag_logic_on_the_host():
    """The binding's option handling, no device involved: accumulate subsets map
    to flags, accumulating needs the tensors, frozen W adds its flag and refuses
    accumulating into dW; unknown reductions raise."""
    import torch
    import linear_cross_entropy_chunked_gb300._binding as B
    t = torch.zeros(1)
    assert B._acc_flags((), None, None) == 0
    assert B._acc_flags(("dW",), None, t) == 1
    assert B._acc_flags(("dH", "dW"), t, t) == 3
    assert B._acc_flags(("dH",), t, None, compute_dW=False) == 2 | B.FROZEN_W
    assert B._acc_flags((), None, None, compute_dW=False) == B.FROZEN_W
    with pytest.raises(ValueError):
        B._acc_flags(("dW",), None, None)               # nothing to add into
    with pytest.raises(ValueError):
        B._acc_flags(("dW",), None, t, compute_dW=False)
    with pytest.raises(ValueError):
        B._acc_flags(("dx",), t, t)
    assert [B._reduction(r) for r in ("mean", "sum", "none")] == [0, 1, 2]
    with pytest.raises(ValueError):
        B._reduction("avg")


def test_count_valid_refuses_host_tensors():
    """The valid-row count runs in the library (lce_count_valid): a host tensor is
    refused before the library is touched."""
    import torch
    from linear_cross_entropy_chunked_gb300 import count_valid
    with pytest.raises(ValueError):
        count_valid(torch.tensor([0, 5, -100]), 10)


def test_count_and_sharded_argument_errors(L):
    """lce_count_valid and lce_fwd_bwd_sharded reject bad arguments before any
    launch (fake device pointers, never dereferenced)."""
    fake = ctypes.c_void_p(1 << 20)
    out = ctypes.c_void_p(1 << 21)
    assert L.lce_count_valid(fake, -1, 10, -100, out, None) == INVALID
    assert L.lce_count_valid(fake, 4, 0, -100, out, None) == INVALID
    assert L.lce_count_valid(fake, 4, 10, -100, None, None) == INVALID
    assert L.lce_count_valid(ctypes.c_void_p((1 << 20) + 8), 4, 10, -100, out, None) == ALIGN
    assert L.lce_count_valid(fake, 4, 10, -100, ctypes.c_void_p((1 << 21) + 4), None) == ALIGN
    p = [ctypes.c_void_p((1 << 20) + 4096 * i) for i in range(10)]
    # no n_valid_total
    assert L.lce_fwd_bwd_sharded(p[0], p[1], p[2], None, None, 8, 64, 100, -100, 64, 0, p[3], p[4],
                                 p[5], p[6], p[7], 1 << 30, None) == INVALID
    # n_valid_total not 8-byte aligned
    assert L.lce_fwd_bwd_sharded(p[0], p[1], p[2], None, ctypes.c_void_p((1 << 20) + 3), 8, 64,
                                 100, -100, 64, 0, p[3], p[4], p[5], p[6], p[7], 1 << 30,
                                 None) == ALIGN
    # workspace too small
    assert L.lce_fwd_bwd_sharded(p[0], p[1], p[2], None, p[8], 8, 64, 100, -100, 64, 0, p[3], p[4],
                                 p[5], p[6], p[7], 16, None) == WORKSPACE


def test_forward_workspace_is_the_forward_share(L):
    """lce_forward needs no chunk buffer: its workspace is the header, the row
    losses, the chunk's target logits and slab partials, far below the full size."""
    for N, D, V, chunk in ((16384, 4096, 128256, 1024), (4096, 4096, 32000, 1024),
                           (77, 128, 100, 1024), (0, 64, 300, 128)):
        full = ctypes.c_size_t(0)
        fwd = ctypes.c_size_t(0)
        assert L.lce_workspace_size(N, D, V, chunk, ctypes.byref(full)) == OK
        assert L.lce_forward_workspace_size(N, D, V, chunk, ctypes.byref(fwd)) == OK
        C = min(chunk, max(N, 1))
        parts = C * ((V + 127) // 128) * 8
        assert parts + 4 * max(N, 1) <= fwd.value <= parts + 4 * max(N, 1) + 4 * C + 16 * 1024
        assert fwd.value < full.value
    assert L.lce_forward_workspace_size(8, 7, 100, 64, ctypes.byref(fwd)) == INVALID
    # 16384 x 128256 at chunk 1024: ~8.3 MB, within the no-alloc entry point's 64 MiB
    assert L.lce_forward_workspace_size(16384, 4096, 128256, 1024, ctypes.byref(fwd)) == OK
    assert fwd.value < 9 << 20


def test_no_library_means_loud_failure(monkeypatch):
    """Without the built library every call raises (there is no fallback), and
    every entry point refuses CPU tensors before touching the library."""
    import torch
    import linear_cross_entropy_chunked_gb300._binding as B
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.setattr(B, "LIB_PATH", "/nonexistent/liblce_gb300.so")
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
    with pytest.raises(RuntimeError):
        B.workspace_size(8, 64, 100, 64)
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(16, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    for call in (lambda: B.lce_fwd_bwd(H, W, y), lambda: B.lce_backward(H, W, y, torch.zeros(4)),
                 lambda: B.ce_logits(torch.zeros(4, 16), y), lambda: B.rmsnorm_forward(H, H[0]),
                 lambda: B.norm_fwd_bwd(H, H[0], W, y)):
        with pytest.raises(ValueError):
            call()
