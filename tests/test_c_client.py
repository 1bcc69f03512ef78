"""The C ABI used from plain C: tests/c_client/lce_c_client.c includes only
include/lce.h and the CUDA runtime, links liblce_gb300.so and libcudart, and runs
lce_fwd_bwd on inputs read from files. On the CPU it must compile and link; on
the GPU its outputs must match the fp64 oracle and, bit for bit, the same call
made through the Python binding (the same kernels on the same inputs)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from lce_synth import make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "lce_c_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    import linear_cross_entropy_chunked_gb300 as pkg
    try:
        lib = pkg.build()
    except RuntimeError as e:   # no nvcc here
        pytest.skip(str(e))
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib)
    exe = os.path.join(out_dir, "lce_c_client")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-L", libdir, "-llce_gb300",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 1 and "usage" in r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,V,chunk", [(300, 264, 1000, 128), (1000, 1024, 8229, 256)])
def test_c_client_matches_oracle_and_binding(tmp_path, N, D, V, chunk):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle import lce_oracle as O
    from tests.gpu_util import check_grad, check_loss, check_lse
    import linear_cross_entropy_chunked_gb300 as lce

    exe = _compile(str(tmp_path))
    H, W, y = make_inputs(N, D, V, seed=N + V, n_ignored=N // 25, w_std=0.05)
    d = str(tmp_path)
    H.view(torch.int16).numpy().tofile(os.path.join(d, "H.bin"))
    W.view(torch.int16).numpy().tofile(os.path.join(d, "W.bin"))
    y.numpy().astype(np.int64).tofile(os.path.join(d, "y.bin"))
    r = subprocess.run([exe, str(N), str(D), str(V), str(chunk), d], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    loss = np.fromfile(os.path.join(d, "loss.bin"), dtype=np.float32)[0]
    lse = np.fromfile(os.path.join(d, "lse.bin"), dtype=np.float32)
    dH = torch.from_numpy(np.fromfile(os.path.join(d, "dH.bin"), dtype=np.int16).reshape(N, D))
    dH = dH.view(torch.bfloat16)
    dW = np.fromfile(os.path.join(d, "dW.bin"), dtype=np.float32).reshape(V, D)

    ref = O.forward_backward(H, W, y)
    check_loss(float(loss), ref["loss"])
    check_lse(lse.astype(np.float64), ref["lse"])
    check_grad("dH", dH.float().double().numpy(), ref["dH"])
    check_grad("dW", dW.astype(np.float64), ref["dW"])

    b_loss, b_lse, b_dH, b_dW = lce.lce_fwd_bwd(H.cuda(), W.cuda(), y.cuda(), chunk=chunk)
    torch.cuda.synchronize()
    assert np.float32(b_loss.item()) == loss
    assert np.array_equal(b_lse.cpu().numpy(), lse)
    assert torch.equal(b_dH.cpu(), dH)
    assert np.array_equal(b_dW.cpu().numpy(), dW)
