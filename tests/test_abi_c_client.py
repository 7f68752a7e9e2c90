"""The C ABI from a plain C99 program (tests/abi_c/awq_client.c), compiled with
gcc against include/awq.h and linked with libawq.so: the header is valid C,
every declared call links, the GPU-free calls behave as documented, and on a
B300 a search run from C -- on device buffers, or through the host-buffer
pipeline -- gives exactly what the Python binding gives."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import post_weight_quantization_33_b300 as awq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib_dir = os.path.dirname(awq.library_path())
    if not os.path.exists(awq.library_path()):
        pytest.skip("libawq.so not built")
    exe = str(tmp_path / "awq_client")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "abi_c", "awq_client.c"), "-o", exe,
           "-L", lib_dir, "-lawq", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_cpu_calls(tmp_path):
    exe = _build(tmp_path)
    out = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert "c client ok" in out.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["gpu", "host"])
def test_c_client_search_matches_binding(tmp_path, mode):
    """mode gpu: awq_search_layer on device buffers the C program filled;
    mode host: awq_search_host_layers from plain host buffers (three copies
    of the layer in one call, which the program checks agree)."""
    import torch
    import workloads
    exe = _build(tmp_path)
    W, X = workloads.random_layer(192, 512, 96, seed=901, outliers=(3, 200), factor=25.0)
    X.tofile(tmp_path / "x.bin")
    W.tofile(tmp_path / "w.bin")
    T, K = X.shape
    N = W.shape[0]
    out = subprocess.run([exe, mode, str(T), str(K), str(N), str(tmp_path / "x.bin"),
                          str(tmp_path / "w.bin"), str(tmp_path / "losses.bin"),
                          str(tmp_path / "codes.bin")], capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    losses = np.fromfile(tmp_path / "losses.bin", dtype=np.float64)
    codes = np.fromfile(tmp_path / "codes.bin", dtype=np.uint32)
    r = awq.search(torch.from_numpy(X).cuda(), [torch.from_numpy(W).cuda()], 4, 128, 20)
    r.check()
    assert np.array_equal(losses, r.losses)
    assert np.array_equal(codes, r.codes(0).cpu().numpy().view(np.uint32))
    assert f"best {r.best}" in out.stdout
    r.free()
