"""Register and spill budget of the hot kernels, from ptxas's resource report
(nvcc -Xptxas -v; no GPU needed).  A change that makes a hot kernel spill, or
pushes the pair GEMM past the registers its 192-thread CTAs can have, fails
here before it is ever timed.  The INT3 final quantizer (run once per search,
after the grid) is allowed its measured 16 bytes under its 3-blocks-per-SM
bound."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "post_weight_quantization_33_b300", "csrc")

# (source, kernel-name pattern in the mangled name, max registers, max spill bytes)
BUDGET = [
    ("awq_gemm.cu", r"k_gemm_err_pair", 168, 0),
    ("awq_gemm.cu", r"k_gemm_ref", 168, 0),
    ("awq_quant.cu", r"k_quant_residual", 128, 0),
    ("awq_quant.cu", r"k_quant_finalILi4E", 85, 0),
    ("awq_quant.cu", r"k_quant_finalILi3E", 85, 16),
    ("awq_stats.cu", r"k_stats_accumulate", 112, 0),   # 2 blocks of 288 threads per SM
    # Decode product: one block of 16 warps per SM, or of 8 warps (255
    # registers each) for 16 tokens with x read through L1 (NT 2, XPERM false).
    ("awq_matvec.cu", r"k_wq_mmaILi1E|k_wq_mmaILi2ELi-?\d+ELi\dELb1E", 128, 0),
    ("awq_matvec.cu", r"k_wq_mmaILi2ELi-?\d+ELi\dELb0E", 255, 0),
    # TMA ring: 16 warps per SM for x staged in shared memory and up to 8
    # tokens, else 8 (255 registers each).
    ("awq_matvec.cu", r"k_wq_tmaILi1ELi-?\d+ELi\dELb1E", 128, 0),
    ("awq_matvec.cu", r"k_wq_tmaILi2E|k_wq_tmaILi1ELi-?\d+ELi\dELb0E", 255, 0),
    ("awq_reduce.cu", r"k_losses", 64, 0),
]


def _ptxas_report(src: str):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", os.devnull,
           "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    kernels, name = {}, None
    for line in out.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            name = m.group(1)
            kernels[name] = {"spill": 0, "regs": None}
            continue
        if name is None:
            continue
        m = re.search(r"(\d+) bytes spill stores", line)
        if m:
            kernels[name]["spill"] = int(m.group(1))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            kernels[name]["regs"] = int(m.group(1))
    return kernels


@pytest.fixture(scope="module")
def reports():
    return {src: _ptxas_report(src) for src in sorted({b[0] for b in BUDGET})}


@pytest.mark.parametrize("src,pattern,max_regs,max_spill", BUDGET,
                         ids=[b[1] for b in BUDGET])
def test_hot_kernel_register_and_spill_budget(reports, src, pattern, max_regs, max_spill):
    hits = {k: v for k, v in reports[src].items() if re.search(pattern, k)}
    assert hits, f"no kernel matching {pattern} in {src}"
    for name, r in hits.items():
        assert r["regs"] is not None and r["regs"] <= max_regs, (name, r)
        assert r["spill"] <= max_spill, (name, r)
