"""The bounds-checked build on the GPU.  In libawq_checked.so every computed
global index of the statistic, scales, quantizers, decode product, losses and
fold kernels is compared with its buffer's extent before the access (a miss
is recorded, not trapped).  A fresh process loads that library, shows the
record path working (a synthetic out-of-range index), then runs the parity
suite's shape families -- odd and ragged sizes, padding between weights,
INT3 / INT4, groups of 64 / 128 / one per row, symmetric codes, the Gram form,
1-16 tokens with x staged, split or read through L1, 64- and 128-channel units
-- and expects no out-of-range access and finite results."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import post_weight_quantization_33_b300 as awq
from post_weight_quantization_33_b300 import build as awq_build
import workloads

awq._LIB_PATH = awq_build.CHECKED_LIB_PATH
L = awq.lib()
assert L.awq_bounds_checked() == 1
out = {}
torch.cuda.set_device(0)
awq._check(L.awq_bounds_selftest())
out["selftest"] = awq.bounds_report(reset=True)
out["after_reset"] = awq.bounds_report(reset=True)
g = torch.Generator(device="cuda").manual_seed(3)
finite = True

def fin(t):
    global finite
    finite = finite and bool(torch.isfinite(t.float()).all())

# statistic and scales
for T, K in ((1, 8), (17, 264), (4099, 264), (33, 1024), (640, 8192)):
    X = (torch.randn(T, K, generator=g, device="cuda") * 3).half()
    sX = awq.stats(X); fin(sX)
    fin(awq.stats_noalloc(X))
    fin(awq.scales(sX, 20))
# quantize + pack, unpack, fold
for N, K, bits, group, zp in ((37, 256, 4, 64, True), (300, 1024, 3, 128, True),
                              (129, 512, 4, -1, True), (45, 704, 4, 64, False),
                              (1, 128, 3, 128, True), (77, 2048, 4, 128, True)):
    W = (torch.randn(N, K, generator=g, device="cuda") * 0.02).half()
    s = torch.rand(K, generator=g, device="cuda") + 0.5
    codes, sc, z = awq.quantize_pack(W, s, bits, group, zero_point=zp)
    fin(sc)
    awq.unpack_codes(codes, N, K, bits)
for rows, cols in ((33, 24), (5, 1), (1000, 1), (17, 4096), (19, 13)):
    V = torch.randn(rows, cols, generator=g, device="cuda").half()
    s = torch.rand(rows, generator=g, device="cuda") + 0.5
    fin(awq.fold_scale(V.reshape(-1) if cols == 1 else V, s))
# searches
for n_rows, K, T, bits, group, zp, gram in (
        ((128,), 256, 64, 4, 128, True, False), ((96, 64), 512, 40, 4, 128, True, False),
        ((300,), 256, 17, 3, 64, True, False), ((64,), 1024, 1, 4, 128, False, False),
        ((200, 56), 512, 300, 4, -1, True, False), ((256,), 512, 1024, 4, 128, True, True),
        ((37,), 2048, 77, 3, 128, True, True)):
    Ws = [(torch.randn(n, K, generator=g, device="cuda") * 0.02).half() for n in n_rows]
    X = torch.randn(T, K, generator=g, device="cuda").half()
    X[:, : max(1, K // 100)] *= 20
    r = awq.search(X, Ws, bits, group, 20, zero_point=zp, gram=gram)
    r.check()
    fin(torch.tensor(r.losses))
    r.free()
# decode product
for M in (1, 5, 8, 9, 16):
    for bits in (4, 3):
        for N, K, group in ((37, 256, 64), (300, 1024, 128), (129, 4096, -1), (45, 704, 64),
                            (33, 192, -1), (70, 8192, 64), (520, 12288, 128), (40, 12416, 64),
                            (19000, 1152, 64)):
            if bits == 3 and K % 32:
                continue
            W = (torch.randn(N, K, generator=g, device="cuda") * 0.02).half()
            s = torch.ones(K, device="cuda")
            codes, sc, z = awq.quantize_pack(W, s, bits, group)
            x = torch.randn(M, K, generator=g, device="cuda").half()
            fin(awq.w4a16_matvec(codes, sc, z, N, K, x, group, bits=bits))
torch.cuda.synchronize()
out["suite"] = awq.bounds_report(reset=True)
out["finite"] = finite
print("RESULT " + json.dumps(out))
"""


def test_checked_build_reports_no_out_of_range_access():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    res = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + SCRIPT], cwd=ROOT,
                         env=env, capture_output=True, text=True, timeout=1200)
    assert res.returncode == 0, res.stderr[-3000:]
    line = [l for l in res.stdout.splitlines() if l.startswith("RESULT ")][-1]
    out = json.loads(line[len("RESULT "):])
    st = out["selftest"]
    assert st["checked"] and st["count"] == 1 and st["site"] == 0
    assert st["index"] == -1 and st["extent"] == 0
    assert out["after_reset"]["count"] == 0
    assert out["suite"]["count"] == 0, out["suite"]
    assert out["finite"]
