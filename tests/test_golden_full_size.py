"""The stored full-size oracle results (tests/golden/full_size_*.json) on
CPU: they are well formed, their argmin is the first minimum of their
losses, and the oracle as it stands reproduces a sample of their row losses
on the very inputs the generator produces (same SHA-256).  The GPU compares
its searches with these files in tests/test_gpu_full_size.py."""
import hashlib
import json
import os

import numpy as np
import pytest

import workloads
from oracle import awq_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NAMES = ["llama7b_mlp", "llama70b", "int3_stress"]


def load(name):
    with open(os.path.join(GOLDEN, f"full_size_{name}.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("name", NAMES)
def test_golden_well_formed(name):
    g = load(name)
    wl = workloads.WORKLOADS[name]
    assert g["workload"] == name and g["n_grid"] == 20
    assert len(g["calls"]) == len(wl.calls)
    for c, call in zip(g["calls"], wl.calls):
        assert (c["x"], tuple(c["ws"]), c["bits"], c["group"]) == \
            (call.x, call.ws, call.bits, call.group)
        losses = np.asarray(c["losses"])
        assert losses.shape == (20,) and np.all(np.isfinite(losses)) and np.all(losses > 0)
        assert c["best"] == O.first_argmin(losses)
        order = np.sort(losses)
        assert c["gap_rel"] == pytest.approx((order[1] - order[0]) / order[0], rel=1e-12)
        for i, w in enumerate(call.ws):
            rows = np.asarray(c["sample_rows"][i])
            assert rows.ndim == 1 and rows.min() >= 0 and rows.max() < wl.spec(w).rows
            assert np.asarray(c["sample_row_losses"][i]).shape == (rows.size, 20)


@pytest.mark.parametrize("name", NAMES)
def test_golden_rows_reproduced_by_the_oracle(name):
    """First call of each workload: the generator's inputs hash as stored,
    and the oracle's row losses of the first sampled row of every weight equal
    the stored ones (the same code on the same inputs; 1e-12 allows for a
    different BLAS blocking)."""
    g = load(name)
    wl = workloads.WORKLOADS[name]
    c, call = g["calls"][0], wl.calls[0]
    data = workloads.generate(name, only=[call.x, *call.ws])
    for t, h in c["sha256"].items():
        assert hashlib.sha256(np.ascontiguousarray(data[t]).tobytes()).hexdigest() == h, t
    X = data[call.x]
    for i, w in enumerate(call.ws):
        row = int(c["sample_rows"][i][0])
        r = O.search(X, [data[w]], call.bits, call.group, 20, rows=[np.array([row])])
        np.testing.assert_allclose(r["row_losses"][0][:, 0], np.asarray(
            c["sample_row_losses"][i][0]), rtol=1e-12)
