"""Write the oracle's full-size search results for the large workloads.

    python tests/golden/make_full_size_goldens.py [workload ...] [--workers N]

For every call of each workload (default: llama7b_mlp, llama70b,
int3_stress) the CPU oracle searches EVERY output row of every weight
(``oracle.row_pool`` runs ``awq_oracle.search`` on row blocks in worker
processes and adds the rows' losses).  It writes
``tests/golden/full_size_<workload>.json`` with, per call:

* ``sha256``: a digest of each input tensor's fp16 bytes, so a test can tell
  whether ``workloads.generate`` still produces the same inputs;
* ``losses``: the n_grid per-grid-point losses, sum_i ||E_i||^2 / (N_i T);
* ``best``: the first index of their minimum; ``gap_rel``: the relative gap
  between the two smallest losses;
* ``sample_rows`` / ``sample_row_losses``: a fixed sample of output rows per
  weight and their per-grid-point row losses sum_t E[n, t]^2.

This script imports only ``oracle/`` and ``workloads.py``; nothing in it comes
from the CUDA path.  The quantizer, loss and argmin are the oracle's
("AWQ Explained", multigrid.ai, "How the scale is chosen").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402
from oracle import awq_oracle as O  # noqa: E402
from oracle.row_pool import OraclePool  # noqa: E402

N_GRID = 20
DEFAULT = ("llama7b_mlp", "llama70b", "int3_stress")


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def sample_rows(n: int, seed: int) -> np.ndarray:
    """Tile edges (0, 1, 127, 128, 255, 256), the middle, the last rows, and
    seven seeded rows."""
    fixed = [0, 1, 127, 128, 255, 256, n // 2, n - 129, n - 1]
    extra = workloads.weight_rng(seed).choice(n, 7, replace=False)
    return np.unique(np.clip(np.concatenate([fixed, extra]), 0, n - 1)).astype(np.int64)


def path_for(name: str) -> str:
    return os.path.join(HERE, f"full_size_{name}.json")


def make(name: str, workers: int | None) -> dict:
    wl = workloads.WORKLOADS[name]
    data = workloads.generate(name)
    out = {"workload": name, "description": wl.description, "n_grid": N_GRID, "calls": [],
           "made_by": "tests/golden/make_full_size_goldens.py (CPU oracle, every output row)"}
    with OraclePool(data, workers) as pool:
        for ci, call in enumerate(wl.calls):
            t0 = time.time()
            X = data[call.x]
            sX = O.channel_magnitude(X)
            rows_all = [np.arange(wl.spec(w).rows) for w in call.ws]
            block = min(1024, -(-sum(len(r) for r in rows_all) // pool.workers))
            r = pool.search_rows(call.x, call.ws, call.bits, call.group, N_GRID, rows_all,
                                 sX=sX, block_rows=block)
            losses = r["losses"]
            order = np.argsort(losses, kind="stable")
            samples = [sample_rows(wl.spec(w).rows, 1000 * wl.index + 10 * ci + j)
                       for j, w in enumerate(call.ws)]
            out["calls"].append({
                "x": call.x, "ws": list(call.ws), "bits": call.bits, "group": call.group,
                "T": int(X.shape[0]), "K": int(X.shape[1]),
                "N": [int(wl.spec(w).rows) for w in call.ws],
                "sha256": {n: digest(data[n]) for n in (call.x, *call.ws)},
                "losses": [float(v) for v in losses],
                "best": int(r["best"]),
                "gap_rel": float((losses[order[1]] - losses[order[0]]) / losses[order[0]]),
                "sample_rows": [s.tolist() for s in samples],
                "sample_row_losses": [rl[:, s].T.tolist()
                                      for rl, s in zip(r["row_losses"], samples)],
            })
            print(f"{name} call {ci}: best {r['best']} gap {out['calls'][-1]['gap_rel']:.3e} "
                  f"({time.time() - t0:.0f} s)", flush=True)
    return out


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("workloads", nargs="*", default=list(DEFAULT))
    ap.add_argument("--workers", type=int, default=None)
    a = ap.parse_args()
    for name in a.workloads:
        res = make(name, a.workers)
        with open(path_for(name), "w") as f:
            json.dump(res, f, indent=1)
            f.write("\n")
        print(f"wrote {path_for(name)}", flush=True)


if __name__ == "__main__":
    main()
