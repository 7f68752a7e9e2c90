"""Row-parallel driver for the CPU oracle.

TEST AND BASELINE INFRASTRUCTURE, like the rest of ``oracle/``: only the
tests, the scripts under ``tests/golden/`` and the benchmark's CPU legs use
it.  It adds no arithmetic of the method.  It runs ``awq_oracle.search``
unchanged on blocks of output rows in worker processes and adds up the rows'
losses.

The search loss is a sum over output rows ("AWQ Explained", multigrid.ai,
"How the scale is chosen": the error is the norm of the whole layer-output
difference).  Quantization and the error are per-row, so each row's loss from
a search over a block of rows is that row's loss from the full search.  A
call's loss at a grid point is then sum_i (sum over rows of W_i) / (N_i T) in
fp64, and alpha* is the first index of its minimum (``first_argmin``).

Workers are started with the ``spawn`` method, so a process that has already
initialised CUDA can use this safely.  Each worker runs its BLAS on
``blas_threads`` threads (default 1), so ``workers * blas_threads`` is the
number of cores the oracle uses.  The inputs are placed once in shared
memory, and workers map them read-only.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory
from typing import Dict, List, Optional, Sequence

import numpy as np

_ARRAYS: Dict[str, np.ndarray] = {}
_SHMS: List[shared_memory.SharedMemory] = []


def _attach(layout):
    # Spawned workers share the parent's resource tracker, so mapping a block
    # here adds no second owner: the parent alone unlinks it in close().
    for name, (shm_name, shape, dtype) in layout.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _SHMS.append(shm)
        a = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
        a.flags.writeable = False
        _ARRAYS[name] = a


def _block_task(task):
    from oracle import awq_oracle as O
    x_name, w_name, rows, bits, group, n_grid, sX, zero_point = task
    X = _ARRAYS[x_name]
    W = _ARRAYS[w_name]
    r = O.search(X, [W], bits, group, n_grid, sX=sX, rows=[rows], zero_point=zero_point)
    return r["row_losses"][0]


def default_workers() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


class OraclePool:
    """A pool of oracle worker processes over a fixed set of named arrays.

    Use as a context manager; ``close()`` ends the workers and frees the
    shared memory."""

    def __init__(self, arrays: Dict[str, np.ndarray], workers: Optional[int] = None,
                 blas_threads: int = 1):
        self.workers = int(workers or default_workers())
        self.blas_threads = max(1, int(blas_threads))
        self.cores = self.workers * self.blas_threads
        self._own: List[shared_memory.SharedMemory] = []
        layout = {}
        self.arrays: Dict[str, np.ndarray] = {}
        for name, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            view = np.ndarray(a.shape, a.dtype, buffer=shm.buf)
            view[...] = a
            self._own.append(shm)
            self.arrays[name] = view
            layout[name] = (shm.name, a.shape, a.dtype.str)
        # The workers' BLAS threads: the children read these at numpy import.
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS",
                                                "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = str(self.blas_threads)
        try:
            ctx = mp.get_context("spawn")
            self._pool = ctx.Pool(self.workers, initializer=_attach, initargs=(layout,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def close(self) -> None:
        self.arrays = {}
        if self._pool is not None:
            self._pool.close()
            self._pool.join()
            self._pool = None
        for shm in self._own:
            shm.close()
            shm.unlink()
        self._own = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def search_rows(self, x_name: str, w_names: Sequence[str], bits: int, group: int,
                    n_grid: int, rows: Sequence[np.ndarray], sX: Optional[np.ndarray] = None,
                    zero_point: bool = True, block_rows: Optional[int] = None) -> Dict:
        """Row losses of the selected rows of each weight, the call's losses
        over those rows, and the first argmin.

        ``rows[i]`` are the output rows of weight ``w_names[i]`` to search;
        they are cut into blocks (about one per worker, or ``block_rows``) that
        run in parallel.  ``sX`` is computed once here if not given."""
        call = dict(x=x_name, ws=list(w_names), bits=bits, group=group, n_grid=n_grid,
                    rows=rows, sX=sX, zero_point=zero_point)
        return self.search_calls([call], block_rows)[0]

    def search_calls(self, calls: Sequence[Dict], block_rows: Optional[int] = None) -> List[Dict]:
        """``search_rows`` for several calls at once: the row blocks of every
        call go to the workers in one batch.  Each call is a dict with keys
        x, ws, bits, group, n_grid, rows and optionally sX, zero_point."""
        from oracle import awq_oracle as O
        tasks, owners = [], []
        total_rows = sum(len(r) for c in calls for r in c["rows"])
        if block_rows is None:
            block_rows = max(1, -(-total_rows // self.workers))
        sxs = []
        for ci, c in enumerate(calls):
            sX = c.get("sX")
            if sX is None:
                sX = O.channel_magnitude(self.arrays[c["x"]])
            sxs.append(sX)
            for wi, (w_name, r) in enumerate(zip(c["ws"], c["rows"])):
                r = np.asarray(r, np.int64)
                for b0 in range(0, len(r), block_rows):
                    tasks.append((c["x"], w_name, r[b0:b0 + block_rows], c["bits"], c["group"],
                                  c["n_grid"], sX, c.get("zero_point", True)))
                    owners.append((ci, wi))
        results = self._pool.map(_block_task, tasks, chunksize=1)
        out = []
        for ci, c in enumerate(calls):
            T = self.arrays[c["x"]].shape[0]
            row_losses = []
            for wi in range(len(c["ws"])):
                parts = [res for res, o in zip(results, owners) if o == (ci, wi)]
                row_losses.append(np.concatenate(parts, axis=1) if parts
                                  else np.zeros((c["n_grid"], 0)))
            losses = np.zeros(c["n_grid"])
            for rl in row_losses:
                losses += rl.sum(axis=1) / (rl.shape[1] * T)
            out.append(dict(row_losses=row_losses, losses=losses, best=O.first_argmin(losses),
                            sX=sxs[ci]))
        return out
