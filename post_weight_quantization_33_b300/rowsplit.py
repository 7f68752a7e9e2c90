"""One scale search split over the output rows of its weights, across ranks.

The search loss is a sum over output rows ("AWQ Explained", multigrid.ai, "How
the scale is chosen": the error is the norm of the whole layer-output
difference, here sum_i ||E_i||^2 / (N_i T) over the weights W_i sharing X).
Quantization and the error are per row, so a rank that holds rows
[r0, r1) of every weight and the whole X searches its rows alone; the only
exchange is one all-reduce of the per-weight, per-grid-point sums of its row
losses (n_w x n_grid fp64 values).  Every rank then takes the same first
argmin and quantizes its rows at the chosen grid point; s depends on X alone,
so every rank holds the same s.

Used from one process per GPU (torch.distributed, nccl or gloo); the host
logic (``shard_rows``, ``combine``) is plain numpy and runs anywhere.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import quantize_pack, search


def shard_rows(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Rows [r0, r1) of an N-row weight held by `rank` of `world`: contiguous
    blocks, the first N % world ranks one row longer."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    base, extra = divmod(N, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def partial_sums(row_losses: np.ndarray, rows_per_weight: Sequence[int]) -> np.ndarray:
    """Per weight and grid point, the sum of this rank's row losses:
    row_losses [n_grid][sum of local rows] (weights concatenated) ->
    [n_w][n_grid] fp64."""
    out = np.zeros((len(rows_per_weight), row_losses.shape[0]), np.float64)
    off = 0
    for i, n in enumerate(rows_per_weight):
        out[i] = row_losses[:, off:off + n].sum(axis=1)
        off += n
    return out


def combine(partials: np.ndarray, N_total: Sequence[int], T: int,
            process_group=None, device=None) -> Tuple[np.ndarray, int]:
    """The call's losses from every rank's partial sums, and their first
    argmin (NaN as +inf).

    ``partials``: this rank's [n_w][n_grid] sums, or, without a process group,
    an array [ranks][n_w][n_grid] holding every rank's (one process standing
    for all of them).  With a process group the sums are all-reduced (one
    collective of n_w * n_grid fp64 values), on ``device`` (a CUDA device for
    nccl, the CPU for gloo)."""
    p = np.asarray(partials, np.float64)
    if process_group is not None:
        import torch.distributed as dist
        t = torch.from_numpy(np.ascontiguousarray(p)).to(device or "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=process_group)
        total = t.cpu().numpy()
    else:
        total = p.sum(axis=0) if p.ndim == 3 else p
    losses = np.zeros(total.shape[1], np.float64)
    for i, n in enumerate(N_total):
        losses += total[i] / (float(n) * float(T))
    best, best_v = 0, None
    for i, v in enumerate(losses):
        v = np.inf if np.isnan(v) else v
        if best_v is None or v < best_v:
            best, best_v = i, v
    return losses, best


def search_row_shard(X: torch.Tensor, Ws_local: Sequence[torch.Tensor], N_total: Sequence[int],
                     bits: int = 4, group: int = 128, n_grid: int = 20,
                     zero_point: bool = True, process_group=None) -> Dict:
    """This rank's part of one search: ``Ws_local[i]`` are its rows of weight
    i (full weight: ``N_total[i]`` rows), X the whole calibration batch on
    this rank's GPU.  Returns the call's losses and alpha (identical on every
    rank) and this rank's codes, scales and zeros at the chosen grid point."""
    r = search(X, Ws_local, bits, group, n_grid, zero_point=zero_point)
    try:
        r.check()
        rows = r.row_losses().cpu().numpy()
        s_grid = r.s_grid()
    finally:
        r.free()
    part = partial_sums(rows, [W.shape[0] for W in Ws_local])
    losses, best = combine(part, N_total, X.shape[0], process_group,
                           device=X.device if process_group is not None and
                           _is_nccl(process_group) else None)
    s = s_grid[best].contiguous()
    out: Dict = {"losses": losses, "best": best, "alpha": best / n_grid, "s": s,
                 "codes": [], "scales": [], "zeros": []}
    for W in Ws_local:
        c, sc, z = quantize_pack(W, s, bits, group, zero_point=zero_point)
        out["codes"].append(c)
        out["scales"].append(sc)
        out["zeros"].append(z)
    return out


def _is_nccl(process_group) -> bool:
    import torch.distributed as dist
    try:
        return dist.get_backend(process_group) == "nccl"
    except Exception:
        return False
