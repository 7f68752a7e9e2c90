"""The row split of one search across ranks (post_weight_quantization_33_b300
.rowsplit), host logic on CPU: the row partition, and the combine (one
all-reduce of the per-weight sums of row losses, then the first argmin) with
world-size-2 gloo process groups.  The per-rank searches are the CPU oracle
over each rank's rows, so the combined result must equal the oracle's search
over all rows."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from oracle import awq_oracle as O  # noqa: E402
from post_weight_quantization_33_b300 import rowsplit  # noqa: E402


def _layer():
    """A two-weight call with ragged row counts and outlier channels."""
    Ws, X = [], None
    for j, n in enumerate((131, 70)):
        W, X0 = workloads.random_layer(n, 256, 90, seed=610 + j, outliers=(3, 100), factor=30.0)
        Ws.append(W)
        X = X0 if X is None else X
    return X, Ws


def _rank_partials(X, Ws, world, rank):
    rows = [np.arange(*rowsplit.shard_rows(W.shape[0], world, rank)) for W in Ws]
    r = O.search(X, Ws, 4, 128, 20, rows=rows)
    rl = np.concatenate(r["row_losses"], axis=1)
    return rowsplit.partial_sums(rl, [len(x) for x in rows])


@pytest.mark.parametrize("N,world", [(1, 1), (7, 2), (256, 2), (131, 3), (5, 8)])
def test_shard_rows_partition(N, world):
    spans = [rowsplit.shard_rows(N, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == N
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in spans]
    assert max(sizes) - min(sizes) <= 1 and all(s >= 0 for s in sizes)
    with pytest.raises(ValueError):
        rowsplit.shard_rows(N, world, world)


def test_combine_of_stacked_partials_equals_full_search():
    X, Ws = _layer()
    full = O.search(X, Ws, 4, 128, 20)
    parts = np.stack([_rank_partials(X, Ws, 3, r) for r in range(3)])
    losses, best = rowsplit.combine(parts, [W.shape[0] for W in Ws], X.shape[0])
    np.testing.assert_allclose(losses, full["losses"], rtol=1e-12)
    assert best == full["best"]


def test_combine_first_argmin_nan_as_inf():
    p = np.array([[[np.nan, 2.0, 1.0, 1.0]]])
    losses, best = rowsplit.combine(p, [1], 1)
    assert best == 2 and np.isnan(losses[0])


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, Ws = _layer()
        part = _rank_partials(X, Ws, world, rank)
        losses, best = rowsplit.combine(part, [W.shape[0] for W in Ws], X.shape[0],
                                        process_group=dist.group.WORLD)
        results[rank] = (losses.tolist(), best)
    finally:
        dist.destroy_process_group()


def test_combine_all_reduce_gloo_world_2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0, f"rank exited with {p.exitcode}"
        out = dict(results)
    X, Ws = _layer()
    full = O.search(X, Ws, 4, 128, 20)
    assert set(out) == {0, 1}
    assert out[0] == out[1]                      # every rank holds the same result
    np.testing.assert_allclose(out[0][0], full["losses"], rtol=1e-12)
    assert out[0][1] == full["best"]
