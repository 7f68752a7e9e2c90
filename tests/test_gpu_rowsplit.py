"""The row split of one search (post_weight_quantization_33_b300.rowsplit) on
one B300, one process standing for the ranks: each rank's rows searched on
the GPU, the per-weight sums of row losses combined, every rank's rows
quantized at the chosen grid point.  The combined losses equal the whole
search's (both are sums of the same row losses), the chosen alpha is the
same, and the ranks' codes, scales and zeros, concatenated, are bit-exact
those of the whole search."""
import numpy as np
import pytest
import torch

import post_weight_quantization_33_b300 as awq
import workloads
from post_weight_quantization_33_b300 import rowsplit

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("bits,group", [(4, 128), (3, 64)])
def test_row_split_equals_whole_search(world, bits, group):
    Ws, X = [], None
    for j, n in enumerate((300, 130)):
        W, X0 = workloads.random_layer(n, 512, 200, seed=720 + j, outliers=(4, 300), factor=30.0)
        Ws.append(torch.from_numpy(W).cuda())
        X = X0 if X is None else X
    Xd = torch.from_numpy(X).cuda()
    whole = awq.search(Xd, Ws, bits, group, 20)
    whole.check()
    parts, shards = [], []
    for rank in range(world):
        spans = [rowsplit.shard_rows(W.shape[0], world, rank) for W in Ws]
        local = [W[a:b].contiguous() for W, (a, b) in zip(Ws, spans)]
        r = awq.search(Xd, local, bits, group, 20)
        r.check()
        parts.append(rowsplit.partial_sums(r.row_losses().cpu().numpy(),
                                           [W.shape[0] for W in local]))
        s_grid = r.s_grid()
        r.free()
        shards.append((local, s_grid))
    losses, best = rowsplit.combine(np.stack(parts), [W.shape[0] for W in Ws], X.shape[0])
    np.testing.assert_allclose(losses, whole.losses, rtol=1e-12)
    assert best == whole.best
    for i, W in enumerate(Ws):
        codes, scales, zeros = [], [], []
        for local, s_grid in shards:
            c, sc, z = awq.quantize_pack(local[i], s_grid[best].contiguous(), bits, group)
            codes.append(c.cpu())
            scales.append(sc.cpu())
            zeros.append(z.cpu())
        # every row is whole words (K/8 for INT4, 3K/32 for INT3): the ranks'
        # codes concatenate
        assert torch.equal(torch.cat(codes), whole.codes(i).cpu())
        assert torch.equal(torch.cat(scales), whole.scales(i).cpu())
        assert torch.equal(torch.cat(zeros), whole.zeros(i).cpu())
    whole.free()
