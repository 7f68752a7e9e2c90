"""Failure paths of the library on a B300, made on the host (no GPU fault):
device allocations that fail as out of memory (awq_inject_allocation_failures
fakes the pool's answer without reaching the allocator) and non-finite
inputs.  Each failing call returns its error, releases every device buffer it
held (the pool's used bytes come back to where they were), and the next call
is correct."""
import numpy as np
import pytest
import torch

import post_weight_quantization_33_b300 as awq
import workloads
from oracle import awq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    awq.lib()
    torch.cuda.set_device(0)
    yield
    awq.inject_allocation_failures(0, 0)
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def disarm():
    yield
    awq.inject_allocation_failures(0, 0)


def used_after_sync():
    torch.cuda.synchronize()
    return awq.pool_usage()[0]


def tiny():
    t = workloads.generate("tiny")
    return t["X"], t["W"]


@pytest.mark.parametrize("skip", [0, 1], ids=["result-block", "scratch"])
def test_search_out_of_memory_releases_everything(skip):
    """skip 0: the result block's allocation fails; skip 1: the result block
    is allocated, the scratch fails, and the result block is released."""
    X, W = tiny()
    Xd, Wd = torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda()
    before = used_after_sync()
    awq.inject_allocation_failures(skip, 1)
    with pytest.raises(awq.AwqError) as e:
        awq.search(Xd, [Wd], 4, 128, 20)
    assert e.value.status == awq.AWQ_ERR_OOM
    assert used_after_sync() == before
    r = awq.search(Xd, [Wd], 4, 128, 20)
    r.check()
    ref = O.search(X, [W], 4, 128, 20)
    np.testing.assert_allclose(r.losses, ref["losses"], rtol=1e-3)
    r.free()
    assert used_after_sync() == before


def test_stats_out_of_memory_then_exact():
    X, _ = tiny()
    Xd = torch.from_numpy(X).cuda()
    before = used_after_sync()
    awq.inject_allocation_failures(0, 1)
    with pytest.raises(awq.AwqError) as e:
        awq.stats(Xd)
    assert e.value.status == awq.AWQ_ERR_OOM
    assert used_after_sync() == before
    assert np.array_equal(awq.stats(Xd).cpu().numpy(), O.channel_magnitude(X))


def _host_layers(n):
    out = []
    for j in range(n):
        W, X = workloads.random_layer(128 + 64 * j, 256, 64 + 40 * j, seed=500 + j,
                                      outliers=(2, 100), factor=20.0)
        out.append((torch.from_numpy(X).pin_memory(), [torch.from_numpy(W).pin_memory()]))
    return out


def test_host_pipeline_out_of_memory_mid_sequence():
    """The host pipeline allocates its input slots, then a result block and a
    scratch block per layer: skipping 3 allocations fails layer 1's result
    while layer 0 is in flight.  The call returns AWQ_ERR_OOM after layer 0's
    work completed, and nothing stays allocated."""
    layers = _host_layers(3)
    before = used_after_sync()
    awq.inject_allocation_failures(3, 1)
    with pytest.raises(awq.AwqError) as e:
        awq.search_host_stream(layers, 4, 128, 20)
    assert e.value.status == awq.AWQ_ERR_OOM
    assert used_after_sync() == before
    got = awq.search_host_stream(layers, 4, 128, 20)
    for (X, Ws), g in zip(layers, got):
        r = awq.search(X.cuda(), [W.cuda() for W in Ws], 4, 128, 20)
        r.check()
        assert g["best"] == r.best and np.array_equal(g["losses"], r.losses)
        assert torch.equal(g["codes"][0], r.codes(0).cpu())
        r.free()
    assert used_after_sync() == before


def test_host_pipeline_non_finite_layer():
    """A layer with a NaN activation in the middle of the sequence: the call
    reports AWQ_ERR_INVALID (a non-finite loss) and releases everything."""
    layers = _host_layers(3)
    X1 = layers[1][0].clone()
    X1[5, 17] = float("nan")
    bad = [layers[0], (X1.pin_memory(), layers[1][1]), layers[2]]
    before = used_after_sync()
    with pytest.raises(awq.AwqError) as e:
        awq.search_host_stream(bad, 4, 128, 20)
    assert e.value.status == awq.AWQ_ERR_INVALID and "non-finite" in str(e.value)
    assert used_after_sync() == before
