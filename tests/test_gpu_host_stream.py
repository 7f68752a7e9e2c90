"""The pipelined host-buffer search (search_host_stream) against one device
search per layer: identical codes, scales, zeros, s, losses and alpha, for a
sequence of layers of different shapes (more layers than input slots, one
call with two weights sharing X)."""
import numpy as np
import pytest
import torch

import post_weight_quantization_33_b300 as awq
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    awq.lib()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _layers():
    shapes = [((128,), 256, 64), ((96, 64), 512, 40), ((256,), 256, 300), ((64,), 1024, 17),
              ((128,), 256, 64)]
    out = []
    for j, (ns, k, t) in enumerate(shapes):
        Ws, X = [], None
        for i, n in enumerate(ns):
            W, X0 = workloads.random_layer(n, k, t, seed=300 + 7 * j + i, outliers=(1, k // 3),
                                          factor=20.0)
            Ws.append(torch.from_numpy(W).pin_memory())
            X = X0 if X is None else X
        out.append((torch.from_numpy(X).pin_memory(), Ws))
    return out


@pytest.mark.parametrize("bits,group", [(4, 128), (3, 64)])
def test_search_host_stream_matches_device_search(bits, group):
    layers = _layers()
    got = awq.search_host_stream(layers, bits, group, 20)
    assert len(got) == len(layers)
    for (X, Ws), g in zip(layers, got):
        r = awq.search(X.cuda(), [W.cuda() for W in Ws], bits, group, 20)
        r.check()
        assert g["best"] == r.best and g["alpha"] == r.alpha
        assert np.array_equal(g["losses"], r.losses)
        assert torch.equal(g["s"], r.s().cpu())
        for i in range(len(Ws)):
            assert torch.equal(g["codes"][i], r.codes(i).cpu())
            assert torch.equal(g["scales"][i], r.scales(i).cpu())
            assert torch.equal(g["zeros"][i], r.zeros(i).cpu())
        r.free()


def test_search_host_stream_empty_and_single():
    assert awq.search_host_stream([], 4, 128) == []
    (X, Ws), = _layers()[:1]
    g, = awq.search_host_stream([(X, Ws)], 4, 128)
    ref = awq.search_host(X, Ws, 4, 128)
    assert g["best"] == ref["best"]
    assert np.array_equal(g["losses"], ref["losses"])
    assert torch.equal(g["codes"][0], ref["codes"][0])


def test_search_host_stream_failure_frees_in_flight_results():
    """A layer that fails validation in the middle of the sequence raises;
    the layers already in flight are completed and freed, and the library
    keeps working."""
    layers = _layers()[:3]
    # K = 96 passes the host-side checks but is not a multiple of the group
    # size: the library refuses it after the first layer is already in flight.
    bad = (torch.zeros((32, 96), dtype=torch.float16).pin_memory(),
           [torch.zeros((64, 96), dtype=torch.float16).pin_memory()])
    seq = [layers[0], bad, layers[2]]
    with pytest.raises(awq.AwqError):
        awq.search_host_stream(seq, 4, 128)
    torch.cuda.synchronize()
    got = awq.search_host_stream(layers, 4, 128)
    ref = awq.search_host(*layers[2], 4, 128)
    assert np.array_equal(got[2]["losses"], ref["losses"])
    assert torch.equal(got[2]["codes"][0], ref["codes"][0])


def test_resumable_search_matches_host_stream(tmp_path):
    """Checkpoint / resume: a run in chunks of two stores every layer; a
    rerun reads them all back; after one file is removed only that layer is
    searched again.  Every result equals the plain pipelined search's."""
    from post_weight_quantization_33_b300 import checkpoint

    layers = _layers()
    ref = awq.search_host_stream(layers, 4, 128, 20)

    def same(a, b):
        assert a["best"] == b["best"] and a["alpha"] == b["alpha"]
        assert np.array_equal(np.asarray(a["losses"]), np.asarray(b["losses"]))
        assert np.array_equal(np.asarray(a["s"]), b["s"].numpy())
        for key in ("codes", "scales", "zeros"):
            for x, y in zip(a[key], b[key]):
                assert np.array_equal(np.asarray(x), y.numpy())

    first = checkpoint.search_layers_resumable(layers, str(tmp_path), 4, 128, 20, chunk=2)
    assert not any(r["resumed"] for r in first)
    again = checkpoint.search_layers_resumable(layers, str(tmp_path), 4, 128, 20, chunk=2)
    assert all(r["resumed"] for r in again)
    (tmp_path / "layer_00002.npz").unlink()
    third = checkpoint.search_layers_resumable(layers, str(tmp_path), 4, 128, 20, chunk=2)
    assert [r["resumed"] for r in third] == [True, True, False, True, True]
    def host(v):
        return v.numpy() if isinstance(v, torch.Tensor) else v

    for runs in (first, again, third):
        for r, g in zip(runs, ref):
            same({k: [host(x) for x in v] if isinstance(v, list) else host(v)
                  for k, v in r.items()}, g)
