"""Checkpoint / resume of multi-layer searches (host logic, no GPU): a stand-in
search records which layers it was asked for; the tests check that finished
layers are stored and skipped on a rerun, that a missing, stale or torn file
is searched again, and that an interrupted run resumes where it stopped."""
import os

import numpy as np
import pytest
import torch

from post_weight_quantization_33_b300 import checkpoint as ck


def _layers(n, seed=0):
    g = torch.Generator().manual_seed(seed)
    out = []
    for i in range(n):
        X = torch.randn(8 + i, 64, generator=g).half()
        Ws = [torch.randn(16, 64, generator=g).half(), torch.randn(32, 64, generator=g).half()]
        out.append((X, Ws))
    return out


class FakeSearch:
    """Deterministic results from the inputs; remembers the layers searched;
    can fail after a number of calls (an interrupted run)."""

    def __init__(self, fail_after=None):
        self.seen = []
        self.calls = 0
        self.fail_after = fail_after

    def __call__(self, part, bits, group, n_grid, zero_point):
        if self.fail_after is not None and self.calls >= self.fail_after:
            raise RuntimeError("interrupted")
        self.calls += 1
        out = []
        for X, Ws in part:
            self.seen.append(int(X.shape[0]))
            key = float(X.float().sum()) + sum(float(W.float().sum()) for W in Ws)
            best = int(abs(key) * 1000) % n_grid
            out.append({"best": best, "alpha": best / n_grid,
                        "losses": np.linspace(1.0, 2.0, n_grid) + key,
                        "s": torch.full((X.shape[1],), key, dtype=torch.float32),
                        "codes": [torch.full((W.shape[0], 8), best, dtype=torch.int32) for W in Ws],
                        "scales": [torch.full((W.shape[0], 1), 0.5, dtype=torch.float16) for W in Ws],
                        "zeros": [torch.full((W.shape[0], 1), 7, dtype=torch.uint8) for W in Ws]})
        return out


def _same(a, b):
    assert a["best"] == b["best"] and a["alpha"] == b["alpha"]
    assert np.array_equal(np.asarray(a["losses"]), np.asarray(b["losses"]))
    assert np.array_equal(ck._to_numpy(a["s"]), ck._to_numpy(b["s"]))
    for key in ("codes", "scales", "zeros"):
        assert len(a[key]) == len(b[key])
        for x, y in zip(a[key], b[key]):
            assert np.array_equal(ck._to_numpy(x), ck._to_numpy(y))


def test_second_run_searches_nothing(tmp_path):
    calls = _layers(5)
    f1 = FakeSearch()
    r1 = ck.search_layers_resumable(calls, str(tmp_path), chunk=2, search=f1)
    assert sorted(f1.seen) == [8, 9, 10, 11, 12] and f1.calls == 3
    assert all(not r["resumed"] for r in r1)
    assert sorted(os.listdir(tmp_path)) == [f"layer_{i:05d}.npz" for i in range(5)]
    f2 = FakeSearch()
    r2 = ck.search_layers_resumable(calls, str(tmp_path), chunk=2, search=f2)
    assert f2.seen == [] and all(r["resumed"] for r in r2)
    for a, b in zip(r1, r2):
        _same(a, b)


def test_missing_stale_and_torn_files_are_searched_again(tmp_path):
    calls = _layers(4)
    ck.search_layers_resumable(calls, str(tmp_path), search=FakeSearch())
    os.remove(tmp_path / "layer_00001.npz")                          # missing
    with open(tmp_path / "layer_00003.npz", "wb") as f:              # torn
        f.write(b"PK\x03\x04 not a whole archive")
    changed = list(calls)
    X2 = changed[2][0].clone()
    X2[0, 0] += 1.0                                                  # stale (first bytes changed)
    changed[2] = (X2, changed[2][1])
    f = FakeSearch()
    r = ck.search_layers_resumable(changed, str(tmp_path), search=f)
    assert sorted(f.seen) == [9, 10, 11]
    assert [x["resumed"] for x in r] == [True, False, False, False]
    f3 = FakeSearch()
    ck.search_layers_resumable(changed, str(tmp_path), search=f3)
    assert f3.seen == []


def test_config_is_part_of_the_fingerprint(tmp_path):
    calls = _layers(2)
    ck.search_layers_resumable(calls, str(tmp_path), bits=4, search=FakeSearch())
    f = FakeSearch()
    ck.search_layers_resumable(calls, str(tmp_path), bits=3, search=f)
    assert sorted(f.seen) == [8, 9]
    f = FakeSearch()
    ck.search_layers_resumable(calls, str(tmp_path), bits=3, zero_point=False, search=f)
    assert sorted(f.seen) == [8, 9]


def test_interrupted_run_resumes_after_the_last_whole_chunk(tmp_path):
    calls = _layers(7)
    f = FakeSearch(fail_after=2)                   # chunks of 2: layers 0-3 stored, then stop
    with pytest.raises(RuntimeError, match="interrupted"):
        ck.search_layers_resumable(calls, str(tmp_path), chunk=2, search=f)
    assert sorted(f.seen) == [8, 9, 10, 11]
    assert not [p for p in os.listdir(tmp_path) if p.endswith(".tmp")]
    f2 = FakeSearch()
    r = ck.search_layers_resumable(calls, str(tmp_path), chunk=2, search=f2)
    assert sorted(f2.seen) == [12, 13, 14]
    assert [x["resumed"] for x in r] == [True] * 4 + [False] * 3
    fresh = ck.search_layers_resumable(calls, str(tmp_path / "fresh"), chunk=3,
                                       search=FakeSearch())
    for a, b in zip(r, fresh):
        _same(a, b)


def test_bad_chunk_and_short_search_are_errors(tmp_path):
    with pytest.raises(ValueError):
        ck.search_layers_resumable(_layers(1), str(tmp_path), chunk=0, search=FakeSearch())
    with pytest.raises(RuntimeError):
        ck.search_layers_resumable(_layers(2), str(tmp_path / "b"),
                                   search=lambda part, **kw: [])
