"""Checkpoint / resume for multi-layer scale searches.

A model's layers are searched independently ("AWQ explained", hungho77.github.io,
"Scaling instead of mixed precision": one activation statistic and one scale
vector per linear layer), so a long run over many layers can keep each finished
layer's results on disk and, when it is restarted, search only the layers that
have none.  ``search_layers_resumable`` does that around ``search_host_stream``
(the library's pipelined host-buffer search): layers are searched in chunks,
and after each chunk every layer's result is written to ``checkpoint_dir`` as
``layer_<index>.npz`` (written to a temporary name and renamed, so a file is
either complete or absent).

A checkpoint is used only if its fingerprint matches the layer: the shapes of
X and of every W, the quantizer configuration, and a SHA-256 over sampled
bytes of every input (the first, middle and last 64 KiB of each tensor; a
change elsewhere in a tensor goes unnoticed, so a run over changed inputs
should use a fresh directory).  A mismatching checkpoint is searched again and
overwritten.  The results returned for a resumed layer are the stored arrays,
bit-identical to the ones the search wrote.
"""
from __future__ import annotations

import hashlib
import json
import os
import zipfile
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

_SAMPLE = 64 * 1024
_KEYS_PER_W = ("codes", "scales", "zeros")


def _tensor_bytes(t) -> np.ndarray:
    """Flat uint8 view of a contiguous host tensor (torch or numpy)."""
    a = t.numpy() if hasattr(t, "numpy") else np.asarray(t)
    return np.ascontiguousarray(a).view(np.uint8).reshape(-1)


def layer_fingerprint(X, Ws: Sequence, bits: int, group: int, n_grid: int,
                      zero_point: bool) -> str:
    """SHA-256 over the layer's shapes, the quantizer configuration and the
    first, middle and last 64 KiB of every input tensor."""
    h = hashlib.sha256()
    h.update(json.dumps({"X": list(X.shape), "W": [list(W.shape) for W in Ws], "bits": bits,
                         "group": group, "n_grid": n_grid, "zero_point": bool(zero_point)},
                        sort_keys=True).encode())
    for t in (X, *Ws):
        b = _tensor_bytes(t)
        n = b.size
        for start in (0, max(0, n // 2 - _SAMPLE // 2), max(0, n - _SAMPLE)):
            h.update(b[start:start + _SAMPLE].tobytes())
    return h.hexdigest()


def _path(checkpoint_dir: str, i: int) -> str:
    return os.path.join(checkpoint_dir, f"layer_{i:05d}.npz")


def _to_numpy(v):
    return v.numpy() if hasattr(v, "numpy") else np.asarray(v)


def save_layer(checkpoint_dir: str, i: int, fingerprint: str, result: dict) -> None:
    """Write one layer's result atomically (temporary file, then rename)."""
    arrays = {"fingerprint": np.frombuffer(fingerprint.encode(), dtype=np.uint8),
              "best": np.array([result["best"]], dtype=np.int64),
              "alpha": np.array([result["alpha"]], dtype=np.float64),
              "losses": _to_numpy(result["losses"]).astype(np.float64),
              "s": _to_numpy(result["s"]),
              "n_w": np.array([len(result["codes"])], dtype=np.int64)}
    for key in _KEYS_PER_W:
        for j, t in enumerate(result[key]):
            arrays[f"{key}_{j}"] = _to_numpy(t)
    final = _path(checkpoint_dir, i)
    tmp = final + ".tmp"
    with open(tmp, "wb") as f:
        np.savez(f, **arrays)
        f.flush()
        os.fsync(f.fileno())
    os.replace(tmp, final)


def load_layer(checkpoint_dir: str, i: int, fingerprint: str) -> Optional[dict]:
    """The stored result of layer i, or None if there is none or it belongs
    to other inputs (fingerprint mismatch) or cannot be read."""
    p = _path(checkpoint_dir, i)
    if not os.path.exists(p):
        return None
    try:
        with np.load(p) as z:
            if z["fingerprint"].tobytes().decode() != fingerprint:
                return None
            n_w = int(z["n_w"][0])
            out = {"best": int(z["best"][0]), "alpha": float(z["alpha"][0]),
                   "losses": z["losses"].copy(), "s": z["s"].copy()}
            for key in _KEYS_PER_W:
                out[key] = [z[f"{key}_{j}"].copy() for j in range(n_w)]
            return out
    except (OSError, KeyError, ValueError, EOFError, zipfile.BadZipFile):
        return None


def search_layers_resumable(calls: Sequence[Tuple[object, Sequence[object]]],
                            checkpoint_dir: str, bits: int = 4, group: int = 128,
                            n_grid: int = 20, zero_point: bool = True, chunk: int = 4,
                            search: Optional[Callable[..., List[dict]]] = None,
                            device="cuda") -> List[dict]:
    """Search every layer ``(X, [W, ...])`` (host tensors, as
    ``search_host_stream`` takes them), reusing the results stored in
    ``checkpoint_dir`` and storing each new one as soon as its chunk of
    ``chunk`` layers is done.  Returns one dict per layer (``best``,
    ``alpha``, ``losses``, ``s``, ``codes``, ``scales``, ``zeros``), in layer
    order; a dict also has ``resumed`` = True when it came from disk.
    ``search`` replaces ``search_host_stream`` (tests use a stand-in)."""
    if chunk < 1:
        raise ValueError("chunk must be >= 1")
    if search is None:
        from . import search_host_stream

        def search(part, **kw):
            return search_host_stream(part, device=device, **kw)
    os.makedirs(checkpoint_dir, exist_ok=True)
    cfg = dict(bits=bits, group=group, n_grid=n_grid, zero_point=zero_point)
    prints = [layer_fingerprint(X, list(Ws), **cfg) for X, Ws in calls]
    results: List[Optional[dict]] = []
    todo: List[int] = []
    for i, fp in enumerate(prints):
        r = load_layer(checkpoint_dir, i, fp)
        if r is not None:
            r["resumed"] = True
        else:
            todo.append(i)
        results.append(r)
    for c in range(0, len(todo), chunk):
        idx = todo[c:c + chunk]
        part = search([calls[i] for i in idx], **cfg)
        if len(part) != len(idx):
            raise RuntimeError(f"search returned {len(part)} results for {len(idx)} layers")
        for i, r in zip(idx, part):
            save_layer(checkpoint_dir, i, prints[i], r)
            r = dict(r)
            r["resumed"] = False
            results[i] = r
    return results  # type: ignore[return-value]
