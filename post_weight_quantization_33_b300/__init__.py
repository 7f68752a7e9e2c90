"""AWQ activation-aware scale search on one B300 (sm_103a).

A thin ctypes binding over ``libawq.so`` (declared in ``include/awq.h``).  It
only marshals arguments: every step of the search runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no
CPU fallback: if the library is missing or the device cannot run it, calls
raise.

Functions mirror the C entry points:

``stats(X)``                      sX = mean_t |X[t, k]|                (awq_stats)
``scales(sX, n_grid)``            s for every grid point               (awq_scales)
``quantize_pack(W, s, bits, g)``  packed codes, fp16 scales, u8 zeros  (awq_quantize_pack)
``unpack_codes(codes, N, K, b)``  codes as uint8 [N, K]                (awq_unpack_codes)
``reference_output(W, X)``        Y = W X^T in fp32                    (awq_reference_output)
``fold_scale(V, s)``              V / s along rows (deploy step)       (awq_fold_scale)
``w4a16_matvec(codes, sc, z, x)`` y = deq(Q) x for 1..8 tokens         (awq_w4a16_matvec)
``search(X, Ws, ...)``            the full per-layer search            (awq_search_layer)
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = [
    "AwqError", "lib", "library_path", "groups_per_row", "stats", "stats_noalloc", "scales", "quantize_pack", "unpack_codes",
    "reference_output", "fold_scale", "w4a16_matvec", "search", "search_host", "SearchResult", "packed_words",
    "release_cached_memory", "selftest_bounded_wait", "set_stage_timing", "STAGES",
    "EXPORTED_SYMBOLS", "search_host_stream", "HostLayer", "inject_allocation_failures",
    "pool_usage", "MAX_STAT_TOKENS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libawq.so")
_lib = None

AWQ_OK, AWQ_ERR_INVALID, AWQ_ERR_UNSUPPORTED, AWQ_ERR_CUDA, AWQ_ERR_OOM, AWQ_ERR_TIMEOUT = range(6)
MAX_STAT_TOKENS = 1 << 22     # AWQ_MAX_STAT_TOKENS

# Every symbol include/awq.h declares.
EXPORTED_SYMBOLS = (
    "awq_abi_version", "awq_last_error", "awq_status_string", "awq_packed_words",
    "awq_stats", "awq_scales", "awq_quantize_pack", "awq_unpack_codes",
    "awq_reference_output", "awq_search_layer", "awq_result_check", "awq_result_n_grid",
    "awq_result_n_weights", "awq_result_best_index", "awq_result_alpha", "awq_result_losses",
    "awq_result_s", "awq_result_s_grid", "awq_result_row_losses", "awq_result_codes",
    "awq_result_scales", "awq_result_zeros", "awq_free", "awq_release_cached_memory",
    "awq_selftest_bounded_wait", "awq_result_kernel_launches", "awq_set_stage_timing",
    "awq_result_stage_ms", "awq_stats_noalloc", "awq_fold_scale", "awq_w4a16_matvec",
    "awq_search_layer_gram", "awq_search_host_layers", "awq_inject_allocation_failures",
    "awq_pool_usage", "awq_bounds_checked", "awq_bounds_report", "awq_bounds_selftest",
)

# Stage ids of awq_result_stage_ms (AWQ_STAGE_* in include/awq.h).
STAGES = ("stats", "scales", "residual", "error_gemm", "loss", "final")


class AwqError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(message)


class QConfig(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int), ("group_size", ctypes.c_int),
                ("zero_point", ctypes.c_int), ("n_grid", ctypes.c_int)]


class Weight(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("N", ctypes.c_int64)]


class HostLayer(ctypes.Structure):
    """awq_host_layer: one layer of awq_search_host_layers (host memory)."""
    _fields_ = [("X", ctypes.c_void_p), ("T", ctypes.c_int64), ("K", ctypes.c_int64),
                ("Ws", ctypes.POINTER(Weight)), ("n_w", ctypes.c_int),
                ("codes", ctypes.POINTER(ctypes.c_void_p)),
                ("scales", ctypes.POINTER(ctypes.c_void_p)),
                ("zeros", ctypes.POINTER(ctypes.c_void_p)),
                ("s", ctypes.c_void_p), ("losses", ctypes.c_void_p), ("best", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libawq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -m post_weight_quantization_33_b300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int
    sig = {
        "awq_abi_version": (i32, []),
        "awq_last_error": (ctypes.c_char_p, []),
        "awq_status_string": (ctypes.c_char_p, [i32]),
        "awq_packed_words": (i64, [i64, i64, i32]),
        "awq_stats": (st, [vp, i64, i64, vp, vp]),
        "awq_stats_noalloc": (st, [vp, i64, i64, vp, vp]),
        "awq_scales": (st, [vp, i64, i32, vp, vp]),
        "awq_quantize_pack": (st, [vp, i64, i64, vp, ctypes.POINTER(QConfig), vp, vp, vp, vp]),
        "awq_unpack_codes": (st, [vp, i64, i64, i32, vp, vp]),
        "awq_reference_output": (st, [vp, i64, vp, i64, i64, vp, vp, vp]),
        "awq_fold_scale": (st, [vp, i64, i64, vp, vp, vp]),
        "awq_w4a16_matvec": (st, [vp, vp, vp, i64, i64, ctypes.POINTER(QConfig), vp, i32, vp,
                                  vp]),
        "awq_search_layer": (st, [vp, i64, i64, vp, ctypes.POINTER(Weight), i32,
                                  ctypes.POINTER(QConfig), vp, ctypes.POINTER(vp)]),
        "awq_search_layer_gram": (st, [vp, i64, i64, vp, ctypes.POINTER(Weight), i32,
                                       ctypes.POINTER(QConfig), vp, ctypes.POINTER(vp)]),
        "awq_result_check": (st, [vp]),
        "awq_result_n_grid": (i32, [vp]),
        "awq_result_n_weights": (i32, [vp]),
        "awq_result_best_index": (i32, [vp]),
        "awq_result_alpha": (ctypes.c_double, [vp]),
        "awq_result_losses": (ctypes.POINTER(ctypes.c_double), [vp]),
        "awq_result_s": (vp, [vp]),
        "awq_result_s_grid": (vp, [vp]),
        "awq_result_row_losses": (vp, [vp]),
        "awq_result_codes": (vp, [vp, i32]),
        "awq_result_scales": (vp, [vp, i32]),
        "awq_result_zeros": (vp, [vp, i32]),
        "awq_free": (None, [vp]),
        "awq_release_cached_memory": (st, []),
        "awq_selftest_bounded_wait": (st, [i64]),
        "awq_result_kernel_launches": (i32, [vp]),
        "awq_set_stage_timing": (None, [i32]),
        "awq_result_stage_ms": (st, [vp, i32, ctypes.POINTER(ctypes.c_float)]),
        "awq_search_host_layers": (st, [ctypes.POINTER(HostLayer), i32, ctypes.POINTER(QConfig),
                                        vp]),
        "awq_inject_allocation_failures": (None, [i32, i32]),
        "awq_pool_usage": (st, [ctypes.POINTER(i64), ctypes.POINTER(i64)]),
        "awq_bounds_checked": (i32, []),
        "awq_bounds_selftest": (st, []),
        "awq_bounds_report": (st, [ctypes.POINTER(i64), ctypes.POINTER(i32), ctypes.POINTER(i64),
                                   ctypes.POINTER(i64), i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int) -> None:
    if status != AWQ_OK:
        L = lib()
        name = L.awq_status_string(status).decode()
        msg = L.awq_last_error().decode()
        raise AwqError(status, f"{name}: {msg}")


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _require(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cfg(bits: int, group: int, n_grid: int = 20, zero_point: bool = True) -> QConfig:
    return QConfig(bits, group, 1 if zero_point else 0, n_grid)


def groups_per_row(K: int, group: int) -> int:
    """Quantization groups in a row of K channels (group -1: the whole row)."""
    return 1 if group == -1 else K // group


def packed_words(N: int, K: int, bits: int) -> int:
    """uint32 words of N packed rows (-1 for an invalid shape)."""
    return int(lib().awq_packed_words(N, K, bits))


def stats(X: torch.Tensor) -> torch.Tensor:
    """sX [K] fp64 = mean over tokens of |X| (X: fp16 [T, K] on the GPU)."""
    _require(X, "X", torch.float16, 2)
    T, K = X.shape
    sX = torch.empty(K, dtype=torch.float64, device=X.device)
    _check(lib().awq_stats(X.data_ptr(), T, K, sX.data_ptr(), _stream()))
    return sX


def stats_noalloc(X: torch.Tensor) -> torch.Tensor:
    """As stats(), through awq_stats_noalloc: the library allocates no device
    memory (its accumulator is a fixed array inside the library; K <= 65536).
    Calls must not overlap on the GPU."""
    _require(X, "X", torch.float16, 2)
    T, K = X.shape
    sX = torch.empty(K, dtype=torch.float64, device=X.device)
    _check(lib().awq_stats_noalloc(X.data_ptr(), T, K, sX.data_ptr(), _stream()))
    return sX


def scales(sX: torch.Tensor, n_grid: int = 20) -> torch.Tensor:
    """s [n_grid, K] fp32, row i at alpha = i / n_grid."""
    _require(sX, "sX", torch.float64, 1)
    K = sX.shape[0]
    s = torch.empty((n_grid, K), dtype=torch.float32, device=sX.device)
    _check(lib().awq_scales(sX.data_ptr(), K, n_grid, s.data_ptr(), _stream()))
    return s


def quantize_pack(W: torch.Tensor, s: torch.Tensor, bits: int = 4, group: int = 128,
                  zero_point: bool = True):
    """(codes int32 [words] holding the uint32 bit patterns, scales fp16 [N, K/g], zeros u8)."""
    _require(W, "W", torch.float16, 2)
    _require(s, "s", torch.float32, 1)
    N, K = W.shape
    words = packed_words(N, K, bits)
    if words < 0:
        raise ValueError(f"cannot pack K={K} at {bits} bits")
    codes = torch.empty(max(words, 1), dtype=torch.int32, device=W.device)[:words]
    G = groups_per_row(K, group)
    sc = torch.empty((N, G), dtype=torch.float16, device=W.device)
    z = torch.empty((N, G), dtype=torch.uint8, device=W.device)
    cfg = _cfg(bits, group, 20, zero_point)
    _check(lib().awq_quantize_pack(W.data_ptr(), N, K, s.data_ptr(), ctypes.byref(cfg),
                                   codes.data_ptr(), sc.data_ptr(), z.data_ptr(), _stream()))
    return codes, sc, z


def unpack_codes(codes: torch.Tensor, N: int, K: int, bits: int) -> torch.Tensor:
    """uint8 [N, K] codes from the packed words."""
    _require(codes, "codes", torch.int32, 1)
    q = torch.empty((N, K), dtype=torch.uint8, device=codes.device)
    _check(lib().awq_unpack_codes(codes.data_ptr(), N, K, bits, q.data_ptr(), _stream()))
    return q


def reference_output(W: torch.Tensor, X: torch.Tensor, check: bool = True) -> torch.Tensor:
    """Y = W X^T in fp32 [N, T] on the tensor cores."""
    _require(W, "W", torch.float16, 2)
    _require(X, "X", torch.float16, 2)
    N, K = W.shape
    T = X.shape[0]
    Y = torch.empty((N, T), dtype=torch.float32, device=W.device)
    status = torch.zeros(1, dtype=torch.int32, device=W.device)
    _check(lib().awq_reference_output(W.data_ptr(), N, X.data_ptr(), T, K, Y.data_ptr(),
                                      status.data_ptr(), _stream()))
    if check and int(status.item()) != 0:
        raise AwqError(AWQ_ERR_TIMEOUT, f"bounded device wait expired (code {int(status.item())})")
    return Y


def fold_scale(V: torch.Tensor, s: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fp16 V / s along the first axis (a norm weight or bias [K], or a
    preceding linear layer's weight [K, M]); `out` may be V (in place)."""
    if V.dtype != torch.float16 or V.dim() not in (1, 2) or not V.is_cuda or not V.is_contiguous():
        raise ValueError("V must be a contiguous CUDA fp16 tensor [K] or [K, M]")
    _require(s, "s", torch.float32, 1)
    rows = V.shape[0]
    cols = 1 if V.dim() == 1 else V.shape[1]
    if out is None:
        out = torch.empty_like(V)
    elif out.shape != V.shape or out.dtype != torch.float16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp16 tensor shaped like V")
    _check(lib().awq_fold_scale(V.data_ptr(), rows, cols, s.data_ptr(), out.data_ptr(), _stream()))
    return out


def w4a16_matvec(codes: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, N: int, K: int,
                 x: torch.Tensor, group: int = 128, bits: int = 4) -> torch.Tensor:
    """y [M, N] fp32 = deq(codes) x^T for x fp16 [M, K], 1 <= M <= 16, INT4 or
    INT3 packed codes (awq_w4a16_matvec)."""
    _require(codes, "codes", torch.int32, 1)
    _require(x, "x", torch.float16, 2)
    if x.shape[1] != K:
        raise ValueError(f"x has K={x.shape[1]}, expected {K}")
    M = x.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    cfg = _cfg(bits, group)
    _check(lib().awq_w4a16_matvec(codes.data_ptr(), scales.data_ptr(), zeros.data_ptr(), N, K,
                                  ctypes.byref(cfg), x.data_ptr(), M, y.data_ptr(), _stream()))
    return y


class _DevArray:
    """__cuda_array_interface__ over library-owned device memory (no copy)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (int(ptr), False), "version": 2, "strides": None}


def _alias(ptr: int, shape, typestr: str, device) -> torch.Tensor:
    if int(np.prod(shape)) == 0:
        dt = {"<f4": torch.float32, "<f8": torch.float64, "<f2": torch.float16,
              "<i4": torch.int32, "|u1": torch.uint8}[typestr]
        return torch.empty(shape, dtype=dt, device=device)
    with torch.cuda.device(device):
        return torch.as_tensor(_DevArray(ptr, shape, typestr), device=device)


class SearchResult:
    """Owns one awq_result.  Host values need the stream synchronised (the
    accessors below do it); tensors returned are copies owned by torch."""

    def __init__(self, handle: int, Ns: Sequence[int], K: int, T: int, bits: int, group: int,
                 n_grid: int, device):
        self._h = ctypes.c_void_p(handle)
        self.Ns = list(Ns)
        self.K, self.T, self.bits, self.group, self.n_grid = K, T, bits, group, n_grid
        self.device = device

    def _handle(self):
        if not self._h:
            raise RuntimeError("result already freed")
        return self._h

    def synchronize(self) -> "SearchResult":
        torch.cuda.current_stream(self.device).synchronize()
        return self

    def check(self) -> None:
        self.synchronize()
        _check(lib().awq_result_check(self._handle()))

    @property
    def best(self) -> int:
        self.synchronize()
        return int(lib().awq_result_best_index(self._handle()))

    @property
    def alpha(self) -> float:
        self.synchronize()
        return float(lib().awq_result_alpha(self._handle()))

    @property
    def losses(self) -> np.ndarray:
        self.synchronize()
        p = lib().awq_result_losses(self._handle())
        return np.array([p[i] for i in range(self.n_grid)], dtype=np.float64)

    def s(self) -> torch.Tensor:
        return _alias(lib().awq_result_s(self._handle()), (self.K,), "<f4", self.device).clone()

    def s_grid(self) -> torch.Tensor:
        return _alias(lib().awq_result_s_grid(self._handle()), (self.n_grid, self.K), "<f4",
                      self.device).clone()

    def row_losses(self) -> torch.Tensor:
        return _alias(lib().awq_result_row_losses(self._handle()), (self.n_grid, sum(self.Ns)),
                      "<f8", self.device).clone()

    def codes(self, i: int = 0) -> torch.Tensor:
        words = packed_words(self.Ns[i], self.K, self.bits)
        return _alias(lib().awq_result_codes(self._handle(), i), (words,), "<i4",
                      self.device).clone()

    def scales(self, i: int = 0) -> torch.Tensor:
        return _alias(lib().awq_result_scales(self._handle(), i),
                      (self.Ns[i], groups_per_row(self.K, self.group)), "<f2",
                      self.device).clone()

    def zeros(self, i: int = 0) -> torch.Tensor:
        return _alias(lib().awq_result_zeros(self._handle(), i),
                      (self.Ns[i], groups_per_row(self.K, self.group)), "|u1",
                      self.device).clone()

    def host_values(self) -> dict:
        """best, alpha, losses and the status check, without synchronising
        the stream: valid once the search's work has completed (the caller
        waits on an event recorded after it)."""
        h = self._handle()
        _check(lib().awq_result_check(h))
        p = lib().awq_result_losses(h)
        return {"best": int(lib().awq_result_best_index(h)),
                "alpha": float(lib().awq_result_alpha(h)),
                "losses": np.array([p[i] for i in range(self.n_grid)], dtype=np.float64)}

    def device_views(self) -> dict:
        """Library-owned device tensors (no copy) of s and of each weight's
        codes, scales and zeros; valid until free()."""
        h = self._handle()
        gpr = groups_per_row(self.K, self.group)
        return {
            "s": _alias(lib().awq_result_s(h), (self.K,), "<f4", self.device),
            "codes": [_alias(lib().awq_result_codes(h, i), (packed_words(n, self.K, self.bits),),
                             "<i4", self.device) for i, n in enumerate(self.Ns)],
            "scales": [_alias(lib().awq_result_scales(h, i), (n, gpr), "<f2", self.device)
                       for i, n in enumerate(self.Ns)],
            "zeros": [_alias(lib().awq_result_zeros(h, i), (n, gpr), "|u1", self.device)
                      for i, n in enumerate(self.Ns)],
        }

    @property
    def kernel_launches(self) -> int:
        return int(lib().awq_result_kernel_launches(self._handle()))

    def stage_ms(self) -> dict:
        """GPU milliseconds per stage (needs set_stage_timing(True) before the search)."""
        self.synchronize()
        out = {}
        for i, name in enumerate(STAGES):
            v = ctypes.c_float()
            _check(lib().awq_result_stage_ms(self._handle(), i, ctypes.byref(v)))
            out[name] = float(v.value)
        return out

    def free(self) -> None:
        if self._h:
            lib().awq_free(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def search(X: torch.Tensor, Ws: Sequence[torch.Tensor], bits: int = 4, group: int = 128,
           n_grid: int = 20, sX: Optional[torch.Tensor] = None,
           zero_point: bool = True, gram: bool = False) -> SearchResult:
    """Run awq_search_layer for the weights ``Ws`` sharing activations ``X``
    (group -1: one group per output row; zero_point False: symmetric;
    gram True: awq_search_layer_gram, the loss as d^T (X^T X) d)."""
    _require(X, "X", torch.float16, 2)
    T, K = X.shape
    arr = (Weight * len(Ws))()
    for i, W in enumerate(Ws):
        _require(W, f"Ws[{i}]", torch.float16, 2)
        if W.shape[1] != K:
            raise ValueError(f"Ws[{i}] has K={W.shape[1]}, X has K={K}")
        arr[i].W = W.data_ptr()
        arr[i].N = W.shape[0]
    sxp = None
    if sX is not None:
        _require(sX, "sX", torch.float64, 1)
        sxp = sX.data_ptr()
    cfg = _cfg(bits, group, n_grid, zero_point)
    out = ctypes.c_void_p()
    entry = lib().awq_search_layer_gram if gram else lib().awq_search_layer
    _check(entry(X.data_ptr(), T, K, sxp, arr, len(Ws), ctypes.byref(cfg), _stream(),
                 ctypes.byref(out)))
    return SearchResult(out.value, [W.shape[0] for W in Ws], K, T, bits, group, n_grid, X.device)


def search_host(X: torch.Tensor, Ws: Sequence[torch.Tensor], bits: int = 4, group: int = 128,
                n_grid: int = 20, device="cuda", zero_point: bool = True) -> dict:
    """Search with host (CPU, ideally pinned) inputs; returns host outputs.

    Copies X and the weights to the device, runs ``search`` and copies the
    results back (codes, scales, zeros per weight, s, losses, alpha)."""
    Xd = X.to(device, non_blocking=True)
    Wd = [W.to(device, non_blocking=True) for W in Ws]
    r = search(Xd, Wd, bits, group, n_grid, zero_point=zero_point)
    try:
        out = {
            "codes": [r.codes(i).to("cpu", non_blocking=True) for i in range(len(Ws))],
            "scales": [r.scales(i).to("cpu", non_blocking=True) for i in range(len(Ws))],
            "zeros": [r.zeros(i).to("cpu", non_blocking=True) for i in range(len(Ws))],
            "s": r.s().to("cpu", non_blocking=True),
        }
        r.check()
        out["losses"] = r.losses
        out["best"] = r.best
        out["alpha"] = r.alpha
    finally:
        r.free()
    return out


def search_host_stream(calls: Sequence[Tuple[torch.Tensor, Sequence[torch.Tensor]]],
                       bits: int = 4, group: int = 128, n_grid: int = 20, device="cuda",
                       zero_point: bool = True) -> List[dict]:
    """awq_search_host_layers over a sequence of layers ``(X, [W, ...])`` in
    host memory (pinned for overlapped copies): the library searches layer i
    on the current stream of ``device`` while its own streams copy layer i+1's
    inputs in and layer i-1's results out.  Returns one dict per layer, as
    search_host does, with the outputs in pinned host tensors."""
    calls = [(X, list(Ws)) for X, Ws in calls]
    if not calls:
        return []
    for i, (X, Ws) in enumerate(calls):
        if not isinstance(X, torch.Tensor) or X.is_cuda or X.dim() != 2:
            raise ValueError(f"calls[{i}]: X must be a 2-D host tensor")
        if not Ws or any(not isinstance(W, torch.Tensor) or W.is_cuda or W.dim() != 2
                         or W.shape[1] != X.shape[1] for W in Ws):
            raise ValueError(f"calls[{i}]: weights must be 2-D host tensors with K = {X.shape[1]}")
        for t in (X, *Ws):
            if t.dtype != torch.float16 or not t.is_contiguous():
                raise TypeError(f"calls[{i}]: inputs must be contiguous float16")
    device = torch.device(device)
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    keep = []                    # ctypes arrays referenced by the layer structs
    layers = (HostLayer * len(calls))()
    out: List[dict] = []
    for i, (X, Ws) in enumerate(calls):
        T, K = X.shape
        gpr = groups_per_row(K, group)
        o = {"codes": [torch.empty(packed_words(W.shape[0], K, bits), dtype=torch.int32,
                                   pin_memory=True) for W in Ws],
             "scales": [torch.empty((W.shape[0], gpr), dtype=torch.float16, pin_memory=True)
                        for W in Ws],
             "zeros": [torch.empty((W.shape[0], gpr), dtype=torch.uint8, pin_memory=True)
                       for W in Ws],
             "s": torch.empty(K, dtype=torch.float32, pin_memory=True),
             "losses": np.zeros(n_grid, dtype=np.float64),
             "best": np.zeros(1, dtype=np.int32)}
        warr = (Weight * len(Ws))()
        for j, W in enumerate(Ws):
            warr[j].W = W.data_ptr()
            warr[j].N = W.shape[0]
        ptrs = [(ctypes.c_void_p * len(Ws))(*[t.data_ptr() for t in o[key]])
                for key in ("codes", "scales", "zeros")]
        keep += [warr, *ptrs]
        L = layers[i]
        L.X, L.T, L.K = X.data_ptr(), T, K
        L.Ws, L.n_w = warr, len(Ws)
        L.codes, L.scales, L.zeros = ptrs
        L.s = o["s"].data_ptr()
        L.losses = o["losses"].ctypes.data
        L.best = o["best"].ctypes.data
        out.append(o)
    cfg = _cfg(bits, group, n_grid, zero_point)
    with torch.cuda.device(device):
        _check(lib().awq_search_host_layers(layers, len(calls), ctypes.byref(cfg), _stream()))
    for o in out:
        o["best"] = int(o["best"][0])
        o["alpha"] = o["best"] / n_grid
    return out


def inject_allocation_failures(skip: int, count: int) -> None:
    """After ``skip`` pool allocations, make the next ``count`` fail as out of
    memory (awq_inject_allocation_failures; count 0 disarms)."""
    lib().awq_inject_allocation_failures(int(skip), int(count))


def pool_usage() -> Tuple[int, int]:
    """(used, reserved) bytes of the library pool on the current device."""
    used, reserved = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().awq_pool_usage(ctypes.byref(used), ctypes.byref(reserved)))
    return int(used.value), int(reserved.value)


def set_stage_timing(enable: bool) -> None:
    """Record CUDA events at stage boundaries of later searches (see stage_ms)."""
    lib().awq_set_stage_timing(1 if enable else 0)


def release_cached_memory() -> None:
    _check(lib().awq_release_cached_memory())


def bounds_report(reset: bool = True) -> dict:
    """Out-of-range accesses recorded by the bounds-checked build
    (libawq_checked.so) since the last reset: ``count``, and the first one's
    ``site``, ``index`` and ``extent``; ``checked`` is False (and the count 0)
    for libawq.so."""
    c, site, idx, ext = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().awq_bounds_report(ctypes.byref(c), ctypes.byref(site), ctypes.byref(idx),
                                   ctypes.byref(ext), int(reset)))
    return {"checked": bool(lib().awq_bounds_checked()), "count": c.value, "site": site.value,
            "index": idx.value, "extent": ext.value}


def selftest_bounded_wait(limit_ns: int = 20_000_000) -> int:
    """Run the bounded-wait self-test; returns the status (AWQ_ERR_TIMEOUT expected)."""
    return int(lib().awq_selftest_bounded_wait(limit_ns))
