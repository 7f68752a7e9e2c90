"""Seeded synthetic inputs for the AWQ scale search.

This module only draws random numbers and shapes them into fp16 arrays.  It
holds none of the method's arithmetic: no statistic, scale, quantizer or loss
lives here.  Both the CPU oracle (``oracle/``) and the CUDA path consume the
same bytes produced here, so parity tests compare like with like.

The five workloads mirror the layer shapes the AWQ pages motivate (LLaMA-class
linear layers; "AWQ explained", multigrid.ai, section "The premise: 1% of
channels", on the ~1 % of salient channels) and are described in words:

``tiny``
    W 256x512 ~ N(0, 0.02^2); X 64x512 ~ N(0, 1) with channels
    {3, 64, 130, 257, 511} multiplied by 20 (3 and 64 share the first group
    of 128, so two salient channels meet inside one group); INT4, group 128.
``llama7b_attn``
    W 4096x4096 ~ N(0, 0.02^2); X 4096x4096 ~ N(0, 1) with 1 % of the
    channels (41) multiplied by a log-uniform factor 10^(1+U[0,1)); INT4, g128.
``llama7b_mlp``
    call A: up and gate W 11008x4096 ~ N(0, 0.02^2) sharing one X 4096x4096
    drawn as in ``llama7b_attn``; call B: down W 4096x11008 ~ N(0, 0.02^2)
    with X 4096x11008 = |N(0,1)| * Laplace(0,1) elementwise (heavy tail);
    INT4, g128.
``llama70b``
    W 8192x8192 and 28672x8192 ~ N(0, 0.015^2), one X 8192x8192 ~ N(0, 1)
    with 0.5 % of the channels (41) multiplied by 50; two calls; INT4, g128.
``int3_stress``
    W 4096x4096 and 11008x4096 = 0.02 * Student-t(nu=4); X 16384x4096 ~
    N(0, 1) with 1 % of the channels (41) multiplied by 30; each W searched at
    group 64 and group 128; INT3 (codes 0..7).

Seeds: workload i draws from ``numpy.random.Generator(PCG64(SeedSequence(
20250 + i)))`` spawned into one child stream per tensor, in the order the
tensors are listed.  Draws happen in fp64 and are rounded to fp16 with
round-to-nearest-even (``astype(float16)``).  Large tensors are drawn in fixed
row chunks so memory stays bounded; the chunking is part of the recipe.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Sequence, Tuple

import numpy as np

SEED_BASE = 20250
_CHUNK_ROWS = 2048


@dataclass(frozen=True)
class TensorSpec:
    """How one tensor is drawn.

    kind: "normal" (sigma * N(0,1)), "student_t" (sigma * t(nu)),
          "act_outliers" (N(0,1) with selected columns multiplied),
          "abs_normal_laplace" (|N(0,1)| * Laplace(0,1)).
    """
    name: str
    rows: int
    cols: int
    kind: str
    sigma: float = 1.0
    nu: float = 4.0
    outlier_channels: Tuple[int, ...] = ()   # fixed channel list, or empty
    outlier_fraction: float = 0.0            # seeded pick when no fixed list
    outlier_factor: float = 1.0              # fixed factor ...
    outlier_log_uniform: Tuple[float, float] = ()  # ... or 10^(a + (b-a) U)


@dataclass(frozen=True)
class Call:
    """One search call: the weights in ``ws`` share the activations ``x``."""
    x: str
    ws: Tuple[str, ...]
    bits: int
    group: int


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    tensors: Tuple[TensorSpec, ...]
    calls: Tuple[Call, ...]
    description: str = ""

    def spec(self, name: str) -> TensorSpec:
        for t in self.tensors:
            if t.name == name:
                return t
        raise KeyError(name)

    def weights_searched(self) -> int:
        """Sum over calls of N*K for every weight searched (the metric's unit)."""
        total = 0
        for c in self.calls:
            for w in c.ws:
                s = self.spec(w)
                total += s.rows * s.cols
        return total

    def gemm_flops(self, n_grid: int = 20) -> int:
        """Algorithmic error-GEMM flops of the whole workload: n_grid * sum 2*N*K*T."""
        total = 0
        for c in self.calls:
            t = self.spec(c.x).rows
            for w in c.ws:
                s = self.spec(w)
                total += 2 * s.rows * s.cols * t
        return n_grid * total


def _n_outliers(frac: float, k: int) -> int:
    return int(round(frac * k))


WORKLOADS: Dict[str, Workload] = {}


def _register(w: Workload) -> None:
    WORKLOADS[w.name] = w


_register(Workload(
    name="tiny", index=0,
    tensors=(
        TensorSpec("W", 256, 512, "normal", sigma=0.02),
        TensorSpec("X", 64, 512, "act_outliers",
                   outlier_channels=(3, 64, 130, 257, 511), outlier_factor=20.0),
    ),
    calls=(Call("X", ("W",), 4, 128),),
    description="W 256x512 N(0,0.02); X 64x512 N(0,1), 5 fixed channels x20; INT4 g128",
))

_register(Workload(
    name="llama7b_attn", index=1,
    tensors=(
        TensorSpec("W", 4096, 4096, "normal", sigma=0.02),
        TensorSpec("X", 4096, 4096, "act_outliers", outlier_fraction=0.01,
                   outlier_log_uniform=(1.0, 2.0)),
    ),
    calls=(Call("X", ("W",), 4, 128),),
    description="W 4096x4096 N(0,0.02); X 4096x4096 N(0,1), 1% channels x 10^(1+U); INT4 g128",
))

_register(Workload(
    name="llama7b_mlp", index=2,
    tensors=(
        TensorSpec("W_up", 11008, 4096, "normal", sigma=0.02),
        TensorSpec("W_gate", 11008, 4096, "normal", sigma=0.02),
        TensorSpec("X_in", 4096, 4096, "act_outliers", outlier_fraction=0.01,
                   outlier_log_uniform=(1.0, 2.0)),
        TensorSpec("W_down", 4096, 11008, "normal", sigma=0.02),
        TensorSpec("X_mid", 4096, 11008, "abs_normal_laplace"),
    ),
    calls=(Call("X_in", ("W_up", "W_gate"), 4, 128),
           Call("X_mid", ("W_down",), 4, 128)),
    description="up/gate 11008x4096 sharing X 4096x4096; down 4096x11008 with |N|*Laplace X; INT4 g128",
))

_register(Workload(
    name="llama70b", index=3,
    tensors=(
        TensorSpec("W_sq", 8192, 8192, "normal", sigma=0.015),
        TensorSpec("W_up", 28672, 8192, "normal", sigma=0.015),
        TensorSpec("X", 8192, 8192, "act_outliers", outlier_fraction=0.005,
                   outlier_factor=50.0),
    ),
    calls=(Call("X", ("W_sq",), 4, 128), Call("X", ("W_up",), 4, 128)),
    description="W 8192x8192 and 28672x8192 N(0,0.015); X 8192x8192, 0.5% channels x50; INT4 g128",
))

_register(Workload(
    name="int3_stress", index=4,
    tensors=(
        TensorSpec("W_a", 4096, 4096, "student_t", sigma=0.02, nu=4.0),
        TensorSpec("W_b", 11008, 4096, "student_t", sigma=0.02, nu=4.0),
        TensorSpec("X", 16384, 4096, "act_outliers", outlier_fraction=0.01,
                   outlier_factor=30.0),
    ),
    calls=(Call("X", ("W_a",), 3, 64), Call("X", ("W_a",), 3, 128),
           Call("X", ("W_b",), 3, 64), Call("X", ("W_b",), 3, 128)),
    description="W 4096x4096, 11008x4096 0.02*t(4); X 16384x4096, 1% channels x30; INT3 g64 and g128",
))

WORKLOAD_ORDER: Tuple[str, ...] = tuple(
    sorted(WORKLOADS, key=lambda n: WORKLOADS[n].index))


def _draw_rows(gen: np.random.Generator, spec: TensorSpec, r0: int, r1: int,
               cols: np.ndarray, factors: np.ndarray) -> np.ndarray:
    shape = (r1 - r0, spec.cols)
    if spec.kind == "normal":
        a = gen.standard_normal(shape) * spec.sigma
    elif spec.kind == "student_t":
        a = gen.standard_t(spec.nu, shape) * spec.sigma
    elif spec.kind == "act_outliers":
        a = gen.standard_normal(shape)
        if cols.size:
            a[:, cols] *= factors[None, :]
    elif spec.kind == "abs_normal_laplace":
        a = np.abs(gen.standard_normal(shape)) * gen.laplace(0.0, 1.0, shape)
    else:
        raise ValueError(f"unknown kind {spec.kind}")
    return a.astype(np.float16)


def outlier_plan(spec: TensorSpec, gen: np.random.Generator) -> Tuple[np.ndarray, np.ndarray]:
    """Seeded outlier channels and their factors (empty for other kinds)."""
    if spec.kind != "act_outliers":
        return np.zeros(0, np.int64), np.zeros(0)
    if spec.outlier_channels:
        cols = np.asarray(spec.outlier_channels, np.int64)
    else:
        n = _n_outliers(spec.outlier_fraction, spec.cols)
        cols = np.sort(gen.permutation(spec.cols)[:n]).astype(np.int64)
    if spec.outlier_log_uniform:
        a, b = spec.outlier_log_uniform
        factors = 10.0 ** (a + (b - a) * gen.random(cols.size))
    else:
        factors = np.full(cols.size, spec.outlier_factor)
    return cols, factors


def draw_tensor(spec: TensorSpec, seed_seq: np.random.SeedSequence) -> np.ndarray:
    """Draw one tensor as a C-contiguous fp16 array [rows, cols]."""
    gen = np.random.Generator(np.random.PCG64(seed_seq))
    cols, factors = outlier_plan(spec, gen)
    out = np.empty((spec.rows, spec.cols), np.float16)
    for r0 in range(0, spec.rows, _CHUNK_ROWS):
        r1 = min(spec.rows, r0 + _CHUNK_ROWS)
        out[r0:r1] = _draw_rows(gen, spec, r0, r1, cols, factors)
    return out


def generate(name: str, only: Sequence[str] | None = None) -> Dict[str, np.ndarray]:
    """All tensors of one workload (or the subset ``only``), keyed by name."""
    w = WORKLOADS[name]
    children = np.random.SeedSequence(SEED_BASE + w.index).spawn(len(w.tensors))
    out = {}
    for spec, child in zip(w.tensors, children):
        if only is not None and spec.name not in only:
            continue
        out[spec.name] = draw_tensor(spec, child)
    return out


def random_layer(n: int, k: int, t: int, seed: int, *, w_sigma: float = 0.02,
                 outliers: Sequence[int] = (), factor: float = 20.0,
                 w_kind: str = "normal") -> Tuple[np.ndarray, np.ndarray]:
    """A small ad-hoc layer (W [n,k], X [t,k]) for edge-case tests."""
    seeds = np.random.SeedSequence(seed).spawn(2)
    wspec = TensorSpec("W", n, k, w_kind, sigma=w_sigma)
    xspec = TensorSpec("X", t, k, "act_outliers",
                       outlier_channels=tuple(int(c) for c in outliers),
                       outlier_factor=factor)
    if not outliers:
        xspec = TensorSpec("X", t, k, "normal", sigma=1.0)
    return draw_tensor(wspec, seeds[0]), draw_tensor(xspec, seeds[1])


def weight_rng(seed: int) -> np.random.Generator:
    """A plain seeded generator for tests that need extra random draws."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
