"""CPU oracle for the AWQ activation-aware scale search.

TEST INFRASTRUCTURE.  This module exists to check the CUDA path.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it; the library path never calls it and has no CPU fallback.  It shares
no code, table or constant generator with the CUDA sources.

It is deliberately plain: numpy, fp64 wherever the pages leave precision open,
fp32/fp16 exactly where the stored format fixes it, one library matmul as the
only heavy step, no blocking or fusion.  Each function names the page passage
it follows.  Pages (by title):

* [AWQX]  "AWQ explained" (hungho77.github.io), section "Scaling instead of
  mixed precision": W' = W diag(s), X' = diag(s)^-1 X, W'X' = WX; the error
  ratio ~1/s when the group step is unchanged; s = sX^alpha with sX the mean
  activation magnitude per input channel; grid search of alpha in [0, 1] to
  minimise the layer-output error after quantization.
* [MG]    "AWQ Explained: Protecting the Weights That Matter Most"
  (multigrid.ai), sections "Scaling instead of mixed precision" (the grid
  step is the group's range divided by the number of levels) and "How the
  scale is chosen" (s = mean(|x_j|)^alpha; alpha* = argmin over a small grid
  of ||W x - Q(W diag(s)) diag(s)^-1 x||; the AwqConfig knobs bits=4,
  group_size=128, zero_point=true).
* [RP]    "activation-aware weight quantization (AWQ)" (realpython.com
  glossary): 3- or 4-bit packing in groups, commonly 128.
* [AI360] "AWQ" (ai360xpert.com), section "How It Works", step 4: the scaled
  weights are quantized with plain round-to-nearest.
* [AWQX-DEC] "AWQ explained" (hungho77.github.io), "Why weight-only
  quantization fits decoding": at small batch the weights dominate the
  memory traffic; 4-bit weights with 16-bit activations (W4A16) cut it about
  four times.
* [MG-FOLD] "AWQ Explained" (multigrid.ai), "Scaling instead of mixed
  precision": diag(s)^-1 is folded offline into the operation that produces
  the layer's input (the preceding LayerNorm / RMSNorm weight, or a preceding
  linear layer), so what ships is the quantized matrix and a modified norm.

Readings where the pages are silent:

1. Normalisation of s: u_j = max(sX_j, 1e-4)^alpha in fp64, then
   s_j = fp32(u_j / sqrt(max_j u * min_j u)).  A global factor on s leaves the
   loss unchanged in exact arithmetic; this choice only keeps W' and the
   inverse-scaled activations near unit range.  alpha = 0 gives s == 1.
2. Grid: alpha_i = i / n_grid for i = 0 .. n_grid-1 (20 points; alpha = 1 is
   not evaluated).
3. Quantizer: per group of ``group`` consecutive input channels of one output
   row, asymmetric min/max round-to-nearest in fp32 with no fused
   multiply-add:  w' = fp32(w * s);  rng = fp32(max - min);
   step32 = fp32(max(rng, 1e-5) / (2^b - 1));  scale = fp16_rne(step32);
   sf = float(scale);  rcp = fp32(1 / sf);  z = clamp(rne(fp32(-min * rcp)),
   0, 2^b - 1);  q = clamp(rne(fp32(w' * rcp)) + z, 0, 2^b - 1).  rne is
   round-half-to-even.
4. Error: squared Frobenius norm divided by N*T (the page writes the unsquared
   norm; the argmin is the same).  Several weights sharing one X share one s
   and sum their per-weight losses.
5. argmin: the first grid index holding the minimum; NaN counts as +inf.
6. Packing: INT4 row n, word j holds codes 8j..8j+7 in nibbles 0..7 (code 8j
   in bits 0-3).  INT3 row n is a little-endian bit stream, code k in bits
   [3k, 3k+3), 32 codes per 3 uint32 words.
7. Folding: V'[k] = fp16(fp32(V[k]) / s_k) for a norm weight or bias; for a
   preceding linear layer [K][M] (its output row k feeds input channel k)
   every entry of row k is divided by s_k.  One correctly rounded fp32
   division, then round-to-nearest-even to fp16.
8. Symmetric quantizer (zero_point false; AI360 "The Idea": quantization
   groups weights and scales them by their maximum value):
   step = max(max|w'|, 1e-5) / (2^(b-1) - 1), scale = fp16_rne(step),
   rcp = fp32(1 / scale), the zero point is the fixed mid-code 2^(b-1), and
   q = clamp(rne(w' * rcp) + 2^(b-1), 0, 2^b - 1) -- the same stored layout
   and dequantization (q - z) * scale.
9. group_size -1 (the AwqConfig knob in [MG] "How the scale is chosen",
   "-1 meaning per-column"): one group spans an output row's K channels.  The
   pages write the layer as W x; the packed AWQ format stores the transpose
   W^T [in x out], whose column is one output channel, so a per-column group
   is one output row of W [N x K] here.
10. Non-finite inputs: the pages assume finite activations and weights.
   ``channel_magnitude`` keeps the IEEE fp64 sum's answer for a channel that
   holds an infinity (+inf) or a NaN (NaN); ``search`` rejects X or W with a
   non-finite value (ValueError): its steps have no meaning there.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

SX_FLOOR = 1e-4          # reading 1: clamp for dead channels
RANGE_FLOOR = np.float32(1e-5)   # reading 3: step floor for constant groups


# --------------------------------------------------------------------------
# Step 1: per-input-channel activation statistic ([AWQX]; [MG] "How the
# scale is chosen": s = mean(|x_j|)^alpha).
# --------------------------------------------------------------------------
def channel_magnitude(X: np.ndarray) -> np.ndarray:
    """sX_j = (1/T) * sum_t |X[t, j]| in fp64.

    Every fp16 value is an integer multiple of 2^-24, so every partial sum is
    too; for |sum| < 2^29 the fp64 sum is exact and independent of order.
    The mean is then one correctly rounded division.  A channel holding an
    infinity gives +inf, one holding a NaN gives NaN (reading 10).
    """
    X = np.asarray(X)
    if X.ndim != 2 or X.shape[0] == 0:
        raise ValueError("X must be [T, K] with T >= 1")
    total = np.abs(X.astype(np.float64)).sum(axis=0)
    return total / np.float64(X.shape[0])


# --------------------------------------------------------------------------
# Step 2: the scale for one alpha ([AWQX]: s = sX^alpha; reading 1).
# --------------------------------------------------------------------------
def alpha_grid(n_grid: int = 20) -> np.ndarray:
    """alpha_i = i / n_grid, i = 0 .. n_grid-1 (reading 2)."""
    return np.arange(n_grid, dtype=np.float64) / np.float64(n_grid)


def scale_vector(sX: np.ndarray, alpha: float) -> np.ndarray:
    """s_j = fp32(u_j / sqrt(max u * min u)), u_j = max(sX_j, 1e-4)^alpha."""
    u = np.power(np.maximum(np.asarray(sX, np.float64), SX_FLOOR), np.float64(alpha))
    u = u / np.sqrt(u.max() * u.min())
    return u.astype(np.float32)


# --------------------------------------------------------------------------
# Step 3: scale W by s and group-quantize along K ([AWQX] W' = W diag(s);
# [MG] "the grid step is the group's range divided by the number of levels";
# [AI360] step 4 round-to-nearest; [MG] AwqConfig zero_point = true).
# --------------------------------------------------------------------------
def quantize_groups(W: np.ndarray, s: np.ndarray, bits: int, group: int,
                    zero_point: bool = True):
    """Return (codes uint8 [N,K], scales fp16 [N,K/group], zeros uint8 [N,K/group]).

    ``group`` = -1 makes one group of each output row (reading 9).
    ``zero_point`` False is the symmetric form of reading 8.
    All arithmetic is fp32 (numpy evaluates each operation separately and
    rounds it; nothing is fused), following readings 3 and 8 step by step.
    """
    W = np.asarray(W, np.float16)
    N, K = W.shape
    if group == -1:
        group = K
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    levels = np.float32((1 << bits) - 1)
    s32 = np.asarray(s, np.float32)
    w_scaled = W.astype(np.float32) * s32[None, :]                 # w' = w * s
    g = w_scaled.reshape(N, K // group, group)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    if zero_point:
        rng = mx - mn                                              # fp32
        step32 = np.maximum(rng, RANGE_FLOOR) / levels             # fp32 divide
    else:
        amax = np.maximum(-mn, mx)                                 # max |w'|
        step32 = np.maximum(amax, RANGE_FLOOR) / np.float32((1 << (bits - 1)) - 1)
    scale16 = step32.astype(np.float16)                            # fp16 RNE
    sf = scale16.astype(np.float32)
    rcp = np.float32(1.0) / sf                                     # fp32 reciprocal
    if zero_point:
        zero = np.clip(np.rint(-mn * rcp), 0, levels)              # integer zero point
    else:
        zero = np.full(mn.shape, np.float32(1 << (bits - 1)))      # fixed mid-code
    q = np.rint(g * rcp[:, :, None]) + zero[:, :, None]
    q = np.clip(q, 0, levels)
    return (q.reshape(N, K).astype(np.uint8), scale16,
            zero.astype(np.uint8))


def dequantize_scaled(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                      group: int) -> np.ndarray:
    """deq(Q(W')) in the scaled units of W': (q - z) * scale, fp64."""
    codes = np.asarray(codes)
    N, K = codes.shape
    if group == -1:
        group = K
    q = codes.astype(np.float64).reshape(N, K // group, group)
    z = np.asarray(zeros).astype(np.float64)[:, :, None]
    sf = np.asarray(scales, np.float16).astype(np.float64)[:, :, None]
    return ((q - z) * sf).reshape(N, K)


# --------------------------------------------------------------------------
# Step 4: packing ([RP] "packed at 3 or 4 bits in groups"; reading 6).
# --------------------------------------------------------------------------
def packed_words(K: int, bits: int) -> int:
    """uint32 words per row."""
    if bits == 4:
        if K % 8:
            raise ValueError("INT4 packing needs K % 8 == 0")
        return K // 8
    if bits == 3:
        if K % 32:
            raise ValueError("INT3 packing needs K % 32 == 0")
        return 3 * K // 32
    raise ValueError("bits must be 3 or 4")


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [N, K] into uint32 words [N, packed_words(K, bits)].

    Written as a plain bit stream: code k of a row occupies bits
    [bits*k, bits*k + bits) of the row, word w holding bits [32w, 32w+32).
    """
    codes = np.asarray(codes, np.uint64)
    N, K = codes.shape
    nw = packed_words(K, bits)
    out = np.zeros((N, nw), np.uint64)
    for k in range(K):
        bit = bits * k
        w, off = divmod(bit, 32)
        out[:, w] |= (codes[:, k] << np.uint64(off)) & np.uint64(0xFFFFFFFF)
        spill = off + bits - 32
        if spill > 0:
            out[:, w + 1] |= codes[:, k] >> np.uint64(bits - spill)
    return out.astype(np.uint32)


def unpack_codes(words: np.ndarray, bits: int, K: int) -> np.ndarray:
    """Inverse of ``pack_codes``."""
    words = np.asarray(words, np.uint64)
    N = words.shape[0]
    mask = np.uint64((1 << bits) - 1)
    out = np.zeros((N, K), np.uint8)
    for k in range(K):
        bit = bits * k
        w, off = divmod(bit, 32)
        v = words[:, w] >> np.uint64(off)
        spill = off + bits - 32
        if spill > 0:
            v = v | (words[:, w + 1] << np.uint64(bits - spill))
        out[:, k] = (v & mask).astype(np.uint8)
    return out


# --------------------------------------------------------------------------
# Step 5: the layer-output error ([MG] "How the scale is chosen":
# || W x - Q(W diag(s)) diag(s)^-1 x ||; reading 4).
# --------------------------------------------------------------------------
def output_error_rows(W: np.ndarray, X: np.ndarray, s: np.ndarray,
                      codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                      group: int, Y: Optional[np.ndarray] = None) -> np.ndarray:
    """Per output row n: sum_t (W X^T - deq(Q(W')) diag(s)^-1 X^T)[n, t]^2, fp64.

    ``Y`` may carry a precomputed W X^T (it does not depend on alpha).
    """
    X64 = np.asarray(X).astype(np.float64)
    if Y is None:
        Y = np.asarray(W).astype(np.float64) @ X64.T            # W x
    x_inv = X64 / np.asarray(s, np.float32).astype(np.float64)[None, :]   # diag(s)^-1 x
    Yhat = dequantize_scaled(codes, scales, zeros, group) @ x_inv.T
    E = Y - Yhat
    return np.einsum("nt,nt->n", E, E)


def layer_loss(W, X, s, bits, group) -> float:
    """||W X^T - deq(Q(W diag(s))) diag(s)^-1 X^T||^2 / (N T)."""
    codes, scales, zeros = quantize_groups(W, s, bits, group)
    rows = output_error_rows(W, X, s, codes, scales, zeros, group)
    N = np.asarray(W).shape[0]
    return float(rows.sum() / (N * np.asarray(X).shape[0]))


# --------------------------------------------------------------------------
# Step 6: grid search ([AWQX]; [MG] alpha* = argmin over the grid).
# --------------------------------------------------------------------------
def first_argmin(losses: Sequence[float]) -> int:
    """Smallest index achieving the minimum; NaN compares as +inf (reading 5)."""
    best, best_v = 0, None
    for i, v in enumerate(losses):
        v = float("inf") if np.isnan(v) else float(v)
        if best_v is None or v < best_v:
            best, best_v = i, v
    return best


def search(X: np.ndarray, Ws: Sequence[np.ndarray], bits: int = 4, group: int = 128,
           n_grid: int = 20, sX: Optional[np.ndarray] = None,
           rows: Optional[Sequence[Optional[np.ndarray]]] = None,
           zero_point: bool = True) -> Dict:
    """The full search for the weights ``Ws`` sharing activations ``X``.

    ``rows`` (optional, one entry per weight) restricts the loss to a subset of
    output rows.  Quantization and the error are independent per row, so the
    per-row losses of a subset equal those rows of the full computation; the
    total loss and the argmin are then those of the subset.

    Returns a dict with ``sX``, ``alphas``, ``s_grid`` [n_grid, K] fp32,
    ``row_losses`` (per weight, [n_grid, rows]) fp64, ``losses`` [n_grid],
    ``best``, ``alpha``, ``s`` and per-weight ``codes``/``scales``/``zeros``
    (of the selected rows) at the chosen alpha, plus ``packed``.
    """
    X = np.asarray(X, np.float16)
    T, K = X.shape
    if not np.all(np.isfinite(X)) or not all(np.all(np.isfinite(np.asarray(W))) for W in Ws):
        raise ValueError("X and W must be finite (reading 10)")
    if sX is None:
        sX = channel_magnitude(X)
    alphas = alpha_grid(n_grid)
    sel = []
    for i, W in enumerate(Ws):
        r = None if rows is None else rows[i]
        sel.append(np.asarray(W, np.float16) if r is None
                   else np.asarray(W, np.float16)[np.asarray(r)])
    X64 = X.astype(np.float64)
    grp = K if group == -1 else group
    Yref = [w.astype(np.float64) @ X64.T for w in sel]
    s_grid = np.stack([scale_vector(sX, a) for a in alphas])
    row_losses = [np.zeros((n_grid, w.shape[0])) for w in sel]
    losses = np.zeros(n_grid)
    for i in range(n_grid):
        s = s_grid[i]
        total = 0.0
        for wi, w in enumerate(sel):
            c, sc, z = quantize_groups(w, s, bits, group, zero_point)
            rl = output_error_rows(w, X, s, c, sc, z, grp, Y=Yref[wi])
            row_losses[wi][i] = rl
            total += rl.sum() / (w.shape[0] * T)
        losses[i] = total
    best = first_argmin(losses)
    s_best = s_grid[best]
    codes, scales, zeros, packed = [], [], [], []
    for w in sel:
        c, sc, z = quantize_groups(w, s_best, bits, group, zero_point)
        codes.append(c)
        scales.append(sc)
        zeros.append(z)
        packed.append(pack_codes(c, bits))
    return dict(sX=sX, alphas=alphas, s_grid=s_grid, row_losses=row_losses,
                losses=losses, best=best, alpha=float(alphas[best]), s=s_best,
                codes=codes, scales=scales, zeros=zeros, packed=packed)


# --------------------------------------------------------------------------
# Step 7: deploy ([MG-FOLD]; reading 7): fold diag(s)^-1 into the producer
# of the layer's input.
# --------------------------------------------------------------------------
def fold_inverse_scale(V: np.ndarray, s: np.ndarray) -> np.ndarray:
    """V / s along the first axis: a vector [K] (norm weight or bias) or a
    preceding linear layer [K, M]; fp32 division, fp16 result."""
    V = np.asarray(V, np.float16)
    s32 = np.asarray(s, np.float32)
    if V.shape[0] != s32.shape[0]:
        raise ValueError("V's first axis must match s")
    d = s32 if V.ndim == 1 else s32.reshape((-1,) + (1,) * (V.ndim - 1))
    return (V.astype(np.float32) / d).astype(np.float16)


# --------------------------------------------------------------------------
# Step 8: consuming the packed layer ([AWQX-DEC]): the W4A16 product.
# --------------------------------------------------------------------------
def w4a16_matvec(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray, group: int,
                 x: np.ndarray) -> np.ndarray:
    """y[m, n] = sum_k (q[n, k] - z[n, g(k)]) * scale[n, g(k)] * x[m, k] in fp64.

    ``codes`` are unpacked [N, K]; ``x`` is fp16 [M, K] (the activations with
    diag(s)^-1 already folded into their producer)."""
    deq = dequantize_scaled(codes, scales, zeros, group)
    return np.asarray(x, np.float16).astype(np.float64) @ deq.T
