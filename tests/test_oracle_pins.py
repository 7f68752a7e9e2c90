"""Pins for the CPU oracle: what the AWQ pages and plain mathematics fix.

None of these tests compares the oracle with itself.  Each checks it against
a hand-derived value, a closed form, an invariant, a brute-force evaluation
on tiny inputs, or a statistical claim the pages make.  A planted-mistake
test at the end shows that plausible bugs in the oracle fail them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import awq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Hand-worked examples (tests/golden/hand_examples.json)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", golden()["quantizer"], ids=lambda c: c["name"])
def test_quantizer_hand_examples(case):
    W = np.array([case["w"]], np.float16)
    s = np.array(case["s"], np.float32)
    codes, scales, zeros = O.quantize_groups(W, s, case["bits"], case["group"])
    assert codes[0].tolist() == case["codes"]
    assert int(scales.view(np.uint16)[0, 0]) == case["scale_fp16_bits"]
    assert int(zeros[0, 0]) == case["zero"]


@pytest.mark.parametrize("case", golden()["quantizer_symmetric"], ids=lambda c: c["name"])
def test_symmetric_quantizer_hand_examples(case):
    w = np.array(case["w"], np.float16)[None, :]
    codes, sc, z = O.quantize_groups(w, np.array(case["s"], np.float32), case["bits"],
                                     case["group"], zero_point=False)
    assert codes[0].tolist() == case["codes"]
    assert int(sc.view(np.uint16)[0, 0]) == case["scale_fp16_bits"]
    assert int(z[0, 0]) == case["zero"]


@pytest.mark.parametrize("case", golden()["packing"], ids=lambda c: c["name"])
def test_packing_hand_examples(case):
    codes = np.array([case["codes"]], np.uint8)
    words = O.pack_codes(codes, case["bits"])
    assert words[0].tolist() == case["words"]
    back = O.unpack_codes(words, case["bits"], codes.shape[1])
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("case", golden()["statistic"], ids=lambda c: c["name"])
def test_statistic_hand_examples(case):
    sX = O.channel_magnitude(np.array(case["X"], np.float16))
    assert sX.tolist() == case["sX"]


@pytest.mark.parametrize("case", golden()["scale"], ids=lambda c: c["name"])
def test_scale_hand_examples(case):
    s = O.scale_vector(np.array(case["sX"]), case["alpha"])
    assert s.tolist() == case["s"]


@pytest.mark.parametrize("case", golden()["loss"], ids=lambda c: c["name"])
def test_loss_hand_examples(case):
    W = np.array(case["W"], np.float16)
    X = np.array(case["X"], np.float16)
    s = O.scale_vector(O.channel_magnitude(X), case["alpha"])
    assert O.layer_loss(W, X, s, case["bits"], case["group"]) == case["loss"]


# --------------------------------------------------------------------------
# Statistic and scale: closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", golden()["fold"], ids=lambda c: c["name"])
def test_fold_hand_examples(case):
    out = O.fold_inverse_scale(np.array(case["V"], np.float16), np.array(case["s"], np.float32))
    assert out.view(np.uint16).tolist() == case["out_fp16_bits"]


def test_statistic_constant_columns_and_order_independence():
    rng = workloads.weight_rng(1)
    c = rng.standard_normal(16).astype(np.float16)
    X = np.tile(c, (37, 1))
    assert np.array_equal(O.channel_magnitude(X), np.abs(c.astype(np.float64)))
    # Exact sum: a permutation of the tokens gives the bit-identical mean.
    X2 = rng.standard_normal((333, 64)).astype(np.float16) * np.float16(50)
    perm = rng.permutation(333)
    assert np.array_equal(O.channel_magnitude(X2), O.channel_magnitude(X2[perm]))
    # and equals the exact rational mean rounded once.
    col = [Fraction(float(v)) for v in X2[:, 5]]
    exact = sum(abs(v) for v in col) / 333
    assert O.channel_magnitude(X2)[5] == float(exact)


def test_statistic_non_finite_channels_follow_ieee_sums():
    """Reading 10: +inf for a channel holding an infinity of either sign, NaN
    for one holding a NaN (also together with an infinity); the other
    channels keep their exact means."""
    X = np.ones((5, 8), np.float16)
    X[2, 1] = np.float16(np.inf)
    X[4, 2] = np.float16(-np.inf)
    X[0, 3] = np.float16(np.nan)
    X[1, 4] = np.float16(np.inf)
    X[3, 4] = np.float16(np.nan)
    sx = O.channel_magnitude(X)
    assert sx[1] == np.inf and sx[2] == np.inf
    assert np.isnan(sx[3]) and np.isnan(sx[4])
    assert np.array_equal(sx[[0, 5, 6, 7]], np.ones(4))


def test_search_rejects_non_finite_inputs():
    W, X = workloads.random_layer(8, 128, 4, seed=12)
    for bad in ("X", "W"):
        Xb, Wb = X.copy(), W.copy()
        (Xb if bad == "X" else Wb)[1, 3] = np.float16(np.nan if bad == "X" else np.inf)
        with pytest.raises(ValueError):
            O.search(Xb, [Wb], 4, 128, 4)


def test_scale_closed_form_ratios():
    rng = workloads.weight_rng(2)
    sX = np.exp(rng.uniform(-2, 4, 300))
    for a in (0.05, 0.35, 0.95):
        s = O.scale_vector(sX, a).astype(np.float64)
        # s_i / s_j = (sX_i / sX_j)^alpha, up to fp32 rounding of each s.
        ratio = s[:, None] / s[None, :]
        want = (sX[:, None] / sX[None, :]) ** a
        assert np.allclose(ratio, want, rtol=3e-7, atol=0)
        # normalisation: max * min = 1 up to the same rounding
        assert abs(s.max() * s.min() - 1.0) < 3e-7
        # monotone in sX
        order = np.argsort(sX)
        assert np.all(np.diff(s[order]) >= 0)


def test_scale_dead_channel_floor():
    s = O.scale_vector(np.array([0.0, 1e-4, 1.0]), 0.5)
    assert s[0] == s[1]
    assert np.isclose(s[0], 0.1, rtol=1e-6) and np.isclose(s[2], 10.0, rtol=1e-6)


def test_alpha_grid_definition():
    a = O.alpha_grid(20)
    assert a[0] == 0.0 and len(a) == 20
    assert [Fraction(x).limit_denominator(20) for x in a] == [Fraction(i, 20) for i in range(20)]
    assert 1.0 not in a


# --------------------------------------------------------------------------
# Transform: W'X' = WX (AWQ explained, 'Scaling instead of mixed precision')
# --------------------------------------------------------------------------
def on_grid_layer(n, k, group, bits, seed):
    """W and power-of-two s such that W diag(s) lies exactly on its 2^-3 grid.

    Every group holds codes 0 and 2^b-1, so its range is (2^b-1)*step and the
    quantizer must return the grid step 1/8 and reproduce W' exactly.
    """
    rng = workloads.weight_rng(seed)
    levels = (1 << bits) - 1
    step = 0.125
    q = rng.integers(0, levels + 1, (n, k))
    q = q.reshape(n, k // group, group)
    q[:, :, 0] = 0
    q[:, :, 1] = levels
    q = q.reshape(n, k)
    z = rng.integers(0, levels + 1, (n, k // group))
    w_scaled = (q - np.repeat(z, group, axis=1)) * step
    s = 2.0 ** rng.integers(-3, 4, k)
    W = (w_scaled / s[None, :]).astype(np.float16)
    assert np.array_equal(W.astype(np.float64) * s[None, :], w_scaled)
    return W, s.astype(np.float32)


@pytest.mark.parametrize("bits", [3, 4])
def test_transform_cancels_exactly_on_grid(bits):
    W, s = on_grid_layer(6, 64, 16, bits, seed=3)
    rng = workloads.weight_rng(4)
    X = rng.standard_normal((9, 64)).astype(np.float16)
    codes, scales, zeros = O.quantize_groups(W, s, bits, 16)
    assert np.all(scales.astype(np.float64) == 0.125)
    rows = O.output_error_rows(W, X, s, codes, scales, zeros, 16)
    # W' X' equals W X, and quantization is exact here, so the error is 0
    # up to fp64 rounding of the two matmuls.
    Y = W.astype(np.float64) @ X.astype(np.float64).T
    assert rows.max() <= 1e-24 * max(1.0, float((Y ** 2).sum()))


def test_transform_identity_random_s():
    rng = workloads.weight_rng(5)
    W = rng.standard_normal((7, 32))
    X = rng.standard_normal((11, 32))
    s = np.exp(rng.uniform(-2, 2, 32))
    lhs = (W * s[None, :]) @ (X / s[None, :]).T
    rhs = W @ X.T
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Quantizer properties
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bits,group", [(4, 128), (4, 64), (3, 128), (3, 64)])
def test_codes_range_and_nearest_level(bits, group):
    rng = workloads.weight_rng(6 + bits + group)
    W = (rng.standard_normal((24, 4 * group)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, 4 * group)).astype(np.float32)
    codes, scales, zeros = O.quantize_groups(W, s, bits, group)
    levels = (1 << bits) - 1
    assert codes.max() <= levels and zeros.max() <= levels
    # Brute force: each code is the nearest of all 2^b levels (ties within
    # the fp32 rounding of w' * (1/step) may go either way).
    w_scaled = (W.astype(np.float32) * s[None, :]).astype(np.float64)
    sf = np.repeat(scales.astype(np.float64), group, axis=1)
    z = np.repeat(zeros.astype(np.float64), group, axis=1)
    lv = np.arange(levels + 1, dtype=np.float64)
    dist = np.abs(w_scaled[:, :, None] - (lv[None, None, :] - z[:, :, None]) * sf[:, :, None])
    best = dist.min(axis=2)
    got = np.abs(w_scaled - (codes - z) * sf)
    assert np.all(got <= best + 1e-6 * sf)


def test_step_is_range_over_levels_and_widens():
    """AWQ Explained (multigrid.ai): the step is range / levels; pushing one
    weight past the group max widens the step for every other weight
    (activation-aware weight quantization (AWQ), realpython, slider text)."""
    rng = workloads.weight_rng(7)
    w = (rng.standard_normal((1, 128)) * 0.02).astype(np.float16)
    ones = np.ones(128, np.float32)
    _, sc0, _ = O.quantize_groups(w, ones, 4, 128)
    w_big = w.copy()
    j = int(np.argmax(w[0]))
    w_big[0, j] = np.float16(float(w[0, j]) * 3)
    _, sc1, _ = O.quantize_groups(w_big, ones, 4, 128)
    r0 = float(w.max()) - float(w.min())
    r1 = float(w_big.max()) - float(w_big.min())
    assert math.isclose(float(sc0[0, 0]), r0 / 15, rel_tol=1e-3)
    assert math.isclose(float(sc1[0, 0]), r1 / 15, rel_tol=1e-3)
    assert float(sc1[0, 0]) > float(sc0[0, 0])


@pytest.mark.parametrize("k", [-3, 2, 5])
def test_homogeneity_power_of_two(k):
    """Min/max RTN is positively homogeneous: s -> 2^k s keeps the codes and
    zeros and multiplies the scales by 2^k exactly."""
    rng = workloads.weight_rng(8)
    W = (rng.standard_normal((16, 256)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, 256)).astype(np.float32)
    c0, sc0, z0 = O.quantize_groups(W, s, 4, 128)
    c1, sc1, z1 = O.quantize_groups(W, (s * np.float32(2.0 ** k)).astype(np.float32), 4, 128)
    assert np.array_equal(c0, c1) and np.array_equal(z0, z1)
    assert np.array_equal(sc1.astype(np.float64), sc0.astype(np.float64) * 2.0 ** k)


def test_alpha_zero_is_plain_rtn_of_w():
    """alpha = 0 gives s = 1, so the search's alpha-0 candidate is plain group
    round-to-nearest of W itself (AWQ, ai360xpert, 'How It Works' step 4)."""
    W, X = workloads.random_layer(8, 256, 16, seed=9)
    res = O.search(X, [W], 4, 128, n_grid=4)
    assert np.all(res["s_grid"][0] == 1.0)
    c, sc, z = O.quantize_groups(W, np.ones(256, np.float32), 4, 128)
    # code = nearest level of w itself on the grid (q - z) * step
    deq = O.dequantize_scaled(c, sc, z, 128)
    err = np.abs(W.astype(np.float64) - deq)
    assert np.all(err <= np.repeat(sc.astype(np.float64), 128, axis=1) * (0.5 + 1e-6))


# --------------------------------------------------------------------------
# The pages' analysis: error ratio ~ 1/s when the step is unchanged, and
# over-scaling hurts (AWQ explained, 'Scaling instead of mixed precision').
# --------------------------------------------------------------------------
def _salient_errors(scale_factor, span=None, rows=20000, seed=10):
    """Errors of one salient column j inside groups whose min and max are set
    by two fixed columns (+-0.04), before and after scaling column j.

    The salient weights are drawn across several grid steps (|w| up to
    ``span``), the regime where rounding error is uniform and the pages'
    analysis applies."""
    rng = workloads.weight_rng(seed)
    g = 128
    W = (rng.uniform(-0.01, 0.01, (rows, g))).astype(np.float16)
    W[:, 0] = np.float16(0.04)
    W[:, 1] = np.float16(-0.04)
    j = 5
    span = 0.95 * 0.04 / scale_factor if span is None else span
    W[:, j] = rng.uniform(-span, span, rows).astype(np.float16)
    s = np.ones(g, np.float32)
    s[j] = scale_factor
    c, sc, z = O.quantize_groups(W, s, 4, g)
    deq = O.dequantize_scaled(c, sc, z, g) / s.astype(np.float64)[None, :]
    err = np.abs(deq - W.astype(np.float64))
    others = np.delete(err, [0, 1, j], axis=1)
    return err[:, j].mean(), others.mean(), sc


@pytest.mark.parametrize("sfac", [2.0, 3.0, 4.0])
def test_salient_error_ratio_one_over_s(sfac):
    span = 0.95 * 0.04 / sfac
    e1, _, sc1 = _salient_errors(1.0, span=span)
    es, _, scs = _salient_errors(sfac, span=span)
    assert np.array_equal(sc1, scs)        # step unchanged (delta' = delta)
    assert abs((es / e1) * sfac - 1.0) < 0.1


def test_over_scaling_hurts_other_weights():
    _, o1, sc1 = _salient_errors(1.0, span=0.004)
    _, o_big, sc_big = _salient_errors(40.0, span=0.004)   # 0.004*40 > group max 0.04
    assert np.all(sc_big.astype(np.float64) >= sc1.astype(np.float64))
    assert o_big > 1.5 * o1


# --------------------------------------------------------------------------
# Loss: brute force, Gram form, special cases
# --------------------------------------------------------------------------
def test_loss_brute_force_loops():
    W, X = workloads.random_layer(3, 16, 5, seed=11, outliers=(2,), factor=10.0)
    s = O.scale_vector(O.channel_magnitude(X), 0.45)
    bits, group = 4, 8
    codes, scales, zeros = O.quantize_groups(W, s, bits, group)
    N, K = W.shape
    T = X.shape[0]
    total = Fraction(0)
    for n in range(N):
        for t in range(T):
            acc = Fraction(0)
            for k in range(K):
                gi = k // group
                deq = (int(codes[n, k]) - int(zeros[n, gi])) * Fraction(float(scales[n, gi]))
                acc += (Fraction(float(W[n, k])) - deq / Fraction(float(s[k]))) * Fraction(float(X[t, k]))
            total += acc * acc
    exact = float(total / (N * T))
    got = O.layer_loss(W, X, s, bits, group)
    assert math.isclose(got, exact, rel_tol=1e-11)


def test_loss_gram_form():
    W, X = workloads.random_layer(12, 256, 40, seed=12, outliers=(7, 99), factor=30.0)
    s = O.scale_vector(O.channel_magnitude(X), 0.3)
    codes, scales, zeros = O.quantize_groups(W, s, 4, 128)
    delta = W.astype(np.float64) - O.dequantize_scaled(codes, scales, zeros, 128) / s.astype(np.float64)
    X64 = X.astype(np.float64)
    G = X64.T @ X64
    gram = np.einsum("nk,kl,nl->n", delta, G, delta)
    rows = O.output_error_rows(W, X, s, codes, scales, zeros, 128)
    assert np.allclose(rows, gram, rtol=1e-9, atol=0)


def test_identity_activations_give_weight_mse():
    K = 128
    rng = workloads.weight_rng(13)
    W = (rng.standard_normal((5, K)) * 0.02).astype(np.float16)
    X = np.eye(K, dtype=np.float16)
    s = np.ones(K, np.float32)
    codes, scales, zeros = O.quantize_groups(W, s, 4, 64)
    mse = ((W.astype(np.float64) - O.dequantize_scaled(codes, scales, zeros, 64)) ** 2).sum() / (5 * K)
    assert math.isclose(O.layer_loss(W, X, s, 4, 64), mse, rel_tol=1e-12)


def test_statistical_loss_at_alpha_zero():
    """With X ~ N(0,1) independent of the rounding, E[loss] is the mean
    squared weight error times K (each output sums K independent terms)."""
    rng = workloads.weight_rng(14)
    N, K, T = 64, 512, 2048
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    X = rng.standard_normal((T, K)).astype(np.float16)
    s = np.ones(K, np.float32)
    codes, scales, zeros = O.quantize_groups(W, s, 4, 128)
    d = W.astype(np.float64) - O.dequantize_scaled(codes, scales, zeros, 128)
    expect = (d ** 2).sum() / N * np.mean(X.astype(np.float64) ** 2)
    got = O.layer_loss(W, X, s, 4, 128)
    assert abs(got / expect - 1.0) < 0.05


def test_argmin_first_minimum_and_nan():
    assert O.first_argmin([3.0, 1.0, 1.0, 2.0]) == 1
    assert O.first_argmin([float("nan"), 5.0, 4.0]) == 2
    assert O.first_argmin([float("nan"), float("nan")]) == 0
    assert O.first_argmin([2.0]) == 0


def test_search_row_subset_consistent():
    W, X = workloads.random_layer(40, 256, 24, seed=15, outliers=(3, 130), factor=25.0)
    full = O.search(X, [W], 4, 128, n_grid=5)
    rows = np.array([0, 7, 39])
    sub = O.search(X, [W], 4, 128, n_grid=5, rows=[rows])
    assert np.array_equal(sub["row_losses"][0], full["row_losses"][0][:, rows])


def test_shared_x_sums_losses():
    W1, X = workloads.random_layer(16, 256, 20, seed=16, outliers=(5,), factor=20.0)
    W2, _ = workloads.random_layer(24, 256, 20, seed=17)
    both = O.search(X, [W1, W2], 4, 128, n_grid=6)
    a = O.search(X, [W1], 4, 128, n_grid=6)
    b = O.search(X, [W2], 4, 128, n_grid=6)
    assert np.allclose(both["losses"], a["losses"] + b["losses"], rtol=1e-13, atol=0)


def test_activation_aware_scaling_helps_on_tiny_workload():
    """The pages' claim (AWQ explained; AWQ Explained, multigrid): with
    outlier input channels, some alpha > 0 beats plain RTN (alpha = 0)."""
    t = workloads.generate("tiny")
    res = O.search(t["X"], [t["W"]], 4, 128, n_grid=20)
    assert res["best"] > 0
    assert res["losses"][res["best"]] < 0.9 * res["losses"][0]


def test_weight_magnitude_saliency_does_worse():
    """The pages' ablation (AWQ explained, "Salient weights are
    activation-aware"; AWQ Explained, multigrid.ai, "Why the activations
    pick, not the weights"): picking the scale by weight magnitude does worse
    than by activation magnitude.  With s built from the mean |W| of each
    input channel, the best loss on the tiny workload (whose salient channels
    come from the activations) stays above the activation-aware best."""
    t = workloads.generate("tiny")
    act = O.search(t["X"], [t["W"]], 4, 128, n_grid=20)
    wmag = O.search(t["X"], [t["W"]], 4, 128, n_grid=20,
                    sX=O.channel_magnitude(t["W"]))
    assert wmag["losses"].min() > 1.05 * act["losses"].min()


def test_fold_keeps_the_layer_output():
    """AWQ Explained (multigrid.ai), "Scaling instead of mixed precision": with
    diag(s)^-1 folded into the producer of x, the scaled layer W diag(s)
    computes the same output.  With power-of-two s every step is exact, so
    the identity holds bit for bit in fp64, for a norm weight and for a
    preceding linear layer."""
    rng = workloads.weight_rng(91)
    K, M, N = 64, 48, 16
    s = (2.0 ** rng.integers(-3, 4, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16).astype(np.float64)
    gamma = rng.uniform(0.5, 2.0, K).astype(np.float16)
    h = rng.standard_normal(K)
    y = W @ (gamma.astype(np.float64) * h)
    g2 = O.fold_inverse_scale(gamma, s).astype(np.float64)
    assert np.array_equal((W * s.astype(np.float64)) @ (g2 * h), y)
    P = (rng.standard_normal((K, M)) * 0.1).astype(np.float16)
    u = rng.standard_normal(M)
    y2 = W @ (P.astype(np.float64) @ u)
    P2 = O.fold_inverse_scale(P, s).astype(np.float64)
    np.testing.assert_allclose((W * s.astype(np.float64)) @ (P2 @ u), y2, rtol=1e-12, atol=1e-15)


def test_fold_rounds_once_to_fp16():
    rng = workloads.weight_rng(92)
    V = rng.standard_normal((37, 5)).astype(np.float16)
    s = np.exp(rng.uniform(-2, 2, 37)).astype(np.float32)
    out = O.fold_inverse_scale(V, s)
    exact = V.astype(np.float64) / s.astype(np.float64)[:, None]
    # within half an fp16 ulp (plus the fp32 rounding before it)
    ulp = np.spacing(np.abs(out).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 0.5 * ulp + np.abs(exact) * 2.0 ** -24)
    with pytest.raises(ValueError):
        O.fold_inverse_scale(V, s[:-1])


@pytest.mark.parametrize("bits", [3, 4])
def test_symmetric_alpha_zero_is_plain_absmax_rtn(bits):
    """alpha = 0 (s == 1), zero_point false: a separately written symmetric
    round-to-nearest by the group's maximum magnitude, loop by loop."""
    rng = workloads.weight_rng(70 + bits)
    W = (rng.standard_t(4, (6, 256)) * 0.02).astype(np.float16)
    codes, sc, z = O.quantize_groups(W, np.ones(256, np.float32), bits, 64, zero_point=False)
    half = 1 << (bits - 1)
    for n in range(6):
        for g in range(4):
            blk = W[n, 64 * g:64 * g + 64].astype(np.float32)
            amax = max(float(np.max(np.abs(blk))), 1e-5)
            step = np.float16(np.float32(amax) / np.float32(half - 1))
            r = np.float32(1) / np.float32(step)
            assert sc[n, g] == step and z[n, g] == half
            for j in range(64):
                q = int(np.rint(np.float32(blk[j] * r))) + half
                assert codes[n, 64 * g + j] == min(max(q, 0), 2 * half - 1)


@pytest.mark.parametrize("bits", [3, 4])
def test_symmetric_codes_nearest_level(bits):
    rng = workloads.weight_rng(80 + bits)
    W = (rng.standard_normal((5, 128)) * 0.05).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, 128)).astype(np.float32)
    codes, sc, z = O.quantize_groups(W, s, bits, 128, zero_point=False)
    assert codes.max() <= (1 << bits) - 1 and np.all(z == 1 << (bits - 1))
    ws = W.astype(np.float32) * s
    levels = (np.arange(1 << bits)[None, :] - (1 << (bits - 1))) * sc.astype(np.float64)
    for n in range(5):
        d = np.abs(ws[n][:, None].astype(np.float64) - levels[n][None, :])
        best = d.min(axis=1)
        got = d[np.arange(128), codes[n]]
        assert np.all(got <= best + 1e-6 * sc[n, 0])


def test_per_row_group_is_one_group_of_k():
    rng = workloads.weight_rng(88)
    W = (rng.standard_normal((9, 512)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, 512)).astype(np.float32)
    for zp in (True, False):
        a = O.quantize_groups(W, s, 4, -1, zero_point=zp)
        b = O.quantize_groups(W, s, 4, 512, zero_point=zp)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
        assert a[1].shape == (9, 1)


@pytest.mark.parametrize("k", [-2, 3])
def test_symmetric_homogeneity_power_of_two(k):
    rng = workloads.weight_rng(89)
    W = (rng.standard_normal((4, 256)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, 256)).astype(np.float32)
    c1, s1, z1 = O.quantize_groups(W, s, 4, 128, zero_point=False)
    c2, s2, z2 = O.quantize_groups(W, s * np.float32(2.0 ** k), 4, 128, zero_point=False)
    assert np.array_equal(c1, c2) and np.array_equal(z1, z2)
    assert np.array_equal(s2.astype(np.float64), s1.astype(np.float64) * 2.0 ** k)


def test_w4a16_matvec_hand_example():
    """AWQ explained, "Why weight-only quantization fits decoding" (W4A16):
    codes [15, 0], scale 0.5, zero 8, x = [1, 2]:
    (15 - 8) * 0.5 * 1 + (0 - 8) * 0.5 * 2 = 3.5 - 8 = -4.5."""
    y = O.w4a16_matvec(np.array([[15, 0]], np.uint8), np.array([[0.5]], np.float16),
                       np.array([[8]], np.uint8), 2, np.array([[1.0, 2.0]], np.float16))
    assert y.shape == (1, 1) and y[0, 0] == -4.5


@pytest.mark.parametrize("zp,group", [(True, 128), (False, 64), (True, -1)])
def test_w4a16_matvec_within_rounding_of_dense(zp, group):
    """y from the packed layer differs from W x by at most the rounding of
    each weight: |y - W x| <= sum_k |w_k - deq_k| |x_k| with |w - deq| <=
    scale / 2 per weight (unclamped codes), checked row by row."""
    rng = workloads.weight_rng(93 + group)
    W = (rng.standard_normal((24, 256)) * 0.02).astype(np.float16)
    x = rng.standard_normal((3, 256)).astype(np.float16)
    c, sc, z = O.quantize_groups(W, np.ones(256, np.float32), 4, group, zero_point=zp)
    y = O.w4a16_matvec(c, sc, z, group, x)
    dense = x.astype(np.float64) @ W.astype(np.float64).T
    g = 256 if group == -1 else group
    half_step = np.repeat(sc.astype(np.float64), g, axis=1) / 2
    bound = np.abs(x.astype(np.float64)) @ half_step.T
    assert np.all(np.abs(y - dense) <= bound * (1 + 1e-9))
    assert np.abs(y - dense).max() > 0


@pytest.mark.parametrize("bits", [3, 4])
def test_pack_roundtrip_random(bits):
    rng = workloads.weight_rng(18 + bits)
    codes = rng.integers(0, 1 << bits, (5, 256)).astype(np.uint8)
    words = O.pack_codes(codes, bits)
    assert words.shape == (5, O.packed_words(256, bits))
    assert np.array_equal(O.unpack_codes(words, bits, 256), codes)


# --------------------------------------------------------------------------
# Planted mistakes: each mutant of the oracle must fail at least one pin.
# --------------------------------------------------------------------------
def _pins_pass():
    try:
        for case in golden()["quantizer"]:
            test_quantizer_hand_examples(case)
        for case in golden()["loss"]:
            test_loss_hand_examples(case)
        for case in golden()["scale"]:
            test_scale_hand_examples(case)
        test_transform_cancels_exactly_on_grid(4)
        test_loss_gram_form()
        test_codes_range_and_nearest_level(4, 128)
    except AssertionError:
        return False
    return True


def test_pins_catch_planted_mistakes(monkeypatch):
    assert _pins_pass()
    real_deq = O.dequantize_scaled
    real_rows = O.output_error_rows
    real_scale = O.scale_vector
    real_quant = O.quantize_groups

    def deq_no_zero(codes, scales, zeros, group):          # dropped term
        return real_deq(codes, scales, np.zeros_like(zeros), group)

    def rows_no_inverse(W, X, s, codes, scales, zeros, group, Y=None):   # dropped 1/s
        return real_rows(W, X, np.ones_like(s), codes, scales, zeros, group, Y)

    def scale_no_norm(sX, alpha):                          # dropped normalisation
        u = np.power(np.maximum(np.asarray(sX, np.float64), 1e-4), alpha)
        return u.astype(np.float32)

    def quant_neg_zero(W, s, bits, group):                 # wrong sign of zero point
        c, sc, z = real_quant(W, s, bits, group)
        levels = (1 << bits) - 1
        return np.clip(c.astype(int) - 2 * np.repeat(z, group, axis=1).astype(int) + levels, 0, levels).astype(np.uint8), sc, z

    for name, mutant in [("dequantize_scaled", deq_no_zero),
                         ("output_error_rows", rows_no_inverse),
                         ("scale_vector", scale_no_norm),
                         ("quantize_groups", quant_neg_zero)]:
        with monkeypatch.context() as m:
            m.setattr(O, name, mutant)
            assert not _pins_pass(), f"mutant {name} passed every pin"
