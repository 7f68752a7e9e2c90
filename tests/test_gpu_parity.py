"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bars: bit-exact for codes, packed words, zeros, fp16 scales, the exact
channel statistic and s; per-grid-point loss within 1e-3 relative; the
chosen alpha equal unless the oracle's two best losses are within 1e-3
relative.
"""
import numpy as np
import pytest
import torch

import post_weight_quantization_33_b300 as awq
import workloads
from oracle import awq_oracle as O

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    awq.lib()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def words_u32(t):
    return host(t).view(np.uint32)


# --------------------------------------------------------------------------
# Failure path: the bounded wait expires, reports, and the context survives.
# --------------------------------------------------------------------------
def test_bounded_wait_expires_and_context_survives():
    assert awq.selftest_bounded_wait(20_000_000) == awq.AWQ_ERR_TIMEOUT
    X = cuda(np.ones((4, 64), np.float16))
    assert np.all(host(awq.stats(X)) == 1.0)


# --------------------------------------------------------------------------
# Channel statistic: exact.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T,K", [(1, 8), (17, 64), (64, 512), (333, 4104), (2048, 1024)])
def test_stats_bit_exact(T, K):
    rng = workloads.weight_rng(T * 7 + K)
    X = (rng.standard_normal((T, K)) * rng.uniform(0.01, 100, K)).astype(np.float16)
    assert np.array_equal(host(awq.stats(cuda(X))), O.channel_magnitude(X))


def test_stats_extreme_values():
    X = np.zeros((40, 64), np.float16)
    X[:, 0] = np.float16(65504.0)
    X[:, 1] = np.float16(-65504.0)
    X[:, 2] = np.float16(2.0 ** -24)          # smallest subnormal
    X[::2, 3] = np.float16(-(2.0 ** -14))     # smallest normal
    X[:, 4] = np.float16(1.0)
    assert np.array_equal(host(awq.stats(cuda(X))), O.channel_magnitude(X))


@pytest.mark.parametrize("T,K", [(31, 256), (1000, 8200), (64, 65536)])
def test_stats_across_box_edges_and_many_slabs(T, K):
    """Token counts and widths that cut the 32-token x 256-channel boxes
    (zero-filled past T and K), and a wide layer whose blocks meet several
    slabs each."""
    rng = workloads.weight_rng(T + K + 3)
    X = (rng.standard_normal((T, K)) * rng.uniform(0.01, 300, K)).astype(np.float16)
    assert np.array_equal(host(awq.stats(cuda(X))), O.channel_magnitude(X))


def test_stats_non_finite_channels():
    """An infinity (either sign) gives +inf, a NaN gives NaN, as the oracle's
    fp64 sum does; the other channels stay exact."""
    rng = workloads.weight_rng(9)
    X = rng.standard_normal((200, 1024)).astype(np.float16)
    X[3, 7] = np.float16(np.inf)
    X[150, 300] = np.float16(-np.inf)
    X[17, 511] = np.float16(np.nan)
    X[5, 600] = np.float16(np.inf)
    X[199, 600] = np.float16(np.nan)
    X[:, 900] = np.float16(np.inf)
    got = host(awq.stats(cuda(X)))
    want = O.channel_magnitude(X)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[7] == np.inf and np.isnan(got[600])


@pytest.mark.parametrize("where", ["X_nan", "X_inf", "W_inf", "W_nan"])
def test_search_rejects_non_finite_inputs(where):
    """X or W with an infinity or a NaN: every grid point's loss is then not
    finite, and the result check reports AWQ_ERR_INVALID; the context stays
    usable and the next search is correct."""
    W, X = workloads.random_layer(128, 256, 64, seed=44, outliers=(5,), factor=20.0)
    Xb, Wb = X.copy(), W.copy()
    bad = np.float16(np.nan if where.endswith("nan") else np.inf)
    if where.startswith("X"):
        Xb[10, 33] = bad
    else:
        Wb[77, 200] = bad
    res = awq.search(cuda(Xb), [cuda(Wb)], 4, 128, 20)
    with pytest.raises(awq.AwqError) as e:
        res.check()
    assert e.value.status == awq.AWQ_ERR_INVALID
    assert "non-finite" in str(e.value)
    res.free()
    _compare_search(X, [W], 4, 128)


# --------------------------------------------------------------------------
# Scales.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n_grid", [5, 20, 64])
@pytest.mark.parametrize("K", [1, 100, 4096, 11008, 65536])
def test_scales_match_oracle(K, n_grid):
    """s equal, bit for bit, to the oracle's fp32 rounding of its fp64 power,
    at every grid point: both sides stay far within half an fp32 ulp of the
    exact value (the GPU's log/exp recurrence to about 2^-47 relative), so
    they round alike except within ~2^-23 of a rounding boundary -- measured
    on a B300: no value differs in 21.5 million (these inputs and two more
    seeds)."""
    rng = workloads.weight_rng(K)
    sX = np.exp(rng.uniform(-3, 5, K))
    if K > 4:
        sX[:3] = [0.0, 1e-7, 1e-4]
    s = host(awq.scales(cuda(sX), n_grid))
    assert np.all(s[0] == 1.0)
    for i, a in enumerate(O.alpha_grid(n_grid)):
        want = O.scale_vector(sX, a)
        assert np.array_equal(s[i], want), (i, int(np.sum(s[i] != want)))


# --------------------------------------------------------------------------
# Quantize + pack: bit-exact.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("zp", [True, False], ids=["asym", "sym"])
@pytest.mark.parametrize("bits,group", [(4, 128), (4, 64), (3, 128), (3, 64), (4, -1), (3, -1)])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (300, 1024), (129, 4096)])
def test_quantize_pack_bit_exact(bits, group, N, K, zp):
    rng = workloads.weight_rng(N * 31 + K + bits * 7 + group + 3 * zp)
    W = (rng.standard_t(4, (N, K)) * 0.02).astype(np.float16)
    W[0, :(K if group == -1 else group)] = 0          # a constant (all-zero) group
    if N > 2:
        W[1, :64] = np.abs(W[1, :64]) + np.float16(0.01)    # an all-positive stretch
        W[2] = -np.abs(W[2]) - np.float16(0.01)             # an all-negative row
    s = np.exp(rng.uniform(-1.5, 1.5, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, group, zero_point=zp)
    oc, osc, oz = O.quantize_groups(W, s, bits, group, zero_point=zp)
    assert np.array_equal(words_u32(codes).reshape(N, -1), O.pack_codes(oc, bits))
    assert np.array_equal(host(sc).view(np.uint16), osc.view(np.uint16))
    assert np.array_equal(host(z), oz)


def test_quantize_pack_empty():
    W = torch.empty((0, 128), dtype=torch.float16, device="cuda")
    s = torch.ones(128, dtype=torch.float32, device="cuda")
    codes, sc, z = awq.quantize_pack(W, s, 4, 128)
    assert codes.numel() == 0 and sc.numel() == 0 and z.numel() == 0


@pytest.mark.parametrize("bits", [3, 4])
def test_unpack_roundtrip(bits):
    rng = workloads.weight_rng(40 + bits)
    q = rng.integers(0, 1 << bits, (37, 512)).astype(np.uint8)
    packed = O.pack_codes(q, bits).reshape(-1).view(np.int32)
    got = host(awq.unpack_codes(cuda(packed), 37, 512, bits))
    assert np.array_equal(got, q)


# --------------------------------------------------------------------------
# Deploy: fold diag(s)^-1 into the producer of the layer's input: bit-exact.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1,), (4096,), (11008,), (64, 256), (300, 13), (7, 8200)])
def test_fold_bit_exact(shape):
    rng = workloads.weight_rng(sum(shape) + len(shape))
    V = (rng.standard_normal(shape) * rng.uniform(0.01, 10)).astype(np.float16)
    s = np.exp(rng.uniform(-4, 4, shape[0])).astype(np.float32)
    got = host(awq.fold_scale(cuda(V), cuda(s)))
    assert np.array_equal(got.view(np.uint16), O.fold_inverse_scale(V, s).view(np.uint16))


def test_fold_in_place_and_misaligned():
    rng = workloads.weight_rng(5150)
    V = rng.standard_normal((33, 24)).astype(np.float16)
    s = np.exp(rng.uniform(-2, 2, 33)).astype(np.float32)
    want = O.fold_inverse_scale(V, s)
    t = cuda(V)
    awq.fold_scale(t, cuda(s), out=t)                    # in place
    assert np.array_equal(host(t).view(np.uint16), want.view(np.uint16))
    # a 2-byte offset view: not 16-byte aligned, takes the scalar path
    flat = cuda(np.concatenate([np.zeros(1, np.float16), V.reshape(-1)]))
    Vm = flat[1:].view(33, 24)
    got = host(awq.fold_scale(Vm, cuda(s)))
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_fold_after_search_keeps_layer_output():
    """A norm weight folded with the chosen s, the quantized layer at that s:
    deq(Q(W diag(s))) applied to the folded activations approximates W x,
    and equals the search's own error path (W - deq/s) x within rounding."""
    t = workloads.generate("tiny")
    W, X = t["W"], t["X"]
    res = awq.search(cuda(X), [cuda(W)], 4, 128, 20)
    res.check()
    s = host(res.s())
    gamma = workloads.weight_rng(7).uniform(0.5, 1.5, W.shape[1]).astype(np.float16)
    g2 = host(awq.fold_scale(cuda(gamma), cuda(s)))
    assert np.array_equal(g2.view(np.uint16), O.fold_inverse_scale(gamma, s).view(np.uint16))
    codes = O.unpack_codes(words_u32(res.codes()).reshape(W.shape[0], -1), 4, W.shape[1])
    deq = O.dequantize_scaled(codes, host(res.scales()), host(res.zeros()), 128)
    x = X.astype(np.float64)
    y_ref = W.astype(np.float64) @ (gamma.astype(np.float64) * x).T
    y_dep = deq @ (g2.astype(np.float64) * x).T
    rel = np.linalg.norm(y_dep - y_ref) / np.linalg.norm(y_ref)
    assert rel < 0.2            # INT4 g128: a few percent of the output norm
    res.free()


# --------------------------------------------------------------------------
# Decode product with the packed layer (W4A16 / W3A16): within a derived
# fp32 rounding bound.
# --------------------------------------------------------------------------
def _matvec_bound(codes, sc, z, group, x):
    """Every product (code - zero) * x is exact in fp32 (a 4-bit integer
    times an fp16 value).  A group of g channels is summed in fp32 on the
    tensor cores (at most g additions, each off by at most 2^-23 of the sum of
    magnitudes so far), scaled once, and added to the row's running sum (one
    addition per group), and at most two partial results meet in y.  So
    |y - y_exact| <= (g + K/g + 4) * 2^-23 * sum_k |deq_k x_k|."""
    K = codes.shape[1]
    g = K if group == -1 else group
    deq = O.dequantize_scaled(codes, sc, z, group)
    mag = np.abs(x.astype(np.float64)) @ np.abs(deq).T
    return (g + K / g + 4) * 2.0 ** -23 * mag


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("M", [1, 2, 8, 9, 16])
@pytest.mark.parametrize("N,K,group", [(1, 128, 128), (37, 256, 64), (300, 1024, 128),
                                       (129, 4096, -1), (64, 11008, 64), (50, 1408, 128),
                                       # 16 groups per row: parameters by TMA
                                       (300, 2048, 128), (40, 1024, 64),
                                       # K % 128 == 64: 64-channel units
                                       (45, 704, 64), (33, 192, -1)])
def test_decode_product(M, N, K, group, bits):
    rng = workloads.weight_rng(M * 100 + N + K + group + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, group)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, cuda(x), group, bits=bits))
    oc, osc, oz = O.quantize_groups(W, s, bits, group)
    want = O.w4a16_matvec(oc, osc, oz, group, x)
    err = np.abs(y.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, group, x) + 1e-30), float(err.max())


@pytest.mark.parametrize("bits", [4, 3])
def test_decode_product_large_and_deterministic(bits):
    """A 70B-class MLP shape (K = 28672) at 16 tokens, where every warp's
    range spans tile boundaries: within the bound, and identical on a
    second run (at most two partial sums meet in an output)."""
    rng = workloads.weight_rng(4242 + bits)
    N, K, M = 520, 28672, 16
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.ones(K, np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, 128)
    x = rng.standard_normal((M, K)).astype(np.float16)
    xd = cuda(x)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, xd, 128, bits=bits))
    y2 = host(awq.w4a16_matvec(codes, sc, z, N, K, xd, 128, bits=bits))
    assert np.array_equal(y, y2)
    oc, osc, oz = O.quantize_groups(W, s, bits, 128)
    want = O.w4a16_matvec(oc, osc, oz, 128, x)
    err = np.abs(y.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, 128, x) + 1e-30)


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("M,N,K,group", [(8, 50, 12416, 64), (8, 40, 12352, 64),
                                         (16, 30, 6208, -1), (5, 20, 40064, 128)])
def test_decode_product_x_through_l1(M, N, K, group, bits):
    """M x K fp16 above the 192 KiB staged in shared memory: x is read
    through L1 and permuted in registers (128- and 64-channel units, 8 and
    16 tokens)."""
    rng = workloads.weight_rng(M + N + K + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, group)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, cuda(x), group, bits=bits))
    oc, osc, oz = O.quantize_groups(W, s, bits, group)
    want = O.w4a16_matvec(oc, osc, oz, group, x)
    err = np.abs(y.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, group, x) + 1e-30), float(err.max())


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("M,N,K,group,unaligned", [
    (8, 300, 8192, 128, False), (6, 2048, 8192, 64, False), (7, 37, 8192, -1, False),
    (5, 520, 12288, 128, False), (8, 17, 8192, 128, False), (8, 100, 9216, 128, False),
    (8, 70, 8192, 64, True),
    # 9-16 tokens (8 warps, two MMAs of 8 tokens per step)
    (16, 300, 8192, 128, False), (10, 37, 12288, -1, False), (12, 2048, 8192, 64, False),
    (12, 100, 9216, 128, False), (16, 70, 8192, 64, True), (16, 17, 8192, 128, False)])
def test_decode_product_split_k(M, N, K, group, unaligned, bits):
    """M x K fp16 too large for shared memory but half of it fits (K a
    multiple of 1024), at 5-8 and 9-16 tokens: half the blocks take the first K/2 channels,
    half the rest, over whole row tiles (2 row tiles upwards, ragged N; parameters by
    TMA, by vector loads (72 groups per row), one by one (unaligned arrays),
    and whole-row groups): within the bound, and identical on a second run."""
    rng = workloads.weight_rng(M * 7 + N + K + group + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, group)
    if unaligned:
        zbuf = torch.zeros(z.numel() + 1, dtype=z.dtype, device=z.device)
        zbuf[1:] = z.reshape(-1)
        sbuf = torch.zeros(sc.numel() + 1, dtype=sc.dtype, device=sc.device)
        sbuf[1:] = sc.reshape(-1)
        z, sc = zbuf[1:], sbuf[1:]
    x = rng.standard_normal((M, K)).astype(np.float16)
    xd = cuda(x)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, xd, group, bits=bits))
    assert np.array_equal(y, host(awq.w4a16_matvec(codes, sc, z, N, K, xd, group, bits=bits)))
    oc, osc, oz = O.quantize_groups(W, s, bits, group)
    want = O.w4a16_matvec(oc, osc, oz, group, x)
    err = np.abs(y.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, group, x) + 1e-30), float(err.max())


@pytest.mark.parametrize("bits", [4, 3])
@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("N,K,group", [(18981, 1024, 128), (19000, 1152, 64),
                                       (20000, 1280, -1)])
def test_decode_product_many_tiles(M, N, K, group, bits):
    """About 1200 row tiles of 16 over the SMs (ragged N; 8, 9 and 10 units
    per row, so ranges start and end mid-tile; three group layouts, x staged
    or split in halves): within the bound, and identical on a second run."""
    rng = workloads.weight_rng(M * 11 + N + K + group + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, group)
    x = rng.standard_normal((M, K)).astype(np.float16)
    xd = cuda(x)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, xd, group, bits=bits))
    assert np.array_equal(y, host(awq.w4a16_matvec(codes, sc, z, N, K, xd, group, bits=bits)))
    oc, osc, oz = O.quantize_groups(W, s, bits, group)
    want = O.w4a16_matvec(oc, osc, oz, group, x)
    err = np.abs(y.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, group, x) + 1e-30), float(err.max())


@pytest.mark.parametrize("bits", [4, 3])
def test_decode_product_unaligned_group_parameters(bits):
    """Zeros at an odd address and scales at 2 mod 4 (slices of larger
    buffers): 64-channel groups are then read one at a time (64-channel
    units, so another split of the work and another fp32 rounding order than
    from aligned copies): within the bound, and deterministic."""
    rng = workloads.weight_rng(515 + bits)
    N, K, M = 70, 1024, 3
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), bits, 64)
    zbuf = torch.zeros(z.numel() + 1, dtype=z.dtype, device=z.device)
    zbuf[1:] = z.reshape(-1)
    sbuf = torch.zeros(sc.numel() + 1, dtype=sc.dtype, device=sc.device)
    sbuf[1:] = sc.reshape(-1)
    zu, su = zbuf[1:], sbuf[1:]
    assert zu.data_ptr() % 2 == 1 and su.data_ptr() % 4 == 2
    x = cuda(rng.standard_normal((M, K)).astype(np.float16))
    y_un = host(awq.w4a16_matvec(codes, su, zu, N, K, x, 64, bits=bits))
    assert np.array_equal(y_un, host(awq.w4a16_matvec(codes, su, zu, N, K, x, 64, bits=bits)))
    oc, osc, oz = O.quantize_groups(W, s, bits, 64)
    xh = x.cpu().numpy()
    want = O.w4a16_matvec(oc, osc, oz, 64, xh)
    err = np.abs(y_un.astype(np.float64) - want)
    assert np.all(err <= _matvec_bound(oc, osc, oz, 64, xh) + 1e-30), float(err.max())


def test_decode_product_symmetric_codes():
    """Symmetric codes (zero point 2^(b-1)) use the same product."""
    rng = workloads.weight_rng(77)
    N, K = 200, 512
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.ones(K, np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W), cuda(s), 4, 64, zero_point=False)
    x = rng.standard_normal((5, K)).astype(np.float16)
    y = host(awq.w4a16_matvec(codes, sc, z, N, K, cuda(x), 64))
    oc, osc, oz = O.quantize_groups(W, s, 4, 64, zero_point=False)
    want = O.w4a16_matvec(oc, osc, oz, 64, x)
    assert np.all(np.abs(y - want) <= _matvec_bound(oc, osc, oz, 64, x) + 1e-30)


# --------------------------------------------------------------------------
# Reference GEMM Y = W X^T (tcgen05).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N,T,K", [(128, 256, 64), (1, 1, 64), (200, 300, 192), (256, 64, 512),
                                   (1000, 1000, 1024), (384, 520, 4096)])
def test_reference_output(N, T, K):
    rng = workloads.weight_rng(N + T + K)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    X = rng.standard_normal((T, K)).astype(np.float16)
    Y = host(awq.reference_output(cuda(W), cuda(X)))
    W64, X64 = W.astype(np.float64), X.astype(np.float64)
    want = W64 @ X64.T
    mag = np.abs(W64) @ np.abs(X64).T
    err = np.abs(Y - want)
    assert np.all(err <= 1e-6 * mag + 1e-30), float((err / (mag + 1e-30)).max())


# --------------------------------------------------------------------------
# Full search vs the oracle.
# --------------------------------------------------------------------------
def _argmin_ok(gpu_best, oracle_losses):
    ob = int(np.argmin(oracle_losses))
    if gpu_best == ob:
        return True
    order = np.argsort(oracle_losses)
    lo, second = oracle_losses[order[0]], oracle_losses[order[1]]
    close = (second - lo) <= LOSS_RTOL * lo
    return close and gpu_best in (order[0], order[1])


def _compare_search(X, Ws, bits, group, n_grid=20, rows_rtol=LOSS_RTOL, zero_point=True, gram=False):
    res = awq.search(cuda(X), [cuda(W) for W in Ws], bits, group, n_grid, zero_point=zero_point,
                     gram=gram)
    res.check()
    ref = O.search(X, Ws, bits, group, n_grid, zero_point=zero_point)
    losses = res.losses
    np.testing.assert_allclose(losses, ref["losses"], rtol=LOSS_RTOL, atol=0)
    assert _argmin_ok(res.best, ref["losses"]), (res.best, ref["losses"])
    assert res.best == O.first_argmin(losses)
    assert res.alpha == res.best / n_grid
    s_best = host(res.s())
    s_grid = host(res.s_grid())
    assert np.array_equal(s_grid, ref["s_grid"])
    assert np.array_equal(s_best, s_grid[res.best])
    rl = host(res.row_losses())
    off = 0
    for i, W in enumerate(Ws):
        n = W.shape[0]
        np.testing.assert_allclose(rl[:, off:off + n], ref["row_losses"][i], rtol=rows_rtol,
                                   atol=1e-12 * max(1.0, float(ref["row_losses"][i].max())))
        off += n
        # codes at the GPU's alpha, bit-exact against the oracle quantizer fed the GPU's s
        oc, osc, oz = O.quantize_groups(W, s_best, bits, group, zero_point)
        assert np.array_equal(words_u32(res.codes(i)).reshape(n, -1), O.pack_codes(oc, bits))
        assert np.array_equal(host(res.scales(i)).view(np.uint16), osc.view(np.uint16))
        assert np.array_equal(host(res.zeros(i)), oz)
    # and the loss vector is the normalised sum of the row losses
    tot = np.zeros(n_grid)
    off = 0
    T = X.shape[0]
    for W in Ws:
        n = W.shape[0]
        tot += rl[:, off:off + n].sum(axis=1) / (n * T)
        off += n
    np.testing.assert_allclose(losses, tot, rtol=1e-12)
    res.free()
    return ref


def test_search_tiny_workload():
    t = workloads.generate("tiny")
    ref = _compare_search(t["X"], [t["W"]], 4, 128)
    assert ref["best"] > 0


@pytest.mark.parametrize("bits,group,zp", [(4, 128, False), (4, -1, True), (4, -1, False),
                                          (3, 64, False), (3, -1, True)],
                         ids=lambda v: str(v))
def test_search_quantizer_modes_tiny(bits, group, zp):
    """The AwqConfig knobs beyond the default: symmetric (zero_point false)
    and one group per output row (group_size -1)."""
    t = workloads.generate("tiny")
    _compare_search(t["X"], [t["W"]], bits, group, zero_point=zp)


@pytest.mark.parametrize("T", [64, 77, 1024])
def test_search_gram_form(T):
    """The loss in its Gram form d^T (X^T X) d (awq_search_layer_gram): the
    same losses within 1e-3, the same argmin rule, codes bit-exact at the
    GPU's alpha -- for T below, at and above K (ragged T pads X^T)."""
    W, X = workloads.random_layer(200, 512, T, seed=700 + T, outliers=(5, 300), factor=30.0)
    _compare_search(X, [W], 4, 128, gram=True)


def test_search_gram_form_tiny_and_two_weights():
    t = workloads.generate("tiny")
    _compare_search(t["X"], [t["W"]], 4, 128, gram=True)
    Ws = []
    X = None
    for j, n in enumerate((130, 60)):
        W, X0 = workloads.random_layer(n, 256, 300, seed=310 + j, outliers=(3, 200), factor=40.0)
        Ws.append(W)
        X = X0 if X is None else X
    _compare_search(X, Ws, 3, 64, gram=True, zero_point=False)


def test_search_per_row_two_weights_ragged():
    Ws = []
    X = None
    for j, n in enumerate((130, 60)):
        W, X0 = workloads.random_layer(n, 256, 77, seed=300 + j, outliers=(3, 200), factor=30.0)
        Ws.append(W)
        X = X0 if X is None else X
    _compare_search(X, Ws, 4, -1, zero_point=False)
    _compare_search(X, Ws, 3, -1, zero_point=True)


@pytest.mark.parametrize("case", [
    dict(N=(1,), K=128, T=64, bits=4, group=128),
    dict(N=(200,), K=256, T=300, bits=4, group=128),
    dict(N=(130, 60), K=256, T=77, bits=4, group=64),
    dict(N=(96,), K=512, T=40, bits=3, group=64),
    dict(N=(128,), K=384, T=256, bits=3, group=128),
    dict(N=(256,), K=64, T=513, bits=4, group=64),
], ids=lambda c: f"N{c['N']}-K{c['K']}-T{c['T']}-b{c['bits']}-g{c['group']}")
def test_search_edge_shapes(case):
    Ws = []
    X = None
    for j, n in enumerate(case["N"]):
        W, X0 = workloads.random_layer(n, case["K"], case["T"], seed=100 + j + n,
                                       outliers=(1, case["K"] // 2), factor=25.0)
        Ws.append(W)
        X = X0 if X is None else X
    _compare_search(X, Ws, case["bits"], case["group"])


def test_search_single_row_single_token_within_rounding_bound():
    """N = T = 1: the loss of each grid point is one squared dot product
    E = sum_k delta_k x_k, which can cancel to almost nothing, so a relative
    bar does not apply.  The residual is rounded to fp16 (|error| <= 2^-11 of
    each term) and accumulated in fp32, so |E_gpu - E| <= B with
    B = (2^-11 + K 2^-23) * sum_k |delta_k x_k|; check |sqrt(loss)| within B."""
    W, X = workloads.random_layer(1, 128, 1, seed=101, outliers=(1, 64), factor=25.0)
    res = awq.search(cuda(X), [cuda(W)], 4, 128)
    res.check()
    ref = O.search(X, [W], 4, 128)
    s_grid = host(res.s_grid())
    for a in range(20):
        c, sc, z = O.quantize_groups(W, s_grid[a], 4, 128)
        delta = W.astype(np.float64) - O.dequantize_scaled(c, sc, z, 128) / s_grid[a].astype(
            np.float64)
        mag = float(np.abs(delta[0] * X[0].astype(np.float64)).sum())
        bound = (2.0 ** -11 + 128 * 2.0 ** -23) * mag
        assert abs(np.sqrt(res.losses[a]) - np.sqrt(ref["losses"][a])) <= bound, a
    res.free()


def test_search_degenerate_inputs():
    rng = workloads.weight_rng(77)
    W = (rng.standard_normal((64, 256)) * 0.02).astype(np.float16)
    W[:5] = 0                                  # all-zero rows: exact, zero loss
    X = rng.standard_normal((50, 256)).astype(np.float16)
    X[:, 7] = 0                                # a dead input channel (sX = 0)
    X[:, 200] *= np.float16(300)               # a huge outlier channel
    _compare_search(X, [W], 4, 128)


def test_search_given_sx_and_small_grid():
    W, X = workloads.random_layer(128, 256, 64, seed=5, outliers=(9,), factor=40.0)
    sX = O.channel_magnitude(X)
    res = awq.search(cuda(X), [cuda(W)], 4, 128, n_grid=5, sX=cuda(sX))
    res.check()
    ref = O.search(X, [W], 4, 128, n_grid=5, sX=sX)
    np.testing.assert_allclose(res.losses, ref["losses"], rtol=LOSS_RTOL)
    res.free()


def test_search_weight_magnitude_ablation():
    """Weight-magnitude saliency (the pages' ablation): the statistic entry
    point applied to W gives the mean |W| of each input channel, which the
    search takes in place of the activation statistic."""
    t = workloads.generate("tiny")
    W, X = cuda(t["W"]), cuda(t["X"])
    sxw = awq.stats(W)
    want_sx = O.channel_magnitude(t["W"])
    assert np.array_equal(host(sxw), want_sx)
    res = awq.search(X, [W], 4, 128, 20, sX=sxw)
    res.check()
    ref = O.search(t["X"], [t["W"]], 4, 128, 20, sX=want_sx)
    np.testing.assert_allclose(res.losses, ref["losses"], rtol=LOSS_RTOL, atol=0)
    assert _argmin_ok(res.best, ref["losses"])
    res.free()


def test_search_deterministic():
    t = workloads.generate("tiny")
    a = awq.search(cuda(t["X"]), [cuda(t["W"])])
    b = awq.search(cuda(t["X"]), [cuda(t["W"])])
    assert np.array_equal(a.losses, b.losses)
    assert np.array_equal(host(a.row_losses()), host(b.row_losses()))
    assert np.array_equal(words_u32(a.codes()), words_u32(b.codes()))


def test_stage_timing_and_launch_count():
    W, X = workloads.random_layer(256, 512, 300, seed=6)
    awq.set_stage_timing(True)
    try:
        r = awq.search(cuda(X), [cuda(W)])
        r.check()
        ms = r.stage_ms()
        assert set(ms) == set(awq.STAGES) and all(v >= 0 for v in ms.values())
        assert ms["error_gemm"] > 0
        assert r.kernel_launches == 8   # 3 stats, 1 scales, 1 residual, 1 GEMM, 1 loss, 1 final
        r.free()
    finally:
        awq.set_stage_timing(False)
    r = awq.search(cuda(X), [cuda(W)])
    with pytest.raises(awq.AwqError):
        r.stage_ms()
    r.free()


def test_bad_pointers_rejected_on_gpu():
    X = cuda(np.ones((8, 128), np.float16))
    Xmis = X.view(-1)[1:1 + 8 * 64].view(8, 64)      # 2-byte offset: misaligned for TMA
    with pytest.raises(awq.AwqError) as e:
        awq.stats(Xmis)
    assert e.value.status == awq.AWQ_ERR_INVALID
    L = awq.lib()
    sx = torch.empty(128, dtype=torch.float64, device="cuda")
    host_buf = np.ones((8, 128), np.float16)
    assert L.awq_stats(host_buf.ctypes.data, 8, 128, sx.data_ptr(), None) == awq.AWQ_ERR_INVALID


# --------------------------------------------------------------------------
# Programmatic dependent launch: the calls chain their kernels to the
# stream's previous kernel and wait for it before reading their inputs, so an
# input written by the kernel just before the call must be seen.
# --------------------------------------------------------------------------
def test_inputs_written_just_before_the_call_are_seen():
    rng = workloads.weight_rng(909)
    N, K = 520, 8192
    W0 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    s = np.exp(rng.uniform(-1, 1, K)).astype(np.float32)
    codes, sc, z = awq.quantize_pack(cuda(W0), cuda(s), 4, 128)
    oc, osc, oz = O.quantize_groups(W0, s, 4, 128)
    big = torch.randn(64 << 20, device="cuda")          # a long producer kernel before each call
    # 1-3 tokens stage x whole; 5 and 8 tokens (one MMA of 8 tokens) and 16
    # (two) stage it in two halves of K.
    for it, M in enumerate((1, 2, 3, 5, 8, 16)):
        x_host = rng.standard_normal((M, K)).astype(np.float16)
        src = cuda(x_host)
        x = torch.empty_like(src)
        big.mul_(1.0)                                     # keeps the stream busy
        x.copy_(src)                                      # the producer of x, just before the call
        y = host(awq.w4a16_matvec(codes, sc, z, N, K, x, 128))
        want = O.w4a16_matvec(oc, osc, oz, 128, x_host)
        err = np.abs(y.astype(np.float64) - want)
        assert np.all(err <= _matvec_bound(oc, osc, oz, 128, x_host) + 1e-30), it
    # quantize + pack of a weight written by the previous kernel
    Wd = torch.empty(N, K, dtype=torch.float16, device="cuda")
    src = cuda(W0)
    big.mul_(1.0)
    Wd.copy_(src)
    c2, s2, z2 = awq.quantize_pack(Wd, cuda(s), 4, 128)
    assert np.array_equal(words_u32(c2), words_u32(codes))
    assert np.array_equal(host(s2).view(np.uint16), host(sc).view(np.uint16))
    # the statistic of activations written by the previous kernel
    X0 = (rng.standard_normal((4096, 1024)) * 3).astype(np.float16)
    Xd = torch.empty(4096, 1024, dtype=torch.float16, device="cuda")
    srcx = cuda(X0)
    big.mul_(1.0)
    Xd.copy_(srcx)
    assert np.array_equal(host(awq.stats(Xd)), O.channel_magnitude(X0))
