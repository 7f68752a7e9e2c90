"""awq_stats_noalloc: the channel statistic for callers that cannot let the
library allocate device memory (see include/awq.h).  Called through the C ABI
and compared with awq_stats, which takes its scratch from the library's pool.
The statistic is exact on both paths, so the comparison is bit for bit,
and it is also checked directly against the CPU oracle.

This file is collected last so that a stop-at-first-failure run has already
run every other test when it gets here; it also passes on its own."""
import numpy as np
import pytest
import torch

import post_weight_quantization_33_b300 as awq
import workloads
from oracle import awq_oracle as O

pytestmark = pytest.mark.gpu


def _stats_through_abi(entry: str, X: torch.Tensor) -> np.ndarray:
    L = awq.lib()
    T, K = X.shape
    sX = torch.empty(K, dtype=torch.float64, device=X.device)
    status = getattr(L, entry)(X.data_ptr(), T, K, sX.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert status == awq.AWQ_OK, L.awq_last_error().decode()
    torch.cuda.synchronize()
    return sX.cpu().numpy()


def _activations(T, K, seed, scale):
    rng = workloads.weight_rng(seed)
    return torch.from_numpy((rng.standard_normal((T, K)) * scale).astype(np.float16)).cuda()


def test_noalloc_matches_pool_version_on_two_calls_in_a_row():
    assert torch.cuda.is_available()
    # First call: a wide layer with large values, filling many scratch entries.
    X1 = _activations(300, 11008, seed=1, scale=200.0)
    # Second call: narrower, smaller values; its entries still hold the first
    # call's sums, which the entry point must clear before accumulating.
    X2 = _activations(77, 4096, seed=2, scale=0.5)
    got1 = _stats_through_abi("awq_stats_noalloc", X1)
    got2 = _stats_through_abi("awq_stats_noalloc", X2)
    assert np.array_equal(got1, _stats_through_abi("awq_stats", X1))
    assert np.array_equal(got2, _stats_through_abi("awq_stats", X2))
    # and directly against the CPU oracle's exact mean
    assert np.array_equal(got1, O.channel_magnitude(X1.cpu().numpy()))
    assert np.array_equal(got2, O.channel_magnitude(X2.cpu().numpy()))


def test_noalloc_rejects_more_channels_than_its_scratch():
    L = awq.lib()
    K = 65536 + 8
    X = torch.zeros((2, K), dtype=torch.float16, device="cuda")
    sX = torch.empty(K, dtype=torch.float64, device="cuda")
    status = L.awq_stats_noalloc(X.data_ptr(), 2, K, sX.data_ptr(), None)
    assert status == awq.AWQ_ERR_INVALID
    assert b"exceeds the fixed scratch" in L.awq_last_error()
