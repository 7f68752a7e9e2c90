"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/awq.h declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest
import torch

import post_weight_quantization_33_b300 as awq
from post_weight_quantization_33_b300 import build as awq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq.h")


@pytest.fixture(scope="module")
def L():
    awq_build.build()
    return awq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(awq_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(awq.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_bounds_checked_build_exports_the_same_interface(L):
    """libawq_checked.so (the same sources with -DAWQ_CHECK_BOUNDS) loads and
    exports every declared symbol; awq_bounds_checked tells the two apart, and
    the report of the normal build is empty (no GPU needed for either)."""
    path = awq_build.build(checked=True)
    C = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(C, name), name
    assert C.awq_bounds_checked() == 1
    assert L.awq_bounds_checked() == 0
    assert L.awq_bounds_selftest() == awq.AWQ_ERR_UNSUPPORTED


def test_no_oracle_in_library_sources():
    csrc = os.path.join(ROOT, "post_weight_quantization_33_b300")
    for dirpath, _, files in os.walk(csrc):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_version_and_status_strings(L):
    assert L.awq_abi_version() == 1
    assert L.awq_status_string(0) == b"AWQ_OK"
    assert L.awq_status_string(5) == b"AWQ_ERR_TIMEOUT"
    assert L.awq_status_string(99) == b"AWQ_ERR_UNKNOWN"


def test_packed_words(L):
    assert L.awq_packed_words(4096, 4096, 4) == 4096 * 512
    assert L.awq_packed_words(3, 4096, 3) == 3 * 384
    assert L.awq_packed_words(1, 100, 4) == -1
    assert L.awq_packed_words(1, 48, 3) == -1
    assert L.awq_packed_words(1, 64, 5) == -1
    assert L.awq_packed_words(0, 64, 4) == 0


def _cfg(bits=4, group=128, zp=1, n_grid=20):
    return ctypes.byref(awq.QConfig(bits, group, zp, n_grid))


def test_invalid_arguments_rejected_before_launch(L):
    INVALID, UNSUPPORTED = awq.AWQ_ERR_INVALID, awq.AWQ_ERR_UNSUPPORTED
    assert L.awq_stats(None, 16, 64, None, None) == INVALID
    assert b"X" in L.awq_last_error()
    assert L.awq_stats(None, 0, 64, None, None) == INVALID
    assert b"T=0" in L.awq_last_error()
    assert L.awq_stats(None, 4, 60, None, None) == INVALID
    assert L.awq_scales(None, 64, 0, None, None) == INVALID
    assert L.awq_scales(None, 64, 65, None, None) == INVALID
    assert L.awq_quantize_pack(None, 4, 256, None, _cfg(bits=5), None, None, None, None) == UNSUPPORTED
    assert L.awq_quantize_pack(None, 4, 256, None, _cfg(group=32), None, None, None, None) == UNSUPPORTED
    assert L.awq_quantize_pack(None, 4, 256, None, _cfg(zp=2), None, None, None, None) == UNSUPPORTED
    assert L.awq_quantize_pack(None, 4, 256, None, _cfg(group=-2), None, None, None, None) == UNSUPPORTED
    # one group per row needs K % 64 == 0; symmetric and per-row are accepted
    assert L.awq_quantize_pack(None, 4, 96, None, _cfg(group=-1), None, None, None, None) == INVALID
    assert L.awq_quantize_pack(None, 4, 256, None, _cfg(group=-1, zp=0), None, None, None,
                               None) == INVALID        # NULL W: reaches the pointer checks
    assert L.awq_quantize_pack(None, 4, 200, None, _cfg(), None, None, None, None) == INVALID
    assert L.awq_quantize_pack(None, 4, 256, None, None, None, None, None, None) == INVALID
    # N = 0 is a valid no-op and touches no pointer.
    assert L.awq_quantize_pack(None, 0, 256, None, _cfg(), None, None, None, None) == 0
    assert L.awq_unpack_codes(None, 2, 100, 4, None, None) == INVALID
    assert L.awq_reference_output(None, 4, None, 4, 100, None, None, None) == INVALID
    assert L.awq_w4a16_matvec(None, None, None, 4, 256, _cfg(bits=5), None, 1, None,
                              None) == UNSUPPORTED
    # 1..16 tokens; K a multiple of 64 (the product's 64-channel unit)
    assert L.awq_w4a16_matvec(None, None, None, 4, 256, _cfg(), None, 17, None, None) == INVALID
    assert b"M=17" in L.awq_last_error()
    assert L.awq_w4a16_matvec(None, None, None, 4, 256, _cfg(), None, 0, None, None) == INVALID
    assert L.awq_w4a16_matvec(None, None, None, 4, 200, _cfg(), None, 1, None, None) == INVALID
    assert L.awq_w4a16_matvec(None, None, None, 4, 96, _cfg(group=-1), None, 1, None,
                              None) == INVALID
    # INT3 codes and 16 tokens pass the argument checks (NULL codes fail next)
    assert L.awq_w4a16_matvec(None, None, None, 4, 256, _cfg(bits=3), None, 16, None,
                              None) == INVALID
    assert b"codes" in L.awq_last_error()
    assert L.awq_w4a16_matvec(None, None, None, 4, 256, _cfg(), None, 1, None, None) == INVALID
    # codes are read 16 bytes at a time: a 4-byte aligned pointer is refused
    assert L.awq_w4a16_matvec(ctypes.c_void_p(0x1004), None, None, 4, 256, _cfg(), None, 1, None,
                              None) == INVALID
    assert b"codes is not 16-byte aligned" in L.awq_last_error()
    assert L.awq_fold_scale(None, 0, 8, None, None, None) == INVALID
    assert L.awq_fold_scale(None, 8, 0, None, None, None) == INVALID
    assert L.awq_fold_scale(None, 8, 8, None, None, None) == INVALID
    assert b"V" in L.awq_last_error()
    out = ctypes.c_void_p()
    w = (awq.Weight * 1)()
    assert L.awq_search_layer(None, 16, 256, None, w, 1, _cfg(), None, None) == INVALID
    assert L.awq_search_layer(None, 0, 256, None, w, 1, _cfg(), None, ctypes.byref(out)) == INVALID
    assert L.awq_search_layer(None, 16, 256, None, w, 0, _cfg(), None, ctypes.byref(out)) == INVALID
    assert L.awq_search_layer(None, 16, 256, None, w, 17, _cfg(), None, ctypes.byref(out)) == INVALID
    assert L.awq_search_layer(None, 16, 256, None, w, 1, _cfg(n_grid=0), None,
                              ctypes.byref(out)) == INVALID
    assert out.value is None
    assert L.awq_selftest_bounded_wait(10) == INVALID
    assert L.awq_result_check(None) == INVALID
    L.awq_free(None)   # ignored


def test_statistic_token_bound(L):
    """The exact 64-bit channel sums hold at most AWQ_MAX_STAT_TOKENS tokens
    (|x| * 2^24 < 2^40 per token, the top two bits of each sum are flags):
    every entry point that computes the statistic refuses more, before
    touching its pointers; a search given sX has no such bound."""
    INVALID = awq.AWQ_ERR_INVALID
    T = awq.MAX_STAT_TOKENS + 1
    assert awq.MAX_STAT_TOKENS == 1 << 22
    for entry in ("awq_stats", "awq_stats_noalloc"):
        assert getattr(L, entry)(None, T, 64, None, None) == INVALID
        assert b"AWQ_MAX_STAT_TOKENS" in L.awq_last_error()
        assert getattr(L, entry)(None, T - 1, 64, None, None) == INVALID
        assert b"AWQ_MAX_STAT_TOKENS" not in L.awq_last_error()
    out = ctypes.c_void_p()
    w = (awq.Weight * 1)()
    assert L.awq_search_layer(None, T, 256, None, w, 1, _cfg(), None, ctypes.byref(out)) == INVALID
    assert b"AWQ_MAX_STAT_TOKENS" in L.awq_last_error()
    sx = ctypes.c_void_p(0x1000)
    assert L.awq_search_layer(None, T, 256, sx, w, 1, _cfg(), None, ctypes.byref(out)) == INVALID
    assert b"AWQ_MAX_STAT_TOKENS" not in L.awq_last_error()


def test_host_pointer_rejected(L):
    # A host buffer must be refused by the pointer check, never launched on.
    buf = (ctypes.c_char * 4096)()
    sx = (ctypes.c_double * 64)()
    st = L.awq_stats(ctypes.addressof(buf), 16, 64, ctypes.addressof(sx), None)
    assert st == awq.AWQ_ERR_INVALID
    st = L.awq_fold_scale(ctypes.addressof(buf), 64, 1, ctypes.addressof(sx),
                          ctypes.addressof(buf), None)
    assert st == awq.AWQ_ERR_INVALID


def test_binding_validates_tensors():
    X = torch.zeros((4, 64), dtype=torch.float16)
    with pytest.raises(ValueError):
        awq.stats(X)                       # CPU tensor
    with pytest.raises(TypeError):
        awq.stats(X.float())
    with pytest.raises(ValueError):
        awq.stats(torch.zeros(64, dtype=torch.float16))


def test_binding_validates_search_arguments_before_any_cuda_call():
    X = torch.zeros((8, 128), dtype=torch.float16)
    W = torch.zeros((16, 128), dtype=torch.float16)
    with pytest.raises(ValueError):
        awq.search(X, [W])                          # host tensors
    with pytest.raises(TypeError):
        awq.search(X.float(), [W])
    with pytest.raises(TypeError):
        awq.quantize_pack(W.float(), torch.ones(128))
    # the pipelined host search checks its layers on the host first
    assert awq.search_host_stream([], 4, 128) == []
    with pytest.raises(ValueError):
        awq.search_host_stream([(X, [torch.zeros((16, 64), dtype=torch.float16)])], 4, 128)
    with pytest.raises(ValueError):
        awq.search_host_stream([(X, [])], 4, 128)


def test_last_error_is_per_thread(L):
    """Two host threads fail different calls; each reads back its own message."""
    import threading
    barrier = threading.Barrier(2)
    seen = {}

    def worker(name, call, expect):
        barrier.wait()
        for _ in range(200):
            assert call() == awq.AWQ_ERR_INVALID
            msg = L.awq_last_error()
            if expect not in msg:
                seen[name] = msg
                return
        seen[name] = "ok"

    t1 = threading.Thread(target=worker, args=(
        "stats", lambda: L.awq_stats(None, 0, 64, None, None), b"T=0"))
    t2 = threading.Thread(target=worker, args=(
        "fold", lambda: L.awq_fold_scale(None, 8, 0, None, None, None), b"cols"))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert seen == {"stats": "ok", "fold": "ok"}, seen
