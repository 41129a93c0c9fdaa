"""Argument rules of the newer entry points (observer statistics, top-k and
block-shared candidates, region drop), checked on the host: every case here
returns before anything is enqueued, so no GPU is needed and nothing runs on
the placeholder addresses."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def k():
    import os
    from quantized_sparse_kv_gb300 import build, kvq
    if not os.path.exists(kvq.LIB_PATH):
        build.build()
    kvq.load_library()
    return kvq


ADDR = ctypes.c_void_p(1 << 20)   # 16-byte aligned placeholder, never dereferenced


def cache(k, n=256, d=128, recent=256, kwin=1, hkv=2, b=1):
    return k.KvqCacheStruct(b, hkv, n, d, recent, kwin, 1, ADDR, ADDR, ADDR, ADDR, ADDR, ADDR, ADDR,
                            (ctypes.c_uint32 * 4)(0, 0, 0, 0), 0, 0)


def test_stats_rules(k):
    lib = k.load_library()
    sz = ctypes.c_size_t(0)
    c = cache(k)
    # the workspace query answers with two fp32 copies of every key, in
    # 32-key tiles, and both fp32 score rows of every query row, each of the
    # four arrays rounded up to 256 bytes
    round256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for (b, hkv, n, d, hq, nq) in ((1, 2, 256, 128, 4, 8), (2, 1, 700, 64, 3, 5), (1, 4, 33, 32, 8, 1)):
        cc = cache(k, n=n, d=d, recent=n, hkv=hkv, b=b)
        assert lib.kv_attend_stats(ctypes.byref(cc), ADDR, 1, hq, nq, 0.0, None, ADDR, None,
                                   ctypes.byref(sz), None, None) == 0
        tiles = 4 * b * hkv * (-(-n // 32)) * 32 * d
        scores = 4 * b * hq * nq * n
        assert sz.value == 2 * round256(tiles) + 2 * round256(scores)
    c96 = cache(k, d=96)
    assert lib.kv_attend_stats(ctypes.byref(c96), ADDR, 1, 4, 8, 0.0, None, ADDR, None,
                               ctypes.byref(sz), None, None) == 3       # D not a power of two
    long_rows = cache(k, n=20000, recent=20000)   # rows past shared memory: swept in place
    assert lib.kv_attend_stats(ctypes.byref(long_rows), ADDR, 1, 4, 8, 0.0, None, ADDR, None,
                               ctypes.byref(sz), None, None) == 0
    big = cache(k, n=(1 << 20) + 32, recent=128)
    assert lib.kv_attend_stats(ctypes.byref(big), ADDR, 1, 4, 8, 0.0, None, ADDR, None,
                               ctypes.byref(sz), None, None) == 3       # N > 2^20
    assert lib.kv_attend_stats(ctypes.byref(c), ADDR, 1, 3, 8, 0.0, None, ADDR, None,
                               ctypes.byref(sz), None, None) == 1       # 3 q-heads over 2
    small = ctypes.c_size_t(16)
    assert lib.kv_attend_stats(ctypes.byref(c), ADDR, 1, 4, 8, 0.0, None, ADDR, ADDR,
                               ctypes.byref(small), None, None) == 4    # workspace too small


def test_topk_rules(k):
    lib = k.load_library()
    c = cache(k, recent=128)
    call = lambda cc, C, top: lib.kv_attend_candidates_topk(  # noqa: E731
        ctypes.byref(cc), ADDR, 1, 16, 1, ADDR, C, top, 0.0, ADDR, 1, None, None, None)
    assert call(c, 64, 0) == 1           # top_k < 1
    assert call(c, 64, 65) == 1          # top_k > C
    assert call(c, 5000, 32) == 3        # C beyond the sort's 4,096
    mx = cache(k, recent=128, kwin=2)
    assert call(mx, 64, 32) == 3         # MXFP8 K window


def test_block_and_region_drop_rules(k):
    lib = k.load_library()
    c = cache(k)
    sz = ctypes.c_size_t(0)
    assert lib.kv_attend_candidates_block(ctypes.byref(c), ADDR, 1, 4, 300, ADDR, 64, 0, 0.0,
                                          ADDR, 1, None, ctypes.byref(sz), None, None) == 1
    bounds = (ctypes.c_int32 * 4)(0, 60, 200, 256)
    drop = lambda mask, b=bounds, n=3: lib.kv_attend_region_drop(  # noqa: E731
        ctypes.byref(c), ADDR, 1, 4, 300, 0.0, b, n, mask, ADDR, 1, None, ctypes.byref(sz), None,
        None)
    assert drop(0b111) == 1              # nothing left
    assert drop(0b1000) == 1             # a region that does not exist
    bad = (ctypes.c_int32 * 4)(0, 60, 200, 250)
    assert drop(0b001, bad) == 1         # bounds must end at N
    d64 = cache(k, d=64)
    assert lib.kv_attend_region_drop(ctypes.byref(d64), ADDR, 1, 4, 300, 0.0, bounds, 3, 1, ADDR,
                                     1, None, ctypes.byref(sz), None, None) == 3


def test_grid_limits_are_argument_errors(k):
    # shapes whose launch grids would pass CUDA's 65,535 limit on y or z are
    # refused before anything is enqueued
    lib = k.load_library()
    sz = ctypes.c_size_t(0)
    c1 = cache(k, n=256, d=128, recent=256, hkv=1)
    assert lib.kv_attend(ctypes.byref(c1), ADDR, 1, 65536, 1, 0.0, ADDR, 1, None, 0, None, None,
                         ctypes.byref(sz), None, None) == 3
    assert lib.kv_attend_stats(ctypes.byref(c1), ADDR, 1, 65536, 1, 0.0, None, ADDR, None,
                               ctypes.byref(sz), None, None) == 3
    assert lib.kv_attend_candidates(ctypes.byref(c1), ADDR, 1, 65536, 1, ADDR, 8, 0, 0.0, ADDR,
                                    1, None, ctypes.byref(sz), None, None) == 3
    # a large but valid head count still answers the workspace query
    assert lib.kv_attend(ctypes.byref(c1), ADDR, 1, 64, 1, 0.0, ADDR, 1, None, 0, None, None,
                         ctypes.byref(sz), None, None) == 0
