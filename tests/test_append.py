"""kv_append: online update of a cache laid out with reserved room.

The oracle has no separate arithmetic for it: after any sequence of appends,
the cache must hold exactly what kv_pack of the whole token sequence holds for
the window length the append rule leaves (the largest multiple of 32 of
quantized tokens that keeps at least `window` in the window). Codes, scales
and windows are compared byte for byte; attention over the appended cache is
compared with the oracle like any other cache. The CPU tests check the
argument rules, which return before any launch."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O

TOL_F32 = 1e-5
TOL_BF16 = 1e-2


def expected_recent(n, window, cut_before):
    cut = 32 * ((n - window) // 32) if n > window else 0
    return n - max(cut, cut_before)


# ------------------------------------------------------------------ host-side rules (no GPU)

@pytest.fixture(scope="module")
def lib():
    from quantized_sparse_kv_gb300 import build, kvq as k
    import os
    if not os.path.exists(k.LIB_PATH):
        build.build()
    return k


def fake_cache(k, n, recent, cap_groups, cap_window, kwin=1, vwin=1, d=128):
    # aligned placeholder addresses: the calls below fail before touching them
    p = ctypes.c_void_p(1 << 20)
    return k.KvqCacheStruct(2, 2, n, d, recent, kwin, vwin, p, p, p, p, p, p, p,
                            (ctypes.c_uint32 * 4)(0, 0, 0, 0), cap_groups, cap_window)


@pytest.mark.parametrize("case,status", [
    (dict(n=96, recent=32, cap_groups=0, cap_window=0), 3),      # tight cache
    (dict(n=96, recent=32, cap_groups=8, cap_window=40, kwin=2), 3),  # MXFP8 K window
    (dict(n=100, recent=32, cap_groups=8, cap_window=40), 3),    # padded last K group
    (dict(n=96, recent=32, cap_groups=2, cap_window=40), 4),     # no room for another group
    (dict(n=96, recent=32, cap_groups=8, cap_window=32), 4),     # no room in the window
    (dict(n=96, recent=32, cap_groups=1, cap_window=40), 1),     # reserve below the contents
])
def test_append_argument_rules(lib, case, status):
    lib.load_library()
    c = fake_cache(lib, **case)
    before = (c.n_tokens, c.recent)
    x = ctypes.c_void_p(1 << 21)
    # 33 new tokens with window 32 need one more group and 33 window rows
    got = lib.load_library().kv_append(ctypes.byref(c), x, x, 1, 33, 32, None, None)
    assert got == status
    assert (c.n_tokens, c.recent) == before


def test_append_rejects_bad_arguments(lib):
    k = lib.load_library()
    c = fake_cache(lib, 96, 32, 8, 80)
    x = ctypes.c_void_p(1 << 21)
    assert k.kv_append(ctypes.byref(c), x, x, 2, 1, 32, None, None) == 1   # MXFP8 input
    assert k.kv_append(ctypes.byref(c), x, x, 1, 0, 32, None, None) == 1   # nothing to add
    assert k.kv_append(ctypes.byref(c), None, x, 1, 1, 32, None, None) == 1
    assert k.kv_append(ctypes.byref(c), ctypes.c_void_p((1 << 21) + 8), x, 1, 1, 32, None,
                       None) == 2


def test_reserved_sizes(lib):
    s = lib.cache_sizes_reserved(2, 3, 128, lib.BF16, lib.BF16, 10, 60)
    assert s[0] == 6 * 10 * 32 * 64 and s[1] == 6 * 10 * 128 * 4
    assert s[2] == 6 * 320 * 64 and s[3] == 6 * 320 * 4 * 4
    assert s[4] == s[5] == 6 * 60 * 128 * 2 and s[6] == 0 and s[7] == 16
    with pytest.raises(lib.KvqError):
        lib.cache_sizes_reserved(2, 3, 128, lib.BF16, lib.BF16, 0, 60)


# ------------------------------------------------------------------ GPU: bit-exact with kv_pack

@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq as k
    k.load_library()
    return k


def _bytes(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8).reshape(-1)


def assert_matches_pack(cache, k, v, window_dtype):
    """The used part of every array equals the oracle's kv_pack of k, v."""
    n = cache.n_tokens
    heads = O.pack(k[:, :, :n], v[:, :, :n], cache.recent, window_dtype)
    ser = [[O.serialize_head(p) for p in row] for row in heads]
    used = cache.used()
    for key in ("k_codes", "k_scales", "v_codes", "v_scales", "k_window", "v_window"):
        ref = np.stack([np.stack([s[key] for s in row]) for row in ser])
        if ref.size == 0:
            continue
        np.testing.assert_array_equal(_bytes(used[key]), ref.view(np.uint8).reshape(-1),
                                      err_msg=f"{key} at N={n}")


def sequence(seed, b, h, n, d, dtype):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((b, h, n, d)).astype(np.float32)
    v = rng.standard_normal((b, h, n, d)).astype(np.float32)
    k[:, :, 7] *= 40.0  # a large token: its group's scales differ from the others
    if dtype == "bf16":
        k, v = O.round_to_bf16(k), O.round_to_bf16(v)
    return k, v


def to_dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


@pytest.mark.gpu
@pytest.mark.parametrize("b,h,d,window,dtype,n0,steps", [
    (2, 2, 128, 40, "bf16", 100, [1] * 40 + [5, 17, 64, 3, 1]),
    (1, 3, 64, 16, "f32", 48, [1] * 20 + [33, 2, 70]),
    (2, 1, 128, 128, "bf16", 160, [1] * 36 + [100, 1]),
    (1, 2, 32, 0, "f32", 64, [1] * 33 + [7, 40]),
    (1, 2, 256, 32, "bf16", 40, [1] * 34 + [9, 50, 1]),
])
def test_append_equals_pack_of_the_whole_sequence(kvq, b, h, d, window, dtype, n0, steps):
    total = n0 + sum(steps)
    k, v = sequence(200 + d + window, b, h, total, d, dtype)
    r0 = expected_recent(n0, window, 0)
    cap_groups = -(-total // 32)
    cache = kvq.pack(to_dev(k[:, :, :n0], dtype), to_dev(v[:, :, :n0], dtype), r0, dtype, dtype,
                     reserve=(cap_groups, window + 32 + max(steps)))
    assert_matches_pack(cache, k, v, dtype)
    n = n0
    for i, t in enumerate(steps):
        cut_before = cache.cut
        kvq.append(cache, to_dev(k[:, :, n:n + t], dtype), to_dev(v[:, :, n:n + t], dtype), window)
        n += t
        assert cache.n_tokens == n and cache.recent == expected_recent(n, window, cut_before)
        assert cache.header == [n, d, cache.recent, 32]
        if t > 1 or i % 7 == 0 or i == len(steps) - 1:
            assert_matches_pack(cache, k, v, dtype)


@pytest.mark.gpu
def test_attention_over_an_appended_cache(kvq):
    # decode (16 query heads over 2 KV heads, D = 128), candidates and a
    # multi-query call, each on the strided arrays of a cache built by appends
    b, hkv, d, window = 2, 2, 128, 64
    n0, total = 300, 700
    k, v = sequence(77, b, hkv, total, d, "bf16")
    cache = kvq.pack(to_dev(k[:, :, :n0], "bf16"), to_dev(v[:, :, :n0], "bf16"),
                     expected_recent(n0, window, 0), "bf16", "bf16",
                     reserve=(-(-total // 32), window + 64))
    n = n0
    while n < total:
        t = min(37, total - n)
        kvq.append(cache, to_dev(k[:, :, n:n + t], "bf16"), to_dev(v[:, :, n:n + t], "bf16"), window)
        n += t
    packed = O.pack(k, v, cache.recent, "bf16")
    rng = np.random.default_rng(5)
    q = O.round_to_bf16(rng.standard_normal((b, 16, 1, d)).astype(np.float32))
    a = kvq.Attend(cache, to_dev(q, "bf16"), out_dtype="f32")
    a.run()
    assert a.path == "decode"
    ref, _ = O.attend(q, packed)
    assert O.rel_l2(to_np(a.out), ref) <= TOL_BF16
    idx = np.stack([np.stack([rng.choice(total, 50, replace=False) for _ in range(16)])
                    for _ in range(b)])[:, :, None, :].astype(np.int32)
    ac = kvq.AttendCandidates(cache, to_dev(q, "bf16"), torch.from_numpy(idx).cuda(),
                              out_dtype="f32")
    ac.run()
    ref_c = O.attend_candidates(q, packed, idx)
    assert O.rel_l2(to_np(ac.out), ref_c) <= TOL_BF16
    q3 = O.round_to_bf16(rng.standard_normal((b, 4, 70, d)).astype(np.float32))
    out, _, path = kvq.attend(cache, to_dev(q3, "bf16"), out_dtype="f32")
    assert path in ("generic", "chunk_int4")
    ref3, _ = O.attend(q3, packed)
    assert O.rel_l2(to_np(out), ref3) <= TOL_BF16


def to_np(t):
    return t.detach().float().cpu().numpy()
