"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

kv_pack must match the oracle byte for byte; attention must match within
relative L2 1e-5 on the fp32 path and 1e-2 on the bf16 / MXFP8 paths (the
tolerances the workload statement fixes); region masses within 1e-4.
"""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_sparse_kv_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 1e-2
TOL_MASS = 1e-4


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq as k
    k.load_library()
    return k


def to_np(t):
    return t.detach().float().cpu().numpy()


def oracle_pack(k, v, recent, window):
    """Oracle packing of (B, H, N, D) float arrays: serialised bytes per array."""
    heads = O.pack(k, v, recent, window)
    ser = [[O.serialize_head(p) for p in row] for row in heads]
    stack = lambda key: np.stack([np.stack([s[key] for s in row]) for row in ser])  # noqa: E731
    return heads, {key: stack(key) for key in ("k_codes", "k_scales", "v_codes", "v_scales",
                                                "k_window", "v_window")}


def _bytes(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint8)


def assert_pack_bitexact(cache, ref):
    for key in ("k_codes", "k_scales", "v_codes", "v_scales"):
        got = _bytes(getattr(cache, key))
        np.testing.assert_array_equal(got.reshape(-1), ref[key].view(np.uint8).reshape(-1),
                                      err_msg=key)
    if cache.recent:
        for key in ("k_window", "v_window"):
            got = _bytes(getattr(cache, key))
            np.testing.assert_array_equal(got.reshape(-1), ref[key].view(np.uint8).reshape(-1),
                                          err_msg=key)


def bf16_cuda(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)


# ------------------------------------------------------------------ kv_pack


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("n", [128, 512])
@pytest.mark.parametrize("recent", [0, 16, 64])
def test_pack_residual_window_bitexact(kvq, seed, n, recent):
    q, k, v = synth.residual_window_batch(seed, n, 1 if n == 128 else 32)
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), recent, "f32")
    _, ref = oracle_pack(k, v, recent, "f32")
    assert_pack_bitexact(cache, ref)
    assert cache.header == [n, 32, recent, 32]
    if n == 128:
        assert cache.payload_bytes() == {0: 5136, 16: 8912, 64: 18960}[recent]


@pytest.mark.parametrize("shape,recent", [((2, 2, 100, 128), 7), ((1, 3, 65, 64), 0),
                                          ((1, 2, 33, 96), 33), ((3, 1, 31, 256), 1)])
def test_pack_ragged_bf16_bitexact(kvq, shape, recent):
    k = O.round_to_bf16(synth.normal_numpy(10, shape) * 3)
    v = O.round_to_bf16(synth.normal_numpy(11, shape))
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    _, ref = oracle_pack(k, v, recent, "bf16")
    assert_pack_bitexact(cache, ref)


def tie_heavy_bf16(seed, shape, scale=1.0):
    # normal values rounded to quarters: group maxima are small multiples of
    # 1/4, so x / scale lands on half-integers often (and a hair off them)
    return O.round_to_bf16(np.round(synth.normal_numpy(seed, shape) * 4) / 4 * scale)


@pytest.mark.parametrize("shape,recent", [((2, 2, 1100, 128), 76), ((1, 3, 333, 128), 0),
                                          ((3, 1, 40, 128), 8), ((1, 1, 31, 128), 0),
                                          ((4, 2, 4100, 128), 4), ((4, 2, 16400, 128), 16)])
@pytest.mark.parametrize("data", ["normal", "ties"])
def test_pack_bf16_d128_bitexact(kvq, shape, recent, data):
    # the fused bf16 kernel: whole and ragged last groups, one group, and
    # 4 x 2 x 512 items, so that each CTA of the grid reuses its ring of
    # shared-memory stages several times
    if data == "normal":
        k = O.round_to_bf16(synth.normal_numpy(30, shape) * 3)
        v = O.round_to_bf16(synth.normal_numpy(31, shape))
    else:
        k, v = tie_heavy_bf16(32, shape), tie_heavy_bf16(33, shape, 2.0 ** -5)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    _, ref = oracle_pack(k, v, recent, "bf16")
    assert_pack_bitexact(cache, ref)


def test_pack_bf16_d128_edge_groups_bitexact(kvq):
    # groups the reciprocal path leaves to the division (maxima below 2^-100,
    # subnormal bf16), next to zero groups, exact .5 quotients and the largest
    # finite bf16 values; one channel of a lane's four on its own
    k = np.zeros((1, 1, 160, 128), np.float32)
    k[0, 0, :32, 0] = np.arange(-16, 16) * 0.5
    k[0, 0, :32, 1] = synth.normal_numpy(40, (32,)) * np.float32(2.0 ** -110)
    k[0, 0, 32:64, 2] = synth.normal_numpy(41, (32,)) * np.float32(1e-39)   # subnormal
    k[0, 0, 32:64, 3] = np.float32(3.38e38) * np.linspace(-1, 1, 32, dtype=np.float32)
    k[0, 0, 64:96, 4:64] = synth.normal_numpy(42, (32, 60)) * np.float32(2.0 ** -99)
    k[0, 0, 96:128, 64:] = tie_heavy_bf16(43, (32, 64), 2.0 ** -120)
    k[0, 0, 128:, 5] = np.float32(2.0 ** -100)
    k[0, 0, 128:, 6] = np.float32(-(2.0 ** -101))
    k = O.round_to_bf16(k)
    v = np.ascontiguousarray(np.swapaxes(k[:, :, :128], 2, 3)).repeat(2, axis=2)[:, :, :160]
    v = O.round_to_bf16(np.ascontiguousarray(v))
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 0, "bf16")
    _, ref = oracle_pack(k, v, 0, "bf16")
    assert_pack_bitexact(cache, ref)


def test_pack_wait_runs_out_and_reports_timeout(kvq):
    # the bf16 pack loader skips one item, so the wait on it can only end by
    # its limit; afterwards a normal call packs the same cache bit-exactly
    shape = (2, 2, 700, 128)
    k = O.round_to_bf16(synth.normal_numpy(44, shape))
    v = O.round_to_bf16(synth.normal_numpy(45, shape))
    st = kvq.new_status()
    try:
        kvq.debug_set(wait_limit_ns=2_000_000, drop_item=3)
        cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 64, "bf16", status=st)
        code = kvq.read_status(st)
    finally:
        kvq.debug_set(0, -1)
    assert code & kvq.DEV_TIMEOUT
    st.zero_()
    kvq.pack(bf16_cuda(k), bf16_cuda(v), 64, "bf16", out=cache, status=st)
    assert kvq.read_status(st) == 0
    _, ref = oracle_pack(k, v, 64, "bf16")
    assert_pack_bitexact(cache, ref)


def test_pack_edge_values_bitexact(kvq):
    # zero groups, exact .5 quotients, a negative amax, tiny and huge groups
    k = np.zeros((1, 1, 96, 32), np.float32)
    k[0, 0, :32, 0] = np.arange(-16, 16) * 0.5
    k[0, 0, 32:64, 1] = -3.5
    k[0, 0, 40, 2] = 1e-30
    k[0, 0, 64:, 3] = np.linspace(-1e30, 1e30, 32)
    v = np.ascontiguousarray(np.swapaxes(k, 2, 3)[:, :, :, :32].repeat(3, axis=2))
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 0, "f32")
    _, ref = oracle_pack(k, v, 0, "f32")
    assert_pack_bitexact(cache, ref)


def test_pack_near_ties_and_tiny_scales_bitexact(kvq):
    # quotients on and a hair off half-integers (scale 1 and 2^-20), groups
    # whose scale is subnormal (its reciprocal large or infinite), and the
    # largest finite values
    k = np.zeros((1, 1, 192, 32), np.float32)
    base = np.array([2.5, 3.5, -2.5, -0.5, 0.5, 6.5, -6.5, 1.5], np.float32)
    col = np.concatenate([base, np.nextafter(base, np.float32(np.inf)),
                          np.nextafter(base, np.float32(-np.inf)), [7.0] * 8]).astype(np.float32)
    k[0, 0, :32, 0] = col
    k[0, 0, 32:64, 1] = col * np.float32(2.0 ** -20)
    k[0, 0, 64:96, 2] = col * np.float32(2.0 ** -130)     # scale 2^-130: subnormal
    k[0, 0, 96:128, 3] = col * np.float32(1e-44 / 7.0)    # scale rounds to the smallest subnormal
    k[0, 0, 128:160, 4] = np.float32(3.4e38) * np.linspace(-1, 1, 32, dtype=np.float32)
    k[0, 0, 160:, 5] = synth.normal_numpy(14, (32,)) * np.float32(1e-38)
    v = np.ascontiguousarray(np.swapaxes(k, 2, 3)[:, :, :, :192].repeat(1, axis=2))
    v = np.ascontiguousarray(np.tile(v[:, :, :, :32], (1, 1, 6, 1))[:, :, :192])
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 0, "f32")
    _, ref = oracle_pack(k, v, 0, "f32")
    assert_pack_bitexact(cache, ref)


def test_pack_mxfp8_window_bitexact(kvq):
    shape = (1, 2, 70, 128)
    k = O.round_to_bf16(synth.normal_numpy(12, shape) * np.logspace(-3, 3, 128, dtype=np.float32))
    k[0, 0, 5, :32] = 0.0
    v = O.round_to_bf16(synth.normal_numpy(13, shape))
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 70, "mxfp8", "bf16")
    codes, sb = O.mxfp8_quantize(k.astype(np.float64))
    np.testing.assert_array_equal(cache.k_window.cpu().numpy(), codes)
    np.testing.assert_array_equal(cache.k_window_e8m0.cpu().numpy(), sb)


# ------------------------------------------------------------------ fp32 attention (small D)


@pytest.mark.parametrize("variant", ["clean", "early", "recent"])
@pytest.mark.parametrize("n,heads", [(128, 1), (512, 32)])
@pytest.mark.parametrize("recent", [0, 16, 64])
def test_attend_residual_window_fp32(kvq, variant, n, heads, recent):
    for seed in range(3):
        q, k, v = synth.residual_window_batch(seed, n, heads, variant=variant)
        cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), recent, "f32")
        out, _, path = kvq.attend(cache, torch.from_numpy(q).cuda(), out_dtype="f32")
        assert path == "generic"
        ref, _ = O.attend(q, O.pack(k, v, recent, "f32"))
        assert O.rel_l2(to_np(out), ref) <= TOL_F32


def test_attend_region_mass_fp32(kvq):
    q, k, v = synth.residual_window_batch(4, 512, 4, variant="recent")
    bounds = [0, 100, 480, 496, 512]
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 16, "f32")
    out, mass, _ = kvq.attend(cache, torch.from_numpy(q).cuda(), out_dtype="f32",
                              region_bounds=bounds)
    ref, ref_mass = O.attend(q, O.pack(k, v, 16, "f32"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_F32
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)
    np.testing.assert_allclose(to_np(mass).sum(-1), 1.0, atol=1e-5)


def test_attend_sixteen_regions_fp32(kvq):
    # the fp32 kernel with the largest region count the call takes
    q, k, v = synth.residual_window_batch(5, 512, 4, variant="early")
    bounds = [0, 1, 2, 5, 16, 17, 40, 64, 100, 128, 200, 255, 256, 300, 480, 511, 512]
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), 64, "f32")
    out, mass, path = kvq.attend(cache, torch.from_numpy(q).cuda(), out_dtype="f32",
                                 region_bounds=bounds)
    assert path == "generic"
    ref, ref_mass = O.attend(q, O.pack(k, v, 64, "f32"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_F32
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)


# ------------------------------------------------------------------ decode (int4 + bf16 window)


def decode_case(seed, batch, n, hkv=2, d=128):
    q = O.round_to_bf16(synth.normal_numpy(seed, (batch, 8 * hkv, 1, d)))
    k = O.round_to_bf16(synth.normal_numpy(seed + 1, (batch, hkv, n, d)))
    v = O.round_to_bf16(synth.normal_numpy(seed + 2, (batch, hkv, n, d)))
    return q, k, v


@pytest.mark.parametrize("batch,n,recent", [(1, 1024, 128), (3, 1000, 128), (2, 333, 0),
                                            (1, 128, 128), (2, 4109, 37), (1, 40, 17)])
def test_decode_matches_oracle(kvq, batch, n, recent):
    q, k, v = decode_case(20 + n, batch, n)
    tq = bf16_cuda(q)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    ref, _ = O.attend(q, O.pack(k, v, recent, "bf16"))
    for out_dtype in ("f32", "bf16"):
        a = kvq.Attend(cache, tq, out_dtype=out_dtype)
        a.run()
        assert a.path == "decode"
        assert kvq.read_status(a.status) == 0
        err = O.rel_l2(to_np(a.out), ref)
        assert err <= TOL_BF16, err
        per_head = [O.rel_l2(to_np(a.out)[b, h], ref[b, h]) for b in range(batch) for h in range(16)]
        assert max(per_head) <= 3 * TOL_BF16


def test_decode_is_deterministic(kvq):
    q, k, v = decode_case(5, 2, 2000)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 128, "bf16")
    a = kvq.Attend(cache, bf16_cuda(q), out_dtype="f32")
    first = a.run().clone()
    second = a.run().clone()
    assert torch.equal(first, second)


# ------------------------------------------------------------------ candidates


@pytest.mark.parametrize("n,recent,c,sort", [(4096, 128, 96, True), (1000, 128, 256, False),
                                             (300, 0, 64, True), (5000, 37, 8, False)])
def test_candidates_match_oracle(kvq, n, recent, c, sort):
    batch = 2
    q, k, v = decode_case(40 + c, batch, n)
    idx = synth.candidate_indices(3, batch, 16, n, c, sort=sort)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    out, status = kvq.attend_candidates(cache, bf16_cuda(q), torch.from_numpy(idx).cuda(),
                                        out_dtype="f32")
    assert kvq.read_status(status) == 0
    ref = O.attend_candidates(q, O.pack(k, v, recent, "bf16"), idx)
    assert O.rel_l2(to_np(out), ref) <= TOL_BF16


def _cand_run(kvq, cache, tq, idx, validate=False):
    a = kvq.AttendCandidates(cache, tq, torch.from_numpy(idx).cuda(), out_dtype="f32",
                             validate=validate)
    a.run()
    return a.out, a.status, a.lib.kvq_last_path().decode()


@pytest.mark.parametrize("case", ["shared", "disjoint", "window_only", "sink_only", "c512",
                                  "one_unit_many_slices"])
def test_candidates_union_of_head_lists(kvq, case):
    # the pass over the union of a KV head's 8 lists: heads listing the same
    # keys, disjoint keys, only window keys, only the first 64 positions (every
    # later slice empty), the largest list it takes (8 x 512 rows), and one
    # (sequence, KV head) split into many slices
    rng = np.random.default_rng(hash(case) % 1000)
    batch, n, recent, c = 2, 3000, 128, 64
    if case == "c512":
        c = 512
    if case == "one_unit_many_slices":
        batch, n = 1, 20000
    q, k, v = decode_case(50 + len(case), batch, n, hkv=2 if case != "one_unit_many_slices" else 1)
    hq = q.shape[1]
    idx = np.empty((batch, hq, 1, c), dtype=np.int32)
    for b in range(batch):
        for h in range(hq):
            if case == "shared":
                base = np.random.default_rng(b * 100 + h // 8).choice(n, c, replace=False)
                idx[b, h, 0] = rng.permutation(base)
            elif case == "disjoint":
                idx[b, h, 0] = (h % 8) * c + rng.permutation(c)
            elif case == "window_only":
                idx[b, h, 0] = n - recent + rng.choice(recent, c, replace=False)
            elif case == "sink_only":
                idx[b, h, 0] = rng.permutation(64)[:c]
            else:
                idx[b, h, 0] = rng.choice(n, c, replace=False)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    out, status, path = _cand_run(kvq, cache, bf16_cuda(q), idx, validate=True)
    assert path == "candidates_union"
    assert kvq.read_status(status) == 0
    ref = O.attend_candidates(q, O.pack(k, v, recent, "bf16"), idx)
    assert O.rel_l2(to_np(out), ref) <= TOL_BF16


def test_candidates_union_flags_and_skips_bad_indices(kvq):
    # out-of-range positions are skipped and flagged; a duplicate within one
    # head's list is flagged with validate; the other rows are still exact
    q, k, v = decode_case(9, 2, 900)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 64, "bf16")
    rng = np.random.default_rng(9)
    idx = np.stack([np.stack([rng.choice(900, 48, replace=False) for _ in range(16)])
                    for _ in range(2)])[:, :, None].astype(np.int32)
    bad = idx.copy()
    bad[1, 5, 0, 7] = -3
    bad[0, 12, 0, 40] = 900
    out, status, path = _cand_run(kvq, cache, bf16_cuda(q), bad)
    assert path == "candidates_union"
    assert kvq.read_status(status) == kvq.DEV_INDEX
    packed = O.pack(k, v, 64, "bf16")
    keep = [(b, h) for b in range(2) for h in range(16) if (b, h) not in ((1, 5), (0, 12))]
    ref = O.attend_candidates(q, packed, idx)
    got = to_np(out)
    for b, h in keep:
        assert O.rel_l2(got[b, h], ref[b, h]) <= TOL_BF16
    # the flagged rows attend the remaining listed keys
    for b, h, j in ((1, 5, 7), (0, 12, 40)):
        rest = np.delete(idx[b, h, 0], j)
        kh, vh = O.dequantize_head(packed[b][h // 8])
        r = O.candidate_attention(q[b, h].astype(np.float64), kh, vh, rest[None])
        assert O.rel_l2(got[b, h], r) <= TOL_BF16
    dup = idx.copy()
    dup[0, 3, 0, 9] = dup[0, 3, 0, 2]
    _, status, _ = _cand_run(kvq, cache, bf16_cuda(q), dup, validate=True)
    assert kvq.read_status(status) & kvq.DEV_DUP


def test_candidates_over_all_keys_equal_dense(kvq):
    q, k, v = decode_case(7, 1, 700)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 64, "bf16")
    tq = bf16_cuda(q)
    perm = np.stack([np.random.default_rng(h).permutation(700) for h in range(16)])
    idx = torch.from_numpy(perm.astype(np.int32)).reshape(1, 16, 1, 700).cuda()
    out_c, _ = kvq.attend_candidates(cache, tq, idx, out_dtype="f32")
    out_d, _, _ = kvq.attend(cache, tq, out_dtype="f32")
    assert O.rel_l2(to_np(out_c), to_np(out_d)) <= TOL_BF16


def test_candidates_flag_bad_and_duplicate_indices(kvq):
    q, k, v = decode_case(8, 1, 200)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 8, "bf16")
    tq = bf16_cuda(q)
    idx = torch.arange(16, dtype=torch.int32).repeat(1, 16, 1, 1).cuda()
    idx[0, 3, 0, 5] = 200                    # out of range
    _, status = kvq.attend_candidates(cache, tq, idx)
    assert kvq.read_status(status) & kvq.DEV_INDEX
    idx[0, 3, 0, 5] = 4                      # duplicate of position 4
    _, status = kvq.attend_candidates(cache, tq, idx, validate=True)
    assert kvq.read_status(status) & kvq.DEV_DUP
    _, status = kvq.attend_candidates(cache, tq, idx, validate=False)
    assert kvq.read_status(status) == 0


# ------------------------------------------------------------------ argument errors and timeouts


def test_argument_errors_return_before_launch(kvq):
    k = torch.zeros((1, 2, 64, 32), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.pack(k, k, 65, "f32")                                            # R > N
    assert e.value.status == 1
    cache = kvq.pack(k, k, 0, "f32")
    with pytest.raises(kvq.KvqError) as e:
        kvq.attend(cache, torch.zeros((1, 3, 2, 32), device="cuda"))        # 3 q-heads, 2 KV heads
    assert e.value.status == 1
    with pytest.raises(kvq.KvqError) as e:
        kvq.attend(cache, torch.zeros((1, 2, 2, 32), device="cuda"), region_bounds=[0, 70, 64])
    assert e.value.status == 1
    with pytest.raises(ValueError):                                         # caught by the binding
        kvq.attend(cache, torch.zeros((1, 2, 2, 64), device="cuda"))
    base = torch.zeros(2 * 64 * 32 + 4, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.pack(base[1:1 + 2 * 64 * 32].view(1, 2, 64, 32), k, 0, "f32")  # 4-byte offset
    assert e.value.status == 2


def test_decode_wait_runs_out_and_reports_timeout(kvq):
    # the loader skips one item, so the wait on it can only end by its limit
    q, k, v = decode_case(9, 1, 2048)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 128, "bf16")
    a = kvq.Attend(cache, bf16_cuda(q))
    try:
        kvq.debug_set(wait_limit_ns=2_000_000, drop_item=3)
        a.run()
        st = kvq.read_status(a.status)
    finally:
        kvq.debug_set(0, -1)
    assert st & kvq.DEV_TIMEOUT
    # the context is still usable and a normal call succeeds afterwards
    a.status.zero_()
    a.run()
    assert kvq.read_status(a.status) == 0
    ref, _ = O.attend(q, O.pack(k, v, 128, "bf16"))
    assert O.rel_l2(to_np(a.out), ref) <= TOL_BF16


# ------------------------------------------------------------------ chunk attention (tcgen05)


def chunk_case(seed, heads_q, heads_kv, n_q, n_kv, concentrated=0.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, heads_q, n_q, 128))
    k = rng.standard_normal((1, heads_kv, n_kv, 128))
    v = rng.standard_normal((1, heads_kv, n_kv, 128))
    if concentrated:
        u = rng.standard_normal((1, heads_kv, 1, 128))
        u /= np.linalg.norm(u, axis=-1, keepdims=True)
        k = k + concentrated * u
        q = q + concentrated * np.repeat(u, heads_q // heads_kv, axis=1)
    return (O.round_to_bf16(q.astype(np.float32)), O.round_to_bf16(k.astype(np.float32)),
            O.round_to_bf16(v.astype(np.float32)))


@pytest.mark.parametrize("hq,hkv,n_q,n_kv,bounds,conc", [
    (2, 2, 200, 300, [0, 100, 250, 300], 0.0),
    (4, 2, 128, 128, [0, 64, 128], 0.0),
    (1, 1, 64, 1000, [0, 390, 999, 1000], 6.0),
    (2, 1, 333, 777, None, 3.0),
])
def test_chunk_bf16_matches_oracle(kvq, hq, hkv, n_q, n_kv, bounds, conc):
    q, k, v = chunk_case(60 + n_kv, hq, hkv, n_q, n_kv, conc)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "bf16")
    for out_dtype in ("f32", "bf16"):
        out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype=out_dtype, region_bounds=bounds)
        assert path == "chunk_bf16"
        ref, ref_mass = O.attend(q, O.pack(k, v, n_kv, "bf16"), region_bounds=bounds)
        err = O.rel_l2(to_np(out), ref)
        assert err <= TOL_BF16, err
        if bounds is not None:
            np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)


def test_chunk_bf16_growing_and_spiking_scores(kvq):
    # scores that grow along the keys move the softmax reference several times,
    # and a late block of keys far above everything before it (more than 2^64
    # in probability) makes the kernel recompute that tile with a new reference
    rng = np.random.default_rng(11)
    n_q, n_kv = 130, 1100
    u = rng.standard_normal(128)
    u /= np.linalg.norm(u)
    q = rng.standard_normal((1, 2, n_q, 128))
    q += (3.0 - q @ u)[..., None] * u  # every row has the same component along u
    k = rng.standard_normal((1, 1, n_kv, 128)) * (1.0 + 6.0 * np.arange(n_kv) / n_kv)[:, None]
    k[0, 0, 900:910] = 300.0 * u + 0.1 * rng.standard_normal((10, 128))
    v = rng.standard_normal((1, 1, n_kv, 128))
    q, k, v = (O.round_to_bf16(x.astype(np.float32)) for x in (q, k, v))
    bounds = [0, 500, 905, n_kv]
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_bf16"
    ref, ref_mass = O.attend(q, O.pack(k, v, n_kv, "bf16"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_BF16
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)
    # the spike takes almost all of the mass
    assert (ref_mass[..., 1:].sum(-1) > 0.99).all()


def test_chunk_bf16_full_size_sampled_heads(kvq):
    # the video chunk: 32 heads, 2,340 queries over 6,240 keys [1560 | 2340 | 2340]
    bounds = list(synth.CHUNK_REGION_BOUNDS)
    q, k, v = synth.chunk_inputs_torch(7, "cuda")
    cache = kvq.pack(k, v, bounds[-1], "bf16")
    out, mass, path = kvq.attend(cache, q, out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_bf16"
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    for h in (0, 17, 31):
        ref, _, ref_mass = O.attention(qn[0, h], kn[0, h], vn[0, h], region_bounds=bounds)
        assert O.rel_l2(to_np(out)[0, h], ref) <= TOL_BF16
        np.testing.assert_allclose(to_np(mass)[0, h], ref_mass, atol=TOL_MASS, rtol=0)
    np.testing.assert_allclose(to_np(mass).sum(-1), 1.0, atol=1e-4)


@pytest.mark.parametrize("hq,hkv,n_q,n_kv,bounds,conc", [
    # 16 regions of one latent frame each (390 keys), as the page's heatmap
    (2, 1, 200, 6240, list(synth.CHUNK_LF_BOUNDS), 3.0),
    # tiny regions: several bounds inside one 32-key chunk, a region of one
    # key, bounds on tile and chunk edges, a ragged last tile
    (2, 2, 130, 700, [0, 1, 2, 3, 31, 32, 33, 64, 100, 127, 128, 129, 300, 301, 640, 699, 700],
     0.0),
    # five regions (one more than the kernel once carried)
    (4, 2, 128, 1000, [0, 200, 390, 512, 999, 1000], 2.0),
])
def test_chunk_bf16_many_regions(kvq, hq, hkv, n_q, n_kv, bounds, conc):
    q, k, v = chunk_case(100 + len(bounds), hq, hkv, n_q, n_kv, conc)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_bf16"
    ref, ref_mass = O.attend(q, O.pack(k, v, n_kv, "bf16"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_BF16
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)
    np.testing.assert_allclose(to_np(mass).sum(-1), 1.0, atol=1e-4)


def test_chunk_bf16_many_regions_with_redone_tile(kvq):
    # the spike of the growing-scores case inside a run of 16 small regions:
    # the tile that holds it is redone with a new reference, and the region
    # sums counted during the first pass of that tile must not count twice
    rng = np.random.default_rng(12)
    n_q, n_kv = 130, 1100
    u = rng.standard_normal(128)
    u /= np.linalg.norm(u)
    q = rng.standard_normal((1, 2, n_q, 128))
    q += (3.0 - q @ u)[..., None] * u
    k = rng.standard_normal((1, 1, n_kv, 128)) * (1.0 + 6.0 * np.arange(n_kv) / n_kv)[:, None]
    k[0, 0, 900:910] = 300.0 * u + 0.1 * rng.standard_normal((10, 128))
    v = rng.standard_normal((1, 1, n_kv, 128))
    q, k, v = (O.round_to_bf16(x.astype(np.float32)) for x in (q, k, v))
    bounds = [0, 100, 200, 300, 400, 500, 600, 700, 800, 896, 901, 903, 905, 908, 960, 1024, n_kv]
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_bf16"
    ref, ref_mass = O.attend(q, O.pack(k, v, n_kv, "bf16"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_BF16
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)
    assert (ref_mass[..., 9:14].sum(-1) > 0.99).all()


def test_chunk_bf16_full_size_sixteen_frames(kvq):
    # the video chunk with one region per latent frame: each query row's 16
    # key-LF masses (the page's temporal heatmap), sampled heads
    bounds = list(synth.CHUNK_LF_BOUNDS)
    q, k, v = synth.chunk_inputs_torch(13, "cuda", concentrated=4.0)
    cache = kvq.pack(k, v, bounds[-1], "bf16")
    out, mass, path = kvq.attend(cache, q, out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_bf16"
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    for h in (0, 17, 31):
        ref, _, ref_mass = O.attention(qn[0, h], kn[0, h], vn[0, h], region_bounds=bounds)
        assert O.rel_l2(to_np(out)[0, h], ref) <= TOL_BF16
        np.testing.assert_allclose(to_np(mass)[0, h], ref_mass, atol=TOL_MASS, rtol=0)
    np.testing.assert_allclose(to_np(mass).sum(-1), 1.0, atol=1e-4)


def history_reference(q, k, v, recent, bounds):
    """Oracle attention over an int4 history + bf16 window, two ways: with the
    dequantized history exact (fp64), and with it rounded once to bf16, which is
    the operand precision the tensor-core path takes."""
    packed = O.pack(k, v, recent, "bf16")
    exact, _ = O.attend(q, packed, region_bounds=bounds)
    bsz, hq, _, _ = q.shape
    hkv = len(packed[0])
    cut = k.shape[2] - recent
    o_bf = np.empty_like(exact)
    m_bf = None if bounds is None else np.empty(exact.shape[:3] + (len(bounds) - 1,))
    for b in range(bsz):
        for h in range(hq):
            kh, vh = O.dequantize_head(packed[b][h // (hq // hkv)])
            kh[:cut] = O.round_to_bf16(kh[:cut])
            vh[:cut] = O.round_to_bf16(vh[:cut])
            o_bf[b, h], _, mb = O.attention(q[b, h], kh, vh, region_bounds=bounds)
            if bounds is not None:
                m_bf[b, h] = mb
    return exact, o_bf, m_bf


@pytest.mark.parametrize("hq,hkv,n_q,n_kv,recent,bounds,conc", [
    (2, 2, 200, 600, 250, [0, 150, 350, 600], 0.0),
    (4, 2, 130, 1000, 0, [0, 390, 999, 1000], 0.0),
    (2, 1, 333, 777, 100, None, 3.0),
    (2, 2, 130, 640, 256, [0, 100, 384, 640], 0.0),   # window starts on a key tile
])
def test_chunk_int4_history_matches_oracle(kvq, hq, hkv, n_q, n_kv, recent, bounds, conc):
    # int4 groups for the older tokens (a ragged last K group where N - R is
    # not a multiple of 32), a bf16 window for the last R, tensor-core path
    q, k, v = chunk_case(70 + n_kv, hq, hkv, n_q, n_kv, conc)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), recent, "bf16")
    exact, o_bf, m_bf = history_reference(q, k, v, recent, bounds)
    for out_dtype in ("f32", "bf16"):
        out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype=out_dtype, region_bounds=bounds)
        assert path == "chunk_int4"
        assert O.rel_l2(to_np(out), exact) <= TOL_BF16
        assert O.rel_l2(to_np(out), o_bf) <= TOL_BF16
        if bounds is not None:
            np.testing.assert_allclose(to_np(mass), m_bf, atol=TOL_MASS, rtol=0)
            np.testing.assert_allclose(to_np(mass).sum(-1), 1.0, atol=1e-4)


def test_chunk_int4_history_full_size_sampled_heads(kvq):
    # the video chunk with its sink and recent regions (3,900 tokens) in int4
    # and the current 2,340 in the bf16 window
    bounds = list(synth.CHUNK_REGION_BOUNDS)
    recent = bounds[-1] - bounds[2]
    q, k, v = synth.chunk_inputs_torch(9, "cuda")
    cache = kvq.pack(k, v, recent, "bf16")
    out, mass, path = kvq.attend(cache, q, out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_int4"
    heads = (0, 17, 31)
    qn = to_np(q)[:, heads]
    kn, vn = to_np(k)[:, heads], to_np(v)[:, heads]
    exact, o_bf, m_bf = history_reference(qn, kn, vn, recent, bounds)
    got, got_mass = to_np(out)[:, heads], to_np(mass)[:, heads]
    assert O.rel_l2(got, exact) <= TOL_BF16
    assert O.rel_l2(got, o_bf) <= TOL_BF16
    np.testing.assert_allclose(got_mass, m_bf, atol=TOL_MASS, rtol=0)


@pytest.mark.parametrize("hq,hkv,n_q,n_kv,bounds", [
    (2, 2, 200, 300, [0, 100, 250, 300]),
    (4, 2, 130, 1000, [0, 390, 999, 1000]),
    # fewer keys than one 112-key tile; one tile and one key; a ragged tail
    (2, 1, 64, 100, [0, 50, 100]),
    (1, 1, 128, 113, [0, 112, 113]),
    (3, 3, 257, 1233, [0, 1, 112, 500, 1233]),
    # 16 regions, bounds inside and on the edges of 112-key tiles
    (2, 2, 190, 1800, [0, 1, 111, 112, 113, 224, 300, 336, 390, 700, 780, 1000, 1120, 1170,
                       1500, 1799, 1800]),
])
def test_chunk_mxfp8_matches_oracle(kvq, hq, hkv, n_q, n_kv, bounds):
    q, k, v = chunk_case(80 + n_kv, hq, hkv, n_q, n_kv, 2.0)
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "mxfp8", "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_mxfp8"
    # oracle: Q and K rounded to MXFP8 (E4M3 + E8M0 per 32 features), V as given
    qc, qs = O.mxfp8_quantize(q.astype(np.float64))
    kc, ks = O.mxfp8_quantize(k.astype(np.float64))
    qh, kh = O.mxfp8_dequantize(qc, qs), O.mxfp8_dequantize(kc, ks)
    for h in range(hq):
        ref, p_mx, ref_mass = O.attention(qh[0, h], kh[0, h // (hq // hkv)], v[0, h // (hq // hkv)],
                                          region_bounds=bounds)
        assert O.rel_l2(to_np(out)[0, h], ref) <= TOL_BF16
        np.testing.assert_allclose(to_np(mass)[0, h], ref_mass, atol=TOL_MASS, rtol=0)
    # the generic fp32 kernel, which applies the same rounding, agrees too
    cache_g = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "mxfp8", "bf16")
    out_g, _, path_g = kvq.attend(cache_g, bf16_cuda(q[:, :, :63]), out_dtype="f32")
    assert path_g == "generic"
    assert O.rel_l2(to_np(out_g), to_np(out)[:, :, :63]) <= TOL_BF16


def test_chunk_mxfp8_spiking_scores(kvq):
    # a late block of keys far above the rest: the MXFP8 kernel redoes that
    # tile with a new reference, as the bf16 one does
    rng = np.random.default_rng(13)
    n_q, n_kv = 130, 1100
    u = rng.standard_normal(128)
    u /= np.linalg.norm(u)
    q = rng.standard_normal((1, 2, n_q, 128))
    q += (3.0 - q @ u)[..., None] * u
    k = rng.standard_normal((1, 1, n_kv, 128)) * (1.0 + 6.0 * np.arange(n_kv) / n_kv)[:, None]
    k[0, 0, 900:910] = 300.0 * u + 0.1 * rng.standard_normal((10, 128))
    v = rng.standard_normal((1, 1, n_kv, 128))
    q, k, v = (O.round_to_bf16(x.astype(np.float32)) for x in (q, k, v))
    bounds = [0, 500, 905, n_kv]
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), n_kv, "mxfp8", "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_mxfp8"
    qh = O.mxfp8_dequantize(*O.mxfp8_quantize(q.astype(np.float64)))
    kh = O.mxfp8_dequantize(*O.mxfp8_quantize(k.astype(np.float64)))
    for h in range(2):
        ref, _, ref_mass = O.attention(qh[0, h], kh[0, 0], v[0, 0], region_bounds=bounds)
        assert O.rel_l2(to_np(out)[0, h], ref) <= TOL_BF16
        np.testing.assert_allclose(to_np(mass)[0, h], ref_mass, atol=TOL_MASS, rtol=0)


def test_chunk_mxfp8_full_size_sampled_heads(kvq):
    # the video chunk on the MXFP8 Q/K path at full size (32 heads, 2,340
    # queries over 6,240 keys), three sampled heads against the oracle on
    # MXFP8-rounded Q and K
    bounds = list(synth.CHUNK_REGION_BOUNDS)
    q, k, v = synth.chunk_inputs_torch(21, "cuda")
    cache = kvq.pack(k, v, bounds[-1], "mxfp8", "bf16")
    out, mass, path = kvq.attend(cache, q, out_dtype="f32", region_bounds=bounds)
    assert path == "chunk_mxfp8"
    heads = (0, 17, 31)
    qn = to_np(q)[0, heads].astype(np.float64)
    kn = to_np(k)[0, heads].astype(np.float64)
    vn = to_np(v)[0, heads]
    qh = O.mxfp8_dequantize(*O.mxfp8_quantize(qn))
    kh = O.mxfp8_dequantize(*O.mxfp8_quantize(kn))
    got, got_mass = to_np(out), to_np(mass)
    for i, h in enumerate(heads):
        ref, _, ref_mass = O.attention(qh[i], kh[i], vn[i], region_bounds=bounds)
        assert O.rel_l2(got[0, h], ref) <= TOL_BF16
        np.testing.assert_allclose(got_mass[0, h], ref_mass, atol=TOL_MASS, rtol=0)
    np.testing.assert_allclose(got_mass.sum(-1), 1.0, atol=1e-4)


def test_chunk_mxfp8_changes_probabilities_little(kvq):
    # reported, not a parity pin: total variation of MXFP8 vs bf16 softmax rows
    q, k, v = chunk_case(90, 1, 1, 64, 512, 0.0)
    qc, qs = O.mxfp8_quantize(q.astype(np.float64))
    kc, ks = O.mxfp8_quantize(k.astype(np.float64))
    _, p_mx, _ = O.attention(O.mxfp8_dequantize(qc, qs)[0, 0], O.mxfp8_dequantize(kc, ks)[0, 0], v[0, 0])
    _, p_bf, _ = O.attention(q[0, 0], k[0, 0], v[0, 0])
    tv = O.probability_tv(p_mx, p_bf)
    assert np.median(tv) < 0.05


@pytest.mark.parametrize("n,heads,n_q,hq_per_kv", [(512, 4, 33, 1), (77, 2, 5, 3), (1000, 1, 40, 2)])
def test_attend_small_head_dim_kernel_edges(kvq, n, heads, n_q, hq_per_kv):
    # ragged key chunks, many or few queries, GQA, bf16 window, region masses
    rng = np.random.default_rng(n)
    q = O.round_to_bf16(rng.standard_normal((2, heads * hq_per_kv, n_q, 32)).astype(np.float32) * 2)
    k = O.round_to_bf16(rng.standard_normal((2, heads, n, 32)).astype(np.float32))
    v = O.round_to_bf16(rng.standard_normal((2, heads, n, 32)).astype(np.float32))
    bounds = [0, n // 3, n - 5, n]
    cache = kvq.pack(bf16_cuda(k), bf16_cuda(v), 21, "bf16")
    out, mass, path = kvq.attend(cache, bf16_cuda(q), out_dtype="f32", region_bounds=bounds)
    assert path == "generic"
    ref, ref_mass = O.attend(q, O.pack(k, v, 21, "bf16"), region_bounds=bounds)
    assert O.rel_l2(to_np(out), ref) <= TOL_F32
    np.testing.assert_allclose(to_np(mass), ref_mass, atol=TOL_MASS, rtol=0)


# ------------------------------------------------------------------ full-size workloads, sampled


def _unit_np(t, b, h):
    return t[b, h].float().cpu().numpy()


@pytest.mark.parametrize("batch,context", [(64, 32768), (16, 32768), (64, 8192), (1, 32768),
                                           (64, 1024), (1, 8192), (16, 1024)])
def test_decode_full_size_sampled_units(kvq, batch, context):
    # the decode workloads at full size (16 q-heads / 2 KV heads, D=128, R=128):
    # the timed step (64, 32768) and the other graded batch / context sizes,
    # through the same kernels and launch configuration, checked on sampled
    # (sequence, KV head) units
    q, k, v = synth.decode_inputs_torch(1, batch, context, "cuda")
    cache = kvq.pack(k, v, 128, "bf16")
    a = kvq.Attend(cache, q, out_dtype="bf16")
    a.run()
    assert a.path == "decode" and kvq.read_status(a.status) == 0
    out = a.out.float().cpu().numpy()
    for b, kvh in sorted({(0, 0), (min(17, batch - 1), 1), (batch - 1, 1)}):
        kn, vn = _unit_np(k, b, kvh), _unit_np(v, b, kvh)
        p = O.pack_head(kn, vn, 128, "bf16")
        ser = O.serialize_head(p)
        for key in ("k_codes", "k_scales", "v_codes", "v_scales"):
            got = getattr(cache, key)[b, kvh].cpu().numpy()
            np.testing.assert_array_equal(got.reshape(-1)[:ser[key].size],
                                          ser[key].reshape(-1), err_msg=key)
        kh, vh = O.dequantize_head(p)
        for h in range(8 * kvh, 8 * kvh + 8):
            ref, _, _ = O.attention(q[b, h].float().cpu().numpy(), kh, vh)
            assert O.rel_l2(out[b, h], ref) <= TOL_BF16


@pytest.mark.parametrize("context,c", [(131072, 256), (32768, 96), (4096, 256)])
def test_candidates_full_size_sampled_rows(kvq, context, c):
    # the candidate workloads at full size: 32 sequences, 16 q-heads / 2 KV
    # heads, the timed L=131072, C=256 and the other graded sizes
    q, k, v = synth.decode_inputs_torch(31, 32, context, "cuda")
    cache = kvq.pack(k, v, 128, "bf16")
    idx = synth.candidate_indices(5, 32, 16, context, c)
    a = kvq.AttendCandidates(cache, q, torch.from_numpy(idx).cuda(), out_dtype="f32")
    a.run()
    out, status = a.out, a.status
    assert a.lib.kvq_last_path().decode() == "candidates_union"
    assert kvq.read_status(status) == 0
    out = out.cpu().numpy()
    for b, h in ((0, 0), (9, 7), (31, 15)):
        kvh = h // 8
        kh, vh = O.dequantize_head(O.pack_head(_unit_np(k, b, kvh), _unit_np(v, b, kvh), 128, "bf16"))
        ref = O.candidate_attention(q[b, h].float().cpu().numpy(), kh, vh, idx[b, h])
        assert O.rel_l2(out[b, h], ref) <= TOL_BF16
