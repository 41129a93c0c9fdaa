"""kv_attend_stats against the oracle's row statistics (observer metrics of
the Catnip study): entropy support, top-k mass, structural zeros, the MXFP8
probability path and the signed-H128 MXFP8 Q/K path."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_sparse_kv_gb300 import synth


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq as k
    k.load_library()
    return k


def to_np(t):
    return t.detach().float().cpu().numpy()


def check(kvq, got, q, khat, signs, n):
    """Every row of got against O.attention_statistics over the oracle's keys
    khat[b][kv_head] (N, D)."""
    bsz, hq = q.shape[:2]
    hkv = len(khat[0])
    for b in range(bsz):
        for h in range(hq):
            ref = O.attention_statistics(q[b, h], khat[b][h // (hq // hkv)], signs)
            g = to_np(got[b, h])
            col = {name: g[:, i] for i, name in enumerate(kvq.STATS)}
            for key in ("top1", "top5", "top10", "p_tv", "p_sum", "qk_tv"):
                np.testing.assert_allclose(col[key], ref[key], atol=1e-4, rtol=0, err_msg=key)
            np.testing.assert_allclose(col["entropy"], ref["entropy"], atol=2e-4, rtol=0)
            np.testing.assert_allclose(col["support"], ref["support"], rtol=2e-4, atol=0)
            # counts: a probability on an fp32 / E4M3 boundary may land either side
            np.testing.assert_allclose(col["zero"], ref["zero"], atol=2.5 / n, rtol=0)
            np.testing.assert_allclose(col["p_zero"], ref["p_zero"], atol=3.5 / n, rtol=0)
            np.testing.assert_array_equal(col["qk_agree"], ref["qk_agree"])


def cache_case(kvq, seed, b, hkv, n, d, recent, kwin, spike=0.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((b, hkv, n, d)).astype(np.float32)
    v = rng.standard_normal((b, hkv, n, d)).astype(np.float32)
    if spike:
        k[:, :, : n // 10] *= spike   # a block of keys far above the rest: peaky rows
    k, v = O.round_to_bf16(k), O.round_to_bf16(v)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    vwin = "bf16" if kwin != "f32" else "f32"
    cache = kvq.pack(dev(k), dev(v), recent, kwin, vwin)
    # the keys as attention reads them: int4 part dequantized, window as stored
    # (an MXFP8 K window holds the MXFP8 values of the bf16 keys)
    khat = []
    for bi in range(b):
        row = []
        for h in range(hkv):
            kh, _ = O.dequantize_head(O.pack_head(k[bi, h], v[bi, h], recent,
                                                  "f32" if kwin == "f32" else "bf16"))
            if kwin == "mxfp8":
                kh[n - recent:] = O.mxfp8_round(kh[n - recent:])
            row.append(kh)
        khat.append(row)
    return cache, khat


@pytest.mark.gpu
@pytest.mark.parametrize("b,hkv,hq,n,d,recent,kwin,use_signs,spike", [
    (1, 2, 4, 700, 128, 300, "bf16", True, 0.0),     # int4 history + bf16 window, signed-H128
    (2, 1, 2, 129, 32, 129, "f32", False, 0.0),      # ragged last block of 32 keys
    (1, 2, 2, 256, 64, 256, "mxfp8", True, 0.0),     # MXFP8 K window
    (1, 1, 2, 20000, 128, 500, "bf16", True, 0.0),   # rows past shared memory, swept in place
])
def test_stats_match_oracle(kvq, b, hkv, hq, n, d, recent, kwin, use_signs, spike):
    cache, khat = cache_case(kvq, 500 + n + d, b, hkv, n, d, recent, kwin, spike)
    rng = np.random.default_rng(7 + d)
    q = O.round_to_bf16(rng.standard_normal((b, hq, 5, d)).astype(np.float32))
    if spike:
        q *= 3.0
    signs = rng.choice([-1.0, 1.0], d) if use_signs else None
    got = kvq.attend_stats(cache, torch.from_numpy(q).cuda().to(torch.bfloat16),
                           None if signs is None else torch.from_numpy(signs))
    check(kvq, got, q, khat, signs, n)


@pytest.mark.gpu
def test_stats_of_peaky_rows(kvq):
    # three identical keys far above the rest take 1/3 of the mass each (a
    # block maximum away from a power of two, so both sides round the P path
    # the same way); the other 29 keys of their block of 32 sit about 56 nats
    # lower, nonzero in fp32 but 0 on the MXFP8 P path (every other block has
    # its own scale), and the last 500 keys about 113 nats lower, 0 in fp32
    # (structural zeros)
    n, d = 1000, 128
    rng = np.random.default_rng(31)
    k = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    k[0, 0, 5:8] = 0.0
    k[0, 0, 5:8, 0] = 40.0
    k[0, 0, 500:, 0] = -40.0
    q = rng.standard_normal((1, 3, 4, d)).astype(np.float32)
    q[..., 0] = 16.0
    k, q = O.round_to_bf16(k), O.round_to_bf16(q)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(k), n, "bf16")
    signs = rng.choice([-1.0, 1.0], d)
    got = kvq.attend_stats(cache, dev(q), torch.from_numpy(signs))
    check(kvq, got, q, [[k[0, 0]]], signs, n)
    g = to_np(got)
    np.testing.assert_allclose(g[..., kvq.STATS.index("zero")], 500 / n)
    np.testing.assert_allclose(g[..., kvq.STATS.index("p_zero")], 29 / n)
    np.testing.assert_allclose(g[..., kvq.STATS.index("top1")], 1.0, atol=1e-6)


@pytest.mark.gpu
def test_stats_on_the_video_chunk_sampled_queries(kvq):
    # 32 heads, 6,240 keys [1560 | 2340 | 2340] in bf16, 4 sampled query rows per head
    q, k, v = synth.chunk_inputs_torch(13, "cuda")
    n = k.shape[2]
    cache = kvq.pack(k, v, n, "bf16")
    qs = q[:, :, ::600].contiguous()   # rows 0, 600, 1200, 1800
    signs = torch.from_numpy(np.random.default_rng(1).choice([-1.0, 1.0], 128))
    got = kvq.attend_stats(cache, qs, signs)
    kn = to_np(k)
    sel = [0, 9, 31]
    check(kvq, got[:, sel], to_np(qs)[:, sel], [[kn[0, h] for h in sel]], signs.numpy(), n)
