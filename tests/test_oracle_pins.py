"""Pins for the fp64 oracle: what the pages print, closed forms and brute force.

Every test here runs on the CPU. Each one is chosen so that a plausible
mistake in the oracle (a wrong divisor, a transposed operand, a dropped
softmax scale, round-half-up instead of half-even, a wrong window cut) fails.
"""
import itertools
import math

import numpy as np
import pytest

from conftest import golden
from oracle import kvq_oracle as O
from quantized_sparse_kv_gb300 import synth


# ---------------------------------------------------------------- payload (page 2 table)

@pytest.mark.parametrize("recent", [0, 16, 64])
def test_payload_bytes_match_page_table(recent):
    g = golden("payload_bytes.json")
    q, k, v = synth.residual_window_inputs(0, g["n"])
    p = O.pack_head(k, v, recent, "f32")
    assert O.payload_bytes_of(p) == g["payload_bytes"][str(recent)]
    full = 2 * g["n"] * g["head_dim"] * 4
    assert full == g["full_fp32_bytes"]
    red = 100.0 * (1 - O.payload_bytes_of(p) / full)
    assert round(red, 1) == g["reduction_pct"][str(recent)]


def test_zero_window_leaves_no_tail():
    # x[-0:] would be the whole array; the cut N - R must give an empty window
    q, k, v = synth.residual_window_inputs(1, 128)
    p = O.pack_head(k, v, 0)
    assert p["k_window"].shape == (0, 32) and p["v_window"].shape == (0, 32)
    assert p["v_codes"].shape == (128, 32) and p["k_codes"].shape == (4, 32, 32)
    k_hat, v_hat = O.dequantize_head(p)
    assert k_hat.shape == (128, 32) and v_hat.shape == (128, 32)
    # all of K is quantized: no row equals its input exactly across the board
    assert not np.array_equal(k_hat, k.astype(np.float64))


def test_window_holds_exactly_the_last_r_tokens():
    q, k, v = synth.residual_window_inputs(2, 128)
    p = O.pack_head(k, v, 16)
    np.testing.assert_array_equal(p["k_window"], k[112:])
    np.testing.assert_array_equal(p["v_window"], v[112:])
    k_hat, v_hat = O.dequantize_head(p)
    np.testing.assert_array_equal(k_hat[112:], k[112:].astype(np.float64))


# ---------------------------------------------------------------- int4 quantizer

def test_quantizer_hand_case_ties_to_even():
    x = np.zeros(32, dtype=np.float32)
    x[:8] = [7.0, 3.5, 2.5, -0.5, 4.5, 5.5, -1.5, 0.25]
    codes, s = O.int4_quantize_groups(x)
    assert s == np.float32(1.0)
    assert codes[:8].tolist() == [7, 4, 2, 0, 4, 6, -2, 0]
    assert not codes[8:].any()


def test_quantizer_all_zero_group():
    codes, s = O.int4_quantize_groups(np.zeros((3, 32), dtype=np.float32))
    assert (s == 0).all() and not codes.any()
    assert not O.int4_dequantize(codes, s).any()


def test_quantizer_amax_on_negative_value():
    x = np.zeros(32, dtype=np.float32)
    x[0], x[1], x[2] = -3.5, 1.0, 0.75
    codes, s = O.int4_quantize_groups(x)
    assert s == np.float32(0.5)
    assert codes[0] == -7 and codes[1] == 2 and codes[2] == 2  # 1.5 -> 2 (even)


def test_quantizer_single_nonzero():
    x = np.zeros(32, dtype=np.float32)
    x[17] = -0.3
    codes, s = O.int4_quantize_groups(x)
    assert s == np.float32(np.float64(np.float32(0.3)) / 7.0)
    assert codes[17] == -7 and np.count_nonzero(codes) == 1


def test_quantizer_grid_values_reconstruct_exactly():
    s = 0.5
    grid = np.arange(-7, 8)
    x = np.zeros(32, dtype=np.float32)
    x[:15] = grid * s
    codes, sc = O.int4_quantize_groups(x)
    assert sc == np.float32(s)
    np.testing.assert_array_equal(O.int4_dequantize(codes, sc), x.astype(np.float64))


def _brute_codes(x, s):
    """Nearest code in [-7, 7] to the fp32 quotient, ties to the even code, by search."""
    out = []
    for xi in x:
        if s == 0:
            out.append(0)
            continue
        t = float(np.float32(xi) / np.float32(s))  # numpy fp32 division: correctly rounded
        best_d, best_c = None, None
        for c in range(-7, 8):
            d = abs(t - c)
            if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
                best_d, best_c = d, c
        out.append(best_c)
    return out


def test_quantizer_matches_brute_force_search():
    rng = np.random.default_rng(7)
    groups = [rng.standard_normal(32).astype(np.float32) * m for m in (1e-3, 0.7, 3.0, 1e4)]
    # groups built to hit exact .5 quotients
    for s in (0.25, 0.5, 2.0):
        g = (rng.integers(-14, 15, size=32) / 2.0 * s).astype(np.float32)
        g[0] = 7 * s
        groups.append(g)
    groups.append(np.full(32, -2.0, dtype=np.float32))
    for g in groups:
        codes, s = O.int4_quantize_groups(g)
        assert codes.tolist() == _brute_codes(g, s), g


def test_quantizer_error_bound_and_range():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((500, 32)) * rng.uniform(0.01, 100, (500, 1))).astype(np.float32)
    codes, s = O.int4_quantize_groups(x)
    assert codes.min() >= -7 and codes.max() <= 7
    err = np.abs(O.int4_dequantize(codes, s) - x.astype(np.float64))
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-6)).all()
    # the element that sets amax always maps to +-7
    i = np.abs(x).argmax(axis=1)
    assert (np.abs(codes[np.arange(500), i]) == 7).all()


def test_k_is_per_channel_and_v_is_per_token():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((96, 64)).astype(np.float32)
    v = rng.standard_normal((96, 64)).astype(np.float32)
    k[:, 5] *= 1000.0   # one loud channel of K
    v[7, :] *= 1000.0   # one loud token of V
    p = O.pack_head(k, v, 0)
    ks, vs = p["k_scales"], p["v_scales"]
    assert ks.shape == (3, 64) and vs.shape == (96, 2)
    assert (ks[:, 5] > 100 * np.delete(ks, 5, axis=1).max()).all()
    assert (vs[7] > 100 * np.delete(vs, 7, axis=0).max()).all()
    # a K scale is the amax of 32 consecutive tokens of one channel
    for g, c in itertools.product(range(3), (0, 5, 63)):
        amax = np.abs(k[32 * g:32 * g + 32, c]).max()
        assert ks[g, c] == np.float32(np.float64(amax) / 7.0)
    for t, j in itertools.product((0, 7, 95), range(2)):
        amax = np.abs(v[t, 32 * j:32 * j + 32]).max()
        assert vs[t, j] == np.float32(np.float64(amax) / 7.0)


def test_k_group_padding_and_unpadded_v():
    rng = np.random.default_rng(6)
    k = rng.standard_normal((100, 32)).astype(np.float32)
    v = rng.standard_normal((100, 32)).astype(np.float32)
    p = O.pack_head(k, v, 30)                     # 70 quantized tokens -> 3 K groups
    assert p["k_codes"].shape == (3, 32, 32)
    assert not p["k_codes"][2, 6:].any()          # tokens 70..95 are padding
    assert p["k_scales"][2, 0] == np.float32(np.float64(np.abs(k[64:70, 0]).max()) / 7.0)
    assert p["v_codes"].shape == (70, 32)         # V is not padded
    assert O.payload_bytes_of(p) == 3 * 32 * 16 + 3 * 32 * 4 + 70 * 16 + 70 * 4 + 2 * 30 * 32 * 4 + 16


def test_nibble_order():
    codes = np.array([[-7, 7, 0, -1]], dtype=np.int8)
    assert O.nibbles(codes).tolist() == [[0x01 | 0xF0, 0x08 | 0x70]]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5], dtype=np.float32)
    r = O.round_to_bf16(x)
    assert r.tolist() == [1.0, 1.0, 1.0 + 4 * 2 ** -8, 1.0, -2.5]


# ---------------------------------------------------------------- attention

def test_uniform_rows_give_region_masses_of_token_shares():
    g = golden("chunk_layout.json")
    b = g["region_bounds"]
    assert b[1] == 4 * g["tokens_per_lf"] and g["tokens_per_lf"] == 15 * 26
    rng = np.random.default_rng(0)
    n = b[-1]
    q = np.zeros((3, 16))
    k = rng.standard_normal((n, 16))
    v = rng.standard_normal((n, 16))
    o, p, mass = O.attention(q, k, v, region_bounds=b)
    want = [g["uniform_mass_pct"][r] / 100 for r in ("sink", "recent", "current")]
    np.testing.assert_allclose(mass, np.tile(want, (3, 1)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, np.tile(v.mean(axis=0), (3, 1)), atol=1e-12)


def test_dominant_logit_selects_its_value_row():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((20, 8))
    v = rng.standard_normal((20, 8))
    q = np.zeros((1, 8))
    q[0, 0] = 1.0
    k[:, 0] = 0.0
    k[13, 0] = 1000.0 * math.sqrt(8)   # logit of key 13 is +1000 above the rest
    o, p, _ = O.attention(q, k, v)
    np.testing.assert_allclose(o[0], v[13], atol=1e-12)
    assert p[0, 13] == 1.0


def test_rows_sum_to_one_and_masses_partition():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 32)) * 3
    k = rng.standard_normal((50, 32))
    v = rng.standard_normal((50, 32))
    o, p, mass = O.attention(q, k, v, region_bounds=[0, 7, 31, 50])
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-13)
    np.testing.assert_allclose(mass.sum(axis=1), 1.0, atol=1e-13)
    np.testing.assert_allclose(mass[:, 1], p[:, 7:31].sum(axis=1), atol=1e-15)


def _online_softmax_attention(q, k, v, scale):
    """One-pass streaming softmax with running max, in plain Python floats."""
    out = []
    for qi in q:
        m, l, acc = -math.inf, 0.0, [0.0] * len(v[0])
        for kj, vj in zip(k, v):
            s = scale * sum(a * b for a, b in zip(qi, kj))
            m_new = max(m, s)
            c = math.exp(m - m_new) if m != -math.inf else 0.0
            e = math.exp(s - m_new)
            l = l * c + e
            acc = [a * c + e * x for a, x in zip(acc, vj)]
            m = m_new
        out.append([a / l for a in acc])
    return np.array(out)


@pytest.mark.parametrize("n,d", [(1, 4), (3, 4), (8, 6)])
def test_attention_matches_streaming_brute_force(n, d):
    rng = np.random.default_rng(n * 10 + d)
    q = rng.standard_normal((3, d)) * 2
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    o, _, _ = O.attention(q, k, v)
    np.testing.assert_allclose(o, _online_softmax_attention(q, k, v, 1 / math.sqrt(d)),
                               rtol=1e-12, atol=1e-12)


def test_full_window_means_no_quantization():
    q, k, v = synth.residual_window_inputs(3, 128)
    p = O.pack_head(k, v, 128)
    assert p["k_codes"].shape == (0, 32, 32) and p["v_codes"].shape == (0, 32)
    kh, vh = O.dequantize_head(p)
    np.testing.assert_array_equal(kh, k.astype(np.float64))
    o, _, _ = O.attention(q, kh, vh)
    o_ref, _, _ = O.attention(q, k, v)
    np.testing.assert_array_equal(o, o_ref)


def test_quantized_output_differs_from_unquantized():
    # the page's guard: an exact match means the unquantized K/V went in
    q, k, v = synth.residual_window_inputs(0, 128)
    o_ref, _, _ = O.attention(q, k, v)
    kh, vh = O.dequantize_head(O.pack_head(k, v, 16))
    o, _, _ = O.attention(q, kh, vh)
    assert O.rel_l2(o, o_ref) > 0.01


# ---------------------------------------------------------------- candidates

def test_candidates_over_all_keys_equal_dense_in_any_order():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((4, 16))
    k = rng.standard_normal((40, 16))
    v = rng.standard_normal((40, 16))
    idx = np.stack([rng.permutation(40) for _ in range(4)])
    o_dense, _, _ = O.attention(q, k, v)
    np.testing.assert_allclose(O.candidate_attention(q, k, v, idx), o_dense, atol=1e-13)


def test_candidates_equal_masked_brute_force_and_ignore_order():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 6))
    k = rng.standard_normal((9, 6))
    v = rng.standard_normal((9, 6))
    idx = np.array([[0, 4, 8], [7, 1, 2], [5, 3, 6]])
    o = O.candidate_attention(q, k, v, idx)
    np.testing.assert_allclose(O.candidate_attention(q, k, v, idx[:, ::-1]), o, atol=1e-14)
    scale = 1 / math.sqrt(6)
    for i in range(3):
        s = [scale * float(q[i] @ k[j]) if j in idx[i] else -math.inf for j in range(9)]
        m = max(s)
        e = [math.exp(x - m) if x != -math.inf else 0.0 for x in s]
        want = sum(e[j] * v[j] for j in range(9)) / sum(e)
        np.testing.assert_allclose(o[i], want, atol=1e-13)


def test_batched_forms_follow_gqa_head_mapping():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 4, 3, 32)).astype(np.float32)
    k = rng.standard_normal((2, 2, 70, 32)).astype(np.float32)
    v = rng.standard_normal((2, 2, 70, 32)).astype(np.float32)
    packed = O.pack(k, v, 6)
    o, _ = O.attend(q, packed)
    kh, vh = O.dequantize_head(packed[1][1])
    o_ref, _, _ = O.attention(q[1, 3], kh, vh)   # q-head 3 of 4 reads KV head 1 of 2
    np.testing.assert_array_equal(o[1, 3], o_ref)
    idx = np.tile(np.arange(70, dtype=np.int32), (2, 4, 3, 1))
    np.testing.assert_allclose(O.attend_candidates(q, packed, idx), o, atol=1e-13)


# ---------------------------------------------------------------- MXFP8

def test_e4m3_table_definition():
    t = O.E4M3_TABLE
    finite = t[~np.isnan(t)]
    assert finite.size == 254 and np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x38] == 1.0


def _brute_e4m3(y):
    mags = O.E4M3_TABLE[:0x7F]                       # 0x00..0x7E, non-negative finite
    a = np.abs(y)[:, None]
    dist = np.abs(a - mags[None, :])
    best = dist.min(axis=1, keepdims=True)
    tie = dist == best
    even = tie & ((np.arange(0x7F) & 1) == 0)[None, :]
    pick = np.where(even.any(axis=1), even.argmax(axis=1), tie.argmax(axis=1))
    return (pick | (np.signbit(y).astype(np.int64) << 7)).astype(np.uint8)


def test_e4m3_encoder_matches_nearest_search_on_all_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    vals = O.bf16_bits_to_fp32(bits.astype(np.uint16))
    vals = vals[np.isfinite(vals)].astype(np.float64)
    vals = vals[np.abs(vals) < 2.0 ** 12]
    np.testing.assert_array_equal(O.e4m3_encode(vals), _brute_e4m3(vals))
    # exact midpoints between neighbours go to the even mantissa
    mids = (O.E4M3_TABLE[0x30:0x3F:1][:-1] + O.E4M3_TABLE[0x31:0x3F]) / 2
    np.testing.assert_array_equal(O.e4m3_encode(mids), _brute_e4m3(mids))


def test_mxfp8_block_scale_rule():
    rng = np.random.default_rng(11)
    x = O.round_to_bf16(rng.standard_normal((64, 128)) * rng.uniform(1e-3, 1e3, (64, 1)))
    codes, sb = O.mxfp8_quantize(x)
    assert codes.shape == x.shape and sb.shape == (64, 4)
    e = sb.astype(np.int64) - 127
    amax = np.abs(x.reshape(64, 4, 32)).max(axis=-1)
    ratio = amax / np.ldexp(1.0, e)
    assert ((ratio >= 256) & (ratio < 512)).all()    # block max lands in E4M3's top binade
    xh = O.mxfp8_dequantize(codes, sb)
    assert (np.abs(xh) <= 448.0 * np.ldexp(1.0, e).repeat(32, axis=1)).all()
    rel = np.abs(xh - x) / np.maximum(np.abs(x), 1e-30)
    unit = np.ldexp(1.0, e).repeat(32, axis=1)
    normal = (np.abs(x) >= unit * 2.0 ** -6) & (np.abs(x) <= 448.0 * unit)
    assert (rel[normal] <= 2.0 ** -4 + 1e-12).all()  # 3 mantissa bits: half-ulp 2^-4
    sat = np.abs(x) > 464.0 * unit                   # beyond the last midpoint: saturate
    np.testing.assert_array_equal(np.abs(xh[sat]), 448.0 * unit[sat])


def test_mxfp8_zero_block_and_exact_grid():
    x = np.zeros((1, 64))
    x[0, 32:40] = np.array([448, -448, 1.0, 0.5, -0.015625, 2 ** -9, 0, 3.5]) * 2.0 ** -5
    codes, sb = O.mxfp8_quantize(x)
    assert sb[0, 0] == 0 and not codes[0, :32].any()
    assert sb[0, 1] == 127 - 5
    np.testing.assert_array_equal(O.mxfp8_dequantize(codes, sb), x)


# ---------------------------------------------------------------- page 2 statistical bands

def _residual_protocol(variant, mode="add", boost=3.0):
    errs = {0: [], 16: [], 64: []}
    mass = []
    for seed in range(3):
        for n in (128, 512):
            q, k, v = synth.residual_window_inputs(seed, n, variant=variant, mode=mode, boost=boost)
            o_ref, p, _ = O.attention(q, k, v)
            mass.append(p[:, n - 16:].sum(axis=1).mean())
            for r in errs:
                kh, vh = O.dequantize_head(O.pack_head(k, v, r))
                o, _, _ = O.attention(q, kh, vh)
                errs[r].append(O.rel_l2(o, o_ref))
    return [100 * np.mean(errs[r]) for r in (0, 16, 64)], 100 * np.mean(mass)


def test_clean_inputs_land_in_the_page_error_band():
    row = golden("residual_window_table.json")["rows"]["clean"]
    err, mass = _residual_protocol("clean")
    for got, want in zip(err, row["rel_l2_pct"]):
        assert abs(got - want) <= 1.5, (err, row)
    assert abs(mass - row["recent16_mass_pct"]) <= 1.5
    assert err[0] > err[1] > err[2]


def test_page_matched_focus_variants():
    rows = golden("residual_window_table.json")["rows"]
    err, mass = _residual_protocol("recent", mode="set", boost=5.1)
    assert abs(mass - rows["recent"]["recent16_mass_pct"]) <= 2.0
    assert err[1] < 3.0 and err[2] <= err[1] and err[0] - err[1] > 8.0
    err, mass = _residual_protocol("early", mode="set", boost=5.1)
    assert abs(mass - rows["early"]["recent16_mass_pct"]) <= 0.5
    assert max(err) - min(err) < 0.2
    for got, want in zip(err, rows["early"]["rel_l2_pct"]):
        assert abs(got - want) <= 1.5


# ------------------------------------------------------------------ observer statistics
# (Catnip study: entropy support, top-k mass, structural and MXFP8 numerical
# zeros, P-path TV and row sum, signed-H128 + MXFP8 Q/K TV and argmax agreement)

def test_statistics_of_a_uniform_row_in_closed_form():
    n = 100
    st = O.row_statistics(np.zeros((1, n)))
    assert np.isclose(st["entropy"][0], math.log(n)) and np.isclose(st["support"][0], 1.0)
    # ceil(1 %, 5 %, 10 % of 100) = 1, 5, 10 keys of mass 1/100 each
    assert np.allclose([st["top1"][0], st["top5"][0], st["top10"][0]], [0.01, 0.05, 0.10])
    assert st["zero"][0] == 0 and st["p_zero"][0] == 0
    # 1/100 in a block whose scale is 2^(floor(log2 0.01) - 8) = 2^-15: 327.68 -> E4M3 320
    assert np.isclose(st["p_sum"][0], 100 * 320 * 2.0 ** -15)
    assert np.isclose(st["p_tv"][0], 0.5 * 100 * (0.01 - 320 * 2.0 ** -15))


def test_statistics_of_a_one_hot_row():
    n = 64
    s = np.zeros((1, n))
    s[0, 17] = 1000.0
    st = O.row_statistics(s)
    assert abs(st["entropy"][0]) < 1e-12 and np.isclose(st["support"][0], 1.0 / n)
    assert st["top1"][0] == 1.0 and st["top10"][0] == 1.0
    assert st["zero"][0] == (n - 1) / n        # e^-1000 is 0 in fp32
    assert st["p_zero"][0] == 0 and st["p_sum"][0] == 1.0 and st["p_tv"][0] == 0


def test_statistics_of_a_two_level_row():
    # k keys at score a, n - k at 0: p_hi = e^a / Z, p_lo = 1 / Z
    n, k, a = 200, 6, 3.0
    s = np.zeros((1, n))
    s[0, :k] = a
    z = k * math.exp(a) + (n - k)
    ph, pl = math.exp(a) / z, 1.0 / z
    st = O.row_statistics(s)
    h = -(k * ph * math.log(ph) + (n - k) * pl * math.log(pl))
    assert np.isclose(st["entropy"][0], h) and np.isclose(st["support"][0], math.exp(h) / n)
    assert np.isclose(st["top1"][0], 2 * ph)               # ceil(2.0) = 2 keys
    assert np.isclose(st["top5"][0], k * ph + 4 * pl)      # 10 keys
    assert np.isclose(st["top10"][0], k * ph + 14 * pl)    # 20 keys


def test_top_count_rounds_up():
    assert [O.top_count(6240, p) for p in (1, 5, 10)] == [63, 312, 624]
    assert [O.top_count(100, p) for p in (1, 5, 10)] == [1, 5, 10]
    assert O.top_count(101, 1) == 2


def test_mxfp8_round_along_a_row():
    # block max 1 -> scale 2^-8: 2^-17 is the smallest subnormal step (2^-9 * 2^-8),
    # 2^-20 rounds to 0, 0.3 * 256 = 76.8 -> 80 (step 8 in [64, 128))
    x = np.zeros(40)
    x[:4] = [1.0, 2.0 ** -20, 2.0 ** -17, 0.3]
    x[33] = 0.3                                   # partial second block, its own scale
    y = O.mxfp8_round(x)
    assert list(y[:4]) == [1.0, 0.0, 2.0 ** -17, 80 / 256]
    # its own block: scale 2^(floor(log2 0.3) - 8) = 2^-10, 307.2 -> 320 (step 32)
    assert y[33] == 320 * 2.0 ** -10


def test_numerical_zeros_of_the_p_path():
    # one dominant key and 31 at 2^-20 of it: after MXFP8 rounding (block scale
    # 2^-8) the 31 small ones are 0 although they are not 0 in fp32
    n = 32
    s = np.full((1, n), -20 * math.log(2.0))
    s[0, 0] = 0.0
    st = O.row_statistics(s)
    assert st["zero"][0] == 0 and st["p_zero"][0] == 31 / n
    pmax = 1.0 / (1.0 + 31 * 2.0 ** -20)
    assert np.isclose(st["p_sum"][0], O.mxfp8_round(np.array([pmax]))[0])


def test_qk_path_identical_and_disagreeing():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((4, 50))
    st = O.row_statistics(s, s)
    assert np.all(st["qk_tv"] == 0) and np.all(st["qk_agree"] == 1)
    s2 = s.copy()
    s2[0, np.argmin(s2[0])] = 100.0
    st2 = O.row_statistics(s, s2)
    # the spiked key takes almost all the mass on one side and little on the other
    assert st2["qk_agree"][0] == 0 and st2["qk_tv"][0] > 0.9


def test_signed_hadamard_is_orthogonal_and_keeps_dot_products():
    h = O.hadamard(128)
    assert np.array_equal(h @ h.T, 128 * np.eye(128))
    assert np.array_equal(O.hadamard(2), np.array([[1, 1], [1, -1]]))
    rng = np.random.default_rng(4)
    signs = rng.choice([-1.0, 1.0], 128)
    q, k = rng.standard_normal((3, 128)), rng.standard_normal((5, 128))
    qr, kr = O.signed_hadamard(q, signs), O.signed_hadamard(k, signs)
    assert np.allclose(qr @ kr.T, q @ k.T)
    # a spike in one channel becomes a flat vector of magnitude 1/sqrt(128)
    e = np.zeros(128)
    e[5] = 1.0
    assert np.allclose(np.abs(O.signed_hadamard(e, signs)), 1 / math.sqrt(128))
    # H / sqrt(D) undoes itself; the signs then undo themselves
    assert np.allclose(O.signed_hadamard(qr, np.ones(128)) * signs, q)


def test_attention_statistics_reference_path_ignores_the_rotation():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((2, 128)), rng.standard_normal((70, 128))
    signs = rng.choice([-1.0, 1.0], 128)
    a = O.attention_statistics(q, k, signs)
    b = O.attention_statistics(q, k, None)
    for key in ("entropy", "support", "top1", "zero", "p_zero", "p_tv", "p_sum"):
        assert np.allclose(a[key], b[key])
    assert np.all(a["qk_tv"] < 0.1) and np.all(b["qk_tv"] < 0.1)


# ------------------------------------------------------------------ exact top-k inside the candidates

def test_topk_inside_candidates_reduces_to_known_cases():
    rng = np.random.default_rng(12)
    n, d = 300, 32
    k, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    q = rng.standard_normal((3, d))
    idx = np.stack([rng.choice(n, 40, replace=False) for _ in range(3)])
    # keeping all C is plain candidate attention
    assert np.allclose(O.candidate_topk_attention(q, k, v, idx, 40),
                       O.candidate_attention(q, k, v, idx))
    # keeping one is the value row of the best-scoring listed key (brute force)
    best = [idx[i][np.argmax(k[idx[i]] @ q[i])] for i in range(3)]
    assert np.allclose(O.candidate_topk_attention(q, k, v, idx, 1), v[best])
    # the list's order does not matter
    perm = rng.permutation(40)
    assert np.allclose(O.candidate_topk_attention(q, k, v, idx[:, perm], 7),
                       O.candidate_topk_attention(q, k, v, idx, 7))
    # the kept keys are the 7 highest-scoring ones, found by brute force
    keep, _ = O.candidate_topk_select(q, k, idx, 7)
    for i in range(3):
        s = {int(t): float(k[t] @ q[i]) for t in idx[i]}
        top = sorted(s, key=lambda t: -s[t])[:7]
        assert list(keep[i]) == top


def test_topk_ties_go_to_the_key_listed_first():
    k = np.zeros((6, 32))
    k[:, 0] = [1.0, 3.0, 3.0, 2.0, 3.0, 0.0]
    q = np.zeros((1, 32))
    q[0, 0] = 1.0
    keep, _ = O.candidate_topk_select(q, k, np.array([[4, 1, 2, 0]]), 2)
    assert list(keep[0]) == [4, 1]


# ------------------------------------------------------------------ region-drop ablation

def test_full_output_is_the_mass_weighted_mix_of_region_outputs():
    # softmax over a union of disjoint key sets: O = sum_r mass_r * O_r, where
    # O_r attends region r alone -- ties the dropped-region outputs to the
    # region masses without retyping either
    rng = np.random.default_rng(21)
    bounds = [0, 39, 100, 160]
    q, k, v = rng.standard_normal((4, 32)), rng.standard_normal((160, 32)), rng.standard_normal((160, 32))
    o, _, mass = O.attention(q, k, v, region_bounds=bounds)
    mix = np.zeros_like(o)
    for r in range(3):
        keep = O.region_drop_keys(bounds, [x for x in range(3) if x != r])
        o_r = O.candidate_attention(q, k, v, np.tile(keep, (4, 1)))
        mix += mass[:, r:r + 1] * o_r
    assert np.allclose(mix, o)
    # dropping nothing is dense attention; the kept positions are exact
    assert np.array_equal(O.region_drop_keys(bounds, []), np.arange(160))
    assert np.array_equal(O.region_drop_keys(bounds, [0, 2]), np.arange(39, 100))
    rel, cos = O.output_change(o, o)
    assert np.all(rel == 0) and np.allclose(cos, 1)
    rel, cos = O.output_change(-o, o)
    assert np.allclose(rel, 2) and np.allclose(cos, -1)


def test_rel_l2_closed_forms():
    # ||a - b|| / ||b|| over the whole array: a 3-4-5 triangle gives exact
    # values, the reference is the second argument, scaling both leaves it
    # unchanged, and a flattening or per-row mean would give other numbers
    ref = np.array([[3.0, 4.0], [0.0, 0.0]])
    assert O.rel_l2(ref, ref) == 0.0
    assert O.rel_l2(ref + np.array([[0.0, 1.0], [0.0, 0.0]]), ref) == pytest.approx(0.2, abs=0)
    assert O.rel_l2(np.zeros_like(ref), ref) == 1.0
    assert O.rel_l2(2.0 * ref, ref) == 1.0
    assert O.rel_l2(ref, 2.0 * ref) == 0.5           # the second argument is the reference
    got = ref + np.array([[0.0, 0.0], [3.0, 4.0]])   # the error sits in the zero row
    assert O.rel_l2(got, ref) == 1.0
    assert O.rel_l2(7.0 * got, 7.0 * ref) == pytest.approx(1.0, rel=1e-15)
