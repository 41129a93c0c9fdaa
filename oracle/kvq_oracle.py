"""fp64 CPU oracle for attention over a grouped-int4 KV cache.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module. It shares no code with the CUDA library
and imports nothing from it; it is a plain, slow, line-by-line statement of
what the hot path computes, written from these pages:

* "KV殘差窗口：最近Token一定值得高精度嗎？" (huhohoo.com, kv-residual-window) --
  the cache ``[early tokens: grouped 4-bit][last R tokens: float]`` (section
  固定預算，先問它保護了誰), its payload accounting (section
  殘差窗口也會吃掉壓縮收益) and the ``cut = N - R; x[cut:]`` rule (section
  小練習與排錯).
* "Catnip Week 10 KV Cache Attention Study" (cappuccino.cafe/kv-attn.html) --
  the chunk layout [sink 1560 | recent 2340 | current 2340], per-row region
  mass (section "KV Cache 的实际作用") and MXFP8 Q/K with E4M3 elements and an
  E8M0 scale per 32 along the head dim (section "Q/K 与 probability
  quantization 的影响").
* the MiniCPM5-2B attention-predictor study (bjdmk.com.cn/news/5855973) --
  exact attention restricted to top-C candidate keys (sections 6 and 9).

Readings where the pages are silent:
int4 scale = fp32(amax / 7) with codes clamped to [-7, 7] and rounded half to
even; a zero scale gives all-zero codes; nibble = code + 8, even element in the
low nibble; K groups are aligned at token 0 and the last one is zero padded; V
is not padded; softmax scale 1/sqrt(D); no causal mask; q-head h reads KV head
h // (Hq / Hkv); MXFP8 block scale 2^(floor(log2 amax) - 8) clamped to
[-127, 127] (zero block: -127), elements rounded to nearest E4M3, ties to even,
saturating at +-448.

Every function here is pinned by the CPU tests (page-printed values, closed
forms, brute force on tiny inputs). One quantity is parity unpinned: the
MXFP8-vs-bf16 probability total variation is only reported, never asserted.
"""
from __future__ import annotations

import math

import numpy as np

GROUP = 32          # int4 group size (K: 32 tokens of one channel; V: 32 features of one token)
QMAX = 7            # symmetric int4 codes in [-7, 7]
HEADER_BYTES = 16   # shape metadata {N, D, R, 32} as four uint32
E4M3_MAX = 448.0
E4M3_EMAX = 8       # floor(log2(448))


# --------------------------------------------------------------------------------------
# bf16 as a storage format (round to nearest even from fp32)
# --------------------------------------------------------------------------------------

def fp32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bfloat16, nearest-even on the dropped 16 bits; returns uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + keep_lsb) >> 16).astype(np.uint32)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r[nan] = 0x7FC0
    return r.astype(np.uint16)


def bf16_bits_to_fp32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """fp32 array holding the bf16 rounding of ``x``."""
    return bf16_bits_to_fp32(fp32_to_bf16_bits(x))


# --------------------------------------------------------------------------------------
# Grouped symmetric int4 (residual-window page, section 固定預算)
# --------------------------------------------------------------------------------------

def int4_quantize_groups(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantize each length-32 row along the last axis to symmetric int4.

    scale = amax / 7 rounded once to fp32; each element's quotient x / scale is
    rounded once to fp32 (the correctly rounded fp32 division), then to the
    nearest integer with ties to even, then clamped to [-7, 7]. A group whose
    scale is zero (all zeros, or amax / 7 below the fp32 range) keeps scale 0 and
    all-zero codes. Returns (codes int8 (..., 32), scale float32 (...)).
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == GROUP
    amax = np.abs(x).max(axis=-1)
    scale = (amax.astype(np.float64) / float(QMAX)).astype(np.float32)
    nonzero = scale != 0
    divisor = np.where(nonzero, scale, np.float32(1)).astype(np.float64)
    quotient = (x.astype(np.float64) / divisor[..., None]).astype(np.float32)
    codes = np.clip(np.rint(quotient.astype(np.float64)), -QMAX, QMAX).astype(np.int8)
    codes = np.where(nonzero[..., None], codes, np.int8(0)).astype(np.int8)
    return codes, scale


def int4_dequantize(codes, scale) -> np.ndarray:
    """x_hat = code * scale, exact in fp64."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


def pack_head(k, v, recent: int, window_dtype: str = "f32") -> dict:
    """Pack one head's K (N, D) and V (N, D).

    The cache is [tokens 0..N-R-1: grouped int4][tokens N-R..N-1: float]. The
    quantized part is x[:cut] and the window x[cut:] with cut = N - R, so R = 0
    leaves an empty window (the page warns that x[-0:] is the whole array).
    K is quantized per channel over groups of 32 consecutive tokens, groups
    aligned at token 0, the last group zero padded; V per token over groups of
    32 consecutive features. The window keeps the input values (rounded to bf16
    when ``window_dtype == "bf16"``).
    """
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    n, d = k.shape
    if v.shape != (n, d) or d % GROUP or not 0 <= recent <= n:
        raise ValueError("bad shapes")
    cut = n - recent
    gk = -(-cut // GROUP)
    k_pad = np.zeros((gk * GROUP, d), dtype=np.float32)
    k_pad[:cut] = k[:cut]
    # (Gk, 32 tokens, D) -> groups along tokens: (Gk, D, 32)
    kc, ks = int4_quantize_groups(k_pad.reshape(gk, GROUP, d).transpose(0, 2, 1))
    vc, vs = int4_quantize_groups(v[:cut].reshape(cut, d // GROUP, GROUP))
    if window_dtype == "f32":
        kw, vw = k[cut:].copy(), v[cut:].copy()
    elif window_dtype == "bf16":
        kw, vw = round_to_bf16(k[cut:]), round_to_bf16(v[cut:])
    else:
        raise ValueError(window_dtype)
    return {
        "n": n, "d": d, "recent": recent, "window_dtype": window_dtype,
        "k_codes": kc.transpose(0, 2, 1).copy(),   # (Gk, 32, D) int8
        "k_scales": ks,                             # (Gk, D) f32
        "v_codes": vc.reshape(cut, d),              # (N-R, D) int8
        "v_scales": vs,                             # (N-R, D/32) f32
        "k_window": kw,                             # (R, D)
        "v_window": vw,                             # (R, D)
        "header": np.array([n, d, recent, GROUP], dtype=np.uint32),
    }


def nibbles(codes) -> np.ndarray:
    """Serialize int4 codes along the last axis: byte i = (c[2i] + 8) | (c[2i+1] + 8) << 4."""
    u = (np.asarray(codes, dtype=np.int16) + 8).astype(np.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def serialize_head(p: dict) -> dict:
    """The packed arrays as the stored bytes (nibbles, fp32 scales, window, header)."""
    wdt = np.float32 if p["window_dtype"] == "f32" else None
    if wdt is None:
        kw = fp32_to_bf16_bits(p["k_window"])
        vw = fp32_to_bf16_bits(p["v_window"])
    else:
        kw = p["k_window"].astype(np.float32)
        vw = p["v_window"].astype(np.float32)
    return {
        "k_codes": nibbles(p["k_codes"]),
        "k_scales": p["k_scales"].astype(np.float32),
        "v_codes": nibbles(p["v_codes"]),
        "v_scales": p["v_scales"].astype(np.float32),
        "k_window": kw,
        "v_window": vw,
        "header": p["header"],
    }


def payload_bytes_of(p: dict) -> int:
    """Size of the stored arrays of one packed head (codes, scales, window, shape)."""
    return int(sum(a.nbytes for a in serialize_head(p).values()))


def dequantize_head(p: dict) -> tuple[np.ndarray, np.ndarray]:
    """K_hat, V_hat (N, D) in fp64: dequantized int4 part followed by the window."""
    n, d, r = p["n"], p["d"], p["recent"]
    cut = n - r
    k_q = int4_dequantize(p["k_codes"].transpose(0, 2, 1), p["k_scales"])  # (Gk, D, 32)
    k_q = k_q.transpose(0, 2, 1).reshape(-1, d)[:cut]
    v_q = int4_dequantize(p["v_codes"].reshape(cut, d // GROUP, GROUP), p["v_scales"])
    v_q = v_q.reshape(cut, d)
    k_hat = np.concatenate([k_q, p["k_window"].astype(np.float64)], axis=0)
    v_hat = np.concatenate([v_q, p["v_window"].astype(np.float64)], axis=0)
    return k_hat, v_hat


# --------------------------------------------------------------------------------------
# Attention (two-pass softmax in fp64, no mask)
# --------------------------------------------------------------------------------------

def attention(q, k_hat, v_hat, sm_scale: float | None = None, region_bounds=None):
    """O = softmax(sm_scale * Q K^T) V over all keys, plus per-row region masses.

    q (n_q, D), k_hat/v_hat (N, D). Returns (O (n_q, D), P (n_q, N), mass
    (n_q, n_regions) or None). Region k is keys [b_k, b_{k+1}); its mass is the
    sum of that row's probabilities over the region.
    """
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    v_hat = np.asarray(v_hat, dtype=np.float64)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    s = sm_scale * (q @ k_hat.T)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    o = p @ v_hat
    mass = None
    if region_bounds is not None:
        b = list(region_bounds)
        mass = np.stack([p[:, b[i]:b[i + 1]].sum(axis=1) for i in range(len(b) - 1)], axis=1)
    return o, p, mass


def candidate_attention(q, k_hat, v_hat, idx, sm_scale: float | None = None):
    """Exact attention of each query row over its own candidate keys only.

    q (n_q, D), idx (n_q, C) of distinct key positions. Row i attends keys
    idx[i] and nothing else.
    """
    q = np.asarray(q, dtype=np.float64)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    out = np.empty_like(q)
    for i in range(q.shape[0]):
        sel = np.asarray(idx[i], dtype=np.int64)
        s = sm_scale * (k_hat[sel] @ q[i])
        e = np.exp(s - s.max())
        out[i] = (e / e.sum()) @ v_hat[sel]
    return out


def candidate_topk_select(q, k_hat, idx, top_k: int, sm_scale: float | None = None):
    """The keys a two-stage candidate pass keeps (MiniCPM study, section 6:
    a predictor proposes top-C candidates, then the true top-32 inside them is
    taken by exact score): per row, the top_k listed keys by sm_scale q . k,
    ties going to the key listed first. Returns (positions (n_q, top_k),
    scores of every listed key (n_q, C))."""
    q = np.asarray(q, dtype=np.float64)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    idx = np.asarray(idx, dtype=np.int64)
    scores = np.stack([sm_scale * (k_hat[idx[i]] @ q[i]) for i in range(q.shape[0])])
    order = np.argsort(-scores, axis=-1, kind="stable")[:, :top_k]
    return np.take_along_axis(idx, order, axis=-1), scores


def candidate_topk_attention(q, k_hat, v_hat, idx, top_k: int, sm_scale: float | None = None):
    """Exact attention of each row over the top_k of its listed keys
    (candidate_topk_select), and nothing else."""
    keep, _ = candidate_topk_select(q, k_hat, idx, top_k, sm_scale)
    return candidate_attention(q, k_hat, v_hat, keep, sm_scale)


def region_drop_keys(region_bounds, drop) -> np.ndarray:
    """Positions of the keys outside the dropped regions (Catnip study,
    recommended local output ablation: drop sink, drop recent, drop all
    history, renormalise P): region r is [b_r, b_{r+1}); drop lists region
    numbers."""
    keep = [np.arange(region_bounds[r], region_bounds[r + 1])
            for r in range(len(region_bounds) - 1) if r not in set(drop)]
    return np.concatenate(keep) if keep else np.zeros(0, dtype=np.int64)


def output_change(o, o_ref) -> tuple[np.ndarray, np.ndarray]:
    """Per-row relative L2 ||o - o_ref|| / ||o_ref|| and cosine similarity."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    nr = np.linalg.norm(o_ref, axis=-1)
    rel = np.linalg.norm(o - o_ref, axis=-1) / nr
    cos = (o * o_ref).sum(-1) / (np.linalg.norm(o, axis=-1) * nr)
    return rel, cos


# --------------------------------------------------------------------------------------
# Batched forms over (batch, head) in the library's tensor layout
# --------------------------------------------------------------------------------------

def pack(k, v, recent: int, window_dtype: str = "f32") -> list[list[dict]]:
    """K, V (B, Hkv, N, D) -> packed heads [b][h]."""
    return [[pack_head(k[b, h], v[b, h], recent, window_dtype) for h in range(k.shape[1])]
            for b in range(k.shape[0])]


def attend(q, packed, sm_scale=None, region_bounds=None, heads=None):
    """Q (B, Hq, n_q, D) over packed[b][h_kv], h_kv = h // (Hq // Hkv).

    Returns O (B, Hq, n_q, D) and, with ``region_bounds``, mass (B, Hq, n_q, R).
    ``heads`` restricts the work to a list of (b, h) pairs (other rows stay NaN).
    """
    bsz, hq, nq, d = q.shape
    hkv = len(packed[0])
    group = hq // hkv
    o = np.full((bsz, hq, nq, d), np.nan)
    nreg = 0 if region_bounds is None else len(region_bounds) - 1
    mass = np.full((bsz, hq, nq, nreg), np.nan) if nreg else None
    pairs = heads if heads is not None else [(b, h) for b in range(bsz) for h in range(hq)]
    cache = {}
    for b, h in pairs:
        key = (b, h // group)
        if key not in cache:
            cache[key] = dequantize_head(packed[b][h // group])
        kh, vh = cache[key]
        ob, _, mb = attention(q[b, h], kh, vh, sm_scale, region_bounds)
        o[b, h] = ob
        if nreg:
            mass[b, h] = mb
    return o, mass


def attend_candidates(q, packed, idx, sm_scale=None, heads=None):
    """Candidate attention in the batched layout; idx (B, Hq, n_q, C)."""
    bsz, hq, nq, d = q.shape
    hkv = len(packed[0])
    group = hq // hkv
    o = np.full((bsz, hq, nq, d), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(bsz) for h in range(hq)]
    cache = {}
    for b, h in pairs:
        key = (b, h // group)
        if key not in cache:
            cache[key] = dequantize_head(packed[b][h // group])
        kh, vh = cache[key]
        o[b, h] = candidate_attention(q[b, h], kh, vh, idx[b, h], sm_scale)
    return o


def rel_l2(a, b) -> float:
    """||a - b||_2 / ||b||_2 over the whole array (per-input relative L2)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


# --------------------------------------------------------------------------------------
# MXFP8: E4M3 elements with one E8M0 scale per 32 along the head dim
# (Catnip study, section "Q/K 与 probability quantization 的影响")
# --------------------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no
    infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y) -> np.ndarray:
    """Round fp64 values to the nearest E4M3 (ties to even mantissa), saturating to +-448.

    The magnitude is rounded on the grid of its binade: quantum 2^(floor(log2|y|) - 3)
    for normal values and 2^-9 below 2^-6; the sign bit follows the sign of y.
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                      # a = f * 2^ex with f in [0.5, 1)
    binade = np.maximum(ex - 1, -6)          # floor(log2 a), clamped to the subnormal binade
    quantum = np.ldexp(1.0, binade - 3)
    mag = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)
    # magnitude -> exponent/mantissa fields
    _, ex2 = np.frexp(mag)
    e_field = np.where(mag < 2.0 ** -6, 0, ex2 - 1 + 7)
    m_field = np.where(e_field == 0, mag / 2.0 ** -9,
                       (mag / np.ldexp(1.0, np.maximum(e_field, 1) - 7) - 1.0) * 8.0)
    code = (e_field.astype(np.int64) << 3) | np.rint(m_field).astype(np.int64)
    code = code | (np.signbit(y).astype(np.int64) << 7)
    return code.astype(np.uint8)


def mxfp8_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows to MXFP8 with one scale per 32 consecutive elements of the last axis.

    Block exponent e = floor(log2 amax) - 8 (8 = floor(log2 448)), clamped to
    [-127, 127], -127 for an all-zero block; stored as the E8M0 byte e + 127.
    Elements are x / 2^e rounded to E4M3. Returns (codes uint8 like x,
    scale bytes uint8 (..., D/32)).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    xb = x.reshape(x.shape[:-1] + (d // GROUP, GROUP))
    amax = np.abs(xb).max(axis=-1)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex - 1 - E4M3_EMAX, -127)
    e = np.clip(e, -127, 127)
    codes = e4m3_encode(xb / np.ldexp(1.0, e)[..., None])
    return codes.reshape(x.shape), (e + 127).astype(np.uint8)


def mxfp8_dequantize(codes, scale_bytes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    vals = E4M3_TABLE[codes].reshape(codes.shape[:-1] + (d // GROUP, GROUP))
    scale = np.ldexp(1.0, np.asarray(scale_bytes, dtype=np.int64) - 127)
    return (vals * scale[..., None]).reshape(codes.shape)


def probability_tv(p, p_ref) -> np.ndarray:
    """Per-row total variation 0.5 * sum |p - p_ref| (reported only; parity unpinned)."""
    return 0.5 * np.abs(np.asarray(p) - np.asarray(p_ref)).sum(axis=-1)


# --------------------------------------------------------------------------------------
# Observer statistics of attention rows (Catnip study: section 实验设计, step 5 and
# the Structural / Effective / Numerical MXFP8 notes; section "Q/K 与 probability
# quantization 的影响" for the signed-H128 + MXFP8 Q/K path, the P-path proxy and
# the argmax agreement)
# --------------------------------------------------------------------------------------

FP32_HALF_TINY = 2.0 ** -150   # fp64 values below this round to 0 in fp32


def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (a power of two), entries +-1."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def signed_hadamard(x, signs) -> np.ndarray:
    """x -> (x * signs) H / sqrt(D) along the last axis.

    An orthogonal rotation (H / sqrt(D) is symmetric and orthogonal, signs are
    +-1), so q . k is unchanged when both sides are rotated; it spreads a large
    channel over all channels before MXFP8 rounding (the page's signed-H128)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / math.sqrt(d)


def mxfp8_round(x) -> np.ndarray:
    """Every element's MXFP8 value, one scale per 32 along the last axis; a
    partial last block is padded with zeros (which do not change its maximum)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    pad = (-d) % GROUP
    if pad:
        x = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1)
    codes, scales = mxfp8_quantize(x)
    return mxfp8_dequantize(codes, scales)[..., :d]


def top_count(n: int, percent: int) -> int:
    """ceil(percent% of n): how many of the largest probabilities a top-x% mass sums."""
    return (n * percent + 99) // 100


def row_statistics(s, s_mx=None) -> dict:
    """Statistics of softmax rows over scores s (rows, N), already scaled.

    entropy   H = -sum p ln p (nats, over p > 0)
    support   exp(H) / N, the entropy-equivalent share of the keys
    top1/5/10 mass of the top_count(N, 1 / 5 / 10) largest probabilities
    zero      share of keys whose probability is 0 in fp32 (structural zeros)
    p_zero    share of keys whose probability is nonzero in fp32 but 0 after
              MXFP8 rounding along the keys (E4M3, one E8M0 scale per 32 keys)
    p_tv      0.5 sum |p_mx - p|; p_sum = sum p_mx (the P-path proxy row sum)
    With s_mx, the scores of the MXFP8 Q/K path for the same rows:
    qk_tv     0.5 sum |softmax(s_mx) - p|
    qk_agree  1 where argmax s_mx == argmax s (first index of the maximum)
    """
    s = np.asarray(s, dtype=np.float64)
    n = s.shape[-1]
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    p = e / e.sum(axis=-1, keepdims=True)
    live = p >= FP32_HALF_TINY
    plogp = np.where(p > 0, p * np.log(np.where(p > 0, p, 1.0)), 0.0)
    h = -plogp.sum(axis=-1)
    ps = -np.sort(-p, axis=-1)
    out = {"entropy": h, "support": np.exp(h) / n,
           "top1": ps[..., :top_count(n, 1)].sum(-1), "top5": ps[..., :top_count(n, 5)].sum(-1),
           "top10": ps[..., :top_count(n, 10)].sum(-1),
           "zero": (~live).sum(-1) / n}
    p_mx = mxfp8_round(p)
    out["p_zero"] = (live & (p_mx == 0)).sum(-1) / n
    out["p_tv"] = 0.5 * np.abs(p_mx - p).sum(-1)
    out["p_sum"] = p_mx.sum(-1)
    if s_mx is not None:
        s_mx = np.asarray(s_mx, dtype=np.float64)
        e2 = np.exp(s_mx - s_mx.max(axis=-1, keepdims=True))
        out["qk_tv"] = 0.5 * np.abs(e2 / e2.sum(axis=-1, keepdims=True) - p).sum(-1)
        out["qk_agree"] = (np.argmax(s_mx, axis=-1) == np.argmax(s, axis=-1)).astype(np.float64)
    return out


def attention_statistics(q, k_hat, signs=None, sm_scale=None) -> dict:
    """row_statistics of softmax(sm_scale q k_hat^T) for q (n_q, D) over k_hat (N, D),
    with the MXFP8 Q/K path: q and k_hat rotated by signed_hadamard when signs
    are given, then both rounded to MXFP8 along D."""
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(q.shape[-1])
    qr, kr = (q, k_hat) if signs is None else (signed_hadamard(q, signs), signed_hadamard(k_hat, signs))
    s = sm_scale * (q @ k_hat.T)
    s_mx = sm_scale * (mxfp8_round(qr) @ mxfp8_round(kr).T)
    return row_statistics(s, s_mx)
