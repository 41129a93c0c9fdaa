"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds input recipes only: random draws, shapes and the
structure of the workloads (focus variants, candidate index lists). It does
none of the method's arithmetic (no quantization, no attention), so the
oracle and the CUDA path can both be fed from it without sharing any code.

Recipes:

* ``residual_window_inputs`` -- "KV residual window" page (huhohoo.com,
  kv-residual-window), section on where the attention mass lands: one head,
  head dim 32, 16 queries, N in {128, 512}, Q/K/V ~ N(0, 1) in fp32, drawn in
  the order Q, K, V from ``numpy.random.default_rng(seed)``.  The
  ``early``/``recent`` variants raise channel 0 of every Q row and of the K
  rows at the first/last 16 positions; ``mode="add"`` adds ``boost`` (+3),
  ``mode="set"`` sets the channel to ``boost``.
* ``decode_inputs`` -- GQA decode shaped like MiniCPM5-2B (bjdmk.com.cn study,
  section 0): 16 query heads, 2 KV heads, head dim 128, bf16 ~ N(0, 1).
* ``chunk_inputs`` -- the video chunk of the "Catnip Week 10 KV Cache
  Attention Study" page: 32 heads, 2,340 queries over 6,240 keys laid out
  [sink 1560 | recent 2340 | current 2340].
* ``candidate_indices`` -- per-query top-C lists: a quarter of C distinct
  positions from [0, 64), the rest distinct and uniform over [64, L),
  sorted ascending (MiniCPM5-2B study, sections 6, 7 and 9).
"""
from __future__ import annotations

import numpy as np

# Region bounds of the chunk layout [sink 4 LF | recent 6 LF | current 6 LF],
# 390 tokens per latent frame (15 x 26).
CHUNK_TOKENS_PER_LF = 390
CHUNK_REGION_BOUNDS = (0, 4 * 390, 10 * 390, 16 * 390)  # (0, 1560, 3900, 6240)
CHUNK_N_Q = 6 * 390  # 2340
# One region per latent frame: the 16 key-LF columns of the page's temporal
# attention heatmap (each query row's 16 masses sum to 100 %).
CHUNK_LF_BOUNDS = tuple(390 * i for i in range(17))  # (0, 390, ..., 6240)


def residual_window_inputs(seed: int, n: int, *, variant: str = "clean",
                           mode: str = "add", boost: float = 3.0,
                           n_q: int = 16, d: int = 32, focus: int = 16):
    """One head of the residual-window protocol: Q (n_q, d), K (n, d), V (n, d) fp32."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n_q, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    _apply_focus(q, k, variant, mode, boost, focus)
    return q.astype(np.float32), k.astype(np.float32), v.astype(np.float32)


def residual_window_batch(seed: int, n: int, heads: int, *, variant: str = "clean",
                          mode: str = "add", boost: float = 3.0,
                          n_q: int = 16, d: int = 32, focus: int = 16):
    """``heads`` independent heads from one stream, drawn head-major (Q, K, V per head).

    Returns Q (1, heads, n_q, d), K and V (1, heads, n, d) in fp32: the batched
    layout the library takes, with one KV head per query head.
    """
    rng = np.random.default_rng(seed)
    qs, ks, vs = [], [], []
    for _ in range(heads):
        q = rng.standard_normal((n_q, d))
        k = rng.standard_normal((n, d))
        v = rng.standard_normal((n, d))
        _apply_focus(q, k, variant, mode, boost, focus)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    q = np.stack(qs)[None].astype(np.float32)
    k = np.stack(ks)[None].astype(np.float32)
    v = np.stack(vs)[None].astype(np.float32)
    return q, k, v


def _apply_focus(q, k, variant, mode, boost, focus):
    if variant == "clean":
        return
    n = k.shape[0]
    rows = slice(0, focus) if variant == "early" else slice(n - focus, n)
    if variant not in ("early", "recent"):
        raise ValueError(f"unknown variant {variant!r}")
    if mode == "add":
        q[:, 0] += boost
        k[rows, 0] += boost
    elif mode == "set":
        q[:, 0] = boost
        k[rows, 0] = boost
    else:
        raise ValueError(f"unknown mode {mode!r}")


def normal_numpy(seed: int, shape, dtype=np.float32):
    """N(0, 1) draws from ``default_rng(seed)`` (small cases, CPU)."""
    return np.random.default_rng(seed).standard_normal(shape).astype(dtype)


def normal_torch(seed: int, shape, dtype, device):
    """N(0, 1) draws from a seeded ``torch.Generator`` on ``device``.

    Used for the large workloads, which are generated where they are used; a
    test copies the slices it checks back to the host for the oracle.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def decode_shapes(batch: int, context: int, *, q_heads: int = 16, kv_heads: int = 2,
                  head_dim: int = 128):
    """Shapes of the GQA decode workload: (Q, K, V) with one query per sequence."""
    return ((batch, q_heads, 1, head_dim),
            (batch, kv_heads, context, head_dim),
            (batch, kv_heads, context, head_dim))


def decode_inputs_torch(seed: int, batch: int, context: int, device, *, q_heads=16,
                        kv_heads=2, head_dim=128):
    """bf16 Q, K, V ~ N(0, 1) for the decode workload, drawn on ``device``."""
    import torch
    qs, ks, vs = decode_shapes(batch, context, q_heads=q_heads, kv_heads=kv_heads,
                               head_dim=head_dim)
    q = normal_torch(seed, qs, torch.bfloat16, device)
    k = normal_torch(seed + 1, ks, torch.bfloat16, device)
    v = normal_torch(seed + 2, vs, torch.bfloat16, device)
    return q, k, v


def chunk_inputs_torch(seed: int, device, *, heads=32, n_q=CHUNK_N_Q,
                       n_kv=CHUNK_REGION_BOUNDS[-1], head_dim=128,
                       concentrated: float = 0.0):
    """bf16 Q (1, H, n_q, D), K and V (1, H, n_kv, D) ~ N(0, 1) for the chunk workload.

    ``concentrated > 0`` adds ``concentrated`` times one shared random unit
    direction (per head) to every Q and K row, which sharpens the softmax rows
    the way the page's real captures are sharp.
    """
    import torch
    q = normal_torch(seed, (1, heads, n_q, head_dim), torch.float32, device)
    k = normal_torch(seed + 1, (1, heads, n_kv, head_dim), torch.float32, device)
    v = normal_torch(seed + 2, (1, heads, n_kv, head_dim), torch.float32, device)
    if concentrated:
        u = normal_torch(seed + 3, (1, heads, 1, head_dim), torch.float32, device)
        u = u / u.norm(dim=-1, keepdim=True)
        q = q + concentrated * u
        k = k + concentrated * u
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def candidate_indices(seed: int, batch: int, q_heads: int, context: int, c: int, *,
                      n_q: int = 1, early: int = 64, sort: bool = True) -> np.ndarray:
    """Per-query candidate lists, int32 (batch, q_heads, n_q, c).

    A quarter of each list (``c // 4``) is drawn without replacement from the
    first ``early`` positions and the rest without replacement from
    [early, context); each list is sorted ascending unless ``sort`` is False,
    in which case it is shuffled.
    """
    rng = np.random.default_rng(seed)
    n0 = c // 4
    if n0 > early or c - n0 > context - early:
        raise ValueError("candidate count does not fit the context")
    out = np.empty((batch, q_heads, n_q, c), dtype=np.int32)
    for b in range(batch):
        for h in range(q_heads):
            for i in range(n_q):
                a = rng.choice(early, n0, replace=False)
                z = early + _distinct(rng, context - early, c - n0)
                row = np.concatenate([a, z])
                if sort:
                    row.sort()
                else:
                    rng.shuffle(row)
                out[b, h, i] = row
    return out


def _distinct(rng, n: int, k: int) -> np.ndarray:
    """k distinct integers from [0, n) without materialising a permutation of n."""
    if k * 4 >= n:
        return rng.choice(n, k, replace=False)
    got = np.unique(rng.integers(0, n, size=2 * k + 8))
    while got.size < k:
        got = np.unique(np.concatenate([got, rng.integers(0, n, size=k)]))
    return rng.permutation(got)[:k]
