"""Benchmark of the compressed-KV-cache attention path on GB300.

Default (``--impl kvq``): the timed step is one GQA decode attention pass over a
packed int4 cache -- 64 sequences, 16 query heads over 2 KV heads, head dim 128,
context 32,768 with the last 128 tokens in bf16 -- through the C ABI
(kv_attend: split-K decode kernel + log-sum-exp combine). The metric is
attended keys per second (sequences x query heads x context / step time).
The other hot-path rows (packing, fp32 small-head attention, chunk attention
with region mass in bf16 and MXFP8, candidate attention) are timed the same
way and reported under ``rows``.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
decode workload on the host cores (the reference arm).

Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DECODE = dict(batch=64, q_heads=16, kv_heads=2, head_dim=128, context=32768, recent=128)
CHUNK = dict(heads=32, n_q=2340, n_kv=6240, head_dim=128, bounds=(0, 1560, 3900, 6240))
CAND = dict(batch=32, q_heads=16, kv_heads=2, head_dim=128, context=131072, recent=128, c=256)
SMALL = dict(heads=32, n=512, head_dim=32, n_q=16, recent=16)
L2_BYTES = 129 * 2 ** 20
NOMINAL_HBM_GBS = 8000.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def profile_traffic(summary):
    """DRAM bytes per full-size launch recorded in a profiles/ summary, or None
    when the kernel source has changed since those counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", summary)
    try:
        fields = dict(line.split(": ", 1) for line in open(path).read().splitlines()
                      if line.startswith(("source: ", "source_sha256: ", "traffic_bytes_per_full_launch: ")))
        src = open(os.path.join(ROOT, fields["source"].strip()), "rb").read()
        if hashlib.sha256(src).hexdigest() != fields["source_sha256"].strip():
            return None
        return int(fields["traffic_bytes_per_full_launch"])
    except (OSError, KeyError, ValueError):
        return None


def fp8_peak_tflops(torch):
    """Measured dense FP8 tensor throughput (TFLOP/s): a cuBLASLt scaled GEMM
    8192^3, best of 10, with one E8M0 scale per 32 along K (MXFP8) when this
    PyTorch build takes it, else per-tensor E4M3 scaling (the same tensor-core
    rate). Returns (tflops, how) or (None, why) when neither runs."""
    n = 8192
    try:
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()
    except Exception as e:  # noqa: BLE001 - report, do not fail the bench
        return None, f"no fp8 tensors: {type(e).__name__}"
    tries = []
    e8 = getattr(torch, "float8_e8m0fnu", None)
    if e8 is not None:
        sa = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device="cuda").view(e8)
        sb = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device="cuda").view(e8)
        tries.append(("MXFP8 (E4M3, E8M0 per 32)", lambda: torch._scaled_mm(
            a, b, scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)))
    one = torch.ones((), device="cuda")
    tries.append(("E4M3 per-tensor scale", lambda: torch._scaled_mm(
        a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)))
    for how, fn in tries:
        try:
            fn()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            return 2.0 * n ** 3 / (best * 1e-3) / 1e12, f"torch._scaled_mm {how}, 8192^3, best of 10"
        except Exception:  # noqa: BLE001 - try the next form
            continue
    return None, "torch._scaled_mm unavailable for fp8 on this build"


# ---------------------------------------------------------------- algorithmic bytes

def decode_bytes(batch, kv_heads, context, recent, head_dim=128, q_heads=16, out_bytes=2):
    """Bytes one decode pass must move: the packed cache once, Q in, O out."""
    cut = context - recent
    gk = -(-cut // 32)
    per_unit = gk * 32 * head_dim // 2 + gk * head_dim * 4 + cut * head_dim // 2 \
        + cut * head_dim // 32 * 4 + 2 * recent * head_dim * 2
    return batch * kv_heads * per_unit + batch * q_heads * head_dim * (2 + out_bytes)


def candidate_unique_bytes(idx, context, recent, head_dim=128, kv_heads=2):
    """Bytes a candidate pass must read at least: each distinct token row and
    each distinct K-scale group once per (sequence, KV head), plus Q and O."""
    import numpy as np
    b, hq, nq, c = idx.shape
    group = hq // kv_heads
    cut = context - recent
    total = 0
    for bi in range(b):
        for h in range(kv_heads):
            toks = np.unique(idx[bi, h * group:(h + 1) * group].reshape(-1))
            q = toks[toks < cut]
            w = toks.size - q.size
            total += q.size * (head_dim // 2 * 2 + head_dim // 32 * 4)   # K, V codes + V scales
            total += np.unique(q // 32).size * head_dim * 4                # K scale groups
            total += w * head_dim * 2 * 2                                 # bf16 window rows
    return total + b * hq * nq * head_dim * 4


# ---------------------------------------------------------------- clocks sampler

class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------- timing helpers

def time_steps(fn, steps, warmup, flush=None):
    """Mean ms per call with CUDA events on the current stream. Without
    ``flush`` the calls run back to back inside one event pair; with it,
    each call is bracketed by its own events and the flush runs outside them.
    The stream is first held by a short spin kernel while every call, flush
    and event is enqueued, so the GPU never waits for the host inside a pair."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    torch.cuda._sleep(int(2e6 + 4e5 * steps))  # about a millisecond, plus per-step room
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    pairs = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn()
        e1.record(s)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in pairs) / steps


def time_e2e_pipelined(torch, pair, q_hosts, o_hosts, steps, warmup):
    """Mean ms per step of query-in / attend / output-out with the copies on
    two more streams (host-to-device and device-to-host, so neither queues
    behind the other): step i uses buffer pair[i % 2]; its query copy is
    issued one step ahead and waits only for the step that last read that
    buffer's output; the attention waits for its query copy; the output copy
    waits for the attention. CUDA events on the compute stream bracket all
    steps (the copy streams are joined into it at the end); a short spin holds
    the compute stream while the steps are enqueued."""
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731

    def enqueue(n, start_event=None):
        out_done = [None, None]
        q_in = [None, None]

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(h2d):
                if start_event is not None and i == 0:
                    h2d.wait_event(start_event)
                if out_done[b] is not None:
                    h2d.wait_event(out_done[b])  # the buffer's previous output is out
                pair[b].q.copy_(q_hosts[i % len(q_hosts)], non_blocking=True)
                q_in[b] = ev()
                q_in[b].record(h2d)

        copy_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            comp.wait_event(q_in[b])
            pair[b].run()
            done = ev()
            done.record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                o_hosts[b].copy_(pair[b].out, non_blocking=True)
                out_done[b] = ev()
                out_done[b].record(d2h)
        comp.wait_stream(h2d)
        comp.wait_stream(d2h)

    enqueue(warmup)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6 + 4e5 * steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    enqueue(steps, e0)
    e1.record(comp)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def make_flush():
    """Evict L2 between timed calls by READING a buffer of twice its size: a
    write-based flush would leave L2 full of dirty lines whose write-back
    then lands inside the next timed call."""
    import torch
    buf = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        torch.amax(buf, dim=0, out=sink)
    return flush


def rotation(touched_bytes, cap=16):
    """How many independent input sets keep every reuse of a set at least two
    L2 sizes of other traffic away (so a call never finds its inputs in L2):
    one set when a call alone touches twice L2, else enough others that
    (n - 1) sets cover twice L2."""
    if touched_bytes >= 2 * L2_BYTES:
        return 1
    return max(1, min(cap, 1 + math.ceil(2 * L2_BYTES / max(1, touched_bytes))))


def cycling(calls):
    """One callable that runs the given calls in turn."""
    state = {"i": 0}

    def run():
        calls[state["i"] % len(calls)]()
        state["i"] += 1
    return run


def l2_note(n, touched_bytes):
    if n == 1:
        return f"inputs larger than L2 ({touched_bytes / 1e6:.0f} MB per call), back to back"
    return (f"{n} input sets rotated back to back, {touched_bytes / 1e6:.0f} MB each: "
            f"{(n - 1) * touched_bytes / 1e6:.0f} MB of other inputs between reuses")


# ---------------------------------------------------------------- rows

def row_pack(kvq, synth, torch, steps, warmup, pk):
    d = DECODE
    q, k, v = synth.decode_inputs_torch(11, d["batch"], d["context"], "cuda")
    cache = kvq.pack(k, v, d["recent"], "bf16")
    ms = time_steps(lambda: kvq.pack(k, v, d["recent"], "bf16", out=cache), steps, warmup)
    nbytes = 2 * k.numel() * 2 + cache.payload_bytes()
    gbs = nbytes / (ms * 1e-3) / 1e9
    tokens = d["batch"] * d["kv_heads"] * d["context"]
    del q, k, v, cache
    return {"workload": "kv_pack int4 K/V, 64 x 2 KV heads x 32768 tokens x 128, bf16 in, R=128",
            "ms": ms, "tokens_per_s": tokens / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": profile_traffic("pack_kv128_bf16_kernel_B64_L32768.md")},
            "launches": 3}


def row_small(kvq, synth, torch, steps, warmup, pk):
    import numpy as np
    s = SMALL
    q, k, v = synth.residual_window_batch(0, s["n"], s["heads"])
    cache = kvq.pack(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), s["recent"], "f32")
    a = kvq.Attend(cache, torch.from_numpy(q).cuda(), out_dtype="f32")
    ms = time_steps(a.run, steps, warmup, flush=make_flush())
    keys = s["heads"] * s["n_q"] * s["n"]
    nbytes = cache.payload_bytes() + 2 * q.nbytes
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "fp32 attention, 32 heads, N=512, D=32, 16 queries, R=16 fp32",
            "ms": ms, "keys_per_s": keys / (ms * 1e-3), "path": a.path,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": None},
            "launches": a.launches(), "note": "latency-bound: 0.8 MB per call"}


def row_chunk(kvq, synth, torch, steps, warmup, pk, kwin, bounds=None):
    """kwin "bf16" / "mxfp8": every key in the window; "int4": the sink and
    recent regions (3,900 tokens) as int4 groups, the current 2,340 in bf16.
    bounds: the region bounds (default [sink | recent | current]; the 16
    latent frames for the heatmap row)."""
    c = CHUNK
    bounds = list(bounds or c["bounds"])
    recent = c["n_kv"] if kwin != "int4" else c["n_kv"] - c["bounds"][2]
    touched = 2 * c["heads"] * c["head_dim"] * (2 * c["n_q"] + 2 * c["n_kv"])
    n = rotation(touched)
    attends = []
    for i in range(n):
        q, k, v = synth.chunk_inputs_torch(21 + 5 * i, "cuda")
        cache = kvq.pack(k, v, recent, "bf16" if kwin == "int4" else kwin, "bf16")
        del k, v
        attends.append(kvq.Attend(cache, q, out_dtype="bf16", region_bounds=bounds))
    a = attends[0]
    ms = time_steps(cycling([x.run for x in attends]), steps, warmup)
    flops = 4.0 * c["heads"] * c["n_q"] * c["n_kv"] * c["head_dim"]
    tf = flops / (ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    if kwin == "mxfp8":
        # QK^T (half the flops) runs block-scaled E4M3 at the FP8 rate, PV at
        # the bf16 rate: the peak of that mix is 1 / (0.5 / fp8 + 0.5 / bf16)
        fp8 = pk.get("fp8_tflops") or 2.0 * pk["bf16_tflops"]
        peak = 1.0 / (0.5 / fp8 + 0.5 / pk["bf16_tflops"])
    keys = c["heads"] * c["n_q"] * c["n_kv"]
    what = {"bf16": "bf16 Q/K", "mxfp8": "mxfp8 Q/K",
            "int4": "bf16 Q, int4 K/V for sink+recent (3900 tokens) and bf16 current window"}[kwin]
    regions = ("[sink 1560 | recent 2340 | current 2340]" if len(bounds) == 4
               else f"{len(bounds) - 1} regions (one per 390-key latent frame)")
    return {"workload": f"chunk attention {what}, 32 heads, 2340 queries over 6240 keys "
                        f"{regions}, D=128, region mass",
            "ms": ms, "keys_per_s": keys / (ms * 1e-3), "path": a.path, "l2": l2_note(n, touched),
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak,
                         "traffic": {"bf16": profile_traffic("chunk_bf16_kernel_H32_Q2340_K6240.md"),
                                     "mxfp8": profile_traffic("chunk_mxfp8_kernel_H32_Q2340_K6240.md"),
                                     }.get(kwin),
                         "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                         "peak_note": {"bf16": "bf16 measured",
                                       "mxfp8": "half fp8 / half bf16 flops: "
                                                + (f"fp8 {pk['fp8_tflops']:.0f} TFLOP/s measured "
                                                   f"({pk.get('fp8_how')})"
                                                   if pk.get("fp8_tflops") else
                                                   "fp8 taken as 2x the measured bf16 (nominal "
                                                   "ratio)")
                                                + f", bf16 {pk['bf16_tflops']:.0f} measured; "
                                                  "QK^T on tcgen05 kind::mxf8f6f4 block-scaled",
                                       "int4": "bf16 measured: int4 history expanded to bf16 "
                                               "(one pass, inside the timed call), bf16 MMA"}[kwin]},
            "launches": a.launches()}


def row_candidates(kvq, synth, torch, steps, warmup, pk, context, c):
    d = CAND
    idx = synth.candidate_indices(5, d["batch"], d["q_heads"], context, c)
    nbytes = candidate_unique_bytes(idx, context, d["recent"])
    n = rotation(nbytes)
    attends = []
    for i in range(n):
        q, k, v = synth.decode_inputs_torch(31 + 3 * i, d["batch"], context, "cuda")
        cache = kvq.pack(k, v, d["recent"], "bf16")
        del k, v
        attends.append(kvq.AttendCandidates(cache, q, torch.from_numpy(idx).cuda(),
                                            out_dtype="bf16"))
    a = attends[0]
    ms = time_steps(cycling([x.run for x in attends]), steps, warmup)
    gbs = nbytes / (ms * 1e-3) / 1e9
    keys = d["batch"] * d["q_heads"] * c
    return {"workload": f"candidate attention, 32 x 16 heads, L={context}, C={c}, int4 + bf16 R=128",
            "ms": ms, "keys_per_s": keys / (ms * 1e-3), "l2": l2_note(n, nbytes),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": (profile_traffic("candidates_union_kernels_B32_L131072_C256.md")
                                     if (context, c) == (131072, 256) else None),
                         "bytes_note": "distinct rows and K-scale groups per (sequence, KV head)"},
            "launches": a.launches()}


def row_candidates_topk(kvq, synth, torch, steps, warmup, pk, context, c, top_k):
    """Two-stage candidates: exact scores of the C listed keys, attention over
    their top_k (the pages' C -> top-32)."""
    d = CAND
    idx = synth.candidate_indices(5, d["batch"], d["q_heads"], context, c)
    nbytes = candidate_unique_bytes(idx, context, d["recent"])
    n = rotation(nbytes)
    calls = []
    for i in range(n):
        q, k, v = synth.decode_inputs_torch(61 + 3 * i, d["batch"], context, "cuda")
        cache = kvq.pack(k, v, d["recent"], "bf16")
        del k, v
        ti = torch.from_numpy(idx).cuda()
        calls.append(lambda cache=cache, q=q, ti=ti:
                     kvq.attend_candidates_topk(cache, q, ti, top_k, out_dtype="bf16"))
    ms = time_steps(cycling(calls), steps, warmup)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"candidate attention, exact top-{top_k} of C={c} listed keys, 32 x 16 "
                        f"heads, L={context}, int4 + bf16 R=128",
            "ms": ms, "keys_per_s": d["batch"] * d["q_heads"] * top_k / (ms * 1e-3),
            "l2": l2_note(n, nbytes),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": None,
                         "bytes_note": "distinct K rows of the lists once, V rows of the kept keys "
                                       "counted as in the plain candidate row (upper bound)"},
            "launches": 1}


def row_candidates_block(kvq, synth, torch, steps, warmup, pk):
    """Candidate prefill with block-shared lists: L = 4096 query rows of one
    sequence (16 query heads over 2 KV heads, D = 128) over its own int4 +
    bf16 R=128 cache, one list of C = 256 keys per 128-row block, against
    dense kv_attend of the same rows on the same cache."""
    import numpy as np
    L, c, bq, hq = 4096, 256, 128, 16
    q, k, v = synth.decode_inputs_torch(71, 1, L, "cuda")
    q = synth.normal_torch(72, (1, hq, L, 128), torch.bfloat16, "cuda")
    cache = kvq.pack(k, v, 128, "bf16")
    del k, v
    nb = L // bq
    rng = np.random.default_rng(8)
    idx = np.stack([np.stack([np.sort(rng.choice(L, c, replace=False)) for _ in range(nb)])
                    for _ in range(hq)])[None].astype(np.int32)
    blk = kvq.AttendCandidatesBlock(cache, q, torch.from_numpy(idx).cuda(), bq, out_dtype="bf16")
    blk.run()
    dense = kvq.Attend(cache, q, out_dtype="bf16")
    dense.run()
    ms = time_steps(blk.run, steps, warmup)
    ms_dense = time_steps(dense.run, steps, warmup)
    flops = 4.0 * hq * L * c * 128
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": "candidate prefill, block-shared lists: 4096 rows x 16 heads, one list of "
                        "C=256 keys per 128 rows, int4 + bf16 R=128 cache of 4096 tokens",
            "ms": ms, "keys_per_s": hq * L * c / (ms * 1e-3), "path": blk.path,
            "dense_ms": ms_dense, "dense_path": dense.path,
            "speedup_vs_dense": ms_dense / ms,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"], "traffic": None,
                         "note": "gather of the lists (bf16) included; 4 x rows x C x 128 flops"},
            "launches": 2}


def row_region_drop(kvq, synth, torch, steps, warmup, pk):
    """The local output ablation on the video chunk: drop the sink region
    (1,560 keys); time, and the median output change of every variant."""
    c = CHUNK
    q, k, v = synth.chunk_inputs_torch(81, "cuda", concentrated=4.0)
    cache = kvq.pack(k, v, c["n_kv"], "bf16")
    full = kvq.attend(cache, q, out_dtype="f32")[0]
    change = {}
    for name, drop in (("drop_sink", [0]), ("drop_recent", [1]), ("drop_history", [0, 1])):
        o = kvq.AttendRegionDrop(cache, q, c["bounds"], drop, out_dtype="f32").run()
        rel = (o - full).norm(dim=-1) / full.norm(dim=-1)
        cos = (o * full).sum(-1) / (o.norm(dim=-1) * full.norm(dim=-1))
        change[name] = {"median_rel_l2": float(rel.median()), "median_cosine": float(cos.median())}
    a = kvq.AttendRegionDrop(cache, q, c["bounds"], [0], out_dtype="bf16")
    ms = time_steps(a.run, steps, warmup)
    kept = c["n_kv"] - c["bounds"][1]
    flops = 4.0 * c["heads"] * c["n_q"] * kept * 128
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": "region-drop ablation on the video chunk (32 heads, 2340 queries, "
                        "[1560 | 2340 | 2340] keys, concentrated rows): sink dropped",
            "ms": ms, "output_change": change,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / pk["bf16_tflops"], "traffic": None,
                         "note": "gather of the kept rows included"},
            "launches": 2}


def row_decode(kvq, synth, torch, steps, warmup, pk, batch, context):
    """The decode step at another (batch, context) of the decode workload."""
    d = dict(DECODE, batch=batch, context=context)
    nbytes = decode_bytes(batch, d["kv_heads"], context, d["recent"])
    n = rotation(nbytes)
    flush = None
    if n > 1 and (n - 1) * nbytes < 2 * L2_BYTES:
        # too small for the rotation to keep two L2 sizes between reuses:
        # one input set, L2 flushed before every call
        n, flush = 1, make_flush()
    attends = []
    for i in range(n):
        q, k, v = synth.decode_inputs_torch(1 + 7 * i, batch, context, "cuda")
        cache = kvq.pack(k, v, d["recent"], "bf16")
        del k, v
        attends.append(kvq.Attend(cache, q, out_dtype="bf16"))
    a = attends[0]
    a.run()
    ms = time_steps(cycling([x.run for x in attends]), steps, warmup, flush=flush)
    gbs = nbytes / (ms * 1e-3) / 1e9
    keys = batch * d["q_heads"] * context
    # the decode profile's traffic (full-size launch) scaled by this row's
    # algorithmic bytes: the kernel's traffic tracks them (1.02x at every size
    # captured), so the scaling is by the units of work each launch processes
    full = profile_traffic("decode_kernel_B16_L32768.md")
    full_bytes = decode_bytes(DECODE["batch"], d["kv_heads"], DECODE["context"], d["recent"])
    traffic = None if full is None else int(round(full * nbytes / full_bytes))
    return {"workload": f"decode: B={batch}, 16 query heads over 2 KV heads, D=128, L={context}, "
                        "R=128 bf16, int4 groups of 32",
            "ms": ms, "keys_per_s": keys / (ms * 1e-3), "path": a.path,
            "l2": (f"L2 flushed before every call ({nbytes / 1e6:.1f} MB per call)" if flush
                   else l2_note(n, nbytes)),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": traffic,
                         "traffic_note": "ncu DRAM bytes of the B=16, L=32768 decode launch, "
                                         "scaled by algorithmic bytes",
                         "algorithmic_bytes": nbytes,
                         "kernel": "decode_kernel + combine_kernel (one kv_attend call)"},
            "launches": a.launches()}


def row_append(kvq, synth, torch, steps, warmup, pk):
    """kv_append of one decoded token per (sequence, KV head) on the decode
    cache (64 sequences x 2 KV heads, D = 128, window 128): every 32nd call
    also moves a 32-token group from the window into int4."""
    d = DECODE
    n_calls = 32 * max(1, -(-steps // 32))
    extra = n_calls + 32 * (warmup + 2)
    q, k, v = synth.decode_inputs_torch(41, d["batch"], d["context"] + extra, "cuda")
    n0 = d["context"]
    cache = kvq.pack(k[:, :, :n0], v[:, :, :n0], d["recent"], "bf16",
                     reserve=(-(-(n0 + extra) // 32), d["recent"] + 32))
    news = [(k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous())
            for t in range(n0, n0 + extra)]
    del q
    state = {"i": 0}

    def one():
        kn, vn = news[state["i"]]
        kvq.append(cache, kn, vn, d["recent"])
        state["i"] += 1
    ms = time_steps(one, n_calls, 32 * warmup)
    nbytes = 2 * d["batch"] * d["kv_heads"] * d["head_dim"] * 2 * 2  # new rows in, window rows out
    return {"workload": "kv_append: 1 token per (sequence, KV head), 64 x 2 heads, D=128, bf16, "
                        "window 128, int4 groups of 32 (a group migrates every 32nd call)",
            "ms": ms, "tokens_per_s": d["batch"] * d["kv_heads"] / (ms * 1e-3),
            "roofline": {"bound": "latency", "achieved": nbytes / (ms * 1e-3) / 1e9,
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None,
                         "note": "64 KB of new rows per call: launch-latency bound"},
            "launches": "1 per call, 2 on every 32nd"}


def row_stats(kvq, synth, torch, steps, warmup, pk):
    """kv_attend_stats on the video chunk: 96 sampled query rows per head (the
    pages' observer samples 96 queries per head), 32 heads over 6,240 keys,
    with the signed-H128 MXFP8 Q/K path."""
    import numpy as np
    c = CHUNK
    q, k, v = synth.chunk_inputs_torch(51, "cuda")
    cache = kvq.pack(k, v, c["n_kv"], "bf16")
    qs = q[:, :, ::c["n_q"] // 96][:, :, :96].contiguous()
    signs = torch.from_numpy(np.random.default_rng(2).choice([-1.0, 1.0], c["head_dim"]))
    kvq.attend_stats(cache, qs, signs)
    sg = signs.cuda().float()
    ms = time_steps(lambda: kvq.attend_stats(cache, qs, sg), steps, warmup)
    rows = c["heads"] * 96
    flops = rows * c["n_kv"] * 2 * (2 * c["head_dim"])   # the two score dot products
    peak = 152 * 128 * 2 * 2.07e9 / 1e12                  # fp32 FMA issue rate at 2.07 GHz
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": "kv_attend_stats: 32 heads x 96 sampled queries over 6240 bf16 keys, "
                        "signed-H128 MXFP8 Q/K path, MXFP8 P path, top-k by radix select",
            "ms": ms, "rows_per_s": rows / (ms * 1e-3),
            "roofline": {"bound": "alu", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "traffic": None,
                         "peak_note": "fp32 FMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz",
                         "note": "three kernels: keys once per head into 32-key tiles, "
                                 "scores of 48 rows per CTA on the tensor cores (tf32 "
                                 "mma.sync: three products per pair on the fp32 path, one "
                                 "on the exact MXFP8 path), per-row statistics; flops "
                                 "counted are the two score dot products only, against the "
                                 "fp32 FMA rate of a CUDA-core scoring; the statistics "
                                 "passes take about 43 % of the time"},
            "launches": 3}


# ---------------------------------------------------------------- oracle (CPU) arm

def _oracle_unit_worker(args):
    """Time the oracle's attend on one (sequence, KV head) of the decode workload:
    dequantize the packed unit and attend its 8 query heads."""
    seed, context, recent = args
    import numpy as np
    from oracle import kvq_oracle as O
    from quantized_sparse_kv_gb300 import synth
    q = O.round_to_bf16(synth.normal_numpy(seed, (8, 1, 128)))
    k = O.round_to_bf16(synth.normal_numpy(seed + 1, (context, 128)))
    v = O.round_to_bf16(synth.normal_numpy(seed + 2, (context, 128)))
    packed = O.pack_head(k, v, recent, "bf16")
    t0 = time.perf_counter()
    kh, vh = O.dequantize_head(packed)
    for h in range(8):
        O.attention(q[h], kh, vh)
    return time.perf_counter() - t0


def _oracle_pack_worker(args):
    """Time the oracle's kv_pack of one (sequence, KV head) of the decode
    workload (int4 groups of K per channel and of V per token, bf16 window)."""
    seed, context, recent = args
    from oracle import kvq_oracle as O
    from quantized_sparse_kv_gb300 import synth
    k = O.round_to_bf16(synth.normal_numpy(seed + 1, (context, 128)))
    v = O.round_to_bf16(synth.normal_numpy(seed + 2, (context, 128)))
    t0 = time.perf_counter()
    O.pack_head(k, v, recent, "bf16")
    return time.perf_counter() - t0


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_pool(workers):
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    return mp.get_context("spawn").Pool(workers)


def oracle_sample(pool, units, workers, seed0=1000):
    d = DECODE
    t0 = time.perf_counter()
    busy = pool.map(_oracle_unit_worker,
                    [(seed0 + 3 * i, d["context"], d["recent"]) for i in range(units)])
    wall = time.perf_counter() - t0
    keys = units * 8 * d["context"]
    cpu_s = sum(busy)
    # each worker is one core; input generation and packing are not timed
    return {"keys": keys, "wall_s": wall, "cpu_s": cpu_s, "keys_per_s": keys * workers / cpu_s}


def oracle_pack_sample(pool, units, workers, seed0=5000):
    d = DECODE
    busy = pool.map(_oracle_pack_worker,
                    [(seed0 + 3 * i, d["context"], d["recent"]) for i in range(units)])
    tokens = units * d["context"]
    return {"tokens": tokens, "cpu_s": sum(busy), "tokens_per_s": tokens * workers / sum(busy)}


def cpu_baseline_record(workers):
    """The fp64 oracle timed on the host cores (spawned before any GPU work):
    attention of the decode workload's (sequence, KV head) units on all
    workers and on one, and kv_pack of such units, each a bounded sample."""
    d = DECODE
    pool = oracle_pool(workers)
    allc = oracle_sample(pool, 8 * workers, workers)
    pack = oracle_pack_sample(pool, 2 * workers, workers)
    pool.close()
    one = oracle_pool(1)
    single = oracle_sample(one, 4, 1, seed0=3000)
    pack1 = oracle_pack_sample(one, 2, 1, seed0=6000)
    one.close()
    try:
        nproc = len(os.sched_getaffinity(0))
    except AttributeError:
        nproc = os.cpu_count() or 1
    return {"value": allc["keys_per_s"], "unit": "keys/s", "cores": workers, "kind": "oracle",
            "sample": f"{8 * workers} (sequence, KV head) units of the decode workload "
                      f"(8 query heads x L={d['context']} each), oracle dequantize + fp64 "
                      f"attention, {allc['cpu_s']:.1f} s of CPU work",
            "cpu_model": cpu_model(), "nproc": nproc,
            "single_thread": {"value": single["keys_per_s"], "unit": "keys/s", "cores": 1,
                              "sample": f"4 units, {single['cpu_s']:.1f} s"},
            "pack": {"value": pack["tokens_per_s"], "unit": "tokens/s (x 1 KV head)",
                     "cores": workers,
                     "sample": f"{2 * workers} units of {d['context']} tokens packed "
                               f"(int4 K per channel, V per token, bf16 window R={d['recent']}), "
                               f"{pack['cpu_s']:.1f} s",
                     "single_thread": pack1["tokens_per_s"]}}


def cpu_workers():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


# ---------------------------------------------------------------- main arms

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def decode_config(world):
    """The headline workload, as both arms report it."""
    d = DECODE
    nbytes = decode_bytes(d["batch"], d["kv_heads"], d["context"], d["recent"])
    return {"workload": f"decode: B={d['batch']} sequences, 16 query heads over 2 KV heads, "
                        "D=128, L=32768, last R=128 tokens bf16, int4 groups of 32",
            "batch": d["batch"], "context": d["context"], "recent": d["recent"],
            "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per step), no flush",
            "parallelism": f"replicas x{world}, each its own batch"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    workers = cpu_workers()
    pool = oracle_pool(workers)
    units = 2 * workers
    for _ in range(args.warmup):
        oracle_sample(pool, workers, workers)
    res = [oracle_sample(pool, units, workers, seed0=2000 + 97 * i) for i in range(args.steps)]
    pool.close()
    keys = sum(r["keys"] for r in res)
    busy = sum(r["cpu_s"] for r in res) / workers   # timed oracle seconds per core
    wall = busy
    value = keys / busy
    d = DECODE
    sample = (f"{units} of the 128 (sequence, KV head) units per step: oracle dequantize + "
              f"fp64 attention of their 8 query heads over L={d['context']}")
    line = {"metric": "attended keys/s (GQA decode over int4 KV cache)", "value": value,
            "unit": "keys/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), bf16-rounded",
            "impl": "reference",
            "config": decode_config(world),
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": workers, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_kvq(args):
    world, rank, local = dist_setup()
    import numpy as np
    import torch

    from quantized_sparse_kv_gb300 import kvq, synth
    kvq.load_library()
    torch.cuda.set_device(local)
    pk = peaks()
    d = dict(DECODE)
    if args.case == "small":
        d["batch"] = 16   # 169 MB per step: still larger than L2, small enough for ncu sections

    # CPU oracle baseline first (spawned before heavy GPU work), rank 0 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_record(cpu_workers())

    q, k, v = synth.decode_inputs_torch(1 + rank, d["batch"], d["context"], "cuda")
    cache = kvq.pack(k, v, d["recent"], "bf16")
    del k, v
    torch.cuda.synchronize()
    att = kvq.Attend(cache, q, out_dtype="bf16")
    att.run()
    assert att.path == "decode", att.path
    launches_per_step = att.launches()
    nbytes = decode_bytes(d["batch"], d["kv_heads"], d["context"], d["recent"])

    for _ in range(max(3, args.warmup)):
        att.run()
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    def busy(seconds):
        # untimed steps, so that the clock sampler sees the GPU under this load
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(20):
                att.run()
            torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        busy(0.5)
        barrier(world)
        e0.record(s)
        for _ in range(args.steps):
            att.run()
        e1.record(s)
        torch.cuda.synchronize()
        barrier(world)
        busy(0.5)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world)
    clocks = clk.summary()
    keys_per_step = d["batch"] * d["q_heads"] * d["context"]
    value = world * keys_per_step / (ms_max * 1e-3)
    gbs = nbytes / (ms * 1e-3) / 1e9

    # end to end through the same C call with host buffers: every step copies
    # its query rows in from pinned host memory and its outputs back out
    q_hosts = [torch.randn(q.shape).to(q.dtype).pin_memory() for _ in range(2)]
    q_hosts[0].copy_(q.cpu())
    o_hosts = [torch.empty(att.out.shape, dtype=att.out.dtype).pin_memory() for _ in range(2)]
    pair = [att, kvq.Attend(cache, q.clone(), out_dtype="bf16")]
    e2e_ms = time_e2e_pipelined(torch, pair, q_hosts, o_hosts, args.steps, 3)
    e2e = {"value": world * keys_per_step / (max_over_ranks(e2e_ms, world) * 1e-3),
           "unit": "keys/s", "h2d_bytes_per_step": q_hosts[0].numel() * q_hosts[0].element_size(),
           "d2h_bytes_per_step": o_hosts[0].numel() * o_hosts[0].element_size(),
           "note": "KV cache resident in HBM; per step the query rows go in from pinned host "
                   "memory and the outputs come back out, on one copy stream per direction, "
                   "double-buffered, so "
                   "that step i's copies overlap the neighbouring steps' attention"}

    rows = {}
    if rank == 0 and not args.no_rows:
        pk["fp8_tflops"], pk["fp8_how"] = fp8_peak_tflops(torch)
        rsteps = max(3, min(args.steps, 20))
        for name, fn in ROWS.items():
            rows[name] = fn(kvq, synth, torch, rsteps, 3, pk)

    if rank != 0:
        return
    line = {
        "metric": "attended keys/s (GQA decode over int4 KV cache)",
        "value": value, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "dtype_note": "int4 KV codes and bf16 Q/window in; the MMAs take f16 operands (bf16 "
                      "for the window tiles) and accumulate in f32",
        "data": "synthetic N(0,1) bf16 Q/K/V, seeded",
        "config": decode_config(world),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": (profile_traffic("decode_kernel_B16_L32768.md")
                                 if d["batch"] == 64 else None),
                     "kernel": "decode_kernel + combine_kernel (one kv_attend call)",
                     "algorithmic_bytes": nbytes, "peak_source": pk["source"],
                     "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS},
        "peaks": {k: pk.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained",
                                          "source", "fp8_tflops", "fp8_how")},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "rows": rows,
    }
    print(json.dumps(line))


ROWS = {
    "decode_B16_L32768": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 16, 32768),
    "decode_B64_L8192": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 64, 8192),
    "decode_B64_L1024": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 64, 1024),
    "decode_B16_L8192": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 16, 8192),
    "decode_B16_L1024": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 16, 1024),
    "decode_B1_L32768": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 1, 32768),
    "decode_B1_L8192": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 1, 8192),
    "decode_B1_L1024": lambda kvq, synth, torch, st, w, pk:
        row_decode(kvq, synth, torch, st, w, pk, 1, 1024),
    "pack": lambda kvq, synth, torch, st, w, pk: row_pack(kvq, synth, torch, st, w, pk),
    "append": lambda kvq, synth, torch, st, w, pk: row_append(kvq, synth, torch, st, w, pk),
    "small_d_fp32": lambda kvq, synth, torch, st, w, pk: row_small(kvq, synth, torch, st, w, pk),
    "candidates_L131072_C256": lambda kvq, synth, torch, st, w, pk:
        row_candidates(kvq, synth, torch, st, w, pk, 131072, 256),
    "candidates_L32768_C96": lambda kvq, synth, torch, st, w, pk:
        row_candidates(kvq, synth, torch, st, w, pk, 32768, 96),
    "candidates_block_prefill_L4096_C256": lambda kvq, synth, torch, st, w, pk:
        row_candidates_block(kvq, synth, torch, st, w, pk),
    "candidates_top32_of_C256_L131072": lambda kvq, synth, torch, st, w, pk:
        row_candidates_topk(kvq, synth, torch, st, w, pk, 131072, 256, 32),
    "chunk_bf16": lambda kvq, synth, torch, st, w, pk: row_chunk(kvq, synth, torch, st, w, pk, "bf16"),
    "chunk_bf16_16frames": lambda kvq, synth, torch, st, w, pk:
        row_chunk(kvq, synth, torch, st, w, pk, "bf16", synth.CHUNK_LF_BOUNDS),
    "chunk_mxfp8": lambda kvq, synth, torch, st, w, pk:
        row_chunk(kvq, synth, torch, st, w, pk, "mxfp8"),
    "chunk_int4_history": lambda kvq, synth, torch, st, w, pk:
        row_chunk(kvq, synth, torch, st, w, pk, "int4"),
    "stats_chunk_96q": lambda kvq, synth, torch, st, w, pk: row_stats(kvq, synth, torch, st, w, pk),
    "region_drop_chunk": lambda kvq, synth, torch, st, w, pk:
        row_region_drop(kvq, synth, torch, st, w, pk),
}


def run_row(args):
    """Time one hot-path row alone (for profiling); prints its JSON object."""
    import torch

    from quantized_sparse_kv_gb300 import kvq, synth
    kvq.load_library()
    pk = peaks()
    if args.row.startswith("chunk_mxfp8"):
        pk["fp8_tflops"], pk["fp8_how"] = fp8_peak_tflops(torch)
    res = ROWS[args.row](kvq, synth, torch, args.steps, args.warmup, pk)
    print(json.dumps({"row": args.row, **res}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--no-rows", action="store_true", help="time only the decode step")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--case", choices=["full", "small"], default="full",
                    help="small: 16 sequences instead of 64 (for profiler captures)")
    ap.add_argument("--row", choices=sorted(ROWS), help="time only this hot-path row")
    args = ap.parse_args()
    if args.row:
        run_row(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_kvq(args)


if __name__ == "__main__":
    main()
