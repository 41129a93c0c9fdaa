"""kv_attend_decode_static: decode attention for callers that cannot allocate.

Some callers have no device memory to give: a serving runtime that has handed
all free HBM to its KV-cache pool, or a latency-critical caller that cannot
take cudaMalloc's implicit device synchronisation. For them the library keeps
the decode kernel's split-K scratch in a fixed 8 MiB device array of its own.
This test calls that entry point through the C ABI and checks it against
kv_attend (which takes a caller workspace) on two calls in a row with
different queries, so stale scratch from the first call would show in the
second. It runs last so that a run stopping at the first failure has already
run every other test, and it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2   # the bf16-path tolerance of the parity tests


def _bind(lib, kvq):
    fn = lib.kv_attend_decode_static
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(kvq.KvqCacheStruct), vp, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_float, vp, ctypes.c_int32, vp, vp]
    fn.restype = ctypes.c_int32
    return fn


def _rel_l2(a, b):
    a = a.double()
    b = b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def test_static_scratch_decode_matches_kv_attend_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq, synth
    lib = kvq.load_library()
    fn = _bind(lib, kvq)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    batch, n, recent = 3, 3000, 128
    k = torch.from_numpy(synth.normal_numpy(101, (batch, 2, n, 128))).cuda().to(torch.bfloat16)
    v = torch.from_numpy(synth.normal_numpy(102, (batch, 2, n, 128))).cuda().to(torch.bfloat16)
    cache = kvq.pack(k, v, recent, "bf16")
    for call, seed in enumerate((103, 104)):
        q = torch.from_numpy(synth.normal_numpy(seed, (batch, 16, 1, 128))).cuda().to(torch.bfloat16)
        ref = kvq.Attend(cache, q, out_dtype="f32").run().clone()
        out = torch.full_like(ref, float("nan"))
        status = kvq.new_status()
        st = fn(cache.ref, ctypes.c_void_p(q.data_ptr()), kvq.BF16, 16, 0.0,
                ctypes.c_void_p(out.data_ptr()), kvq.F32, ctypes.c_void_p(status.data_ptr()), stream)
        assert st == 0, (call, kvq.STATUS.get(st, st))
        assert kvq.read_status(status) == 0
        assert torch.isfinite(out).all()
        assert _rel_l2(out, ref) <= TOL_BF16, call


def test_static_scratch_decode_rejects_oversized_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq
    lib = kvq.load_library()
    fn = _bind(lib, kvq)
    # 2,048 (sequence, KV head) units need more split-K scratch than 8 MiB
    k = torch.zeros((1024, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    cache = kvq.pack(k, k, 0, "bf16")
    q = torch.zeros((1024, 16, 1, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    st = fn(cache.ref, ctypes.c_void_p(q.data_ptr()), kvq.BF16, 16, 0.0,
            ctypes.c_void_p(out.data_ptr()), kvq.BF16, None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4, kvq.STATUS.get(st, st)   # KVQ_ERR_WORKSPACE, nothing enqueued
    assert not out.any()
