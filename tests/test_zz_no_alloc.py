"""kv_attend_decode_static: decode attention for callers that cannot allocate.

Some callers have no device memory to give: a serving runtime that has handed
all free HBM to its KV-cache pool, or a latency-critical caller that cannot
take cudaMalloc's implicit device synchronisation. For them the library keeps
the decode kernel's split-K scratch in a fixed 8 MiB device array of its own.
This test calls that entry point through the C ABI and checks it against
kv_attend (which takes a caller workspace) on two calls in a row with
different queries, so stale scratch from the first call would show in the
second; that the second call changes neither the device's free memory nor
torch's reservation; and, in a fresh process, that a call still succeeds
after everything but a small margin of HBM has been handed out following the
first kv_pack. It runs last so that a run stopping at the first failure has
already run every other test, and it passes alone in a fresh process too.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

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
        # the reference (kv_attend with a caller workspace) is taken before
        # the memory snapshot, so its workspace is not counted
        ref = kvq.Attend(cache, q, out_dtype="f32").run().clone()
        out = torch.full_like(ref, float("nan"))
        status = kvq.new_status()
        torch.cuda.synchronize()
        free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
        st = fn(cache.ref, ctypes.c_void_p(q.data_ptr()), kvq.BF16, 16, 0.0,
                ctypes.c_void_p(out.data_ptr()), kvq.F32, ctypes.c_void_p(status.data_ptr()), stream)
        assert st == 0, (call, kvq.STATUS.get(st, st))
        torch.cuda.synchronize()
        if call == 1:  # after a warm-up call, a call allocates nothing
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_reserved() == reserved0
        assert kvq.read_status(status) == 0
        assert torch.isfinite(out).all()
        assert _rel_l2(out, ref) <= TOL_BF16, call


_FULL_HBM_SCRIPT = textwrap.dedent("""
    import ctypes, sys
    import torch
    sys.path.insert(0, sys.argv[1])
    from quantized_sparse_kv_gb300 import kvq, synth
    lib = kvq.load_library()
    fn = lib.kv_attend_decode_static
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(kvq.KvqCacheStruct), vp, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_float, vp, ctypes.c_int32, vp, vp]
    fn.restype = ctypes.c_int32
    k = torch.from_numpy(synth.normal_numpy(111, (2, 2, 2000, 128))).cuda().to(torch.bfloat16)
    v = torch.from_numpy(synth.normal_numpy(112, (2, 2, 2000, 128))).cuda().to(torch.bfloat16)
    cache = kvq.pack(k, v, 128, "bf16")          # the first library call on this device
    q = torch.from_numpy(synth.normal_numpy(113, (2, 16, 1, 128))).cuda().to(torch.bfloat16)
    ref = kvq.Attend(cache, q, out_dtype="f32").run().clone()
    out = torch.full_like(ref, float("nan"))
    torch.cuda.synchronize()
    # hand out all free HBM but a small margin, as a KV-cache pool would
    free = torch.cuda.mem_get_info()[0]
    hog = torch.empty(free - (256 << 20), dtype=torch.uint8, device="cuda")
    st = fn(cache.ref, vp(q.data_ptr()), kvq.BF16, 16, 0.0, vp(out.data_ptr()), kvq.F32, None,
            vp(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    err = float(torch.linalg.norm(out.double() - ref.double()) / torch.linalg.norm(ref.double()))
    print("status", st, "rel_l2", err, "left_mib", torch.cuda.mem_get_info()[0] >> 20)
    sys.exit(0 if st == 0 and err <= 1e-2 else 1)
""")


def test_static_scratch_decode_after_hbm_is_handed_out_fresh_process():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FULL_HBM_SCRIPT, root], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


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
