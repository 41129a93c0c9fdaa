"""Run every kernel family once through one build of the library.

python tests/debug_build_cases.py LIB OUT.npz

Loads LIB (libkvq.so or libkvq_debug.so), runs small seeded cases of pack,
append, decode (with a workspace and with the library-owned scratch), the
fp32 kernels, chunk attention (bf16, MXFP8, int4 history, with region
masses), candidate attention (union, per row, top-k, block lists), region
drop and the observer statistics, and saves every output (as raw bytes) and
every status word. test_debug_build compares the files of the two builds.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(lib_path: str, out_path: str) -> None:
    import torch

    from quantized_sparse_kv_gb300 import kvq, synth

    lib = kvq.load_library(lib_path)
    dev = "cuda"
    res = {"checks": np.array(lib.kvq_debug_checks())}

    def keep(name, t):
        t = t.detach().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        res[name] = t.cpu().numpy()

    def status(name, s):
        res["status_" + name] = np.array(kvq.read_status(s))

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(torch.bfloat16)

    # fp32 small-D path with region masses (residual-window shapes)
    q, k, v = synth.residual_window_batch(0, 512, 4)
    s = kvq.new_status()
    c32 = kvq.pack(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), 16, "f32", status=s)
    status("pack_f32", s)
    a = kvq.Attend(c32, torch.from_numpy(q).to(dev), region_bounds=[0, 256, 496, 512])
    a.run()
    keep("small_out", a.out)
    keep("small_mass", a.mass)
    status("small", a.status)
    for name in ("k_codes", "k_scales", "v_codes", "v_scales", "k_window", "v_window"):
        keep("pack_f32_" + name, getattr(c32, name))

    # GQA decode shapes: pack, decode, candidate attention (union, per row, top-k)
    qd, kd, vd = synth.decode_inputs_torch(1, 2, 600, dev)
    s = kvq.new_status()
    cd = kvq.pack(kd, vd, 128, "bf16", status=s)
    status("pack_bf16", s)
    for name in ("k_codes", "k_scales", "v_codes", "v_scales", "k_window", "v_window"):
        keep("pack_bf16_" + name, getattr(cd, name))
    a = kvq.Attend(cd, qd, out_dtype="f32")
    a.run()
    assert a.path == "decode", a.path
    keep("decode_out", a.out)
    status("decode", a.status)
    # the same decode with the library-owned scratch (kv_attend_decode_static)
    import ctypes
    fn = lib.kv_attend_decode_static
    fn.argtypes = [ctypes.POINTER(kvq.KvqCacheStruct), ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    out_s = torch.empty_like(a.out)
    s = kvq.new_status()
    rc = fn(cd.ref, qd.data_ptr(), kvq.BF16, 16, 0.0, out_s.data_ptr(), kvq.F32, s.data_ptr(),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    keep("decode_static_out", out_s)
    status("decode_static", s)
    idx = torch.from_numpy(synth.candidate_indices(0, 2, 16, 600, 96)).to(dev)
    out, s = kvq.attend_candidates(cd, qd, idx, out_dtype="f32")
    keep("cand_union_out", out)
    status("cand_union", s)
    out, s = kvq.attend_candidates(cd, qd.float(), idx, out_dtype="f32")
    keep("cand_row_out", out)
    status("cand_row", s)
    out, sel, s = kvq.attend_candidates_topk(cd, qd, idx, 32, out_dtype="f32")
    keep("topk_out", out)
    keep("topk_sel", sel)
    status("topk", s)
    st = kvq.attend_stats(cd, qd, torch.from_numpy(
        np.random.default_rng(3).choice([-1.0, 1.0], 128)).float())
    keep("stats", st)

    # head dim 64 through the general per-row candidate kernel
    k64 = torch.from_numpy(synth.normal_numpy(5, (1, 2, 300, 64))).to(dev)
    v64 = torch.from_numpy(synth.normal_numpy(6, (1, 2, 300, 64))).to(dev)
    q64 = torch.from_numpy(synth.normal_numpy(7, (1, 4, 2, 64))).to(dev)
    c64 = kvq.pack(k64, v64, 40, "f32")
    i64 = torch.from_numpy(synth.candidate_indices(1, 1, 4, 300, 40, n_q=2)).to(dev)
    out, s = kvq.attend_candidates(c64, q64, i64)
    keep("cand64_out", out)
    status("cand64", s)

    # chunk attention on the tensor cores: bf16 window, MXFP8 K window, int4 history
    qc, kc, vc = synth.chunk_inputs_torch(3, dev, heads=2, n_q=200, n_kv=300)
    bounds = [0, 100, 250, 300]
    for name, recent, kwin in (("chunk_bf16", 300, "bf16"), ("chunk_mxfp8", 300, "mxfp8"),
                               ("chunk_int4", 128, "bf16")):
        cc = kvq.pack(kc, vc, recent, kwin, "bf16")
        a = kvq.Attend(cc, qc, out_dtype="f32", region_bounds=bounds)
        a.run()
        assert a.path == name, (a.path, name)
        keep(name + "_out", a.out)
        keep(name + "_mass", a.mass)
        status(name, a.status)
    # block-shared lists and region drop over the int4-history cache
    ci = kvq.pack(kc, vc, 128, "bf16")
    lists = torch.from_numpy(synth.candidate_indices(2, 1, 2, 300, 64, n_q=2)).to(dev)
    b = kvq.AttendCandidatesBlock(ci, qc, lists, 128, out_dtype="f32")
    b.run()
    keep("block_out", b.out)
    status("block", b.status)
    r = kvq.AttendRegionDrop(ci, qc, bounds, [0], out_dtype="f32")
    keep("drop_out", r.run())
    status("drop", r.status)

    # kv_append: two groups migrate into int4
    kn = torch.from_numpy(synth.normal_numpy(8, (1, 2, 200, 128))).to(dev).to(torch.bfloat16)
    vn = torch.from_numpy(synth.normal_numpy(9, (1, 2, 200, 128))).to(dev).to(torch.bfloat16)
    ca = kvq.pack(kn[:, :, :100], vn[:, :, :100], 100, "bf16", reserve=(8, 160))
    s = kvq.new_status()
    kvq.append(ca, kn[:, :, 100:], vn[:, :, 100:], 64, status=s)
    status("append", s)
    for name, t in ca.used().items():
        keep("append_" + name, t)

    torch.cuda.synchronize()
    np.savez(out_path, **res)


if __name__ == "__main__":
    main(sys.argv[1], sys.argv[2])
