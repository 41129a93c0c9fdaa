"""The bounds-checked build (KVQ_DEBUG, libkvq_debug.so).

CPU: the range check every kernel of that build runs before an access is
compiled as host code and exercised on ranges whose answer follows from its
definition (inside one of the call's buffers, or not); and the debug library
loads, exports what the header declares and reports that it checks.
GPU: the same calls through both libraries give the same bytes and the debug
build flags nothing on valid inputs (tests/debug_build_cases.py).
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# A host program: two buffers A = [0x10000, 0x10800) and B = [0x20000, 0x20010)
# in the table, then one check per line of CASES (address, bytes); prints
# "ok/miss status" for each.
_PROGRAM = textwrap.dedent(r"""
    #include <cstdio>
    #include <cstdint>
    #include "kvq_common.cuh"
    int main(int argc, char **argv) {
      int32_t status = 0;
      kvq::KernelCtl c{};
      c.dev_status = &status;
    #ifdef KVQ_DEBUG
      c.n_bufs = 2;
      c.buf_lo[0] = 0x10000; c.buf_hi[0] = 0x10800;
      c.buf_lo[1] = 0x20000; c.buf_hi[1] = 0x20010;
    #endif
      unsigned long long a, n;
      while (std::scanf("%llx %llx", &a, &n) == 2) {
        status = 0;
        const bool ok = kvq::in_bounds(c, reinterpret_cast<const void *>(uintptr_t(a)), size_t(n));
        std::printf("%s %d\n", ok ? "ok" : "miss", status);
      }
      return 0;
    }
""")

# (address, bytes, inside one buffer?)
CASES = [
    (0x10000, 0x800, True),            # all of A
    (0x10000, 1, True),                # first byte of A
    (0x107FF, 1, True),                # last byte of A
    (0x107FF, 2, False),               # runs one byte past A
    (0x0FFFF, 1, False),               # one byte before A
    (0x0FFFF, 2, False),               # straddles A's start
    (0x10800, 1, False),               # first byte after A
    (0x20000, 0x10, True),             # all of B
    (0x20008, 0x8, True),
    (0x20008, 0x9, False),
    (0x10400, 0x10000, False),         # from inside A into B: not inside one buffer
    (0x18000, 4, False),               # between the buffers
    (0xFFFFFFFFFFFFFFF0, 0x20, False), # the end wraps past the address space
]


def _run(tmp_path, defines):
    from quantized_sparse_kv_gb300 import build
    src = tmp_path / "check.cu"
    src.write_text(_PROGRAM)
    exe = tmp_path / "check"
    cmd = [build.nvcc(), "-std=c++17", *defines, "-I", build.CSRC, "-I",
           os.path.join(ROOT, "include"), str(src), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    inp = "".join(f"{a:x} {n:x}\n" for a, n, _ in CASES)
    out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True)
    return [line.split() for line in out.stdout.splitlines()]


def test_range_check_follows_its_definition(tmp_path):
    got = _run(tmp_path, ["-DKVQ_DEBUG"])
    assert len(got) == len(CASES)
    for (a, n, inside), (word, status) in zip(CASES, got):
        assert word == ("ok" if inside else "miss"), (hex(a), hex(n))
        assert int(status) == (0 if inside else 8), (hex(a), hex(n))  # KVQ_DEV_BOUNDS


def test_release_build_checks_nothing(tmp_path):
    got = _run(tmp_path, [])
    assert all(word == "ok" and status == "0" for word, status in got)


def test_debug_library_exports_and_reports_checks():
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        from quantized_sparse_kv_gb300 import build, kvq
        if not __import__('os').path.exists(kvq.DEBUG_LIB_PATH):
            build.build(debug=True)
        lib = kvq.load_library(kvq.DEBUG_LIB_PATH)
        for n in kvq.header_functions():
            assert hasattr(lib, n), n
        print(lib.kvq_debug_checks())
    """)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().splitlines()[-1] == "1"


@pytest.mark.gpu
def test_debug_build_matches_release_and_flags_nothing(tmp_path):
    """Every kernel family through libkvq.so and libkvq_debug.so on the same
    seeded inputs: the same output bytes, and no status bit in either."""
    from quantized_sparse_kv_gb300 import kvq
    assert os.path.exists(kvq.DEBUG_LIB_PATH), "build() makes libkvq_debug.so"
    script = os.path.join(ROOT, "tests", "debug_build_cases.py")
    outs = {}
    for name, lib in (("release", kvq.LIB_PATH), ("debug", kvq.DEBUG_LIB_PATH)):
        dst = tmp_path / f"{name}.npz"
        r = subprocess.run([sys.executable, script, lib, str(dst)], capture_output=True,
                           text=True, timeout=900)
        assert r.returncode == 0, r.stdout + r.stderr
        outs[name] = np.load(dst)
    rel, dbg = outs["release"], outs["debug"]
    assert sorted(rel.files) == sorted(dbg.files)
    assert int(dbg["checks"]) == 1 and int(rel["checks"]) == 0
    for k in rel.files:
        if k.startswith("status_"):
            assert int(rel[k]) == 0 and int(dbg[k]) == 0, k
        elif k != "checks":
            assert rel[k].tobytes() == dbg[k].tobytes(), k
