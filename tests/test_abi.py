"""Host-side checks of the C ABI: the library loads, exports what the header
declares, and its size arithmetic agrees with the pages and the oracle.
No GPU is used here."""
import os
import re

import numpy as np
import pytest

from conftest import golden
from oracle import kvq_oracle as O
from quantized_sparse_kv_gb300 import synth


@pytest.fixture(scope="session")
def kvq():
    from quantized_sparse_kv_gb300 import build, kvq as k
    srcs = [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    srcs.append(os.path.join(build.ROOT, "include", "kvq.h"))
    if not os.path.exists(k.LIB_PATH) or os.path.getmtime(k.LIB_PATH) < max(map(os.path.getmtime, srcs)):
        build.build()
    k.load_library()
    return k


def test_library_exports_every_declared_function(kvq):
    names = kvq.header_functions()
    assert {"kv_pack", "kv_attend", "kv_attend_candidates", "kvq_cache_sizes",
            "kvq_cache_bytes"} <= set(names)
    lib = kvq.load_library()
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("recent", [0, 16, 64])
def test_cache_bytes_match_page_payload(kvq, recent):
    g = golden("payload_bytes.json")
    n, d = g["n"], g["head_dim"]
    assert kvq.cache_bytes(1, 1, n, d, recent, kvq.F32, kvq.F32) == g["payload_bytes"][str(recent)]


@pytest.mark.parametrize("n,d,recent,kwin", [(512, 32, 16, "f32"), (100, 64, 30, "bf16"),
                                              (32768, 128, 128, "bf16"), (6240, 128, 6240, "bf16"),
                                              (77, 128, 77, "mxfp8"), (40, 32, 0, "f32")])
def test_cache_sizes_match_oracle_arrays(kvq, n, d, recent, kwin):
    vwin = kvq.F32 if kwin == "f32" else kvq.BF16
    sizes = kvq.cache_sizes(2, 3, n, d, recent, kvq.DTYPES[kwin], vwin)
    cut = n - recent
    gk = -(-cut // 32)
    assert sizes[0] == 6 * gk * 32 * d // 2 and sizes[1] == 6 * gk * d * 4
    assert sizes[2] == 6 * cut * d // 2 and sizes[3] == 6 * cut * d // 32 * 4
    assert sizes[6] == (6 * recent * d // 32 if kwin == "mxfp8" else 0)
    assert sizes[7] == 16
    if n <= 512 and kwin != "mxfp8":
        # one head's arrays, serialised by the oracle, have the same byte counts
        k = np.zeros((n, d), np.float32)
        ser = O.serialize_head(O.pack_head(k, k, recent, "f32" if kwin == "f32" else "bf16"))
        assert ser["k_codes"].nbytes * 6 == sizes[0] and ser["k_scales"].nbytes * 6 == sizes[1]
        assert ser["v_codes"].nbytes * 6 == sizes[2] and ser["v_scales"].nbytes * 6 == sizes[3]
        assert ser["k_window"].nbytes * 6 == sizes[4] and ser["v_window"].nbytes * 6 == sizes[5]


@pytest.mark.parametrize("args", [(0, 1, 8, 32, 0), (1, 1, 8, 48, 0), (1, 1, 8, 32, 9),
                                  (1, 1, 8, 288, 0), (1, 0, 8, 32, 0), (1, 1, 0, 32, 0)])
def test_cache_sizes_reject_bad_shapes(kvq, args):
    with pytest.raises(kvq.KvqError):
        kvq.cache_sizes(*args, kvq.F32, kvq.F32)


def test_v_window_cannot_be_mxfp8(kvq):
    with pytest.raises(kvq.KvqError):
        kvq.cache_sizes(1, 1, 8, 32, 4, kvq.F32, kvq.MXFP8)


def test_inputs_module_holds_no_method_arithmetic():
    # the shared generator module must not reach into either side
    src = open(synth.__file__, encoding="utf-8").read()
    imports = re.findall(r"^\s*(?:from|import)\s+([\w\.]+)", src, flags=re.M)
    assert not [m for m in imports if "oracle" in m or "kvq" in m], imports


def test_product_path_never_touches_the_oracle():
    # the library binding and the build must not import or read the oracle
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "quantized_sparse_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, flags=re.M), f
                assert "kvq_oracle" not in text, f


def test_binding_struct_matches_header():
    # the ctypes descriptor lists the header's kvq_cache fields in order
    from quantized_sparse_kv_gb300 import kvq as k
    text = open(k.HEADER, encoding="utf-8").read()
    body = re.search(r"typedef struct kvq_cache \{(.*?)\} kvq_cache;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        for part in decl.split(","):
            names.append(re.findall(r"(\w+)\s*(?:\[\d+\])?\s*$", part.strip())[0])
    assert names == [f[0] for f in k.KvqCacheStruct._fields_]


def test_binding_fails_loudly_without_the_library():
    # no fallback path: a missing libkvq.so is an error at the first call
    import subprocess
    import sys
    code = ("from quantized_sparse_kv_gb300 import kvq\n"
            "try:\n"
            "    kvq.load_library('/nonexistent/libkvq.so')\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'missing' in str(e))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == "raised True"
