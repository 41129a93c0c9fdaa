"""The division-free int4 rounding of the bf16 kv_pack kernel, on the CPU.

int4_round.cuh (host and device code) is compiled as a host program and
checked exhaustively: for every positive finite bf16 group maximum amax with
recip_ok(amax), the scale equals fl(amax / 7), and for every bf16 x with
|x| <= amax (both signs) the code equals clamp(rint(fl(x / s)), -7, 7), the
rule of the residual-window page ("KV殘差窗口", section 固定預算) with the
division correctly rounded in fp32 and ties to even. The same program shows
the correction step is needed: the uncorrected quotient fl(x r) gives other
codes on some pairs.
"""
import os
import shutil
import subprocess
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_sparse_kv_gb300", "csrc")

_PROGRAM = textwrap.dedent(r"""
    #include <cstdio>
    #include <cmath>
    #include "int4_round.cuh"
    static float bf16(uint32_t h) { uint32_t u = h << 16; float f; memcpy(&f, &u, 4); return f; }
    static int ref_code(float x, float s) {  // clamp(rint(fl(x / s)), -7, 7) + 8
      if (s == 0.0f) return 8;
      float c = std::nearbyint(x / s);
      c = c > 7.0f ? 7.0f : (c < -7.0f ? -7.0f : c);
      return static_cast<int>(c) + 8;
    }
    int main() {
      long pairs = 0, bad_code = 0, bad_high = 0, bad_scale = 0, scales = 0, uncorrected = 0;
    #pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, bad_code, bad_high, bad_scale, scales, uncorrected)
      for (int ha = 0; ha < 0x7f80; ++ha) {     // amax: +0 and every positive finite bf16
        const float amax = bf16(ha);
        if (!kvq::recip_ok(amax)) continue;
        ++scales;
        const float s = kvq::scale_recip(amax);
        if (kvq::bits_of(s) != kvq::bits_of(amax / 7.0f)) ++bad_scale;
        const float r = kvq::recip_of(s);
        for (int hx = 0; hx <= ha; ++hx) {
          for (int sg = 0; sg < 2; ++sg) {
            const float x = sg ? -bf16(hx) : bf16(hx);
            const uint32_t c = kvq::code8_recip(x, s, r);
            const int want = ref_code(x, s);
            ++pairs;
            if (static_cast<int>(c & 15u) != want) ++bad_code;
            if (c & 0xf0u) ++bad_high;
            const uint32_t c0 = kvq::bits_of(kvq::add_rn(kvq::mul_rn(x, r), 12582920.0f));
            if (static_cast<int>(c0 & 15u) != want) ++uncorrected;
          }
        }
      }
      std::printf("%ld %ld %ld %ld %ld %ld\n", scales, pairs, bad_scale, bad_code, bad_high,
                  uncorrected);
      return 0;
    }
""")


def test_int4_reciprocal_rounding_exhaustive_bf16(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "round_check.cu"
    src.write_text(_PROGRAM)
    exe = tmp_path / "round_check"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-fopenmp,-ffp-contract=off",
                    "-I", CSRC, str(src), "-o", str(exe), "-lgomp"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    scales, pairs, bad_scale, bad_code, bad_high, uncorrected = map(int, out)
    # every bf16 maximum from 2^-100 to the largest finite value, plus zero
    assert scales == 1 + (0x7f80 - 0x0d80)
    assert pairs > 10 ** 9
    assert (bad_scale, bad_code, bad_high) == (0, 0, 0)
    assert uncorrected > 0
