"""The tensor-core kernels' low-bit -> bf16 conversions (csrc/lowbit.cuh),
built for the host with the byte permute and the rounding written out, against
the formats' definitions as the oracle restates them:

* MXFP4: for every E8M0 scale byte 0..255 and every E2M1 code, the bf16
  pattern is that of e2m1(code) * 2^(e8m0 - 127) (exact: every such product
  has at most two significant bits), infinite where it leaves the fp32 range
  and NaN for the NaN scale byte;
* Q4: for binary16 scales sampled over every exponent (both signs, subnormals
  included) and every code, the pattern is (code - 8) * d rounded once to
  bf16, nearest even."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rows(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("lowbit") / "lowbit_check")
    src = os.path.join(ROOT, "tests", "native", "lowbit_check.cpp")
    inc = os.path.join(ROOT, "sparse_mixture_experts_gb300", "csrc")
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", inc, src, "-o", exe], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return [line.split() for line in out.splitlines()]


def _bf16_rne_bits(v: float) -> int:
    with np.errstate(over="ignore"):
        u = int(np.array([np.float32(v)], dtype=np.float32).view(np.uint32)[0])
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF


def test_mxfp4_every_code_times_every_scale_is_the_exact_bf16(rows):
    m = [(int(s), int(c), int(b)) for k, s, c, b in rows if k == "M"]
    assert len(m) == 256 * 24
    for s, code, bits in m:
        v = oracle.e2m1_value(code) * oracle.e8m0_scale(s)
        if np.isnan(v):
            assert (bits & 0x7f80) == 0x7f80 and (bits & 0x7f) != 0, (s, code, hex(bits))
            continue
        with np.errstate(over="ignore"):
            exact = int(np.array([np.float32(v)], dtype=np.float32).view(np.uint32)[0] >> 16)
        assert bits == exact, (s, code, hex(bits), v)


def test_q4_codes_times_scales_round_once_to_bf16(rows):
    q = [(int(d), int(c), int(b)) for k, d, c, b in rows if k == "Q"]
    assert len(q) > 8000
    seen_sub = False
    for d16, code, bits in q:
        d = oracle.fp16_value(d16)
        seen_sub |= d != 0 and abs(d) < 2.0 ** -14
        v = (code - 8) * d  # exact in double
        assert np.float32(v) == v
        assert bits == _bf16_rne_bits(v), (hex(d16), code, hex(bits), v)
    assert seen_sub
