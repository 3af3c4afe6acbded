"""The tensor-core kernels' MXFP4 -> bf16 conversion (csrc/mxfp4.cuh), built
for the host with its byte permute written out, against the format's
definition as the oracle restates it: for every E8M0 scale byte 0..255 and
every E2M1 code, the bf16 pattern is that of e2m1(code) * 2^(e8m0 - 127)
(exact: every such product has at most two significant bits), infinite where
it leaves the fp32 range and NaN for the NaN scale byte."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "mxfp4_table_check")
    src = os.path.join(ROOT, "tests", "native", "mxfp4_table_check.cpp")
    inc = os.path.join(ROOT, "sparse_mixture_experts_gb300", "csrc")
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", inc, src, "-o", exe], check=True, capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return np.array([[int(v) for v in line.split()] for line in out.splitlines()], dtype=np.int64)


def _bf16_bits_of(v: float) -> int:
    with np.errstate(over="ignore"):
        f = np.float32(v)
    return int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)


def test_every_code_times_every_scale_is_the_exact_bf16(tmp_path):
    rows = _run(tmp_path)
    assert len(rows) == 256 * 24
    for s, code, bits in rows.tolist():
        v = oracle.e2m1_value(code) * oracle.e8m0_scale(s)
        if np.isnan(v):
            assert (bits & 0x7f80) == 0x7f80 and (bits & 0x7f) != 0, (s, code, hex(bits))
            continue
        assert bits == _bf16_bits_of(v), (s, code, hex(bits), v)
