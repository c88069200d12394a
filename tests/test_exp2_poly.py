"""The FMA-pipe exponential of csrc/ssd_exp2.cuh, built for the host (the same operations a
device build runs) and checked against 2^x in double precision (no GPU): relative error
within the stated bound, exact powers of two at integers, monotone, and the edge cases."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_copy_gb300", "csrc")

HARNESS = r"""
#include <stdio.h>
#include <stdlib.h>
#include "ssd_exp2.cuh"
int main(int argc, char** argv) {
  FILE* in = fopen(argv[1], "rb");
  FILE* out = fopen(argv[2], "wb");
  float x, y;
  while (fread(&x, sizeof x, 1, in) == 1) {
    y = ssd::exp2_poly(x);
    fwrite(&y, sizeof y, 1, out);
  }
  fclose(in);
  fclose(out);
  return 0;
}
"""


@pytest.fixture(scope="module")
def exp2_host(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("exp2")
    src, exe = d / "h.cpp", d / "h"
    src.write_text(HARNESS)
    r = subprocess.run([gxx, "-O2", "-std=c++17", "-Wall", "-Werror", "-I", CSRC, str(src), "-o", str(exe), "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    def run(x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        fi, fo = d / "in.bin", d / "out.bin"
        x.tofile(fi)
        subprocess.run([str(exe), str(fi), str(fo)], check=True, timeout=120)
        return np.fromfile(fo, dtype=np.float32)
    return run


def test_relative_error_within_bound(exp2_host):
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-126.0, 127.99, 2_000_001, dtype=np.float64).astype(np.float32),
                        rng.uniform(-30.0, 8.0, 1_000_000).astype(np.float32)])
    y = exp2_host(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= 1.04e-4, rel.max()


def test_exact_at_integers_and_monotone(exp2_host):
    i = np.arange(-126, 128, dtype=np.float32)
    np.testing.assert_array_equal(exp2_host(i), np.exp2(i.astype(np.float64)).astype(np.float32))
    # monotone on a sorted grid crossing many integer steps, including the last ulp below each
    x = np.sort(np.concatenate([np.linspace(-20.0, 8.0, 400_001, dtype=np.float32),
                                np.nextafter(np.arange(-20, 9, dtype=np.float32), np.float32(-np.inf))]))
    y = exp2_host(x)
    assert np.all(np.diff(y) >= 0)


def test_edge_cases(exp2_host):
    x = np.array([-np.inf, -1000.0, -126.5, -126.0, 0.0, -0.0, 127.5, 128.0, np.inf], np.float32)
    y = exp2_host(x)
    assert y[0] == 0 and y[1] == 0 and y[2] == 0
    assert y[3] == np.float32(2.0 ** -126) and y[4] == 1.0 and y[5] == 1.0
    assert np.isfinite(y[6]) and y[7] == np.inf and y[8] == np.inf


def test_compiles_as_device_code(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("no nvcc")
    src = tmp_path / "k.cu"
    src.write_text('#include "ssd_exp2.cuh"\n'
                   '__global__ void k(const float* x, float* y, int n) {\n'
                   '  int i = blockIdx.x * blockDim.x + threadIdx.x;\n'
                   '  if (i < n) y[i] = ssd::exp2_poly(x[i]);\n'
                   '}\n')
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-I", CSRC, "-c", str(src),
                        "-o", str(tmp_path / "k.o")], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
