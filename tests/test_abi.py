"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
function include/ssd.h declares (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "ssd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def libpath():
    from speculative_decoding_copy_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    return build.LIB


def test_header_declares_the_four_step_calls():
    d = _declared()
    for n in ["ssd_gate_match", "ssd_retrieve", "ssd_verify_attn", "ssd_accept"]:
        assert n in d


def test_library_exports_every_declared_symbol(libpath):
    L = ctypes.CDLL(libpath)
    for n in _declared():
        assert hasattr(L, n), n


def test_binding_declares_the_same_symbols(libpath):
    from speculative_decoding_copy_gb300 import _binding
    assert sorted(_binding.EXPORTED) == _declared()
    L = _binding.lib()
    assert _binding.status_string(0) == "ok"
    assert _binding.status_string(-4).startswith("workspace")
    assert L.ssd_version() >= 100


def test_host_validation_without_gpu(libpath):
    # argument errors are caught on the host before anything touches a device
    from speculative_decoding_copy_gb300 import _binding as b
    L = b.lib()
    null = None
    assert L.ssd_gate_match(null, 1, null, 1, null, 0, 1, null, 1, 0.4, 0, null, null, null, null, null) == b.SSD_ERR_INVALID
    assert L.ssd_gate_match(null, 1, null, 0, null, 0, 1, null, 1, 0.4, 5, null, null, null, null, null) == b.SSD_OK
    assert L.ssd_retrieve(null, 1, null, 1, null, null, 5, 0, 4, 0, 0, null, null, null, null, null) == b.SSD_ERR_INVALID
    a = b.AttnArgs()
    a.B, a.NB, a.Dmax, a.Hq, a.Hkv, a.dh, a.dtype = 1, 1, 4, 4, 2, 96, b.SSD_BF16
    assert L.ssd_verify_attn(ctypes.byref(a), null, 0, null) == b.SSD_ERR_UNSUPPORTED
    a.dh, a.Hkv = 128, 3
    assert L.ssd_verify_attn(ctypes.byref(a), null, 0, null) == b.SSD_ERR_INVALID
    a.Hkv, a.skip_absent = 2, 3                     # only 0, 1 or 2
    assert L.ssd_verify_attn(ctypes.byref(a), null, 0, null) == b.SSD_ERR_INVALID
    c = b.AcceptArgs()
    c.mode, c.kind, c.V, c.B, c.NB, c.Dmax, c.chain_blk = 7, 0, 100, 1, 1, 4, -1
    assert L.ssd_accept(ctypes.byref(c), null, 0, null) == b.SSD_ERR_INVALID
    c.mode, c.chain_blk = b.SSD_GREEDY, 3
    assert L.ssd_accept(ctypes.byref(c), null, 0, null) == b.SSD_ERR_INVALID
    c.chain_blk, c.B = -1, 0
    assert L.ssd_accept(ctypes.byref(c), null, 0, null) == b.SSD_OK


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "ssd.h"

int main(void) {
  ssd_attn_args a;
  ssd_accept_args c;
  memset(&a, 0, sizeof a);
  memset(&c, 0, sizeof c);
  if (ssd_version() < 100) return 1;
  if (strcmp(ssd_status_string(SSD_OK), "ok") != 0) return 2;
  /* argument errors come back from host-side validation, before any device work */
  a.B = 1; a.NB = 1; a.Dmax = 4; a.Hq = 4; a.Hkv = 2; a.dh = 96; a.dtype = SSD_BF16;
  if (ssd_verify_attn(&a, NULL, 0, NULL) != SSD_ERR_UNSUPPORTED) return 3;
  c.mode = 7; c.V = 100; c.B = 1; c.NB = 1; c.Dmax = 4; c.chain_blk = -1;
  if (ssd_accept(&c, NULL, 0, NULL) != SSD_ERR_INVALID) return 4;
  c.mode = SSD_GREEDY; c.B = 0;
  if (ssd_accept(&c, NULL, 0, NULL) != SSD_OK) return 5;
  printf("c-abi ok\n");
  return 0;
}
"""


def test_header_is_plain_c_and_links(libpath, tmp_path):
    """A C99 program includes ssd.h with every warning an error, links libssd.so and runs
    host-side calls: the boundary needs no C++ and no torch."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(libpath)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lssd", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c-abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
