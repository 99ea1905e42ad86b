"""The C ABI from plain C: include/sp24.h compiles as C99 and C++17 with every
warning on, and a C program linked against libsp24.so calls the entry points
that need no GPU (status strings, metadata size, decomposition modes)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp24.h")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sp24.h"

int main(void) {
  /* every status has a distinct, non-empty name */
  for (int s = SP24_OK; s <= SP24_ERR_DEVICE_TIMEOUT; ++s) {
    const char* name = sp24_status_string((sp24_status)s);
    if (name == NULL || name[0] == '\0') return 10 + s;
    for (int t = SP24_OK; t < s; ++t)
      if (strcmp(name, sp24_status_string((sp24_status)t)) == 0) return 30 + s;
  }
  /* one 4-bit entry per group of four along K */
  if (sp24_meta_bytes(4096, 4096) != (size_t)4096 * 4096 / 8) return 50;
  if (sp24_meta_bytes(128, 128) != 2048) return 51;
  /* the decomposition modes */
  if (sp24_set_decomposition(SP24_DECOMP_CLUSTER_SPLIT) != SP24_OK) return 60;
  if (sp24_set_decomposition(SP24_DECOMP_STREAM_K) != SP24_OK) return 61;
  if (sp24_set_decomposition(SP24_DECOMP_DATA_PARALLEL) != SP24_OK) return 62;
  if (sp24_set_decomposition(7) != SP24_ERR_INVALID_ARG) return 63;
  if (sp24_set_decomposition(SP24_DECOMP_HEURISTIC) != SP24_OK) return 64;
  /* invalid shapes are refused before any device work */
  if (sp24_fp8_gemm_decomposition(0, 4096, 4096, 0, NULL) != -1) return 70;
  if (sp24_fp8_gemm_workspace_size(16, 100, 4096, 0) != 0) return 71;
  puts("c-abi ok");
  return 0;
}
"""


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    return cc


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_cleanly(lang, std):
    cc = _cc() if lang == "c" else (shutil.which("g++") or pytest.skip("no C++ compiler"))
    r = subprocess.run([cc, std, "-fsyntax-only", "-Wall", "-Wextra", "-Werror", "-pedantic", "-x", lang, HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_runs(tmp_path):
    import semi_structured_sparse_gb300 as sp24
    lib = sp24.build.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([_cc(), "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        lib, "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # host-only entry points: no GPU is touched
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, "exit %d: %s %s" % (r.returncode, r.stdout, r.stderr)
    assert "c-abi ok" in r.stdout
