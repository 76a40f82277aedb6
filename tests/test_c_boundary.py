"""The boundary from C (CPU only): a C99 program that includes both headers compiles with strict
warnings, links against libspecverify.so and calls the entry points that need no GPU (workspace
sizing, host-side argument checks, status strings, the draft-length controller)."""
import os
import shutil
import subprocess

import pytest

import speculative_decoding_rejection_verify_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "spec_verify.h"
#include "spec_control.h"
#include <math.h>
#include <stdio.h>

int main(void) {
  /* workspace sizing: one (max, sum) pair per 16 KB chunk of every row at least, 256-byte multiple */
  size_t n = spec_verify_workspace_bytes(1024, 4, 128256, SPEC_DTYPE_BF16, 0);
  if (n < (size_t)1024 * 9 * 16 * 8 || n % 256 != 0) return 1;
  if (spec_verify_workspace_bytes(-1, 4, 128256, SPEC_DTYPE_BF16, 0) != 0) return 2;
  /* host-checkable errors are returned before any CUDA call */
  spec_status_t s = spec_verify(NULL, NULL, NULL, NULL, NULL, NULL, 1.0f, 0, NULL, NULL, NULL, -1, 4, 100,
                                SPEC_DTYPE_F32, NULL, 0, NULL);
  if (s != SPEC_ERR_INVALID_ARG) return 3;
  if (spec_verify_status_string(s) == NULL) return 4;
  /* the controller: the pages' defaults, then a full window of fully accepted batches raises K */
  spec_ctrl_config_t cfg;
  spec_ctrl_default_config(&cfg);
  if (cfg.k_init != 4 || cfg.k_min != 2 || cfg.k_max != 10 || cfg.window != 100) return 5;
  spec_ctrl_t* c = spec_ctrl_create(&cfg);
  if (c == NULL) return 6;
  const int32_t acc[2] = {4, 4};
  int32_t k = 0;
  for (int i = 0; i < 50; ++i) k = spec_ctrl_update(c, acc, NULL, 2, 4);
  if (k != 4 || fabs(spec_ctrl_window_mean(c) - 1.0) > 1e-12 || spec_ctrl_window_fill(c) != 50) return 8;
  for (int i = 0; i < 50; ++i) k = spec_ctrl_update(c, acc, NULL, 2, 4);
  int64_t a = 0, p = 0, b = 0;
  spec_ctrl_totals(c, &a, &p, &b);
  if (a != 800 || p != 800 || b != 100) return 7;
  if (k <= 4 || k != spec_ctrl_k(c)) return 9;
  spec_ctrl_destroy(c);
  if (spec_ctrl_create(NULL) != NULL || spec_ctrl_k(NULL) != -1) return 10;
  printf("ok %d\n", (int)k);
  return 0;
}
"""


def test_c_program_uses_the_boundary(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = sv.library_path()
    if not os.path.exists(lib):
        sv.load(build_if_missing=True)
    src = tmp_path / "use_boundary.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_boundary"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), f"-L{libdir}", "-l:libspecverify.so", f"-Wl,-rpath,{libdir}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
