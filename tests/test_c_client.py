"""The boundary used from plain C: a C99 program that includes
include/lopt.h, links the in-tree liblopt.so and calls the entry points
that need no device (version, error strings, weight-set size, the launch
schedule of a ragged list).  Compiled with gcc and run on the CPU."""

import os
import shutil
import subprocess

import pytest

from learned_optimizer_step_gb300 import build as B

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "lopt.h"

int main(void) {
  lopt_tensor t[3];
  int32_t n_units[3], n_groups = -1, strips[3];
  int32_t units[2 * 64];
  memset(t, 0, sizeof(t));
  t[0].rows = 300; t[0].cols = 200;       /* 60,000 elements */
  t[1].rows = 1;   t[1].cols = 5000;      /* a [1 x n] view */
  t[2].rows = 7;   t[2].cols = 9;
  if (lopt_version() < 100) return 1;
  if (strcmp(lopt_strerror(LOPT_OK), "ok") != 0) return 2;
  if (lopt_weight_set_size(39, 32) != 39 * 32 + 32 + 32 * 32 + 32 + 64 + 2) return 3;
  if (lopt_schedule_info(t, 3, 0, n_units, NULL, NULL, &n_groups, NULL) != LOPT_OK) return 4;
  if (n_units[0] + n_units[1] + n_units[2] > 64) return 5;
  if (lopt_schedule_info(t, 3, 0, n_units, units, strips, &n_groups, NULL) != LOPT_OK) return 6;
  if (lopt_schedule_info(t, -1, 0, n_units, NULL, NULL, &n_groups, NULL) != LOPT_E_ARG) return 7;
  printf("%d %d %d %d %d %d %d\n", n_units[0], n_units[1], n_units[2], n_groups,
         strips[0], strips[1], strips[2]);
  return 0;
}
"""


def test_c_program_links_the_library_and_reads_the_schedule(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = B.build()
    src = tmp_path / "client.c"
    exe = tmp_path / "client"
    src.write_text(C_SRC)
    libdir = os.path.dirname(lib)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(B.ROOT, "include"), str(src),
                    "-o", str(exe), "-L", libdir, "-l:liblopt.so", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    k0, k1, k2, groups, s0, s1, s2 = map(int, out.stdout.split())
    # K1 chunks of 16,384 and K2 chunks of 4,096 elements per tensor
    assert k1 == 4 + 1 + 1 and k2 == 15 + 2 + 1 and groups == 0
    assert s1 == 1 and 1 <= s0 <= 300 and 1 <= s2 <= 7
    assert k0 == -(-300 // s0) + 1 + -(-7 // s2)
