"""The boundary is plain C: a C99 program includes the header with every
warning an error, links against the library and calls it (CPU only: the
calls below fail or answer before touching a GPU)."""
import os
import shutil
import subprocess

import pytest

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "coli_moe.h"

int main(void) {
  char err[256] = {0};
  coli_moe* h = NULL;
  coli_moe_config cfg = {256, 512, 8, 2, 16, COLI_BF16, COLI_BF16, 0, COLI_PATH_AUTO, 0, 0};
  coli_moe_weights w;
  memset(&w, 0, sizeof w);
  if (strstr(coli_version(), "sm_103a") == NULL) return 10;
  if (strcmp(coli_status_string(COLI_OK), "ok") != 0) return 11;
  /* a NULL config, then weights missing: both rejected before any launch */
  if (coli_moe_create(NULL, &w, NULL, &h, err, sizeof err) != COLI_EINVAL) return 12;
  if (coli_moe_create(&cfg, &w, NULL, &h, err, sizeof err) != COLI_EINVAL) return 13;
  if (h != NULL || err[0] == 0 || coli_last_error()[0] == 0) return 14;
  /* a stage with an impossible size */
  if (coli_route_topk(NULL, NULL, NULL, 4, 100, 8, 2, COLI_BF16, NULL, NULL, NULL, NULL, 0,
                      NULL) != COLI_EINVAL)
    return 15;
  if (coli_permute_scratch_bytes(4, 2, 8) != 0) return 16;
  /* residency query on no handle; a tier with more slots than experts */
  if (coli_moe_residency(NULL, NULL, NULL, NULL) != COLI_EINVAL) return 17;
  cfg.expert_slots = 9;
  if (coli_moe_create(&cfg, &w, NULL, &h, err, sizeof err) != COLI_EINVAL) return 18;
  printf("%s\n", err);
  return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    _build.build()
    return moe.LIB_PATH


def test_c99_program_compiles_links_and_runs(built, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(built)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-l:libcoli_moe.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip()  # the validation message reached the caller's buffer
