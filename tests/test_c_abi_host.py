"""The boundary from plain C: include/pa.h compiles as C11 with warnings as
errors, and a C program linked against libpa.so calls the host packer and the
host-side refusals of the device calls (no GPU needed; nothing is launched)."""
import os
import subprocess

import pytest

from segment_masked_causal_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "segment_masked_causal_gb300", "_build")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pa.h"

#define CHECK(cond) do { if (!(cond)) { printf("FAIL line %d: %s\n", __LINE__, #cond); return 1; } } while (0)

int main(void) {
  /* host packer: three sequences into two rows of 8 tokens */
  const int32_t lengths[3] = {5, 4, 3};
  const int32_t offsets[3] = {2, 0, 1};
  const int32_t tokens[12] = {10, 11, 12, 13, 14, 20, 21, 22, 23, 30, 31, 32};
  int32_t seg[16], rows_tok[16], rows_tgt[16], used = -1;
  uint8_t mask[16];
  int64_t placement[3], placed = -1;
  CHECK(pa_pack_first_fit(lengths, offsets, 3, tokens, -1, 2, 8, 7, 0, seg, mask, rows_tok, rows_tgt, placement,
                          &used, &placed) == PA_OK);
  CHECK(placed == 12 && used == 2);
  int64_t sup = 0;
  for (int i = 0; i < 16; ++i) {
    sup += mask[i];
    CHECK(mask[i] ? rows_tgt[i] == rows_tok[i + 1] : rows_tgt[i] == -1);
  }
  CHECK(sup == (5 - 2) + (4 - 1) + (3 - 1)); /* max(0, L - max(offset, 1)) per sequence */
  for (int s = 0; s < 3; ++s) {
    int64_t at = placement[s], start = 0;
    for (int i = 0; i < s; ++i) start += lengths[i];
    CHECK(at >= 0 && at + lengths[s] <= 16);
    CHECK(memcmp(rows_tok + at, tokens + start, sizeof(int32_t) * (size_t)lengths[s]) == 0);
  }
  CHECK(pa_pack_first_fit(lengths, offsets, 3, NULL, 0, 0, 8, 7, 0, seg, NULL, NULL, NULL, NULL, NULL, NULL) ==
        PA_ERR_SHAPE);
  CHECK(pa_pack_first_fit(lengths, offsets, 3, NULL, 0, 2, 8, 7, 0, seg, NULL, NULL, rows_tgt, NULL, NULL, NULL) ==
        PA_ERR_NULL);

  /* device calls refuse bad arguments on the host, before any device call */
  pa_dims d = {1, 4, 2, 256, 80, 0.0f};
  CHECK(pa_workspace_bytes(&d) == 0);
  void* fake = (void*)0x100000;
  CHECK(pa_fwd(&d, fake, fake, fake, (const int32_t*)fake, fake, (float*)fake, fake, (size_t)1 << 30, NULL) ==
        PA_ERR_HEAD_DIM);
  d.D = 128;
  CHECK(pa_workspace_bytes(&d) > 0 && pa_workspace_bytes_strided(&d) > pa_workspace_bytes(&d));
  CHECK(pa_fwd(&d, fake, fake, fake, NULL, fake, (float*)fake, fake, (size_t)1 << 30, NULL) == PA_ERR_NULL);
  pa_strides st = {4 * 256 * 128, 128, 4 * 128, 2 * 256 * 128, 128, 2 * 128};
  CHECK(pa_fwd_strided(&d, &st, 7, fake, fake, fake, NULL, fake, (float*)fake, fake, (size_t)1 << 30, NULL) ==
        PA_ERR_DTYPE);
  CHECK(pa_lce_workspace_bytes(128, 1000, 96) == 0);
  CHECK(strcmp(pa_status_string(PA_OK), "ok") == 0);
  printf("ok\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    return pabuild.build()


@pytest.fixture(scope="module")
def work_dir(lib_path):
    """Scratch for the C programs, inside the package's (git-ignored) build folder."""
    d = os.path.join(BUILD, "c_abi_test")
    os.makedirs(d, exist_ok=True)
    return d


def test_header_compiles_as_strict_c(work_dir):
    src = os.path.join(work_dir, "h.c")
    exe = os.path.join(work_dir, "h")
    with open(src, "w") as f:
        f.write('#include "pa.h"\nint main(void) { return (int)sizeof(pa_dims) - 24; }\n')
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), "-o", exe, src], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert subprocess.run([exe]).returncode == 0  # pa_dims is 6 x 4 bytes


def test_c_program_against_the_library(lib_path, work_dir):
    src = os.path.join(work_dir, "prog.c")
    exe = os.path.join(work_dir, "prog")
    with open(src, "w") as f:
        f.write(C_PROGRAM)
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        "-o", exe, "-L", os.path.dirname(lib_path), "-lpa",
                        "-Wl,-rpath," + os.path.dirname(lib_path)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip().endswith("ok"), run.stdout + run.stderr
