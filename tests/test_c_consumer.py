"""The C ABI from a plain C program (no GPU): include/fa.h compiles as C99
with warnings as errors, and a program linked against libfa.so gets the
documented answers from the calls that need no device (version, error
strings, workspace sizes, argument checks, empty problems)."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fa.h"

static int fails = 0;
#define CHECK(cond) do { if (!(cond)) { printf("FAIL line %d: %s\n", __LINE__, #cond); ++fails; } } while (0)

int main(void) {
  static unsigned char buf[4096] __attribute__((aligned(256)));
  void* p = buf;
  CHECK(fa_version() >= 100);
  CHECK(strlen(fa_strerror(FA_ERR_INVALID)) > 0);
  CHECK(strlen(fa_strerror(12345)) > 0);
  CHECK(fa_bwd_workspace_bytes(1, 1, 8, 64) > 0);
  CHECK(fa_bwd_workspace_bytes(0, 1, 8, 64) == 0);
  /* argument checks happen before any device is touched */
  CHECK(fa_fwd(NULL, p, p, p, (float*)p, 1, 1, 8, 64, 0, 0.125f) == FA_ERR_INVALID);
  CHECK(fa_fwd(p, p, p, p, (float*)p, 1, 1, 8, 96, 0, 0.125f) == FA_ERR_UNSUPPORTED);
  CHECK(fa_fwd(p, p, p, p, (float*)p, 1, 1, 8, 64, 0, -1.0f) == FA_ERR_INVALID);
  CHECK(fa_fwd_dropout(p, p, p, p, (float*)p, 1, 1, 8, 64, 0, 0.125f, 1.0f, 1ull, 0ull, NULL)
        == FA_ERR_INVALID);
  CHECK(fa_bwd_stream(p, p, p, p, (const float*)p, p, p, p, p, 1, 1, 8, 64, 0, 0.125f, NULL, 0, NULL)
        == FA_ERR_WORKSPACE);
  /* empty problems are no-ops */
  CHECK(fa_fwd(NULL, NULL, NULL, NULL, NULL, 0, 4, 128, 64, 0, 0.125f) == FA_OK);
  CHECK(fa_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 0, 64, 64, 0, 0.125f) == FA_OK);
  printf("%s\n", fails ? "failed" : "ok");
  return fails != 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from exact_io_aware_33_gb300 import build
    return os.path.dirname(build.build())


def test_header_is_c99_and_the_library_links(libdir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lfa", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("ok")
