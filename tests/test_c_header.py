"""include/pkv.h is a plain C header: a C99 program that includes it compiles
with every warning an error, links against libpkv.so and calls entry points
that need no GPU (version, status text, host-side validation)."""
import os
import shutil
import subprocess

import pytest

import paged_kv_attention_31_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PROGRAM = r"""
#include "pkv.h"
#include <stdio.h>
int main(void) {
  pkv_pool_desc d = {0};
  printf("%d|%s\n", (int)pkv_version(), pkv_status_string(PKV_ERR_OUT_OF_BLOCKS));
  /* a zeroed pool descriptor is refused before any CUDA call */
  return pkv_kv_append(0, 0, 0, 1, 0, 0, &d, 0) == PKV_ERR_INVALID_ARG ? 0 : 1;
}
"""


def test_c99_program_builds_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pkv.lib()  # the library must be built
    libdir = os.path.dirname(pkv.LIB_PATH)
    src, exe = tmp_path / "t.c", tmp_path / "t"
    src.write_text(_PROGRAM)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lpkv",
                        f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    version, text = r.stdout.strip().split("|")
    assert int(version) == int(pkv.lib().pkv_version()) and text == "not enough free KV-cache blocks"
