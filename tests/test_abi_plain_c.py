"""The boundary is plain C: include/sv.h compiles as C99 on its own (no C++,
no CUDA or torch headers), and a C program links libsv.so and calls it —
version, status names, workspace sizes and host-side argument checks, which
need no GPU."""

import os
import shutil
import subprocess
import textwrap

import pytest

from speculative_decoding_tree_sv_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = textwrap.dedent(r"""
    #include <stdio.h>
    #include <string.h>
    #include "sv.h"

    int main(void) {
      size_t bytes = 0;
      sv_attn_params p;
      int splits = -1, mode = -1;
      if (sv_abi_version() < 1) return 1;
      if (strncmp(sv_status_string(SV_ERR_WORKSPACE), "SV_ERR_WORKSPACE", 16) != 0) return 2;
      if (sv_greedy_accept_workspace_size(4, 100, &bytes) != SV_OK || bytes < 256 + 800) return 3;
      if (sv_sample_accept_workspace_size(4, 100, &bytes) != SV_OK || bytes < 256) return 4;
      if (sv_tree_attention(NULL, NULL) != SV_ERR_INVALID_ARG) return 5;
      memset(&p, 0, sizeof p);
      p.batch = 1;                      /* q and the other pointers left NULL */
      if (sv_tree_attention_plan(&p, &splits, &mode, NULL) != SV_ERR_INVALID_ARG) return 6;
      if (sv_greedy_accept(NULL, 10, NULL, NULL, NULL, 1, 4, 4, 3, NULL, NULL, NULL, NULL, NULL, 0, NULL)
          != SV_ERR_INVALID_ARG) return 7;
      printf("ok %d\n", sv_abi_version());
      return 0;
    }
""")


@pytest.fixture(scope="module")
def lib_path():
    return build.build()


def test_header_and_library_from_plain_c(tmp_path, lib_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "check.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "check"
    libdir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), str(src),
           "-L", libdir, "-lsv", "-Wl,-rpath," + libdir, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith("ok ")
