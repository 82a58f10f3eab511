"""The boundary as a plain C caller sees it, without a GPU: include/dit_attn.h compiles as
strict C99 and as C++17, and a C program linked against libdit_attn.so builds RoPE tables
(checked against the 1-D angle formula written out in C), reads status strings and gets
the documented status for invalid arguments before any CUDA call."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "video_dit_attention_gb300")

C_CALLER = r"""
#include <math.h>
#include <stdio.h>
#include <string.h>
#include "dit_attn.h"

int main(void) {
  enum { S_PAD = 6, L = 4, D = 8, HALF = D / 2, OFFSET = 3 };
  float c[S_PAD * HALF], s[S_PAD * HALF];
  if (dit_rope_table_1d(c, s, S_PAD, L, D, 10000.0, OFFSET) != DIT_OK) return 10;
  for (int r = 0; r < S_PAD; ++r)
    for (int i = 0; i < HALF; ++i) {
      /* row r < L rotates by (OFFSET + r) * 10000^(-2 i / D); pad rows are the identity */
      const double a = r < L ? (OFFSET + r) * pow(10000.0, -2.0 * i / D) : 0.0;
      if (fabs(c[r * HALF + i] - cos(a)) > 1e-6 || fabs(s[r * HALF + i] - sin(a)) > 1e-6) return 11;
    }
  if (dit_rope_table_1d(c, s, S_PAD, S_PAD + 1, D, 10000.0, 0) != DIT_ERR_INVALID_ARG) return 12;
  if (strlen(dit_status_string(DIT_OK)) == 0 || strlen(dit_status_string(DIT_ERR_ALIGNMENT)) == 0) return 13;
  /* invalid arguments: rejected before any pointer is used or any CUDA call is made */
  if (dit_attn_fwd(NULL, NULL, NULL, 1, 256, 256, 2, 128, 256, 256, NULL, NULL, NULL, NULL,
                   0.088f, NULL, NULL, NULL) != DIT_ERR_INVALID_ARG) return 14;
  void* P = (void*)0x10000;
  if (dit_attn_fwd(P, P, P, 1, 256, 256, 2, 96, 256, 256, NULL, NULL, NULL, NULL,
                   0.088f, P, (float*)P, NULL) != DIT_ERR_UNSUPPORTED) return 15;
  if (dit_attn_lse_merge(P, (const float*)P, 0, 1, 128, 2, 128, P, (float*)P, NULL) != DIT_ERR_INVALID_ARG) return 16;
  printf("ok\n");
  return 0;
}
"""


def _tool(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


@pytest.fixture(scope="module")
def libdir():
    if not os.path.exists(os.path.join(PKG, "libdit_attn.so")):
        from video_dit_attention_gb300.build import build
        build()
    return PKG


@pytest.mark.parametrize("compiler,flags", [("gcc", ["-x", "c", "-std=c99"]), ("g++", ["-x", "c++", "-std=c++17"])])
def test_header_compiles_strictly(tmp_path, compiler, flags):
    src = tmp_path / "inc.txt"
    src.write_text('#include "dit_attn.h"\nint main(void) { return dit_status_string(DIT_OK) == 0; }\n')
    subprocess.run([_tool(compiler), *flags, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", INCLUDE, str(src)], check=True)


def test_plain_c_caller_links_and_runs_host_calls(tmp_path, libdir):
    src, exe = tmp_path / "caller.c", tmp_path / "caller"
    src.write_text(C_CALLER)
    subprocess.run([_tool("gcc"), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                    "-L", libdir, "-ldit_attn", f"-Wl,-rpath,{libdir}", "-lm"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
