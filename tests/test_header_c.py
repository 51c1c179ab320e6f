"""The boundary is plain C: a C11 program that includes include/sageattn.h (no C++, no torch)
compiles with warnings as errors, links against libsageattn.so and calls the host-only
entry points (workspace sizes, status strings, host-side validation) without a GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_attention_mean_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sageattn.h"

int main(void) {
  /* workspace for 2x8 heads, 4096 tokens, head_dim 128, per-warp groups */
  size_t ws = sage_attn_workspace_size(2, 8, 8, 4096, 4096, 128, 1);
  if (ws == 0) return 1;
  /* invalid head_dim: no workspace size */
  if (sage_attn_workspace_size(1, 2, 2, 256, 256, 200, 1) != 0) return 2;
  if (sage_attn_varlen_workspace_size(16, 32, 32, 70000, 70000, 128, 1) == 0) return 3;
  if (strcmp(sage_status_string(SAGE_OK), sage_status_string(SAGE_ERR_INVALID_ARG)) == 0) return 4;
  /* host validation rejects null tensors before touching any device */
  if (sage_attn(NULL, NULL, NULL, NULL, NULL, 1, 2, 2, 8, 8, 64, 0, 0, 0, 0.0f, 0, 1, 0, 1, 0,
                NULL, 0, NULL) != SAGE_ERR_INVALID_ARG) return 5;
  printf("ok %zu\n", ws);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_uses_the_abi(tmp_path):
    lib = os.path.join(PKG, "libsageattn.so")
    if not os.path.exists(lib):
        pytest.skip("libsageattn.so not built")
    src = tmp_path / "abi_demo.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi_demo"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", PKG, "-lsageattn", f"-Wl,-rpath,{PKG}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.startswith("ok ")
