"""The boundary from C itself: a C99 program that includes include/attn_fwd.h,
links the library and calls it (validation paths only: no GPU is needed)."""
import os
import shutil
import subprocess

import pytest

from bf16_forward_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn_fwd.h"

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL %s\n", #cond); ++fails; } } while (0)

int main(void) {
  char buf[64];
  void* q = (void*)buf;  /* never dereferenced on these paths */
  EXPECT(attn_fwd_version() >= 100);
  EXPECT(strcmp(attn_status_str(ATTN_OK), "ok") == 0);
  EXPECT(attn_fwd(NULL, q, q, q, ATTN_LAYOUT_BHSD, 1, 1, 1, 1, 128, 0.1f, ATTN_ROUND_RTNE, NULL)
         == ATTN_ERR_INVALID_ARG);
  EXPECT(attn_fwd((void*)0x100000, (void*)0x200000, (void*)0x300000, (void*)0x400000,
                  ATTN_LAYOUT_BSHD, 1, 1, 1, 1, 64, 0.1f, ATTN_ROUND_RTZ, NULL)
         == ATTN_ERR_UNSUPPORTED);
  EXPECT(attn_fwd_ex((void*)0x100000, (void*)0x200000, (void*)0x300000, (void*)0x400000,
                     ATTN_LAYOUT_BHSD, 1, 6, 4, 16, 16, 128, 0.1f, ATTN_ROUND_RTNA,
                     ATTN_FLAG_CAUSAL, NULL) == ATTN_ERR_INVALID_ARG);
  EXPECT(attn_fwd_splitkv_workspace_bytes(1, 2, 256, 1000, 128, 2) > 0);
  EXPECT(attn_fwd_split_tail_items(0, 1, 1, 1) == ATTN_ERR_INVALID_ARG);
  EXPECT(ATTN_FLAG_SPLIT_TAIL == 2 && (ATTN_FLAG_SPLIT_TAIL & ATTN_FLAG_CAUSAL) == 0);
  EXPECT(attn_fwd_host_workspace_bytes(1, 2, 2, 256, 256, 128) == 4 * 2 * 256 * 256);
  EXPECT(attn_fwd_debug_build() == 0 || attn_fwd_debug_build() == 1);
  printf("%s\n", fails ? "C-ABI FAILED" : "C-ABI OK");
  return fails != 0;
}
"""


def test_c_program_links_and_calls_the_library(tmp_path):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    if not build.up_to_date():
        build.build()
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(build.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", lib_dir, "-lattn_fwd", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C-ABI OK" in r.stdout
