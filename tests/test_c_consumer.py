"""A plain C program compiles against include/smla.h, links libsmla.so and calls its host-only
entry points (CPU only): the boundary is a C ABI, not only what ctypes sees."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "sparse_mla_decode_smla_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "smla.h"

/* the struct layouts the Python binding assumes */
_Static_assert(sizeof(smla_desc) == 64, "smla_desc");
_Static_assert(sizeof(smla_launch_plan) == 40, "smla_launch_plan");

int main(void) {
  smla_desc d;
  smla_launch_plan p;
  memset(&d, 0, sizeof d);
  /* 64 requests x 4 query tokens, 128 heads, top-k 2048, fp8_ds */
  d.num_tokens = 256; d.num_heads = 128; d.topk = 2048; d.num_requests = 64; d.next_n = 4;
  d.page_size = 64; d.num_pages = 4096; d.page_table_stride = 2048;
  d.kv_format = SMLA_KV_FP8_DS; d.sm_scale = 0.0416666f; d.kv_scale = 1.0f; d.q_scale = 1.0f;
  smla_status st = smla_plan_launches(&d, 152, &p);
  printf("abi %d\n", (int)smla_abi_version());
  printf("status %d %s\n", (int)st, smla_status_string(st));
  printf("plan %d %d %d %d %d %d %d %d %llu\n", (int)p.kernel, (int)p.num_splits, (int)p.split_len,
         (int)p.merge, (int)p.num_launches, (int)p.ctas[0], (int)p.ctas[1], (int)p.tail_items,
         (unsigned long long)p.workspace_bytes);
  d.num_heads = 8; /* not a multiple of 16: rejected on the host */
  st = smla_plan_launches(&d, 152, &p);
  printf("bad %d %d\n", (int)st, (int)p.kernel);
  return 0;
}
"""


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = os.path.join(LIB_DIR, "libsmla.so")
    if not os.path.exists(lib):
        pytest.skip("libsmla.so is not built")
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", LIB_DIR, "-lsmla", f"-Wl,-rpath,{LIB_DIR}"],
                   check=True, capture_output=True, text=True, timeout=120)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout.split("\n")
    assert out[0] == "abi 5"
    assert out[1] == "status 0 ok"
    # head-group kernel, one split of 2048, no merge, 456 CTAs of whole waves + 112 for the last 56 items
    assert out[2] == "plan 1 1 2048 0 2 456 112 56 256"
    assert out[3] == "bad 2 0"
