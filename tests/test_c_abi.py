"""The C ABI from C: a program compiled with gcc against include/wsattn.h and
linked to libwsattn.so builds a plan, reads its geometry, block map and
CSR, checks argument errors and releases it (host-only calls, no GPU)."""
import os
import shutil
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "frame_aligned_window_gb300")

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include "wsattn.h"

int main(void) {
  wsattn_plan_t plan = NULL;
  int rc = wsattn_plan(4, 48, 1, 1, 2, 64, 16, 16, &plan);
  if (rc != WSATTN_OK) { printf("plan %d\n", rc); return 1; }
  int64_t info[10];
  if (wsattn_plan_info(plan, info, 10) != WSATTN_OK) return 2;
  const int64_t nqb = info[3], nkb = info[4], nnz = info[5];
  uint8_t* map = (uint8_t*)malloc((size_t)(nqb * nkb));
  int32_t* rp = (int32_t*)malloc((size_t)(nqb + 1) * sizeof(int32_t));
  int32_t* col = (int32_t*)malloc((size_t)nnz * sizeof(int32_t));
  if (wsattn_get_block_map(plan, map, (size_t)(nqb * nkb)) != WSATTN_OK) return 3;
  if (wsattn_get_csr(plan, rp, col, (size_t)(nqb + 1), (size_t)nnz) != WSATTN_OK) return 4;
  int64_t ones = 0;
  for (int64_t i = 0; i < nqb * nkb; ++i) ones += map[i];
  /* argument errors come back as codes, never as aborts */
  wsattn_plan_t bad = NULL;
  const int e1 = wsattn_plan(4, 48, 1, 1, 2, 64, 24, 16, &bad);   /* 24 is not a multiple of 16 */
  const int e2 = wsattn_plan(4, 48, 1, 1, 2, 96, 16, 16, &bad);   /* head_dim 96 */
  printf("N=%lld nqb=%lld nkb=%lld nnz=%lld ones=%lld rp_last=%d e1=%d e2=%d\n%s\n",
         (long long)info[0], (long long)nqb, (long long)nkb, (long long)nnz, (long long)ones,
         rp[nqb], e1, e2, wsattn_status_string(e1));
  free(map); free(rp); free(col);
  return wsattn_plan_destroy(plan);
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_header(tmp_path):
    src = tmp_path / "use_wsattn.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "use_wsattn"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", PKG, "-lwsattn",
                    "-Wl,-rpath," + PKG], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    first, status_text = r.stdout.splitlines()[:2]
    fields = dict(kv.split("=") for kv in first.split())
    bm = oracle.blockmap(4, 48, 1, 1, 16, 16)
    assert int(fields["N"]) == 240
    assert int(fields["nqb"]) == int(fields["nkb"]) == 15
    assert int(fields["nnz"]) == bm["nnz"] == int(fields["ones"]) == int(fields["rp_last"])
    assert int(fields["e1"]) == 2 and int(fields["e2"]) == 3
    assert status_text.strip()
