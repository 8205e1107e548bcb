"""The boundary from C: a plain C11 program includes include/bsattn.h, links
libbsattn.so and makes host-side calls (sizes, status text, head-configuration
checks, argument rejection before any launch). Nothing here touches a GPU."""
import os
import shutil
import subprocess

import pytest

from long_context_serving_gb300 import bsattn as B
from long_context_serving_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "bsattn.h"

int main(void) {
  bs_dims d;
  memset(&d, 0, sizeof d);
  d.batch = 2; d.n_q_heads = 8; d.n_kv_heads = 2; d.head_dim = 128; d.page_size = 16;
  d.max_pages_per_unit = 64; d.max_blocks_per_unit = 32; d.max_sel_per_unit = 16;
  d.max_subs_per_unit = 128; d.max_gather_pages_per_unit = 32; d.n_pages = 128;
  d.kv_dtype = BS_BF16; d.q_dtype = BS_BF16;
  printf("workspace %zu\n", bs_workspace_size(&d));
  printf("status %s\n", bs_status_string(BS_ERR_CAPACITY));

  int32_t cls[4] = {BS_RETRIEVAL, BS_STREAMING, BS_DUAL, BS_RETRIEVAL};
  int32_t g[4] = {32, 32, 32, 32}, s[4] = {8, 8, 8, 8}, k[4] = {4, 0, 4, 4}, ke[4] = {0, 0, 2, 0};
  int32_t sink[4] = {32, 32, 32, 32}, local[4] = {32, 32, 32, 32}, rows[4] = {128, 128, 128, 128};
  int64_t off[4] = {0, 16384, 32768, 49152};
  bs_head_cfg c = {cls, g, s, k, ke, sink, local, off, rows};
  int32_t lens[2] = {500, 1000};
  printf("cfg_ok %d\n", (int)bs_check_head_cfg(&d, &c, lens));
  g[3] = 24;  /* not a multiple of the 16-token page */
  printf("cfg_bad_g %d\n", (int)bs_check_head_cfg(&d, &c, lens));
  g[3] = 32;
  lens[1] = 5000;  /* more pages than a page-table row holds */
  printf("cfg_long %d\n", (int)bs_check_head_cfg(&d, &c, lens));

  /* Rejected on the host before anything is enqueued. */
  printf("attn_null %d\n", (int)bs_sparse_decode_attn(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                                      NULL, 0, NULL, NULL));
  d.head_dim = 96;
  printf("ws_bad %zu\n", bs_workspace_size(&d));
  printf("setdiff_shape %d\n", (int)bs_block_setdiff(&d, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                                     NULL, NULL));
  return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("needs a C compiler")
    lib = build()
    d = tmp_path_factory.mktemp("c_abi")
    src, exe = d / "main.c", d / "main"
    src.write_text(PROGRAM)
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), lib, "-Wl,-rpath," + libdir], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def _py_dims():
    return B.Dims(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, max_pages_per_unit=64,
                  max_blocks_per_unit=32, max_sel_per_unit=16, max_subs_per_unit=128,
                  max_gather_pages_per_unit=32, n_pages=128, kv_dtype=B.BS_BF16, q_dtype=B.BS_BF16)


def test_sizes_and_status_text(program):
    assert int(program["workspace"]) == B.workspace_size(_py_dims()) > 0
    assert program["status"] == "capacity exceeded"
    assert int(program["ws_bad"]) == 0


def test_head_configuration_checks(program):
    assert int(program["cfg_ok"]) == B.BS_OK
    assert int(program["cfg_bad_g"]) == B.BS_ERR_INVALID_ARG
    assert int(program["cfg_long"]) == B.BS_ERR_CAPACITY


def test_calls_reject_before_launch(program):
    assert int(program["attn_null"]) == B.BS_ERR_INVALID_ARG
    assert int(program["setdiff_shape"]) == B.BS_ERR_SHAPE
