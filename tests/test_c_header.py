"""The boundary from C: include/skv.h compiles as strict C11 (gcc -Wall -Werror
-pedantic), and a C program linked against libskv.so calls the host-side
entry points without a GPU -- the version, the size queries, the p-hat
table builder and the argument checks -- with the same results as the
Python binding."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include "skv.h"

int main(void) {
  skv_params p = {0};
  skv_shape s = {2, 2, 2, 256, 64};
  uint64_t *counts = calloc(65536, sizeof(uint64_t));
  uint32_t *ecdf = malloc(sizeof(uint32_t) * 65283);
  float *phat = malloc(sizeof(float) * 65282);
  size_t enc, ws;
  int rc;
  if (!counts || !ecdf || !phat) return 2;
  p.dtype = SKV_BF16;
  p.token_block = 256;
  p.lanes = 8;
  p.sigma = (const float *)(uintptr_t)(1u << 20);
  p.ecdf = (const uint32_t *)(uintptr_t)(1u << 21);
  enc = skv_max_encoded_bytes(&p, &s);
  ws = skv_workspace_bytes(&p, &s, SKV_OP_ENCODE);
  counts[0x3F80] = 1000;
  rc = skv_build_ecdf(counts, ecdf, phat);
  printf("%d %zu %zu %d %u %u\n", skv_version(), enc, ws, rc, ecdf[0], ecdf[65282]);
  /* a range that ends past the last chunk: refused on the host */
  rc = skv_encode_commit(&p, &s, 0, 9, (void *)(uintptr_t)(1u << 20), 1u << 30, NULL,
                         (void *)(uintptr_t)(1u << 20), 1u << 30, NULL);
  printf("%d %s\n", rc, skv_strerror(rc));
  free(counts);
  free(ecdf);
  free(phat);
  return 0;
}
"""


@pytest.fixture(scope="module")
def skv():
    import lossless_kv_cache_fixed_gb300 as P
    P.build()
    return P


def test_header_compiles_as_c_and_links(skv, tmp_path):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(skv.LIB)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", lib_dir, "-lskv", "-Wl,-rpath," + lib_dir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    P = skv
    params = P.SkvParams(P.SKV_BF16, 256, 8, 0, 1 << 20, 1 << 21, None)
    shape = P.SkvShape(2, 2, 2, 256, 64)
    assert int(out[0]) == P.skv_version() == 1
    assert int(out[1]) == P.skv_max_encoded_bytes(params, shape) > 0
    assert int(out[2]) == P.skv_workspace_bytes(params, shape, P.SKV_OP_ENCODE) > 0
    assert int(out[3]) == P.SKV_OK
    assert int(out[4]) == 0 and int(out[5]) == 1 << 26
    assert int(out[6]) == P.SKV_ERR_ARG and out[7] == P.skv_strerror(P.SKV_ERR_ARG).split()[0]
