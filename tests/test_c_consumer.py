"""The C ABI is usable from plain C.

A C99 program that includes only include/dspark.h (no CUDA headers) is
compiled with gcc, linked against libdspark.so and run; it calls the entry
points that need no GPU: the version, the workspace-size queries and host
validation that rejects bad arguments before any launch.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "dspark.h"

int main(void) {
  int bad = 0;
  if (dspark_version() <= 0) bad |= 1;
  if (dspark_chain_workspace_size(256, 7) < 256 + 256 * 7 * 8) bad |= 2;
  if (dspark_select_workspace_size(256, 7, 8192) == 0) bad |= 4;
  /* NULL pointers: rejected on the host, nothing launched */
  if (dspark_chain_draft(NULL, DSPARK_BF16, 7 * 1024, 1024, NULL, NULL, NULL,
                         4, 7, 1024, 16, NULL, NULL, NULL, 0, NULL)
      != DSPARK_ERR_INVALID_ARG) bad |= 8;
  if (dspark_select_step(NULL, NULL, 4, 7, NULL, 64, NULL, 0.0f, 0u, NULL,
                         NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                         NULL, NULL, NULL, 0, NULL) != DSPARK_ERR_INVALID_ARG) bad |= 16;
  if (dspark_chain_sample(NULL, DSPARK_BF16, 7 * 1024, 1024, NULL, NULL, NULL,
                          4, 7, 1024, 16, 1u, 0u, 0.0f, NULL, NULL, NULL, 0, NULL)
      != DSPARK_ERR_INVALID_ARG) bad |= 32;
  printf("%d\n", bad);
  return bad;
}
"""


def test_plain_c_program_uses_the_abi(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_draft_dspark_gb300 import dspark as D
    lib = D.LIB_PATH
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    lib, "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.stdout, r.stderr)
