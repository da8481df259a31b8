"""The C ABI from C, without Python in between: include/ctxattn.h compiles as
C99 with every warning an error, and a C program links against libctxattn.so
and calls the pure host helpers (no GPU needed), checked on the layouts'
definitions and the DCP page's worked example (block 4, positions 64-79,
wraps to rank 0 with interleave 16 and four ranks)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include "ctxattn.h"

int main(void) {
  int64_t filled = 0;
  int r;
  /* striped storage: row r*Ls + a holds token a*cp + r (cp 4, Ls 8) */
  if (ca_layout_global_index(CA_LAYOUT_STRIPED, 4, 8, 1 * 8 + 3) != 3 * 4 + 1) return 1;
  if (ca_layout_shard_row(CA_LAYOUT_STRIPED, 4, 8, 13) != 1 * 8 + 3) return 2;
  if (ca_layout_global_index(CA_LAYOUT_CONTIGUOUS, 4, 8, 11) != 11) return 3;
  /* ring step 1 of shard 0 meets shard cp - 1 */
  if (ca_ring_kv_shard(0, 1, 8) != 7) return 4;
  /* interleave 16, 4 ranks: positions 64-79 wrap to rank 0, 32-47 on rank 2 */
  if (ca_dcp_owner(70, 4, 16) != 0 || ca_dcp_owner(40, 4, 16) != 2) return 5;
  if (ca_dcp_local_to_global(16, 1, 4, 16) != 80) return 6;
  for (r = 0; r < 4; ++r) filled += ca_dcp_local_filled(100, 4, 16, 16, r);
  if (filled != 100) return 7;
  if (ca_layout_global_index(CA_LAYOUT_STRIPED, 0, 8, 1) != -1) return 8;  /* bad cp */
  printf("%s %d\n", ca_status_string(CA_ERR_SHAPE), ca_version());
  return 0;
}
"""


def test_header_compiles_as_c_and_the_library_links(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    import context_attention_gb300 as ca

    ca.build()
    libdir = os.path.join(ROOT, "context_attention_gb300")
    src = tmp_path / "use_ctxattn.c"
    src.write_text(C_SRC)
    exe = tmp_path / "use_ctxattn"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(exe), f"-L{libdir}", "-lctxattn", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, f"check {r.returncode} failed: {r.stderr}"
    name, version = r.stdout.split()
    assert name == "CA_ERR_SHAPE" and int(version) >= 100
