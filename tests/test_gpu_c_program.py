"""The C ABI driven from a plain C program on the GPU (no PyTorch in the
process): it allocates device memory itself, queries and passes the
workspace, runs a causal striped const-max ring forward on the legacy default
stream, reads back o and lse, and the test compares them with the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "ctxattn.h"

static float* load(const char* path, size_t n) {
  float* h = (float*)malloc(n * sizeof(float));
  FILE* f = fopen(path, "rb");
  if (!h || !f || fread(h, sizeof(float), n, f) != n) exit(10);
  fclose(f);
  return h;
}

int main(int argc, char** argv) {
  const int B = 1, Hq = 4, Hkv = 2, S = 384, D = 64, cp = 3;
  const size_t nq = (size_t)B * Hq * S * D, nk = (size_t)B * Hkv * S * D, nl = (size_t)B * Hq * S;
  float *hq, *hk, *hv, *ho, *hl, *dq, *dk, *dv, *dO, *dl;
  void* ws = NULL;
  size_t wsb;
  ca_status st;
  FILE* f;
  if (argc != 2) return 11;
  (void)argv;
  hq = load("q.bin", nq);
  hk = load("k.bin", nk);
  hv = load("v.bin", nk);
  ho = (float*)malloc(nq * sizeof(float));
  hl = (float*)malloc(nl * sizeof(float));
  if (cudaMalloc((void**)&dq, nq * 4) || cudaMalloc((void**)&dk, nk * 4) || cudaMalloc((void**)&dv, nk * 4) ||
      cudaMalloc((void**)&dO, nq * 4) || cudaMalloc((void**)&dl, nl * 4))
    return 12;
  cudaMemcpy(dq, hq, nq * 4, cudaMemcpyHostToDevice);
  cudaMemcpy(dk, hk, nk * 4, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, hv, nk * 4, cudaMemcpyHostToDevice);
  wsb = ca_ring_attn_fwd_workspace_size(B, Hq, Hkv, S, D, cp, CA_MODE_CONST_MAX);
  if (wsb && cudaMalloc(&ws, wsb)) return 13;
  st = ca_ring_attn_fwd(dq, dk, dv, dO, dl, CA_DTYPE_F32, B, Hq, Hkv, S, D, cp, CA_MODE_CONST_MAX, 1,
                        CA_LAYOUT_STRIPED, 0.0f, ws, wsb, NULL);
  if (st != CA_OK) {
    fprintf(stderr, "%s\n", ca_status_string(st));
    return 14;
  }
  if (cudaDeviceSynchronize() != cudaSuccess || ca_device_status(0) != CA_OK) return 15;
  cudaMemcpy(ho, dO, nq * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(hl, dl, nl * 4, cudaMemcpyDeviceToHost);
  f = fopen("o.bin", "wb");
  if (!f || fwrite(ho, 4, nq, f) != nq) return 16;
  fclose(f);
  f = fopen("lse.bin", "wb");
  if (!f || fwrite(hl, 4, nl, f) != nl) return 17;
  fclose(f);
  printf("ok\n");
  return 0;
}
"""


def test_c_program_runs_the_ring_on_the_gpu(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    import context_attention_gb300 as ca

    ca.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.join(ROOT, "context_attention_gb300")
    rng = np.random.default_rng(71)
    q = rng.standard_normal((1, 4, 384, 64)).astype(np.float32)
    k = rng.standard_normal((1, 2, 384, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 384, 64)).astype(np.float32)
    for name, x in (("q", q), ("k", k), ("v", v)):
        x.tofile(tmp_path / f"{name}.bin")
    src = tmp_path / "ring.c"
    src.write_text(C_SRC)
    exe = tmp_path / "ring"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(cuda, "include"), str(src), "-o", str(exe), f"-L{libdir}", "-lctxattn", f"-Wl,-rpath,{libdir}",
           f"-L{os.path.join(cuda, 'lib64')}", "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe), "run"], capture_output=True, text=True, cwd=tmp_path, timeout=120)
    assert r.returncode == 0, f"step {r.returncode}: {r.stderr}"
    o = np.fromfile(tmp_path / "o.bin", dtype=np.float32).reshape(q.shape)
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32).reshape(q.shape[:3])
    ro, rl, _ = oracle.ring(q, k, v, 3, mode=oracle.MODE_CONST_MAX, causal=True, layout=oracle.LAYOUT_STRIPED)
    import torch

    assert_close(o, ro, lse, rl, dtype=torch.float32, what="C program, fp32 const max causal striped")
