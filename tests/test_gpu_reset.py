"""The library across a device reset.

The library keeps two device addresses per device: the status word that its
kernels' bounded waits write, and the fixed scratch of the no-alloc decode.
Both belong to the CUDA context that looked them up; after cudaDeviceReset the
device's next context loads the library's module again, possibly at other
addresses, so the library keys the cached addresses on the context.  A plain C
caller (no torch: torch keeps its own state in the old context) runs the
no-alloc decode, resets the device, allocates again and runs the same decode:
the two results must be identical byte for byte, and the status word must read
SDPA_OK after each.
"""
import os
import shutil
import subprocess

import pytest
import torch

import scaled_dot_product_sm_gb300 as sdpa

pytestmark = pytest.mark.gpu

CALLER = r"""
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include "sdpa.h"

enum { B = 2, HQ = 8, HKV = 2, S = 1000, E = 128 };

static uint16_t to_bf16(float x) {   /* round to nearest even; the inputs are finite */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* one no-alloc decode of fixed inputs; 0 on success */
static int run(uint16_t* o_host, float* lse_host) {
  const size_t nq = (size_t)B * HQ * E, nkv = (size_t)B * HKV * S * E;
  uint16_t* h = (uint16_t*)malloc((nq + 2 * nkv) * sizeof(uint16_t));
  uint32_t state = 12345u;
  for (size_t i = 0; i < nq + 2 * nkv; ++i) {   /* uniform in [-1, 1) from a 32-bit LCG */
    state = state * 1664525u + 1013904223u;
    h[i] = to_bf16((float)(state >> 8) / 8388608.0f - 1.0f);
  }
  void *q, *k, *v, *o;
  float* lse;
  if (cudaMalloc(&q, nq * 2) || cudaMalloc(&k, nkv * 2) || cudaMalloc(&v, nkv * 2) || cudaMalloc(&o, nq * 2) ||
      cudaMalloc((void**)&lse, (size_t)B * HQ * sizeof(float)))
    return 10;
  if (cudaMemcpy(q, h, nq * 2, cudaMemcpyHostToDevice) || cudaMemcpy(k, h + nq, nkv * 2, cudaMemcpyHostToDevice) ||
      cudaMemcpy(v, h + nq + nkv, nkv * 2, cudaMemcpyHostToDevice))
    return 11;
  sdpa_shape shp = {B, HQ, HKV, 1, S, E, E, SDPA_BF16, 1, 1};
  sdpa_status st = sdpa_decode_noalloc(&shp, q, k, v, NULL, (double)NAN, 1, 0, o, lse, NULL);
  if (st != SDPA_OK) return 12;
  if (cudaDeviceSynchronize() != cudaSuccess) return 13;
  if (sdpa_last_device_status(NULL) != SDPA_OK) return 14;
  if (cudaMemcpy(o_host, o, nq * 2, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(lse_host, lse, (size_t)B * HQ * sizeof(float), cudaMemcpyDeviceToHost))
    return 15;
  cudaFree(q); cudaFree(k); cudaFree(v); cudaFree(o); cudaFree(lse);
  free(h);
  return 0;
}

int main(void) {
  static uint16_t o1[B * HQ * E], o2[B * HQ * E];
  static float l1[B * HQ], l2[B * HQ];
  int rc = run(o1, l1);
  if (rc) return rc;
  if (cudaDeviceReset() != cudaSuccess) return 20;
  rc = run(o2, l2);
  if (rc) return 30 + rc;
  if (memcmp(o1, o2, sizeof(o1)) || memcmp(l1, l2, sizeof(l1))) return 40;
  for (int i = 0; i < B * HQ; ++i)
    if (!(l1[i] > 0.0f && l1[i] < 100.0f)) return 41;   /* finite, plausible log-sum-exp */
  printf("same\n");
  return 0;
}
"""


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_noalloc_decode_and_status_survive_a_device_reset(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    sdpa.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(sdpa.LIB_PATH)
    cuda = _cuda_home()
    cudalib = next((os.path.join(cuda, d) for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
                    if os.path.exists(os.path.join(cuda, d, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("no libcudart.so found")
    src = tmp_path / "reset.c"
    src.write_text(CALLER)
    exe = tmp_path / "reset"
    r = subprocess.run([cc, "-std=c11", "-O1", "-I", os.path.join(root, "include"), "-I", os.path.join(cuda, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lsdpa_gb300", "-L", cudalib, "-lcudart",
                        f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    env.setdefault("CUDA_VISIBLE_DEVICES", str(torch.cuda.current_device()))
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120, env=env)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.strip() == "same"
