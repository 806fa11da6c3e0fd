"""The FMA-pipe 2^x used for part of the forward's exponentials (scalar and paired forms),
against CUDA's exp2f, on the GPU: relative error within the polynomial's minimax bound (7.5e-5)
plus single-precision rounding, over the range the softmax feeds it (scores minus the running
max: at most 8).  The paired form must agree with the scalar one bit for bit."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

from exact_attention_50_gb300 import build

pytestmark = pytest.mark.gpu

PROGRAM = r'''
#include <cstdio>
#include <cmath>
#include "ptx.cuh"
__global__ void k(const float* x, float* a, float* b, float* c, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) { a[i] = attn::exp2_fma(x[i]); b[i] = exp2f(x[i]); }
  if (2 * i + 1 < n) {
    const float2 r = attn::f2_unpack(attn::exp2_fma2(attn::f2_pack(x[2 * i], x[2 * i + 1])));
    c[2 * i] = r.x;
    c[2 * i + 1] = r.y;
  }
}
int main() {
  const int n = 1 << 20;
  float *x, *a, *b, *c;
  cudaMallocManaged(&x, n * 4); cudaMallocManaged(&a, n * 4); cudaMallocManaged(&b, n * 4);
  cudaMallocManaged(&c, n * 4);
  for (int i = 0; i < n; ++i) x[i] = -120.0f + 128.0f * (float)i / (float)(n - 1);  // [-120, 8]
  k<<<(n + 255) / 256, 256>>>(x, a, b, c, n);
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  double worst = 0;
  int mismatch = 0;
  for (int i = 0; i < n; ++i) {
    double r = fabs((double)a[i] - (double)b[i]) / (double)b[i];
    if (r > worst) worst = r;
    if (a[i] != c[i]) ++mismatch;
  }
  printf("%.6e %d\n", worst, mismatch);
  return 0;
}
'''


def test_exp2_fma_relative_error():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "e.cu")
        exe = os.path.join(d, "e")
        open(src, "w").write(PROGRAM)
        subprocess.run([build.nvcc(), *build.ARCH, "-O3", "-std=c++17", "-I" + build.CSRC, "-I" + build.INCLUDE,
                        src, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    worst, mismatch = out.split()
    assert float(worst) <= 7.5e-5 + 4 * 2.0 ** -24, worst
    assert int(mismatch) == 0, mismatch
