"""The C ABI end to end from a plain C program, without Python in the data
path: the client allocates device memory with the CUDA runtime, copies seeded
inputs in, runs moe_route_expand_cast_fp8 (AUTO) on the default stream, reads
every output back and checks what the method fixes (TileKernels article,
sections 2.1-3.2): each token's k experts are the k largest scores, lower
index first on ties, in descending order; the weights sum to 1; counts sum to
T*k and offsets are their exclusive scan; pos and sorted_src are inverse
permutations, stable within each expert; all k copies of a token carry the
same codes and scales.  The oracle comparisons of the same call are in the
other GPU tests."""
import os
import shutil
import subprocess

import pytest

from moe_routing_precision_gb300 import _build

pytestmark = pytest.mark.gpu

CLIENT = r"""
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include "moe_route.h"

#define T 1000
#define E 64
#define K 4
#define H 512
#define G (H / 128)
#define R (T * K)
#define CK(x) do { if ((x) != cudaSuccess) { printf("cuda %d\n", __LINE__); return 10; } } while (0)

static uint32_t lcg = 12345u;
static float uni(void) { lcg = lcg * 1664525u + 1013904223u; return (lcg >> 8) * (1.0f / 16777216.0f); }
static uint16_t to_bf16(float f) { uint32_t b; memcpy(&b, &f, 4); return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16); }

int main(void) {
  static float scores[T * E], w[T * K];
  static uint16_t x[T * H];
  static int32_t idx[T * K], counts[E], offsets[E + 1], pos[T * K], src[R];
  static uint8_t q[(size_t)R * H];
  static float sf[R * G];
  for (int i = 0; i < T * E; ++i) scores[i] = (float)(int)(uni() * 40.0f) * 0.25f;  /* ties */
  for (int i = 0; i < T * H; ++i) x[i] = to_bf16(uni() * 8.0f - 4.0f);
  float *d_s, *d_w, *d_sf; uint16_t *d_x; uint8_t *d_q, *d_ws;
  int32_t *d_idx, *d_counts, *d_off, *d_pos, *d_src;
  size_t wsb = moe_route_expand_cast_fp8_workspace_bytes(T, E, K);
  CK(cudaMalloc((void **)&d_s, sizeof scores)); CK(cudaMalloc((void **)&d_x, sizeof x));
  CK(cudaMalloc((void **)&d_w, sizeof w)); CK(cudaMalloc((void **)&d_idx, sizeof idx));
  CK(cudaMalloc((void **)&d_counts, sizeof counts)); CK(cudaMalloc((void **)&d_off, sizeof offsets));
  CK(cudaMalloc((void **)&d_pos, sizeof pos)); CK(cudaMalloc((void **)&d_src, sizeof src));
  CK(cudaMalloc((void **)&d_q, sizeof q)); CK(cudaMalloc((void **)&d_sf, sizeof sf));
  CK(cudaMalloc((void **)&d_ws, wsb)); CK(cudaMemset(d_ws, 0, wsb));
  CK(cudaMemcpy(d_s, scores, sizeof scores, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));
  moe_status_t st = moe_route_expand_cast_fp8(d_s, T, E, K, d_x, H, d_idx, d_w, d_counts, d_off,
                                              d_pos, d_src, d_q, d_sf, d_ws, wsb, MOE_PATH_AUTO,
                                              128, NULL);
  if (st != MOE_OK) { printf("status %s\n", moe_status_string(st)); return 11; }
  uint32_t bits = 1;
  if (moe_get_device_status(NULL, &bits) != MOE_OK || bits != 0) return 12;
  CK(cudaMemcpy(idx, d_idx, sizeof idx, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(w, d_w, sizeof w, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(counts, d_counts, sizeof counts, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(offsets, d_off, sizeof offsets, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(pos, d_pos, sizeof pos, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(src, d_src, sizeof src, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(q, d_q, sizeof q, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(sf, d_sf, sizeof sf, cudaMemcpyDeviceToHost));
  for (int t = 0; t < T; ++t) {
    /* the k largest, lower index first on ties, in descending order */
    int used[E] = {0};
    float wsum = 0.0f;
    for (int j = 0; j < K; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!used[e] && (best < 0 || scores[t * E + e] > scores[t * E + best])) best = e;
      used[best] = 1;
      if (idx[t * K + j] != best) { printf("topk t=%d j=%d\n", t, j); return 20; }
      wsum += w[t * K + j];
    }
    if (wsum < 0.9999f || wsum > 1.0001f) return 21;
  }
  int64_t tot = 0;
  if (offsets[0] != 0) return 30;
  for (int e = 0; e < E; ++e) { tot += counts[e]; if (offsets[e + 1] != offsets[e] + counts[e]) return 31; }
  if (tot != R) return 32;
  for (int p = 0; p < R; ++p) {
    int r = pos[p];
    if (r < 0 || r >= R || src[r] != p) return 33;
    int e = idx[p];
    if (r < offsets[e] || r >= offsets[e + 1]) return 34;
    if (r > offsets[e] && src[r - 1] > p) return 35;  /* stable: ascending copy index */
  }
  for (int t = 0; t < T; ++t) {
    const int r0 = pos[t * K];
    for (int j = 1; j < K; ++j) {
      const int r = pos[t * K + j];
      if (memcmp(q + (size_t)r * H, q + (size_t)r0 * H, H) != 0) return 40;
      if (memcmp(sf + (size_t)r * G, sf + (size_t)r0 * G, G * sizeof(float)) != 0) return 41;
    }
    for (int g = 0; g < G; ++g) if (!(sf[(size_t)r0 * G + g] > 0.0f)) return 42;
  }
  printf("OK\n");
  return 0;
}
"""


def test_c_client_route_expand_cast():
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("gcc not installed")
    lib = _build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    tmp = os.path.join(os.path.dirname(lib), "_build", "c_client")
    os.makedirs(tmp, exist_ok=True)
    src = os.path.join(tmp, "client.c")
    with open(src, "w") as f:
        f.write(CLIENT)
    exe = os.path.join(tmp, "client")
    libdir = os.path.dirname(lib)
    cudalib = next((d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                os.path.join(cuda, "targets", "sbsa-linux", "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so"))), os.path.join(cuda, "lib64"))
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Werror", f"-I{_build.INCLUDE}",
           f"-I{os.path.join(cuda, 'include')}", src, f"-L{libdir}", "-lmoe_route",
           f"-L{cudalib}", "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "OK", (r.returncode, r.stdout, r.stderr)
