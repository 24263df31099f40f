// peak_copy.cu -- a plain 16-byte vectorised device copy, used only to measure
// the HBM bandwidth the path's kernels are held against (read + write bytes).
// Four independent 16-byte loads per thread are in flight before the stores.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) peak_copy_kernel(const uint4* __restrict__ src,
                                                             uint4* __restrict__ dst, int64_t n) {
  pdl_enter();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream_v4(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_stream_v4(dst + i + u * stride, v[u]);
  }
  for (; i < n; i += stride) st_stream_v4(dst + i, ld_stream_v4(src + i));
}

}  // namespace

cudaError_t launch_peak_copy(const LaunchCtx& c, const void* src, void* dst, size_t bytes) {
  const int64_t n = (int64_t)(bytes / 16);
  int per_sm = 0;
  cudaError_t st =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, peak_copy_kernel, kThreads, 0);
  if (st != cudaSuccess) return st;
  const int64_t need = (n + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(peak_copy_kernel, blocks, kThreads, 0, c.stream,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), n);
}

}  // namespace moe
