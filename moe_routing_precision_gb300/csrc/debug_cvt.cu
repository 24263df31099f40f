// debug_cvt.cu -- the device's f32 -> FP8 E4M3 and f32 -> FP4 E2M1
// conversions on arbitrary values, so that tests can compare them with the
// oracle's encoders over every bit pattern.  The cast kernels use exactly
// these conversions (e4m3x2, e2m1x2 in common.cuh) on x * (1 / scale).
#include "common.cuh"

namespace moe {
namespace {

// Four values per thread: 16-byte loads, one 4-byte store of four codes (one
// code per byte; E2M1 codes in the low nibble).
__global__ void __launch_bounds__(256) cvt_kernel(const float4* __restrict__ in,
                                                  uint32_t* __restrict__ out, int64_t n4,
                                                  int fmt) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = __ldcs(in + i);
    uint32_t c;
    if (fmt == MOE_DEBUG_CVT_E4M3) {
      c = e4m3x2(v.x, v.y) | (e4m3x2(v.z, v.w) << 16);
    } else {
      const uint32_t lo = e2m1x2(v.x, v.y), hi = e2m1x2(v.z, v.w);
      c = (lo & 0xFu) | ((lo >> 4) << 8) | ((hi & 0xFu) << 16) | ((hi >> 4) << 24);
    }
    out[i] = c;
  }
}

}  // namespace

cudaError_t launch_debug_cvt(const LaunchCtx& c, int fmt, const float* in, uint8_t* out,
                             int64_t n) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  const int64_t need = (n4 + 255) / 256;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(cvt_kernel, blocks, 256, 0, c.stream, reinterpret_cast<const float4*>(in),
                    reinterpret_cast<uint32_t*>(out), n4, fmt);
}

}  // namespace moe
