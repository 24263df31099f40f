// swiglu_cast.cu -- SwiGLU fused with the per-group FP8 E4M3 cast.
//
// TileKernels article (itsolotime.com), section 3.3: in f32,
// val_l / (1 + exp(-val_l)) * val_r with val_l from the left (gate) half and
// val_r from the right (up) half of each row, then per-group absmax -> scale
// -> cast in the same kernel (plain form: no clamp, no top-k weight).
//
// Work unit: one (row, 128-channel group) per aligned 8-lane subgroup; each
// lane reads 16 gate and 16 up values (four 16-byte loads) and writes one
// 16-byte code vector.  HBM traffic is ~80% reads.  The grid is persistent and
// strides over tiles of 4 units per warp.  At ~1 GB per 0.15 ms the kernel
// must spend under ~12 instructions per element to stay memory-bound, which is
// why the activation uses the hardware exp2 and reciprocal.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float swiglu(float g, float u) {
  // evaluated in the order written on the page, in f32, with the hardware
  // exp2 and reciprocal (__expf, __fdividef): a few ulps from the correctly
  // rounded value, which moves an E4M3 code only when v / sf lies within those
  // ulps of a rounding midpoint (about 1e-5 of elements).  For g < -88,
  // exp(-g) is +inf and g / inf gives a signed zero, as the IEEE division does.
  const float e = __expf(-g);
  return __fdividef(g, 1.0f + e) * u;
}

__global__ void __launch_bounds__(kThreads) swiglu_cast_kernel(const uint16_t* __restrict__ x,
                                                               uint32_t units, int N,
                                                               uint8_t* __restrict__ out,
                                                               float* __restrict__ out_sf,
                                                               FastDiv fdG) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;
  const int l8 = lane & 7;
  const int G = N >> 7;
  const uint32_t tiles = (units + 3) >> 2;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  for (uint32_t tile = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; tile < tiles; tile += warps) {
    const uint32_t u = tile * 4 + sub;
    const bool active = u < units;
    const uint32_t r = active ? fdG.div(u) : 0;
    const int g = active ? (int)(u - r * G) : 0;
    const uint16_t* gate = x + (int64_t)r * 2 * N + g * kGroup + l8 * 16;
    const uint16_t* up = gate + N;
    uint4 ga = make_uint4(0, 0, 0, 0), gb = ga, ua = ga, ub = ga;
    if (active) {
      ga = ld_stream_v4(gate);
      gb = ld_stream_v4(gate + 8);
      ua = ld_stream_v4(up);
      ub = ld_stream_v4(up + 8);
    }
    float gv[16], uv[16], v[16];
    unpack16(ga, gb, gv);
    unpack16(ua, ub, uv);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = swiglu(gv[i], uv[i]);
    const float amax = max8(absmax16(v));
    const float sf = group_scale(amax);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16(v, inv);
    if (active) {
      st_stream_v4(out + (int64_t)r * N + g * kGroup + l8 * 16, q);
      if (l8 == 0) st_stream_f32(out_sf + (int64_t)r * G + g, sf);
    }
  }
}

}  // namespace

cudaError_t launch_swiglu_cast(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                               float* out_sf) {
  const int G = N / kGroup;
  const uint32_t units = (uint32_t)(M * G);  // < 2^31, checked by the caller
  const uint32_t tiles = (units + 3) / 4;
  const int64_t need = ((int64_t)tiles + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, swiglu_cast_kernel,
                                                                 kThreads, 0);
  if (st != cudaSuccess) return st;
  const int64_t cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(swiglu_cast_kernel, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, N, out, out_sf, FastDiv((uint32_t)G));
}

}  // namespace moe
