// expand_cast.cu -- per-token FP8 E4M3 cast fused with the expand to the
// expert-sorted layout.
//
// TileKernels article (itsolotime.com): section 3.2 per_token_cast (absmax
// over each 128-channel group, scale, multiply by the inverse scale, cast) and
// section 2.2 expand_to_fused (copy each token's row and scales to the rows
// pos[t, j], skipping pos < 0).  The page runs them as two kernels; every
// copy of a token casts identically, so here each token is read and cast once
// and its codes are written k times.
//
// Work unit: one (token, 128-channel group) per aligned 8-lane subgroup; lane
// l of the subgroup holds channels 16l..16l+15 (two 16-byte loads), the group
// amax is a 3-step xor-shuffle, and each lane writes one 16-byte code vector
// per destination row.  A warp handles 4 consecutive units, so a warp's loads
// cover 1 KiB and its stores 512 contiguous bytes per destination row.
// The grid is persistent (a multiple of the SM count) and strides over tiles
// of 4 units; HBM traffic is ~80% writes (k copies of 1 byte per channel plus
// scales, against 2 bytes per channel read once).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) expand_cast_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int k, const int32_t* __restrict__ pos,
    int64_t R, uint8_t* __restrict__ out, float* __restrict__ out_sf, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;  // unit within the warp's tile
  const int l8 = lane & 7;    // 16-channel slice within the group
  const int G = H >> 7;
  const int64_t units = T * G;
  const int64_t tiles = (units + 3) >> 2;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool bad = false;
  for (int64_t tile = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; tile < tiles;
       tile += warps) {
    const int64_t u = tile * 4 + sub;
    const bool active = u < units;
    const int64_t t = active ? u / G : 0;
    const int g = active ? (int)(u - t * G) : 0;
    const uint16_t* src = x + t * H + g * kGroup + l8 * 16;
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (active) {
      a = ld_stream_v4(src);
      b = ld_stream_v4(src + 8);
    }
    float v[16];
    unpack16(a, b, v);
    const float amax = max8(absmax16(v));
    const float sf = group_scale(amax);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16(v, inv);
    if (active) {
      const int32_t* prow = pos + t * k;
      for (int j = 0; j < k; ++j) {
        const int32_t r = __ldg(prow + j);
        if (r < 0) continue;  // dropped copy
        if (r >= R) {
          bad = true;
          continue;
        }
        st_stream_v4(out + (int64_t)r * H + g * kGroup + l8 * 16, q);
        if (l8 == 0) st_stream_f32(out_sf + (int64_t)r * G + g, sf);
      }
    }
  }
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

}  // namespace

cudaError_t launch_expand_cast(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                               const int32_t* pos, int64_t R, uint8_t* out, float* out_sf) {
  const int64_t units = T * (H / kGroup);
  const int64_t tiles = (units + 3) / 4;
  const int64_t need = (tiles + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, expand_cast_kernel,
                                                                 kThreads, 0);
  if (st != cudaSuccess) return st;
  const int64_t cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  const int blocks = (int)(need < cap ? need : cap);
  expand_cast_kernel<<<blocks, kThreads, 0, c.stream>>>(
      static_cast<const uint16_t*>(x), T, H, k, pos, R, out, out_sf, c.err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
