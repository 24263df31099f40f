// combine.cu -- weighted combine of each token's k expert outputs back to
// token order.
//
// "CuTeDSL at Perplexity", MoE combine: using the token positions computed by
// dispatch, accumulate in registers and write the final tokens to the output
// buffer (a vectorised accumulation).  Here:
//   out[t, c] = sum_j w[t, j] * y[pos[t, j], c]
// in f32, slot order j = 0..k-1, one fused multiply-add per term, rounded
// once to bf16 (or stored as f32).
//
// Work unit: 8 channels (16 bytes of one bf16 row) per lane; a warp covers 32
// consecutive 8-channel slices of the flattened [T, H/8] output.  Each lane
// issues its k row loads in batches of 8 before accumulating, so up to 8
// independent 16-byte gathers are in flight per lane.  HBM traffic is ~90%
// reads of y.
#include "common.cuh"

#include <cuda_bf16.h>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ w, const int32_t* __restrict__ pos,
    uint32_t slices, int H, int k, int64_t R, void* __restrict__ out, FastDiv fdS, unsigned* err) {
  pdl_enter();
  const int S = H >> 3;  // 8-channel slices per token
  const uint32_t stride = gridDim.x * blockDim.x;
  bool bad = false;
  for (uint32_t s = blockIdx.x * blockDim.x + threadIdx.x; s < slices; s += stride) {
    const int64_t t = fdS.div(s);
    const int c = (int)(s - (uint32_t)t * S) * 8;
    const int32_t* prow = pos + t * k;
    const float* wrow = w + t * k;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      uint4 v[kBatch];
      float wj[kBatch];
      bool use[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int j = j0 + b;
        use[b] = false;
        wj[b] = 0.0f;
        v[b] = make_uint4(0, 0, 0, 0);
        if (j < k) {
          const int32_t r = __ldg(prow + j);
          if (r >= R) bad = true;
          if (r >= 0 && r < R) {
            use[b] = true;
            wj[b] = __ldg(wrow + j);
            v[b] = ld_stream_v4(y + (int64_t)r * H + c);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (use[b]) {
          const uint32_t wd[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fmaf_rn(wj[b], bf16_lo(wd[i]), acc[2 * i]);
            acc[2 * i + 1] = __fmaf_rn(wj[b], bf16_hi(wd[i]), acc[2 * i + 1]);
          }
        }
      }
    }
    if (kOutF32) {
      float* o = static_cast<float*>(out) + t * H + c;
      st_stream_v4(o, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                 __float_as_uint(acc[2]), __float_as_uint(acc[3])));
      st_stream_v4(o + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                     __float_as_uint(acc[6]), __float_as_uint(acc[7])));
    } else {
      uint16_t* o = static_cast<uint16_t*>(out) + t * H + c;
      st_stream_v4(o, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                 pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    }
  }
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

template <bool kOutF32>
cudaError_t launch_t(const LaunchCtx& c, const void* y, const float* w, const int32_t* pos,
                     int64_t T, int H, int k, int64_t R, void* out) {
  const uint32_t slices = (uint32_t)(T * (H / 8));  // < 2^31, checked by the caller
  const int64_t need = ((int64_t)slices + kThreads - 1) / kThreads;
  int per_sm = 0;
  cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<kOutF32>,
                                                                 kThreads, 0);
  if (st != cudaSuccess) return st;
  const int64_t cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(combine_kernel<kOutF32>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(y), w, pos, slices, H, k, R, out,
                    FastDiv((uint32_t)(H / 8)), c.err);
}

}  // namespace

cudaError_t launch_combine(const LaunchCtx& c, const void* y, const float* w, const int32_t* pos,
                           int64_t T, int H, int k, int64_t R, void* out, bool out_f32) {
  return out_f32 ? launch_t<true>(c, y, w, pos, T, H, k, R, out)
                 : launch_t<false>(c, y, w, pos, T, H, k, R, out);
}

}  // namespace moe
