// topk_gate.cu -- top-k expert selection and softmax top-k weights.
//
// TileKernels article (itsolotime.com), section 2.1 "Top-K Gating": one warp
// per token holds the token's E scores in registers and repeats k times
// "find the maximum, take the lowest index among equal maxima, retire it".
// The weights are the softmax over the k selected scores (the "Weight
// Normalization" that closes the routing chain at the top of section 2).
//
// GB300 form: each lane keeps E/32 scores as order-preserving 32-bit keys,
// so one round is a lane-local max, one redux.sync max (value) and one
// redux.sync min (lowest index among the lanes holding that value) -- two
// warp instructions instead of a 5-step shuffle butterfly on (value, index).
#include "common.cuh"

namespace moe {
namespace {

// Order-preserving map of a non-NaN f32 onto uint32 (larger float -> larger
// key).  -0.0 is folded onto +0.0 first, so the two compare equal as floats
// do.  Every non-NaN key is >= 0x007FFFFF (the key of -inf), so 0 never
// collides with a real score and marks a retired or absent slot.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t key) {
  uint32_t b = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(b);
}

// V = slots per lane: expert e lives in lane e % 32, slot e / 32.
template <int V>
__global__ void __launch_bounds__(256) topk_gate_kernel(const float* __restrict__ scores,
                                                        int64_t T, int E, int k,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const float* row = scores + t * E;
    uint32_t key[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = i * 32 + lane;
      key[i] = (e < E) ? score_key(__ldcs(row + e)) : 0u;
    }
    uint32_t my_key = 0;  // lane j keeps round j's winner
    int my_e = 0;
    uint32_t top_key = 0;
    for (int r = 0; r < k; ++r) {
      // lane-local best: largest key, lowest slot (= lowest expert) on ties
      uint32_t best = 0;
      int best_i = 0;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        if (key[i] > best) {
          best = key[i];
          best_i = i;
        }
      }
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);
      const uint32_t cand = (best == m) ? (uint32_t)(best_i * 32 + lane) : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, cand);
      if ((int)(win & 31u) == lane) {
        const int slot = (int)(win >> 5);
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (i == slot) key[i] = 0u;
      }
      if (r == 0) top_key = m;
      if (lane == r) {
        my_key = m;
        my_e = (int)win;
      }
    }
    if (lane < k) topk_idx[t * k + lane] = my_e;
    if (topk_w != nullptr) {
      const float s0 = key_score(top_key);
      const float ex = (lane < k) ? expf(key_score(my_key) - s0) : 0.0f;
      float sum = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      if (lane < k) topk_w[t * k + lane] = __fdiv_rn(ex, sum);
    }
  }
}

template <int V>
cudaError_t launch_v(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                     int32_t* idx, float* w) {
  const int threads = 256;
  const int64_t need = (T + 7) / 8;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  topk_gate_kernel<V><<<blocks, threads, 0, c.stream>>>(scores, T, E, k, idx, w);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_gate(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                             int32_t* idx, float* w) {
  if (E <= 32) return launch_v<1>(c, scores, T, E, k, idx, w);
  if (E <= 64) return launch_v<2>(c, scores, T, E, k, idx, w);
  if (E <= 128) return launch_v<4>(c, scores, T, E, k, idx, w);
  if (E <= 256) return launch_v<8>(c, scores, T, E, k, idx, w);
  if (E <= 512) return launch_v<16>(c, scores, T, E, k, idx, w);
  return launch_v<32>(c, scores, T, E, k, idx, w);
}

}  // namespace moe
