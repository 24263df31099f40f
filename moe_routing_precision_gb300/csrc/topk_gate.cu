// topk_gate.cu -- top-k expert selection and softmax top-k weights.
//
// TileKernels article (itsolotime.com), section 2.1 "Top-K Gating": one warp
// per token holds the token's E scores in registers and repeats k times
// "find the maximum, take the lowest index among equal maxima, retire it".
// The weights are the softmax over the k selected scores (the "Weight
// Normalization" that closes the routing chain at the top of section 2).
//
// GB300 forms: scores become order-preserving 32-bit integer keys so that a
// warp reduction is one redux.sync instruction.  For E <= 256 each lane sorts
// its E/32 candidates once and the k rounds merge the 32 sorted lists (the
// "sorted-list form" below); otherwise each round rescans the lane's keys
// (lane-local max, redux.sync max on the value, redux.sync min on the index
// among lanes holding it) -- two warp instructions per round either way, in
// place of a 5-step shuffle butterfly on (value, index).
#include "topk_warp.cuh"

namespace moe {
namespace {

// V = slots per lane: expert e lives in lane e % 32, slot e / 32.
template <int V>
__global__ void __launch_bounds__(256) topk_gate_kernel(const float* __restrict__ scores,
                                                        int64_t T, int E, int k,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  pdl_enter();
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

constexpr int kSortedWarps = 8;

// V slots per lane (see topk_token).  KFIX > 0: k is that constant (the
// common k = 8 gets its own instance); VEC implies E = 32 V.
template <int V, bool VEC, int KMAX, int KFIX = 0>
__global__ void __launch_bounds__(kSortedWarps * 32) topk_gate_sorted_kernel(
    const float* __restrict__ scores, int64_t T, int E_, int k_, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w) {
  __shared__ unsigned long long s_list[kSortedWarps][V][32];
  __shared__ unsigned long long s_cand[kSortedWarps][32];
  pdl_enter();
  const int E = VEC ? 32 * V : E_;
  const int k = KFIX > 0 ? KFIX : k_;
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  uint32_t sel_e;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps)
    topk_token<V, VEC, KMAX>(scores + t * E, E, k, lane, s_list[wib], s_cand[wib],
                             topk_idx + t * k, topk_w != nullptr ? topk_w + t * k : nullptr,
                             sel_e);
}

template <int V, bool VEC>
cudaError_t launch_sorted(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                          int32_t* idx, float* w) {
  const int64_t need = (T + kSortedWarps - 1) / kSortedWarps;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  if (k == 8)
    return launch_pdl(topk_gate_sorted_kernel<V, VEC, 8, 8>, blocks, kSortedWarps * 32, 0,
                      c.stream, scores, T, E, k, idx, w);
  if (k <= 8)
    return launch_pdl(topk_gate_sorted_kernel<V, VEC, 8>, blocks, kSortedWarps * 32, 0, c.stream,
                      scores, T, E, k, idx, w);
  return launch_pdl(topk_gate_sorted_kernel<V, VEC, 32>, blocks, kSortedWarps * 32, 0, c.stream,
                    scores, T, E, k, idx, w);
}

// rescan form (E <= 32, E > 256)
template <int V>
cudaError_t launch_v(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                     int32_t* idx, float* w) {
  const int threads = 256;
  const int64_t need = (T + 7) / 8;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(topk_gate_kernel<V>, blocks, threads, 0, c.stream, scores, T, E, k, idx, w);
}

}  // namespace

cudaError_t launch_topk_gate(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                             int32_t* idx, float* w) {
  const bool vec = (E % 128 == 0) && (reinterpret_cast<uintptr_t>(scores) % 16 == 0);
  if (E <= 32) return launch_v<1>(c, scores, T, E, k, idx, w);
  if (E <= 64) return launch_sorted<2, false>(c, scores, T, E, k, idx, w);
  if (E <= 128) return vec ? launch_sorted<4, true>(c, scores, T, E, k, idx, w)
                           : launch_sorted<4, false>(c, scores, T, E, k, idx, w);
  if (E <= 256) return vec ? launch_sorted<8, true>(c, scores, T, E, k, idx, w)
                           : launch_sorted<8, false>(c, scores, T, E, k, idx, w);
  if (E <= 512) return launch_v<16>(c, scores, T, E, k, idx, w);
  return launch_v<32>(c, scores, T, E, k, idx, w);
}

}  // namespace moe
