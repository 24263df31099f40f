// topk_gate.cu -- top-k expert selection and softmax top-k weights.
//
// TileKernels article (itsolotime.com), section 2.1 "Top-K Gating": one warp
// per token holds the token's E scores in registers and repeats k times
// "find the maximum, take the lowest index among equal maxima, retire it".
// The weights are the softmax over the k selected scores (the "Weight
// Normalization" that closes the routing chain at the top of section 2).
//
// GB300 forms: scores become order-preserving 32-bit integer keys.
//   32 < E <= 512: the candidate-filter form (topk_warp.cuh): a lower bound
//     from the lane maxima (k rounds of redux.sync) leaves a few candidates,
//     ranked directly; E = 128, 256, 384 and 512 load whole float4 rows.
//   E <= 16: 8 or 16 lanes per token (several tokens per warp), k rounds of
//     a segmented xor-shuffle max on (key, ~expert).
//   16 < E <= 32 and E > 512: one token per warp, each round rescanning the
//     lane's keys (lane-local max, redux.sync max on the value, redux.sync
//     min on the index among lanes holding it).
#include "topk_warp.cuh"

namespace moe {
namespace {

// E <= 16: S lanes per token (S = 8 or 16, the smallest that holds E), so
// 32 / S tokens share a warp; lane j of a token's segment holds expert j as
// (score key << 32 | ~j), 0 where j >= E.  Each of the k rounds takes the
// segment's largest such value by a butterfly of log2(S) xor shuffles (the
// lower expert wins ties, as its ~j is larger) and retires it; lane r keeps
// round r's winner.  The weights' sum runs over the same lanes in the same
// order as a 32-lane butterfly would, the other lanes adding zeros.
template <int S>
__global__ void __launch_bounds__(256) topk_gate_small_kernel(const float* __restrict__ scores,
                                                              int64_t T, int E, int k,
                                                              int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w) {
  constexpr int TPW = 32 / S;  // tokens per warp
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int j = lane & (S - 1);
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * TPW; t0 < T;
       t0 += warps * TPW) {
    const int64_t t = t0 + lane / S;
    const bool tok = t < T;
    unsigned long long p = 0ull;
    if (tok && j < E)
      p = ((unsigned long long)score_key(__ldcs(scores + t * E + j)) << 32) |
          (uint32_t)~(uint32_t)j;
    unsigned long long mine = 0ull, top = 0ull;
    for (int r = 0; r < k; ++r) {  // k <= E <= S
      unsigned long long m = p;
#pragma unroll
      for (int o = S / 2; o > 0; o >>= 1) {
        const unsigned long long q = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = q > m ? q : m;
      }
      if (p == m) p = 0ull;  // the winner: experts differ, so one lane
      if (r == 0) top = m;
      if (j == r) mine = m;
    }
    if (tok && j < k) topk_idx[t * k + j] = (int32_t)~(uint32_t)mine;
    if (topk_w != nullptr) {
      const float s0 = key_score((uint32_t)(top >> 32));
      const float ex = (tok && j < k) ? expf(key_score((uint32_t)(mine >> 32)) - s0) : 0.0f;
      float sum = ex;
#pragma unroll
      for (int o = S / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      if (tok && j < k) topk_w[t * k + j] = __fdiv_rn(ex, sum);
    }
  }
}

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

template <int S>
cudaError_t launch_small(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                         int32_t* idx, float* w) {
  constexpr int TPB = 256 / S;  // tokens per block
  const int64_t need = (T + TPB - 1) / TPB;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  return launch_pdl(topk_gate_small_kernel<S>, blocks, 256, 0, c.stream, scores, T, E, k, idx, w);
}

// rescan form (16 < E <= 32, E > 512)
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
  // E <= 16: several tokens per warp (at T = 65536, E = 8, k = 2: 8.8 against
  // 17.0 us for one token per warp; E = 16: 12.9 against 17.0); at E = 32 the
  // one-token rescan with redux.sync is the faster (19.2 against 27.3 us)
  if (E <= 8) return launch_small<8>(c, scores, T, E, k, idx, w);
  if (E <= 16) return launch_small<16>(c, scores, T, E, k, idx, w);
  if (E <= 32) return launch_v<1>(c, scores, T, E, k, idx, w);
  if (E <= 64) return launch_sorted<2, false>(c, scores, T, E, k, idx, w);
  if (E <= 128) return vec ? launch_sorted<4, true>(c, scores, T, E, k, idx, w)
                           : launch_sorted<4, false>(c, scores, T, E, k, idx, w);
  if (E <= 256) return vec ? launch_sorted<8, true>(c, scores, T, E, k, idx, w)
                           : launch_sorted<8, false>(c, scores, T, E, k, idx, w);
  // 256 < E <= 512 (T = 65536, k = 8): E = 384 33.4 us and E = 512 37.5 us,
  // against 84.6 and 84.1 us for the rescan form
  if (E == 384 && vec) return launch_sorted<12, true>(c, scores, T, E, k, idx, w);
  if (E <= 512) return vec && E == 512 ? launch_sorted<16, true>(c, scores, T, E, k, idx, w)
                                       : launch_sorted<16, false>(c, scores, T, E, k, idx, w);
  return launch_v<32>(c, scores, T, E, k, idx, w);
}

}  // namespace moe
