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

// ---- filtered form (E <= 256) -----------------------------------------------
//
// Every candidate is packed as a 64-bit integer (score key << 32 | ~expert):
// the larger packed value is the larger score, or on equal scores the lower
// expert, so the packed order is exactly the selection order.
//
// Fast path: theta = the k-th largest of the 32 lane maxima.  At least k
// distinct experts score >= theta, so every top-k expert does too; the lanes
// compact their experts scoring >= theta (usually 8-16 of them) one per lane,
// and each candidate's rank (how many candidates beat it) is its output slot
// if below k.
// Fallback (more than 32 candidates, i.e. heavy ties): each lane sorts its V
// packed candidates and the rounds merge the 32 sorted lists, the winning lane
// advancing its head from shared memory.  Sorting networks: the optimal
// 19-comparator network for 8 inputs (Knuth, TAOCP vol. 3, 5.3.4) and the
// 5-comparator one for 4.
__device__ __forceinline__ void cex(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b;
  const unsigned long long lo = a > b ? b : a;
  a = hi;
  b = lo;
}

template <int V>
__device__ __forceinline__ void sort_desc(unsigned long long (&p)[V]) {
  if constexpr (V == 2) {
    cex(p[0], p[1]);
  } else if constexpr (V == 4) {
    cex(p[0], p[1]); cex(p[2], p[3]); cex(p[0], p[2]); cex(p[1], p[3]); cex(p[1], p[2]);
  } else if constexpr (V == 8) {
    cex(p[0], p[2]); cex(p[1], p[3]); cex(p[4], p[6]); cex(p[5], p[7]);
    cex(p[0], p[4]); cex(p[1], p[5]); cex(p[2], p[6]); cex(p[3], p[7]);
    cex(p[0], p[1]); cex(p[2], p[3]); cex(p[4], p[5]); cex(p[6], p[7]);
    cex(p[2], p[4]); cex(p[3], p[5]);
    cex(p[1], p[4]); cex(p[3], p[6]);
    cex(p[1], p[2]); cex(p[3], p[4]); cex(p[5], p[6]);
  }
}

constexpr int kSortedWarps = 8;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// V slots per lane.  VEC: E % 128 == 0, lane l loads experts h*128 + 4l + j
// (16-byte loads); otherwise expert i*32 + l in slot i.  KMAX >= k bounds the
// unrolled rounds.
template <int V, bool VEC, int KMAX>
__global__ void __launch_bounds__(kSortedWarps * 32) topk_gate_sorted_kernel(
    const float* __restrict__ scores, int64_t T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w) {
  __shared__ unsigned long long s_list[kSortedWarps][V][32];
  __shared__ unsigned long long s_cand[kSortedWarps][32];
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const float* row = scores + t * E;
    unsigned long long p[V];
    if constexpr (VEC) {
#pragma unroll
      for (int h = 0; h < V / 4; ++h) {
        const float4 f = __ldcs(reinterpret_cast<const float4*>(row + h * 128 + 4 * lane));
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t e = (uint32_t)(h * 128 + 4 * lane + j);
          p[h * 4 + j] = ((unsigned long long)score_key(fv[j]) << 32) | (uint32_t)~e;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = i * 32 + lane;
        p[i] = (e < E) ? (((unsigned long long)score_key(__ldcs(row + e)) << 32) |
                          (uint32_t)~(uint32_t)e)
                       : 0ull;  // absent slot: below every real score
      }
    }
    // Each lane ends with at most one output: slot out_j (-1: none) holding
    // expert out_e with score key out_key.
    int out_j = -1;
    uint32_t out_key = 0, out_e = 0;
    // ---- candidate filter: theta = k-th largest of the 32 lane maxima; every
    // top-k element scores >= theta (k distinct lane maxima do)
    uint32_t lmax = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) lmax = max(lmax, (uint32_t)(p[i] >> 32));
    uint32_t theta = 0;
    {
      uint32_t lm = lmax;
#pragma unroll
      for (int r = 0; r < KMAX; ++r) {
        if (r < k) {
          theta = __reduce_max_sync(0xFFFFFFFFu, lm);
          const unsigned holders = __ballot_sync(0xFFFFFFFFu, lm == theta);
          if (lane == __ffs(holders) - 1) lm = 0u;  // retire one holder
        }
      }
    }
    unsigned cmask = 0;  // this lane's candidates (absent slots are 0)
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (p[i] != 0ull && (uint32_t)(p[i] >> 32) >= theta) cmask |= 1u << i;
    const int nc = __popc(cmask);
    const int C = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)nc);
    __syncwarp();  // the previous token is done with shared memory
    if (C <= 32) {
      // compact the candidates one per lane; each counts the candidates that
      // beat it, and that count is its output slot
      int slot = warp_incl_scan(nc, lane) - nc;
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (cmask & (1u << i)) s_cand[wib][slot++] = p[i];
      __syncwarp();
      const unsigned long long cand = (lane < C) ? s_cand[wib][lane] : 0ull;
      int rank = 0;
      for (int j = 0; j < C; ++j) rank += (s_cand[wib][j] > cand) ? 1 : 0;
      if (lane < C && rank < k) {
        out_j = rank;
        out_key = (uint32_t)(cand >> 32);
        out_e = ~(uint32_t)cand;
      }
    } else {
      // many ties: sort each lane's list and merge the 32 lists
      sort_desc<V>(p);
#pragma unroll
      for (int i = 1; i < V; ++i) s_list[wib][i][lane] = p[i];
      __syncwarp();
      unsigned long long head = p[0];
      int taken = 0;
      for (int r = 0; r < k; ++r) {
        const uint32_t hk = (uint32_t)(head >> 32);
        const uint32_t hl = (uint32_t)head;
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, hk);
        const uint32_t wl = __reduce_max_sync(0xFFFFFFFFu, hk == m ? hl : 0u);
        if (lane == r) {
          out_j = r;
          out_key = m;
          out_e = ~wl;
        }
        if (hk == m && hl == wl) {  // this lane supplied the winner
          ++taken;
          head = (taken < V) ? s_list[wib][taken][lane] : 0ull;
        }
      }
    }
    if (out_j >= 0) topk_idx[t * k + out_j] = (int32_t)out_e;
    if (topk_w != nullptr) {
      const uint32_t top_key = __reduce_max_sync(0xFFFFFFFFu, out_j >= 0 ? out_key : 0u);
      const float s0 = key_score(top_key);
      const float ex = (out_j >= 0) ? expf(key_score(out_key) - s0) : 0.0f;
      float sum = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      if (out_j >= 0) topk_w[t * k + out_j] = __fdiv_rn(ex, sum);
    }
  }
}

template <int V, bool VEC>
cudaError_t launch_sorted(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                          int32_t* idx, float* w) {
  const int64_t need = (T + kSortedWarps - 1) / kSortedWarps;
  const int64_t cap = (int64_t)c.num_sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
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
