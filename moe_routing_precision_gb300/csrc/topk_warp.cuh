// topk_warp.cuh -- one warp selects one token's top-k experts (E <= 256) and
// their softmax weights.  Shared by the top-k kernel, the decode kernels and
// the chained route kernel.
//
// TileKernels article (itsolotime.com), section 2.1 "Top-K Gating": the k
// largest scores of a token, the lowest expert index first among equal
// scores, in descending order; the weights are the softmax over the k
// selected scores (the "Weight Normalization" closing section 2's chain).
#pragma once
#include "common.cuh"

namespace moe {

// Order-preserving map of a non-NaN f32 onto uint32 (larger float -> larger
// key).  -0.0 is folded onto +0.0 first, so the two compare equal as floats
// do.  Every non-NaN key is >= 0x007FFFFF (the key of -inf), so 0 never
// collides with a real score and marks a retired or absent slot.
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t b = __float_as_uint(s + 0.0f);  // -0.0 + 0.0 = +0.0 (round to nearest)
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);  // negative: ~b; else b | sign
}

__device__ __forceinline__ float key_score(uint32_t key) {
  uint32_t b = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(b);
}

// ---- filtered form (E <= 256) -----------------------------------------------
//
// Every candidate is packed as a 64-bit integer (score key << 32 | ~expert):
// the larger packed value is the larger score, or on equal scores the lower
// expert, so the packed order is exactly the selection order.
//
// Fast path: theta = the k-th largest distinct value among the 32 lane maxima
// (at most the k-th largest lane maximum).  At least k distinct experts score
// >= theta, so every top-k expert does too; the lanes
// compact their experts scoring >= theta (usually 8-16 of them) one per lane,
// and each candidate's rank (how many candidates beat it) is its output slot
// if below k.
// Fallback (more than 32 candidates, i.e. heavy ties): each lane sorts its V
// packed candidates and the rounds merge the 32 sorted lists, the winning lane
// advancing its head from shared memory.  Sorting networks: the optimal
// 19-comparator network for 8 inputs (Knuth, TAOCP vol. 3, 5.3.4), the
// 5-comparator one for 4, and odd-even transposition for 12 and 16.
__device__ __forceinline__ void cex(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b;
  const unsigned long long lo = a > b ? b : a;
  a = hi;
  b = lo;
}

template <int V>
__device__ __forceinline__ void sort_desc(unsigned long long (&p)[V]) {
  if constexpr (V != 2 && V != 4 && V != 8) {
    // other V (12, 16): odd-even transposition sort, V passes (only the
    // heavy-tie fallback gets here)
#pragma unroll
    for (int pass = 0; pass < V; ++pass) {
#pragma unroll
      for (int i = pass & 1; i + 1 < V; i += 2) cex(p[i], p[i + 1]);
    }
  } else if constexpr (V == 2) {
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

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// One token: row = its E scores; s_list = this warp's [V][32] and s_cand its
// [32] shared-memory scratch; idx_out / w_out = the token's k outputs (w_out
// may be null).  V slots per lane.  VEC: E % 128 == 0 and row 16-byte
// aligned, lane l loads experts h*128 + 4l + j; otherwise expert i*32 + l in
// slot i.  KMAX >= k bounds the unrolled rounds.  Returns the output slot
// this lane wrote (-1: none; every slot j < k is written by exactly one
// lane) and sets sel_expert to that slot's expert.
template <int V, bool VEC, int KMAX>
__device__ __forceinline__ int topk_token(const float* __restrict__ row, int E, int k, int lane,
                                          unsigned long long (*s_list)[32],
                                          unsigned long long* s_cand,
                                          int32_t* __restrict__ idx_out,
                                          float* __restrict__ w_out, uint32_t& sel_expert) {
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
  // ---- candidate filter: theta = the k-th largest distinct value among the
  // 32 lane maxima (each round retires every lane holding the current
  // maximum).  theta <= the k-th largest lane maximum, and the k largest lane
  // maxima are k distinct experts, so every top-k element scores >= theta.
  // With heavy ties theta falls lower and more candidates pass: the sorted
  // merge below handles more than 32.
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
        if (lm == theta) lm = 0u;  // retire every holder
      }
    }
  }
  unsigned cmask = 0;  // this lane's candidates (absent slots are 0)
#pragma unroll
  for (int i = 0; i < V; ++i) {
    // VEC: E = 32 V, so no slot is absent
    const bool present = VEC || p[i] != 0ull;
    if (present && (uint32_t)(p[i] >> 32) >= theta) cmask |= 1u << i;
  }
  const int nc = __popc(cmask);
  const int C = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)nc);
  __syncwarp();  // the previous token is done with shared memory
  if (C <= 32) {
    // compact the candidates one per lane; each counts the candidates that
    // beat it, and that count is its output slot
    int slot = warp_incl_scan(nc, lane) - nc;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (cmask & (1u << i)) s_cand[slot++] = p[i];
    __syncwarp();
    const unsigned long long cand = (lane < C) ? s_cand[lane] : 0ull;
    int rank = 0;
    for (int j = 0; j < C; ++j) rank += (s_cand[j] > cand) ? 1 : 0;
    if (lane < C && rank < k) {
      out_j = rank;
      out_key = (uint32_t)(cand >> 32);
      out_e = ~(uint32_t)cand;
    }
  } else {
    // many ties: sort each lane's list and merge the 32 lists
    sort_desc<V>(p);
#pragma unroll
    for (int i = 1; i < V; ++i) s_list[i][lane] = p[i];
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
        head = (taken < V) ? s_list[taken][lane] : 0ull;
      }
    }
  }
  if (out_j >= 0) idx_out[out_j] = (int32_t)out_e;
  if (w_out != nullptr) {
    const uint32_t top_key = __reduce_max_sync(0xFFFFFFFFu, out_j >= 0 ? out_key : 0u);
    const float s0 = key_score(top_key);
    const float ex = (out_j >= 0) ? expf(key_score(out_key) - s0) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (out_j >= 0) w_out[out_j] = __fdiv_rn(ex, sum);
  }
  sel_expert = out_e;
  return out_j;
}

}  // namespace moe
