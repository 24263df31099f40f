// route_map.cu -- token -> expert mapping: per-expert counts, exclusive
// offsets, the stable expert-sorted slot of every routed copy, and its inverse.
//
// "CuTeDSL at Perplexity", MoE dispatch (TP=1 local kernel): count the tokens
// routed to each expert and give each copy a unique index in its expert's
// list; for prefill the routing is split over many blocks with shared-memory
// counters, then aggregated.  The page's atomics order copies arbitrarily;
// here every slot is fixed by the row-major (token, slot) order, so the
// result is deterministic and stable (ascending token within an expert).
//
// Two launches over chunks of consecutive tokens (a multiple of 32 tokens, at
// most 512, about 128 chunks):
//   1. route_count_kernel: one CTA per chunk builds the chunk's histogram in
//      shared memory (order-free atomics) -> hist[chunk][E] in the workspace.
//   2. route_rank_kernel: one CTA per chunk sums the histogram columns (all
//      chunks for the totals, earlier chunks for its own base) and scans the
//      totals into offsets, all in shared memory.  Warp w owns the chunk's
//      w-th run of 32 tokens and sets bit `lane` of word[w][e] for each expert
//      e its lane's token picked; a copy's rank among its expert's copies is
//      then (copies in earlier words) + popc(word & lanes-below), which is
//      the row-major order because a token's k experts are distinct.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCountThreads = 512;
constexpr int kRankWarps = kRouteMaxChunkTokens / 32;  // 16: one 32-token word each
constexpr int kRankThreads = kRankWarps * 32;

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(
    const int32_t* __restrict__ idx, int64_t R, int E, int chunk_pairs, int32_t* __restrict__ hist,
    unsigned* err) {
  extern __shared__ int32_t s_hist[];
  pdl_enter();
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * chunk_pairs;
  const int64_t p1 = min(p0 + chunk_pairs, R);
  bool bad = false;
  // eight loads in flight per thread, then the shared-memory increments
  for (int64_t base = p0 + threadIdx.x; base < p1; base += 8 * (int64_t)blockDim.x) {
    int e[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t p = base + (int64_t)u * blockDim.x;
      e[u] = (p < p1) ? __ldg(idx + p) : -1;
      if (p < p1 && (unsigned)e[u] >= (unsigned)E) {
        bad = true;
        e[u] = -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (e[u] >= 0) atomicAdd(&s_hist[e[u]], 1);
  }
  if (bad) flag_error(err, MOE_DEVERR_EXPERT_RANGE);
  __syncthreads();
  int32_t* out = hist + (int64_t)blockIdx.x * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = s_hist[e];
}

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// KFIX > 0: k is that constant; ALIGN1: align == 1 (the plain layout).  The
// common k = 8 and the plain layout get instances of their own.
template <int KFIX, bool ALIGN1>
__global__ void __launch_bounds__(kRankThreads) route_rank_kernel(
    const int32_t* __restrict__ idx, int64_t T, int E, int k_, int chunk_tokens, int num_chunks,
    int align_, int64_t num_rows, const int32_t* __restrict__ hist, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ pos, int32_t* __restrict__ sorted_src,
    unsigned* err) {
  const int k = KFIX > 0 ? KFIX : k_;
  const int align = ALIGN1 ? 1 : align_;
  extern __shared__ int32_t smem[];
  int32_t* s_off = smem;                                     // [E] totals, then offsets
  int32_t* s_base = smem + E;                                // [E] copies in earlier chunks
  uint32_t* s_word = reinterpret_cast<uint32_t*>(smem + 2 * E);  // [kRankWarps][E] bitmaps
  int32_t* s_wpre = smem + (2 + kRankWarps) * E;             // [kRankWarps][E] word prefixes
  __shared__ int32_t s_warp_tot[kRankWarps];
  __shared__ int32_t s_carry;
  pdl_enter();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int64_t t = (int64_t)b * chunk_tokens + warp * 32 + lane;  // this lane's token
  const bool tok = (warp * 32 < chunk_tokens) && t < T;

  // the first 8 expert ids of this lane's token, loaded before anything else
  int ids[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ids[j] = (tok && j < k) ? __ldg(idx + t * k + j) : -1;

  for (int i = tid; i < kRankWarps * E; i += kRankThreads) s_word[i] = 0u;
  for (int e = tid; e < E; e += kRankThreads) {
    s_off[e] = 0;
    s_base[e] = 0;
  }
  __syncthreads();

  // ---- bitmap words: bit `lane` of word[warp][e] <=> this lane's token picked e
  if (tok) {
    bool dup = false;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((unsigned)ids[j] < (unsigned)E)
        dup |= (atomicOr(&s_word[warp * E + ids[j]], 1u << lane) >> lane) & 1u;
    for (int j = 8; j < k; ++j) {
      const int e = __ldg(idx + t * k + j);
      if ((unsigned)e < (unsigned)E)
        dup |= (atomicOr(&s_word[warp * E + e], 1u << lane) >> lane) & 1u;
    }
    // a token naming one expert twice cannot be ranked this way (top-k never
    // produces it): flag it; the slot bound check below keeps writes in range
    if (dup) flag_error(err, MOE_DEVERR_DUPLICATE_EXPERT);
  }

  // ---- column sums of the histogram: totals and this chunk's base.  Every
  // CTA reads the whole histogram, so each starts at a different row to spread
  // the reads over L2; 16-byte loads (E % 4 == 0), 16 in flight per thread.
  {
    const int V4 = (E % 4 == 0) ? 4 : 1;  // columns per load
    const int ncol = E / V4;
    const int cols = ncol < kRankThreads ? ncol : kRankThreads;
    const int phases = kRankThreads / cols;
    const int col = tid % cols;
    const int ph = tid / cols;
    const int nrows = (num_chunks - ph + phases - 1) / phases;  // rows in this phase
    if (ph < phases && nrows > 0) {
      const int start = (b / phases) % nrows;
      for (int c4 = col; c4 < ncol; c4 += cols) {
        int4 tot = make_int4(0, 0, 0, 0), base = tot;
        for (int i0 = 0; i0 < nrows; i0 += 16) {
          int4 v[16];
          int cc[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            int i = start + i0 + u;
            if (i >= nrows) i -= nrows;
            cc[u] = ph + i * phases;
            v[u] = make_int4(0, 0, 0, 0);
            if (i0 + u < nrows) {
              const int32_t* src = hist + (int64_t)cc[u] * E + c4 * V4;
              if (V4 == 4)
                v[u] = __ldg(reinterpret_cast<const int4*>(src));
              else
                v[u].x = __ldg(src);
            }
          }
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const bool before = i0 + u < nrows && cc[u] < b;
            tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
            if (before) {
              base.x += v[u].x; base.y += v[u].y; base.z += v[u].z; base.w += v[u].w;
            }
          }
        }
        const int e = c4 * V4;
        atomicAdd(&s_off[e], tot.x);
        atomicAdd(&s_base[e], base.x);
        if (V4 == 4) {
          atomicAdd(&s_off[e + 1], tot.y); atomicAdd(&s_base[e + 1], base.y);
          atomicAdd(&s_off[e + 2], tot.z); atomicAdd(&s_base[e + 2], base.z);
          atomicAdd(&s_off[e + 3], tot.w); atomicAdd(&s_base[e + 3], base.w);
        }
      }
    }
  }
  __syncthreads();

  // ---- offsets: exclusive scan of the totals rounded up to `align` (1 for
  // the plain layout), kRankThreads at a time
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < E; base += kRankThreads) {
    const int e = base + tid;
    const int32_t cnt = (e < E) ? s_off[e] : 0;
    const int32_t v = (cnt + align - 1) / align * align;
    const int32_t incl = warp_incl_scan(v, lane);
    if (lane == 31) s_warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int32_t wt = (lane < kRankWarps) ? s_warp_tot[lane] : 0;
      const int32_t wi = warp_incl_scan(wt, lane);
      if (lane < kRankWarps) s_warp_tot[lane] = wi - wt;  // exclusive
    }
    __syncthreads();
    const int32_t excl = s_carry + s_warp_tot[warp] + incl - v;
    if (e < E) s_off[e] = excl;
    if (b == 0 && e < E) counts[e] = cnt;
    // this expert's padding rows, written by one CTA
    if (e < E && e % num_chunks == b)
      for (int64_t r = (int64_t)excl + cnt; r < (int64_t)excl + v && r < num_rows; ++r)
        sorted_src[r] = -1;
    __syncthreads();
    if (tid == kRankThreads - 1) s_carry = excl + v;
    __syncthreads();
  }
  if (b == 0) {
    for (int e = tid; e < E; e += kRankThreads) offsets[e] = s_off[e];
    if (tid == 0) offsets[E] = s_carry;
    if (tid == 0 && (int64_t)s_carry > num_rows) flag_error(err, MOE_DEVERR_ROWS_SHORT);
  }
  // rows past the padded total, up to num_rows, are not any copy's
  for (int64_t r = (int64_t)s_carry + (int64_t)b * kRankThreads + tid; r < num_rows;
       r += (int64_t)num_chunks * kRankThreads)
    sorted_src[r] = -1;
  // ---- start of each word's copies of e: offset + chunk base + earlier words
  for (int e = tid; e < E; e += kRankThreads) {
    int32_t run = s_off[e] + s_base[e];
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
      s_wpre[w * E + e] = run;
      run += __popc(s_word[w * E + e]);
    }
  }
  __syncthreads();

  // ---- positions
  if (tok) {
    const uint32_t below = (1u << lane) - 1u;
    bool bad = false;
    for (int j = 0; j < k; ++j) {
      const int64_t p = t * k + j;
      int e = -1;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u == j) e = ids[u];
      if (j >= 8) e = __ldg(idx + p);
      if ((unsigned)e >= (unsigned)E) {
        pos[p] = -1;  // out-of-range expert (flagged by the count kernel)
        continue;
      }
      const int32_t slot = s_wpre[warp * E + e] + __popc(s_word[warp * E + e] & below);
      // slot < num_rows whenever num_rows covers the padded total and
      // topk_idx is unchanged since the count kernel read it; otherwise a flag,
      // not a wild write
      if ((int64_t)slot < num_rows && slot >= 0) {
        pos[p] = slot;
        sorted_src[slot] = (int32_t)p;
      } else {
        pos[p] = -1;
        bad = true;
      }
    }
    if (bad) flag_error(err, MOE_DEVERR_EXPERT_RANGE);
  }
}

}  // namespace

cudaError_t launch_route_map_aligned(const LaunchCtx& c, const int32_t* idx, int64_t T, int E,
                                     int k, int align, int64_t num_rows, int32_t* counts,
                                     int32_t* offsets, int32_t* pos, int32_t* sorted_src,
                                     int32_t* ws, int64_t num_chunks) {
  const int64_t R = T * k;
  const int chunk_tokens = (int)route_chunk_tokens(T);
  const size_t count_smem = sizeof(int32_t) * E;
  cudaError_t st = launch_pdl(route_count_kernel, (unsigned)num_chunks, kCountThreads, count_smem,
                              c.stream, idx, R, E, chunk_tokens * k, ws, c.err);
  if (st != cudaSuccess) return st;
  const size_t rank_smem = sizeof(int32_t) * (size_t)E * (2 + 2 * kRankWarps);
  auto kern = k == 8 ? (align == 1 ? route_rank_kernel<8, true> : route_rank_kernel<8, false>)
                     : (align == 1 ? route_rank_kernel<0, true> : route_rank_kernel<0, false>);
  if (rank_smem > 48 * 1024) {
    st = allow_max_dynamic_smem(kern);
    if (st != cudaSuccess) return st;
  }
  return launch_pdl(kern, (unsigned)num_chunks, kRankThreads, rank_smem, c.stream, idx, T, E, k,
                    chunk_tokens, (int)num_chunks, align, num_rows, ws, counts, offsets, pos,
                    sorted_src, c.err);
}

cudaError_t launch_route_map(const LaunchCtx& c, const int32_t* idx, int64_t T, int E, int k,
                             int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* sorted_src,
                             int32_t* ws, int64_t num_chunks) {
  // small T: one launch in which every block builds the whole map itself
  if (route_map_replicated_ok(T, E, k))
    return launch_route_map_replicated(c, idx, T, E, k, counts, offsets, pos, sorted_src);
  return launch_route_map_aligned(c, idx, T, E, k, 1, T * k, counts, offsets, pos, sorted_src, ws,
                                  num_chunks);
}

}  // namespace moe
