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
// Three launches over chunks of kRouteChunkTokens tokens:
//   1. route_count_kernel: one CTA per chunk builds the chunk's histogram in
//      shared memory (order-free atomics) -> hist[chunk][E] in the workspace.
//   2. route_scan_kernel: one CTA per 32 experts scans its columns of hist
//      down the chunks (exclusive) and writes counts[e].
//   3. route_rank_kernel: one CTA per chunk scans counts into offsets (in
//      shared memory), ranks its copies stably within the chunk with
//      __match_any_sync + per-warp counters, and writes pos and sorted_src.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCountThreads = 256;
constexpr int kRankWarps = 16;
constexpr int kRankThreads = kRankWarps * 32;
// Copies a lane ranks per chunk: kRouteChunkTokens * k / kRankThreads rounds
// at most (k <= 32 -> 128 * 32 / 512 = 8).
constexpr int kMaxRounds = (kRouteChunkTokens * 32) / kRankThreads;

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(
    const int32_t* __restrict__ idx, int64_t R, int E, int k, int32_t* __restrict__ hist,
    unsigned* err) {
  extern __shared__ int32_t s_hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * kRouteChunkTokens * k;
  const int64_t p1 = min(p0 + (int64_t)kRouteChunkTokens * k, R);
  bool bad = false;
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = __ldg(idx + p);
    if ((unsigned)e < (unsigned)E)
      atomicAdd(&s_hist[e], 1);
    else
      bad = true;
  }
  if (bad) flag_error(err, MOE_DEVERR_EXPERT_RANGE);
  __syncthreads();
  int32_t* out = hist + (int64_t)blockIdx.x * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = s_hist[e];
}

// blockDim = (32, 32): x = expert within the CTA's 32, y = one of 32 runs of
// consecutive chunks.  hist[c][e] becomes the number of copies of e in chunks
// before c (exclusive down the column); counts[e] gets the column total.
__global__ void __launch_bounds__(1024) route_scan_kernel(int32_t* __restrict__ hist,
                                                          int64_t num_chunks, int E,
                                                          int32_t* __restrict__ counts) {
  __shared__ int32_t part[32][33];
  const int e = blockIdx.x * 32 + threadIdx.x;
  const int64_t per = (num_chunks + 31) / 32;
  const int64_t c0 = threadIdx.y * per;
  const int64_t c1 = min(c0 + per, num_chunks);
  int32_t sum = 0;
  if (e < E)
    for (int64_t c = c0; c < c1; ++c) sum += hist[c * E + e];
  part[threadIdx.y][threadIdx.x] = sum;
  __syncthreads();
  int32_t run = 0;
  for (int y = 0; y < (int)threadIdx.y; ++y) run += part[y][threadIdx.x];
  if (threadIdx.y == 31 && e < E) counts[e] = run + sum;
  if (e < E)
    for (int64_t c = c0; c < c1; ++c) {
      const int32_t v = hist[c * E + e];
      hist[c * E + e] = run;
      run += v;
    }
}

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__global__ void __launch_bounds__(kRankThreads) route_rank_kernel(
    const int32_t* __restrict__ idx, int64_t R, int E, int k, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ offsets, int32_t* __restrict__ pos,
    int32_t* __restrict__ sorted_src, unsigned* err) {
  extern __shared__ int32_t smem[];
  int32_t* s_off = smem;                 // [E] expert offsets
  int32_t* s_wcnt = smem + E;            // [kRankWarps][E] per-warp counters
  __shared__ int32_t s_warp_tot[kRankWarps];
  __shared__ int32_t s_carry;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- offsets: exclusive scan of counts[0..E) in chunks of kRankThreads
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < E; base += kRankThreads) {
    const int e = base + tid;
    const int32_t v = (e < E) ? __ldg(counts + e) : 0;
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
    __syncthreads();
    if (tid == kRankThreads - 1) s_carry = excl + v;
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += kRankThreads) offsets[e] = s_off[e];
    if (tid == 0) offsets[E] = s_carry;
  }
  for (int i = tid; i < kRankWarps * E; i += kRankThreads) s_wcnt[i] = 0;
  __syncthreads();

  // ---- stable ranks inside the chunk: warp w owns a contiguous run of copies
  const int64_t p0 = (int64_t)blockIdx.x * kRouteChunkTokens * k;
  const int64_t p1 = min(p0 + (int64_t)kRouteChunkTokens * k, R);
  const int64_t n = p1 - p0;
  const int64_t per_warp = ((n + kRankWarps * 32 - 1) / (kRankWarps * 32)) * 32;
  const int64_t w0 = p0 + warp * per_warp;
  const int rounds = (int)(per_warp / 32);
  int32_t* wcnt = s_wcnt + warp * E;
  const unsigned lt_mask = (1u << lane) - 1u;
  int32_t r_e[kMaxRounds];
  int32_t r_rank[kMaxRounds];
#pragma unroll
  for (int r = 0; r < kMaxRounds; ++r) {
    r_e[r] = -1;
    r_rank[r] = 0;
    if (r < rounds) {
      const int64_t p = w0 + r * 32 + lane;
      const bool valid = p < p1;
      const int e = valid ? __ldg(idx + p) : -1;
      const bool ok = valid && (unsigned)e < (unsigned)E;
      // invalid lanes get a key no other lane has
      const unsigned key = ok ? (unsigned)e : (0x80000000u | (unsigned)lane);
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
      int32_t before = 0;
      if (ok) before = wcnt[e];
      __syncwarp();
      if (ok && (peers & lt_mask) == 0) wcnt[e] = before + __popc(peers);
      __syncwarp();
      if (ok) {
        r_e[r] = e;
        r_rank[r] = before + __popc(peers & lt_mask);
      } else if (valid) {
        r_e[r] = -2;  // out-of-range expert: dropped copy
      }
    }
  }
  __syncthreads();
  // exclusive scan of the per-warp counters, per expert
  for (int e = tid; e < E; e += kRankThreads) {
    int32_t run = 0;
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
      const int32_t v = s_wcnt[w * E + e];
      s_wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  const int32_t* cbase = chunk_base + (int64_t)blockIdx.x * E;
#pragma unroll
  for (int r = 0; r < kMaxRounds; ++r) {
    if (r < rounds) {
      const int64_t p = w0 + r * 32 + lane;
      const int e = r_e[r];
      if (e >= 0) {
        const int32_t slot = s_off[e] + __ldg(cbase + e) + wcnt[e] + r_rank[r];
        // slot < R whenever topk_idx is unchanged since the count kernel read
        // it; a caller who rewrote it in between gets a flag, not a wild write
        if ((unsigned)slot < (unsigned)R) {
          pos[p] = slot;
          sorted_src[slot] = (int32_t)p;
        } else {
          pos[p] = -1;
          flag_error(err, MOE_DEVERR_EXPERT_RANGE);
        }
      } else if (e == -2) {
        pos[p] = -1;
      }
    }
  }
}

}  // namespace

cudaError_t launch_route_map(const LaunchCtx& c, const int32_t* idx, int64_t T, int E, int k,
                             int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* sorted_src,
                             int32_t* ws, int64_t num_chunks) {
  const int64_t R = T * k;
  const size_t count_smem = sizeof(int32_t) * E;
  route_count_kernel<<<(unsigned)num_chunks, kCountThreads, count_smem, c.stream>>>(idx, R, E, k, ws,
                                                                                  c.err);
  cudaError_t st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  route_scan_kernel<<<(E + 31) / 32, dim3(32, 32), 0, c.stream>>>(ws, num_chunks, E, counts);
  st = cudaGetLastError();
  if (st != cudaSuccess) return st;
  const size_t rank_smem = sizeof(int32_t) * (size_t)E * (1 + kRankWarps);
  if (rank_smem > 48 * 1024) {
    st = cudaFuncSetAttribute(route_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)rank_smem);
    if (st != cudaSuccess) return st;
  }
  route_rank_kernel<<<(unsigned)num_chunks, kRankThreads, rank_smem, c.stream>>>(
      idx, R, E, k, counts, ws, offsets, pos, sorted_src, c.err);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace moe
