// route_chain.cu -- top-k, route map and expand + E4M3 cast in three launches.
//
// TileKernels article (itsolotime.com), section 2: the routing chain Top-K
// Gating -> counting -> token-expert mapping -> fused expand; "CuTeDSL at
// Perplexity", MoE dispatch: the local route kernel counts the tokens of each
// expert while it routes, and for prefill the counts of many blocks are
// aggregated before the copy kernel runs.
//
// The separate calls need four launches (top-k, the route map's histogram
// and rank passes, the expand).  Here:
//   1. chain_topk_kernel: one CTA per chunk of C consecutive tokens (16 warps,
//      C / 16 tokens each) selects the experts of its tokens (topk_token),
//      marks them in a shared-memory bitmap per expert (bit = the token's
//      place in the chunk), and from it writes each copy's rank among its
//      expert's copies in the chunk (into pos) and the chunk's histogram row.
//   2. chain_scan_kernel: for every expert, the exclusive prefix of its
//      histogram column over the chunks (in place: the copies of the expert
//      in earlier chunks) and the total (counts).  One CTA per 32 experts,
//      lane = expert, so each warp load reads 32 consecutive counters of one
//      row; the last CTA to finish scans the totals into the offsets.
//   3. the expand kernel's chained form places every copy itself (its
//      expert's offset + the chunk's base + the copy's rank in the chunk),
//      writes pos and sorted_src, and stores the rows.
// The result is the separate calls' result bit for bit: the copies of an
// expert are ordered by token (a token's k experts are distinct), which is
// the order of (chunk, place in chunk).
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr int kChainWarps = 16;
constexpr int kScanWarps = 32;

// Tokens per chunk: a power of two from 16 (one per warp) to 64 (four per
// warp), chosen so that the histogram stays small while every SM still gets
// several chunks: 16 up to 16K tokens, 32 up to 32K, else 64.
inline int chain_chunk_shift(int64_t T) { return T <= 16384 ? 4 : (T <= 32768 ? 5 : 6); }

// TPW tokens per warp: the chunk is 16 TPW tokens.
template <int V, bool VEC, int KMAX, int TPW>
__global__ void __launch_bounds__(kChainWarps * 32) chain_topk_kernel(
    const float* __restrict__ scores, int64_t T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* __restrict__ rank, int32_t* __restrict__ hist) {
  __shared__ unsigned long long s_list[kChainWarps][V][32];
  __shared__ unsigned long long s_cand[kChainWarps][32];
  constexpr int W = (kChainWarps * TPW + 31) / 32;  // 32-token bitmap words per chunk
  __shared__ uint32_t s_bits[W][256];                // [word][E], E <= 256
  __shared__ int32_t s_sel[TPW][kChainWarps][32];    // slot << 16 | expert, or -1
  pdl_enter();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * (kChainWarps * TPW);
  for (int e = tid; e < E; e += kChainWarps * 32) {
#pragma unroll
    for (int w = 0; w < W; ++w) s_bits[w][e] = 0u;
  }
  __syncthreads();
  // token c0 + i for i = warp, warp + 16, ... (TPW per warp); each lane's
  // selection is kept in shared memory (not registers) until the ranks
  for (int u = 0; u < TPW; ++u) {
    const int i = warp + u * kChainWarps;
    const int64_t t = c0 + i;
    int32_t sel = -1;
    if (t < T) {
      uint32_t e;
      const int j = topk_token<V, VEC, KMAX>(scores + t * E, E, k, lane, s_list[warp],
                                             s_cand[warp], topk_idx + t * k, topk_w + t * k, e);
      if (j >= 0) {
        atomicOr(&s_bits[i >> 5][e], 1u << (i & 31));
        sel = (j << 16) | (int32_t)e;
      }
    }
    s_sel[u][warp][lane] = sel;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < TPW; ++u) {
    const int i = warp + u * kChainWarps;
    const int32_t sel = s_sel[u][warp][lane];
    if (sel >= 0) {
      const int ex = sel & 0xFFFF;
      int r = __popc(s_bits[i >> 5][ex] & ((1u << (i & 31)) - 1u));
#pragma unroll
      for (int w = 0; w < W; ++w) r += w < (i >> 5) ? __popc(s_bits[w][ex]) : 0;
      rank[(c0 + i) * k + (sel >> 16)] = r;
    }
  }
  int32_t* row = hist + (int64_t)blockIdx.x * E;
  for (int e = tid; e < E; e += kChainWarps * 32) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) n += __popc(s_bits[w][e]);
    row[e] = n;
  }
}

// The column scan.  CTA b owns experts 32 b .. 32 b + 31 (lane = expert), and
// warp w rows [w R/32, (w + 1) R/32) of the histogram, held in registers
// between the two passes:
//   1. each warp sums its rows; the warps' partial sums are scanned in shared
//      memory, giving every warp the count of its rows' predecessors and every
//      expert its total (counts[e]);
//   2. each warp rewrites its rows in place as the copies of expert e in
//      earlier chunks;
//   3. the CTA that finishes last (an arrival counter in the caller's
//      workspace, zero before the call and left at zero) scans the totals
//      into offsets.  No CTA waits for another.
// The expand adds offsets[e] to a chunk's base to place the chunk's copies.
constexpr int kScanRowsInRegs = 16;  // rows per warp held in registers

__global__ void __launch_bounds__(kScanWarps * 32) chain_scan_kernel(
    int32_t* __restrict__ hist, int64_t rows, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, unsigned* __restrict__ arrivals) {
  __shared__ int32_t s_part[kScanWarps][32];
  __shared__ int s_last;
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const bool on = e < E;
  const int64_t per = (rows + kScanWarps - 1) / kScanWarps;
  const int64_t r0 = warp * per;
  const int64_t r1 = r0 + per < rows ? r0 + per : rows;
  const bool in_regs = per <= kScanRowsInRegs;
  int32_t v[kScanRowsInRegs];
  int32_t sum = 0;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kScanRowsInRegs; ++u)
      v[u] = (on && r0 + u < r1) ? hist[(r0 + u) * E + e] : 0;
#pragma unroll
    for (int u = 0; u < kScanRowsInRegs; ++u) sum += v[u];
  } else {
    for (int64_t r = r0; r < r1; r += 8) {
      int32_t w8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w8[u] = (on && r + u < r1) ? hist[(r + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += w8[u];
    }
  }
  s_part[warp][lane] = sum;
  __syncthreads();
  int32_t run = 0, total = 0;
#pragma unroll 8
  for (int w = 0; w < kScanWarps; ++w) {
    const int32_t p = s_part[w][lane];
    run += w < warp ? p : 0;
    total += p;
  }
  if (warp == 0 && on) counts[e] = total;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kScanRowsInRegs; ++u) {
      if (on && r0 + u < r1) hist[(r0 + u) * E + e] = run;
      run += v[u];
    }
  } else {
    for (int64_t r = r0; r < r1; r += 8) {
      int32_t w8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w8[u] = (on && r + u < r1) ? hist[(r + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (on && r + u < r1) hist[(r + u) * E + e] = run;
        run += w8[u];
      }
    }
  }
  // ---- the last CTA to finish turns the totals into offsets
  if (warp == 0) __threadfence();  // this CTA's counts are visible before its arrival
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(arrivals, 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  int32_t c[8];  // E <= 256: experts 8 lane .. 8 lane + 7
#pragma unroll
  for (int j = 0; j < 8; ++j) c[j] = lane * 8 + j < E ? __ldcg(counts + lane * 8 + j) : 0;
  int32_t own = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) own += c[j];
  int32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  int32_t excl = incl - own;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (lane * 8 + j < E) offsets[lane * 8 + j] = excl;
    excl += c[j];
  }
  if (lane == 31) {
    offsets[E] = incl;
    *arrivals = 0u;  // ready for the next call
  }
}

template <int V, bool VEC, int TPW>
cudaError_t launch_topk_tpw(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                            int32_t* idx, float* w, int32_t* rank, int32_t* hist) {
  const int64_t chunks = (T + kChainWarps * TPW - 1) / (kChainWarps * TPW);
  if (k <= 8)
    return launch_pdl(chain_topk_kernel<V, VEC, 8, TPW>, (unsigned)chunks, kChainWarps * 32, 0,
                      c.stream, scores, T, E, k, idx, w, rank, hist);
  return launch_pdl(chain_topk_kernel<V, VEC, 32, TPW>, (unsigned)chunks, kChainWarps * 32, 0,
                    c.stream, scores, T, E, k, idx, w, rank, hist);
}

template <int V, bool VEC>
cudaError_t launch_topk_t(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                          int shift, int32_t* idx, float* w, int32_t* rank, int32_t* hist) {
  if (shift == 4) return launch_topk_tpw<V, VEC, 1>(c, scores, T, E, k, idx, w, rank, hist);
  if (shift == 5) return launch_topk_tpw<V, VEC, 2>(c, scores, T, E, k, idx, w, rank, hist);
  return launch_topk_tpw<V, VEC, 4>(c, scores, T, E, k, idx, w, rank, hist);
}

}  // namespace

bool route_chain_ok(int64_t T, int E, int k, int H, const void* out, const void* out_sf) {
  return T > 0 && E > 32 && E <= 256 && k >= 1 && k <= MOE_MAX_TOPK && H <= 16384 &&
         (H / kGroup) % 4 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(out_sf) % 16 == 0;
}

size_t route_chain_workspace_bytes(int64_t T, int E) {
  if (T <= 0) return 0;
  const int shift = chain_chunk_shift(T);
  const int64_t chunks = (T + (1 << shift) - 1) >> shift;
  return (size_t)((chunks * E * 4 + 255) / 256 * 256);
}

cudaError_t launch_route_chain(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                               const void* x, int H, int32_t* idx, float* w, int32_t* counts,
                               int32_t* offsets, int32_t* pos, int32_t* src, uint8_t* out,
                               float* out_sf, int32_t* hist, unsigned* arrivals) {
  const int shift = chain_chunk_shift(T);
  const int64_t chunks = (T + (1 << shift) - 1) >> shift;
  const bool vec = (E % 128 == 0) && (reinterpret_cast<uintptr_t>(scores) % 16 == 0);
  cudaError_t e;
  if (E <= 64)
    e = launch_topk_t<2, false>(c, scores, T, E, k, shift, idx, w, pos, hist);
  else if (E <= 128)
    e = vec ? launch_topk_t<4, true>(c, scores, T, E, k, shift, idx, w, pos, hist)
            : launch_topk_t<4, false>(c, scores, T, E, k, shift, idx, w, pos, hist);
  else
    e = vec ? launch_topk_t<8, true>(c, scores, T, E, k, shift, idx, w, pos, hist)
            : launch_topk_t<8, false>(c, scores, T, E, k, shift, idx, w, pos, hist);
  if (e != cudaSuccess) return e;
  e = launch_pdl(chain_scan_kernel, (unsigned)((E + 31) / 32), kScanWarps * 32, 0, c.stream, hist,
                 chunks, E, counts, offsets, arrivals);
  if (e != cudaSuccess) return e;
  RouteChain rc;
  rc.idx = idx;
  rc.base = hist;
  rc.offsets = offsets;
  rc.sorted_src = src;
  rc.E = E;
  rc.chunk_shift = shift;
  return launch_expand_cast_chain(c, x, T, H, k, pos, out, out_sf, rc);
}

}  // namespace moe
