// decode_replicated.cu -- top-k gate, route map and expand + E4M3 cast of a
// decode batch with no communication between blocks, and the route map alone
// for small T.
//
// "CuTeDSL at Perplexity" (perplexity.ai), the prefill/decode section: decode
// kernels run at launch latency, so the fewer dependent launches the better;
// the MoE dispatch section routes with shared-memory counters.  Here every
// block builds the whole route map in its own shared memory (per-expert
// 32-token bitmaps and popcount ranks), then handles only its own tokens:
// their pos and sorted_src entries, and their cast rows.  There is no grid
// barrier, no wait on another block and no cooperative launch; every launch
// takes part in programmatic dependent launch like the separate kernels.
//
//   * T <= 32: one launch; every block also selects the experts of all T
//     tokens (T / 16 per warp), block 0 writing idx, w, counts and offsets.
//   * larger T (to 2048): the top-k kernel runs first (once, on all SMs), then
//     one launch builds the map in every block from the T*k ids in L2.
//   * the same kernel without the expand is moe_route_map for T <= 1024.
//
// Results are those of moe_topk_gate + moe_route_map + moe_expand_cast_fp8:
// the same top-k routine, the route map's stable order (copies of one expert
// in ascending token order), and the same scale arithmetic.
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr int kRepWarps = 16;
constexpr int kRepThreads = kRepWarps * 32;
constexpr int kRepBatch = 8;  // ids a thread loads before their atomics (two-launch form)

struct RepArgs {
  const float* scores;
  const uint16_t* x;
  int32_t* idx;
  float* w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* pos;
  int32_t* src;
  uint8_t* out;
  float* out_sf;
  unsigned* err;
  int T, E, k, H;
  FastDiv fk;  // division by k
};

// Shared memory beyond the static arrays: idx and pos [T*k], offsets [E],
// bitmaps [W][E] u32 and their word prefixes [W][E] u16 (W = ceil(T/32)).
size_t rep_dyn_smem(int T, int E, int k) {
  const size_t P = (size_t)T * k, W = ((size_t)T + 31) / 32;
  return 4 * (2 * P + E) + 4 * W * E + ((2 * W * E + 15) / 16) * 16;
}

// The block's own tokens are t = blockIdx.x + i * gridDim.x, i < own_tokens().
// H/16 threads cast one token (16 channels each; an 8-lane group is one
// 128-channel group), so kRepThreads / (H/16) tokens go at a time.
__device__ __forceinline__ int own_tokens(int T) {
  return (T - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
}

// The first x loads of this thread's first own token.
__device__ __forceinline__ void own_first_loads(const RepArgs& a, uint4& va, uint4& vb) {
  const int P16 = a.H >> 4, slot = (int)threadIdx.x / P16, c = (int)threadIdx.x - slot * P16;
  va = make_uint4(0, 0, 0, 0);
  vb = va;
  if (slot < kRepThreads / P16 && slot < own_tokens(a.T)) {
    const int64_t t = (int64_t)blockIdx.x + (int64_t)slot * gridDim.x;
    va = ld_stream_v4(a.x + t * a.H + c * 16);
    vb = ld_stream_v4(a.x + t * a.H + c * 16 + 8);
  }
}

// Cast the block's own tokens once each and write their k rows.  The row of
// copy j of own token i (token t) is s_pos[OWN ? i * k + j : t * k + j].
// Every thread runs the same number of iterations (the group maxima shuffle
// across lanes); va/vb hold the first token's loads (own_first_loads).
template <bool OWN>
__device__ __forceinline__ void cast_own_tokens(const RepArgs& a, const int32_t* s_pos, uint4 va,
                                                uint4 vb) {
  const int H = a.H, k = a.k, G = H >> 7, P = a.T * k;
  const int P16 = H >> 4, per = kRepThreads / P16;
  const int slot = (int)threadIdx.x / P16, c = (int)threadIdx.x - slot * P16;
  const int nt = own_tokens(a.T);
  const int iters = (nt + per - 1) / per;
  for (int it = 0; it < iters; ++it) {
    const int i = it * per + slot;
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    const bool live = slot < per && i < nt;
    const uint4 ca = va, cb = vb;
    const int in = i + per;
    if (slot < per && in < nt) {  // the next token's loads stay in flight during this one
      const int64_t tn = (int64_t)blockIdx.x + (int64_t)in * gridDim.x;
      va = ld_stream_v4(a.x + tn * H + c * 16);
      vb = ld_stream_v4(a.x + tn * H + c * 16 + 8);
    }
    const float amax = max8(absmax16_bf16(ca, cb));  // every lane: shuffles over 8 lanes
    const float sf = group_scale(amax);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16_bf16(ca, cb, inv);
    if (live) {
      for (int j = 0; j < k; ++j) {
        const int r = s_pos[OWN ? i * k + j : t * k + j];
        if (r < 0 || r >= P) continue;
        st_stream_v4(a.out + (int64_t)r * H + c * 16, q);
        if ((c & 7) == 0) st_stream_f32(a.out_sf + (int64_t)r * G + (c >> 3), sf);
      }
    }
  }
}

template <int V, bool VEC, int KMAX>
__global__ void __launch_bounds__(kRepThreads, 1) decode_replicated_kernel(RepArgs a) {
  __shared__ unsigned long long s_list[kRepWarps][V][32];
  __shared__ unsigned long long s_cand[kRepWarps][32];
  __shared__ int s_scan[2 * 32];  // warp totals, then exclusive warp prefixes
  extern __shared__ __align__(16) int32_t s_dyn[];
  const int T = a.T, E = a.E, k = a.k;
  const int P = T * k, W = (T + 31) >> 5;
  int32_t* s_idx = s_dyn;
  int32_t* s_pos = s_idx + P;
  int32_t* s_off = s_pos + P;
  uint32_t* bm = reinterpret_cast<uint32_t*>(s_off + E);
  uint16_t* pre = reinterpret_cast<uint16_t*>(bm + W * E);
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;
  const bool b0 = blockIdx.x == 0;
  // this block's first tokens: their loads go out before the selection
  uint4 va, vb;
  own_first_loads(a, va, vb);
  for (int i = tid; i < W * E; i += kRepThreads) bm[i] = 0u;

  // ---- 1: the experts of every token (block 0: also the weights)
  uint32_t sel_e;
  for (int tt = wib; tt < T; tt += kRepWarps)
    topk_token<V, VEC, KMAX>(a.scores + (int64_t)tt * E, E, k, lane, s_list[wib], s_cand[wib],
                             s_idx + tt * k,
                             (b0 && a.w != nullptr) ? a.w + (int64_t)tt * k : nullptr, sel_e);
  __syncthreads();

  // ---- 2: the route map.  Bit (t % 32) of bm[t / 32][e] <=> token t chose e;
  // a copy's row is offsets[e] + (copies in earlier words) + popc(lower bits).
  for (int p = tid; p < P; p += kRepThreads) {
    const int e = s_idx[p];
    if ((unsigned)e < (unsigned)E) {
      const int tt = (int)a.fk.div((uint32_t)p);
      atomicOr(bm + (tt >> 5) * E + e, 1u << (tt & 31));
    }
  }
  __syncthreads();
  int total = 0;
  if (tid < E) {
    for (int w = 0; w < W; ++w) {
      pre[w * E + tid] = (uint16_t)total;
      total += __popc(bm[w * E + tid]);
    }
  }
  const int incl = warp_incl_scan(total, lane);  // exclusive scan of the totals over e
  if (lane == 31) s_scan[wib] = incl;
  __syncthreads();
  if (wib == 0) {
    const int v = lane < kRepWarps ? s_scan[lane] : 0;
    const int sc = warp_incl_scan(v, lane);
    if (lane < kRepWarps) s_scan[32 + lane] = sc - v;
  }
  __syncthreads();
  if (tid < E) {
    const int excl = s_scan[32 + wib] + incl - total;
    s_off[tid] = excl;
    if (b0) {
      a.counts[tid] = total;
      a.offsets[tid] = excl;
    }
  }
  if (b0 && tid == 0) a.offsets[E] = s_scan[32 + kRepWarps - 1] + s_scan[kRepWarps - 1];
  __syncthreads();
  for (int p = tid; p < P; p += kRepThreads) {
    const int e = s_idx[p];
    int r = -1;
    if ((unsigned)e < (unsigned)E) {
      const int tt = (int)a.fk.div((uint32_t)p);
      const int wd = (tt >> 5) * E + e;
      r = s_off[e] + pre[wd] + __popc(bm[wd] & ((1u << (tt & 31)) - 1u));
    } else if (b0) {
      flag_error(a.err, MOE_DEVERR_EXPERT_RANGE);  // top-k never selects one
    }
    s_pos[p] = r;
    if (b0) {
      a.idx[p] = e;
      a.pos[p] = r;
      if (r >= 0 && MOE_DBG_OK(r < P, a.err)) a.src[r] = p;
    }
  }
  __syncthreads();

  // ---- 3: this block's tokens, cast once and written to their k rows
  cast_own_tokens<false>(a, s_pos, va, vb);
}

// Shared memory of the route-only kernel: offsets [E], bitmaps [W][E] u32,
// word prefixes [W][E] u16, and the rows of this block's copies [tpb * k].
size_t route_rep_smem(int T, int E, int k, int tpb) {
  const size_t W = ((size_t)T + 31) / 32;
  return 4 * (size_t)E + 4 * W * E + ((2 * W * E + 15) / 16) * 16 + 4 * (size_t)tpb * k;
}

// The second launch of the two-launch form: a.idx holds the top-k launch's
// expert ids.  Every block builds the route map of all T*k copies in its own
// shared memory, then takes its tokens t = blockIdx.x + i * gridDim.x.  With
// EXPAND = false it is the route map alone (moe_route_map for small T, where
// the ids may come from anywhere: a token naming one expert twice is
// flagged, as the two-kernel route map does).
template <bool EXPAND>
__global__ void __launch_bounds__(kRepThreads, 1) route_expand_replicated_kernel(RepArgs a) {
  __shared__ int s_scan[2 * 32];
  extern __shared__ __align__(16) int32_t s_dyn[];
  const int T = a.T, E = a.E, k = a.k;
  const int P = T * k, W = (T + 31) >> 5;
  int32_t* s_off = s_dyn;
  uint32_t* bm = reinterpret_cast<uint32_t*>(s_off + E);
  uint16_t* pre = reinterpret_cast<uint16_t*>(bm + W * E);
  int32_t* s_pos = reinterpret_cast<int32_t*>(pre + ((W * E + 7) & ~7));
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;
  const bool b0 = blockIdx.x == 0;
  // This block's first tokens: x is read before the wait for the top-k
  // launch.  That launch itself waited for every earlier kernel before it
  // could let this one start, so x (an input of both) is complete here.
  uint4 va = make_uint4(0, 0, 0, 0), vb = va;
  if (EXPAND) own_first_loads(a, va, vb);
  for (int i = tid; i < W * E; i += kRepThreads) bm[i] = 0u;
  __syncthreads();
  pdl_enter();  // the expert ids

  // ---- the route map of every copy, as in the one-launch form.  The ids are
  // loaded kRepBatch at a time before their atomics (one round of L2 latency
  // per batch instead of one per copy).
  bool dup = false;
  for (int p0 = 0; p0 < P; p0 += kRepBatch * kRepThreads) {
    int ev[kRepBatch];
#pragma unroll
    for (int u = 0; u < kRepBatch; ++u) {
      const int p = p0 + tid + u * kRepThreads;
      ev[u] = p < P ? __ldcg(a.idx + p) : -1;
    }
#pragma unroll
    for (int u = 0; u < kRepBatch; ++u) {
      const int p = p0 + tid + u * kRepThreads;
      if (p < P && (unsigned)ev[u] < (unsigned)E) {
        const int tt = (int)a.fk.div((uint32_t)p);
        const uint32_t bit = 1u << (tt & 31);
        dup |= (atomicOr(bm + (tt >> 5) * E + ev[u], bit) & bit) != 0u;
      }
    }
  }
  if (dup && b0) flag_error(a.err, MOE_DEVERR_DUPLICATE_EXPERT);
  __syncthreads();
  int total = 0;
  if (tid < E) {
    for (int w = 0; w < W; ++w) {
      pre[w * E + tid] = (uint16_t)total;
      total += __popc(bm[w * E + tid]);
    }
  }
  const int incl = warp_incl_scan(total, lane);
  if (lane == 31) s_scan[wib] = incl;
  __syncthreads();
  if (wib == 0) {
    const int v = lane < kRepWarps ? s_scan[lane] : 0;
    const int sc = warp_incl_scan(v, lane);
    if (lane < kRepWarps) s_scan[32 + lane] = sc - v;
  }
  __syncthreads();
  if (tid < E) {
    const int excl = s_scan[32 + wib] + incl - total;
    s_off[tid] = excl;
    if (b0) {
      a.counts[tid] = total;
      a.offsets[tid] = excl;
    }
  }
  if (b0) {
    const int all = s_scan[32 + kRepWarps - 1] + s_scan[kRepWarps - 1];  // copies counted
    if (tid == 0) a.offsets[E] = all;
    for (int r = all + tid; r < P; r += kRepThreads) a.src[r] = -1;  // rows no copy takes
  }
  __syncthreads();
  // ---- this block's copies: their rows, pos and sorted_src entries
  const int nt = (T - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // tokens here
  bool bad = false;
  for (int q = tid; q < nt * k; q += kRepThreads) {
    const int i = (int)a.fk.div((uint32_t)q), j = q - i * k;
    const int tt = (int)blockIdx.x + i * (int)gridDim.x;
    const int p = tt * k + j;
    const int e = __ldcg(a.idx + p);
    int r = -1;
    if ((unsigned)e < (unsigned)E) {
      const int wd = (tt >> 5) * E + e;
      r = s_off[e] + pre[wd] + __popc(bm[wd] & ((1u << (tt & 31)) - 1u));
      if (MOE_DBG_OK(r >= 0 && r < P, a.err)) a.src[r] = p;
    } else {
      bad = true;  // top-k never selects one
    }
    s_pos[q] = r;
    a.pos[p] = r;
  }
  if (bad) flag_error(a.err, MOE_DEVERR_EXPERT_RANGE);
  if (!EXPAND) return;
  __syncthreads();

  // ---- cast once, write k rows, as in the one-launch form
  cast_own_tokens<true>(a, s_pos, va, vb);
}

template <int V, bool VEC, int KMAX>
cudaError_t launch_t(const LaunchCtx& c, const RepArgs& a, int blocks, size_t smem) {
  auto kern = decode_replicated_kernel<V, VEC, KMAX>;
  cudaError_t e = allow_max_dynamic_smem(kern);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, blocks, kRepThreads, smem, c.stream, a);
}

}  // namespace

bool decode_replicated_ok(int64_t T, int E, int k, int H) {
  if (T < 1 || E <= 32 || E > 256 || k > 32 || H > 8192) return false;
  if (T <= kDecodeReplicatedInlineTokens) return T * k <= 4096;  // one launch
  return T <= kDecodeReplicatedMaxTokens && T * k <= 16384;      // top-k launch + route/expand
}

cudaError_t launch_decode_replicated(const LaunchCtx& c, const float* scores, int64_t T, int E,
                                     int k, const void* x, int H, int32_t* idx, float* w,
                                     int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                                     uint8_t* out, float* out_sf) {
  if (!decode_replicated_ok(T, E, k, H)) return cudaErrorInvalidValue;
  RepArgs a;
  a.scores = scores;
  a.x = static_cast<const uint16_t*>(x);
  a.idx = idx;
  a.w = w;
  a.counts = counts;
  a.offsets = offsets;
  a.pos = pos;
  a.src = src;
  a.out = out;
  a.out_sf = out_sf;
  a.err = c.err;
  a.T = (int)T;
  a.E = E;
  a.k = k;
  a.H = H;
  a.fk = FastDiv((uint32_t)k);
  const int blocks = (int)(T < c.num_sms ? T : c.num_sms);
  if (T > kDecodeReplicatedInlineTokens) {
    cudaError_t e = launch_topk_gate(c, scores, T, E, k, idx, w);
    if (e != cudaSuccess) return e;
    const int tpb = (int)((T + blocks - 1) / blocks);
    const size_t smem = route_rep_smem((int)T, E, k, tpb);
    e = allow_max_dynamic_smem(route_expand_replicated_kernel<true>);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_expand_replicated_kernel<true>, blocks, kRepThreads, smem, c.stream,
                      a);
  }
  const size_t smem = rep_dyn_smem((int)T, E, k);
  const bool vec = (E % 128 == 0) && (reinterpret_cast<uintptr_t>(scores) % 16 == 0);
  if (E <= 64) return k <= 8 ? launch_t<2, false, 8>(c, a, blocks, smem)
                             : launch_t<2, false, 32>(c, a, blocks, smem);
  if (E <= 128) {
    if (vec) return k <= 8 ? launch_t<4, true, 8>(c, a, blocks, smem)
                           : launch_t<4, true, 32>(c, a, blocks, smem);
    return k <= 8 ? launch_t<4, false, 8>(c, a, blocks, smem)
                  : launch_t<4, false, 32>(c, a, blocks, smem);
  }
  if (vec) return k <= 8 ? launch_t<8, true, 8>(c, a, blocks, smem)
                         : launch_t<8, true, 32>(c, a, blocks, smem);
  return k <= 8 ? launch_t<8, false, 8>(c, a, blocks, smem)
                : launch_t<8, false, 32>(c, a, blocks, smem);
}

bool route_map_replicated_ok(int64_t T, int E, int k) {
  return T >= 1 && T <= kRouteMapReplicatedMaxTokens && E >= 1 && E <= 256 && T * k <= 16384;
}

cudaError_t launch_route_map_replicated(const LaunchCtx& c, const int32_t* idx, int64_t T, int E,
                                        int k, int32_t* counts, int32_t* offsets, int32_t* pos,
                                        int32_t* src) {
  if (!route_map_replicated_ok(T, E, k)) return cudaErrorInvalidValue;
  RepArgs a = {};
  a.idx = const_cast<int32_t*>(idx);  // read only
  a.counts = counts;
  a.offsets = offsets;
  a.pos = pos;
  a.src = src;
  a.err = c.err;
  a.T = (int)T;
  a.E = E;
  a.k = k;
  a.H = 0;
  a.fk = FastDiv((uint32_t)k);
  const int blocks = (int)(T < c.num_sms ? T : c.num_sms);
  const int tpb = (int)((T + blocks - 1) / blocks);
  const size_t smem = route_rep_smem((int)T, E, k, tpb);
  cudaError_t e = allow_max_dynamic_smem(route_expand_replicated_kernel<false>);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_expand_replicated_kernel<false>, blocks, kRepThreads, smem, c.stream, a);
}

}  // namespace moe
