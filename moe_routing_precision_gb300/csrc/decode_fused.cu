// decode_fused.cu -- top-k gate, route map and expand + E4M3 cast of a
// decode-sized batch in ONE cooperative launch.
//
// "CuTeDSL at Perplexity" (perplexity.ai), the prefill/decode section: decode
// kernels run at launch latency, so their work is spread over as many SMs as
// possible and, where every block fits on the device at once, a grid barrier
// replaces the split into several launches; the MoE dispatch section routes
// with one block and copies with the others.  Here the grid is one block per
// SM (cooperative launch, so all blocks are resident) and runs:
//
//   1. every warp: top-k + weights of its tokens (topk_token, as the top-k
//      kernel); every block: the E4M3 cast of its own tokens into shared
//      memory (the codes do not depend on the routing);  then each block
//      arrives on a counter in the workspace;
//   2. block 0, once all blocks arrived: the route map of all T*k copies
//      (counts, offsets, stable pos, sorted_src; per-expert token bitmaps and
//      popcount ranks), then one more arrival as the "routed" signal;
//   3. every block, once routed: its tokens' k code rows and scale rows go
//      out from shared memory, every thread storing 16-byte chunks (measured
//      on GB300: one thread issuing TMA bulk copies of the rows wrote at less
//      than half the rate).
//
// Every wait is bounded (globaltimer and an iteration cap).  A wait that runs
// out sets MOE_DEVERR_TIMEOUT, skips what depends on it and still finishes the
// protocol, so the context stays usable.  The last block to finish resets the
// two control words to zero, which every launch expects to find.
//
// Results are those of moe_topk_gate + moe_route_map + moe_expand_cast_fp8:
// the same top-k routine, the same scale arithmetic, and the route map's
// stable order (copies of one expert in ascending t*k + j).
#include <atomic>

#include "topk_warp.cuh"

namespace moe {

std::atomic<int64_t> g_decode_timeout_ns{1000000000};  // 1 s
std::atomic<int> g_decode_skip_signal{0};

namespace {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kSlices = 4;  // 16-channel slices whose loads a thread keeps in flight
constexpr int kRouteCopies = 16384 / kDecThreads;  // copies per thread in the route map (T*k <= 16384)

struct DecodeArgs {
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
  unsigned* ctl;  // [0]: arrivals (grid, then grid + 1 once routed); [1]: finished blocks
  unsigned* err;
  int64_t timeout_ns;
  int T, E, k, H;
  int tpb;          // tokens cast by each block
  int stage_bytes;  // bytes per staged token: H codes + G f32 scales, rounded to 16
  int skip_signal;  // test hook: block 0 never sends the routed signal
  FastDiv fk;       // division by k
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until *p >= target; false once timeout_ns have passed (or, should the
// timer stall, after an iteration cap of the same order).  (Relaxed polling
// every 200 ns plus a fence was measured no faster than this.)
__device__ bool wait_at_least(const unsigned* p, unsigned target, int64_t timeout_ns) {
  const uint64_t t0 = global_ns();
  const int64_t cap = timeout_ns / 32 + 1024;
  for (int64_t i = 0; i < cap; ++i) {
    if (ld_acquire_gpu(p) >= target) return true;
    if ((int64_t)(global_ns() - t0) > timeout_ns) break;
    __nanosleep(64);
  }
  return ld_acquire_gpu(p) >= target;
}

// Route map of all P = T*k copies by one block.  A token names each of its
// experts once, so per expert and per 32-token word w the tokens that chose
// it form a bitmap bm[w][e] (shared-memory atomicOr: the result does not
// depend on the order).  Thread e then walks its W words, storing before each
// the number of tokens in the earlier words (pre[w][e]); the count is the
// total.  The stable row of copy (t, j) with expert e is
//   offsets[e] + pre[t / 32][e] + popc(bm[t / 32][e] & bits below t % 32),
// i.e. its rank in ascending token order among expert e's copies.
// Shared memory: bm [W][E] u32, pre [W][E] u16 (T <= 2048, W <= 64), and
// sorted_src [T*k]; bm and pre are word-major,
// so that the lanes of a warp (one token word, different experts) hit
// different banks.  In [E][W] order every copy of a warp landed in one bank
// and the atomics serialised.
__device__ void route_block(const DecodeArgs& a, uint32_t* bm, uint16_t* pre, int* s_src,
                            int* s_scan) {
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;
  const int E = a.E, k = a.k, T = a.T;
  const int W = (T + 31) >> 5;
  const int P = T * k;
  // thread tid owns copies tid + u * kDecThreads; all their experts are loaded
  // at once (one round of L2 latency) and kept in registers for both passes
  int ev[kRouteCopies];
#pragma unroll
  for (int u = 0; u < kRouteCopies; ++u) {
    const int p = tid + u * kDecThreads;
    ev[u] = p < P ? __ldcg(a.idx + p) : -1;
  }
  for (int i = tid; i < E * W; i += kDecThreads) bm[i] = 0u;
  for (int i = tid; i < P; i += kDecThreads) s_src[i] = -1;  // rows no copy takes stay -1
  __syncthreads();
  const FastDiv fk = a.fk;
#pragma unroll
  for (int u = 0; u < kRouteCopies; ++u) {
    const int p = tid + u * kDecThreads;
    if (p >= P) continue;
    const int e = ev[u];
    if (e < 0 || e >= E) {
      flag_error(a.err, MOE_DEVERR_EXPERT_RANGE);  // top-k never writes one
      ev[u] = -1;
      continue;
    }
    const int t = (int)fk.div((uint32_t)p);
    atomicOr(bm + (t >> 5) * E + e, 1u << (t & 31));
  }
  __syncthreads();
  int total = 0;
  if (tid < E) {
    for (int w = 0; w < W; ++w) {
      pre[w * E + tid] = (uint16_t)total;
      total += __popc(bm[w * E + tid]);
    }
  }
  // exclusive scan of the totals over e (E <= kDecThreads)
  int incl = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_scan[wib] = incl;
  __syncthreads();
  if (wib == 0) {
    const int v = lane < kDecWarps ? s_scan[lane] : 0;
    int sc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      if (lane >= o) sc += n;
    }
    if (lane < kDecWarps) s_scan[32 + lane] = sc - v;
  }
  __syncthreads();
  int* s_off = s_scan + 64;  // offsets, shared: [E]
  if (tid < E) {
    const int excl = s_scan[32 + wib] + incl - total;
    a.counts[tid] = total;
    a.offsets[tid] = excl;
    s_off[tid] = excl;
  }
  if (tid == 0) a.offsets[E] = P;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kRouteCopies; ++u) {
    const int p = tid + u * kDecThreads;
    if (p >= P) continue;
    const int e = ev[u];
    if (e < 0) {
      a.pos[p] = -1;  // not routed
      continue;
    }
    const int t = (int)fk.div((uint32_t)p);
    const int wd = (t >> 5) * E + e;
    const int r = s_off[e] + pre[wd] + __popc(bm[wd] & ((1u << (t & 31)) - 1u));
    a.pos[p] = r;
    if (MOE_DBG_OK(r >= 0 && r < P, a.err)) s_src[r] = p;
  }
  __syncthreads();
  // sorted_src leaves in row order (coalesced): scattered 4-byte global stores
  // from a single SM were the slowest part of this block's work
  for (int r = tid; r < P; r += kDecThreads) a.src[r] = s_src[r];
}

template <int V, bool VEC, int KMAX>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fused_kernel(DecodeArgs a) {
  __shared__ unsigned long long s_list[kDecWarps][V][32];
  __shared__ unsigned long long s_cand[kDecWarps][32];
  __shared__ int s_scan[64 + 256];  // warp sums, warp prefixes, offsets
  __shared__ int s_ok;
  // tpb staged tokens, then (block 0) the route map's bm, pre and sorted_src
  extern __shared__ __align__(128) uint8_t s_stage[];
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;
  const int H = a.H, G = H >> 7, k = a.k;
  const int nblk = (int)gridDim.x;

  // ---- 1: top-k of some tokens and the cast of this block's tokens.  Slice
  // s (16 channels) of this block's nt * H/16 slices is token s / (H/16),
  // channel slice s % (H/16); 8 consecutive slices form one 128-channel group.
  // Each thread keeps the loads of kSlices slices in flight; the first batch
  // is issued before the top-k so that its latency overlaps the selection.
  const int t0 = (int)blockIdx.x * a.tpb;
  const int nt = max(0, min(a.tpb, a.T - t0));
  const int P = H >> 4;
  const int S = nt * P;
  const uint16_t* xb = a.x + (int64_t)t0 * H;
  uint4 va[kSlices], vb[kSlices];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int u = 0; u < kSlices; ++u) {
      const int sl = s0 + u * kDecThreads + tid;
      va[u] = make_uint4(0, 0, 0, 0);
      vb[u] = va[u];
      if (sl < S) {  // slices are contiguous in x: token rows follow each other
        va[u] = ld_stream_v4(xb + (int64_t)sl * 16);
        vb[u] = ld_stream_v4(xb + (int64_t)sl * 16 + 8);
      }
    }
  };
  load_batch(0);

  // top-k + weights, one warp per token; token t on block t % grid (warp
  // t / grid), so every block selects about T / grid tokens
  uint32_t sel_e;
  for (int t = (int)blockIdx.x + wib * nblk; t < a.T; t += nblk * kDecWarps)
    topk_token<V, VEC, KMAX>(a.scores + (int64_t)t * a.E, a.E, k, lane, s_list[wib], s_cand[wib],
                             a.idx + (int64_t)t * k, a.w != nullptr ? a.w + (int64_t)t * k : nullptr,
                             sel_e);

  for (int s0 = 0; s0 < S; s0 += kDecThreads * kSlices) {
    if (s0 > 0) load_batch(s0);
#pragma unroll
    for (int u = 0; u < kSlices; ++u) {
      const int sl = s0 + u * kDecThreads + tid;
      const float amax = max8(absmax16_bf16(va[u], vb[u]));
      const float sf = group_scale(amax);
      const float inv = __fdiv_rn(1.0f, sf);
      const uint4 q = quant16_bf16(va[u], vb[u], inv);
      if (sl < S) {
        const int i = sl / P, c = sl - i * P;
        uint8_t* st = s_stage + (size_t)i * a.stage_bytes;
        *reinterpret_cast<uint4*>(st + c * 16) = q;
        if ((c & 7) == 0) *reinterpret_cast<float*>(st + H + 4 * (c >> 3)) = sf;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(a.ctl, 1u);  // arrival: this block's top-k rows are written
  }

  // ---- 2: block 0 routes once every block has arrived
  if (blockIdx.x == 0) {
    if (tid == 0) s_ok = wait_at_least(a.ctl, (unsigned)nblk, a.timeout_ns) ? 1 : 0;
    __syncthreads();
    if (s_ok) {
      uint32_t* bm = reinterpret_cast<uint32_t*>(s_stage + (size_t)a.tpb * a.stage_bytes);
      const int W = (a.T + 31) >> 5;
      uint16_t* pre = reinterpret_cast<uint16_t*>(bm + a.E * W);
      int* s_src = reinterpret_cast<int*>(pre + ((a.E * W + 1) & ~1));
      route_block(a, bm, pre, s_src, s_scan);
      __syncthreads();
      if (tid == 0 && !a.skip_signal) {
        __threadfence();
        atomicAdd(a.ctl, 1u);  // routed
      }
    } else if (tid == 0) {
      flag_error(a.err, MOE_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }

  // ---- 3: every block writes its tokens' k rows once routed
  if (tid == 0) s_ok = wait_at_least(a.ctl, (unsigned)nblk + 1u, a.timeout_ns) ? 1 : 0;
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) flag_error(a.err, MOE_DEVERR_TIMEOUT);
  } else {
    // this block's nt*k destination rows, then every 16-byte chunk of every
    // row from shared memory by all threads (many stores in flight per SM)
    int* s_pos = s_scan + 64;
    for (int q = tid; q < nt * k; q += kDecThreads) {
      const int r = __ldcg(a.pos + (int64_t)t0 * k + q);
      s_pos[q] = (r >= 0 && r < a.T * k) ? r : -1;  // -1: a copy the route map skipped
    }
    __syncthreads();
    const int nq = nt * k * P;
    for (int q = tid; q < nq; q += kDecThreads) {
      const int ij = q / P, c = q - ij * P;
      const int r = s_pos[ij];
      if (r < 0) continue;
      const uint8_t* st = s_stage + (size_t)(ij / k) * a.stage_bytes;
      st_stream_v4(a.out + (int64_t)r * H + c * 16, *reinterpret_cast<const uint4*>(st + c * 16));
    }
    const int ns = nt * k * G;
    for (int q = tid; q < ns; q += kDecThreads) {
      const int ij = q / G, g = q - ij * G;
      const int r = s_pos[ij];
      if (r < 0) continue;
      const float* ssf = reinterpret_cast<const float*>(s_stage + (size_t)(ij / k) * a.stage_bytes + H);
      st_stream_f32(a.out_sf + (int64_t)r * G + g, ssf[g]);
    }
  }
  __syncthreads();
  if (tid == 0) {
    const unsigned done = atomicAdd(a.ctl + 1, 1u);
    if (done == (unsigned)nblk - 1u) {  // last block out: leave the control words zero
      atomicExch(a.ctl, 0u);
      atomicExch(a.ctl + 1, 0u);
    }
  }
}

template <int V, bool VEC, int KMAX>
cudaError_t launch_t(const LaunchCtx& c, const DecodeArgs& a, int blocks, size_t smem) {
  auto kern = decode_fused_kernel<V, VEC, KMAX>;
  cudaError_t e = allow_max_dynamic_smem(kern);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// Shared memory the fused kernel needs beyond its static arrays (at most 39 KB),
// or 0 when the shape is not one it handles (T > 2048, E outside (32, 256],
// k > 32, T*k > 16384, H > 16384, or more than 180 KB).
size_t decode_fused_smem(int64_t T, int E, int k, int H, int num_sms, int* blocks, int* tpb) {
  if (T < 1 || T > 2048 || E <= 32 || E > 256 || k > 32 || T * k > 16384 || H > 16384) return 0;
  const int nb = (int)(T < num_sms ? T : num_sms);
  const int per = (int)((T + nb - 1) / nb);
  const int G = H / kGroup;
  const size_t stage = ((size_t)H + 4 * G + 15) / 16 * 16;
  const int W = (int)((T + 31) / 32);
  // + bm, pre and sorted_src (block 0)
  const size_t smem = (size_t)per * stage + (size_t)E * W * 4 + ((size_t)E * W + 1) / 2 * 4 +
                      (size_t)T * k * 4;
  if (smem > 180 * 1024) return 0;
  if (blocks) *blocks = nb;
  if (tpb) *tpb = per;
  return smem;
}

cudaError_t launch_decode_fused(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                                const void* x, int H, int32_t* idx, float* w, int32_t* counts,
                                int32_t* offsets, int32_t* pos, int32_t* src, uint8_t* out,
                                float* out_sf, unsigned* ctl) {
  int blocks = 0, tpb = 0;
  const size_t smem = decode_fused_smem(T, E, k, H, c.num_sms, &blocks, &tpb);
  if (smem == 0) return cudaErrorInvalidValue;
  const int G = H / kGroup;
  DecodeArgs a;
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
  a.ctl = ctl;
  a.err = c.err;
  a.timeout_ns = g_decode_timeout_ns.load();
  a.T = (int)T;
  a.E = E;
  a.k = k;
  a.H = H;
  a.tpb = tpb;
  a.stage_bytes = (int)(((size_t)H + 4 * G + 15) / 16 * 16);
  a.skip_signal = g_decode_skip_signal.load();
  a.fk = FastDiv((uint32_t)k);
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

}  // namespace moe
