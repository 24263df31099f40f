// expand_cast.cu -- per-token FP8 E4M3 cast fused with the expand to the
// expert-sorted layout.
//
// TileKernels article (itsolotime.com): section 3.2 per_token_cast (absmax
// over each 128-channel group, scale, multiply by the inverse scale, cast) and
// section 2.2 expand_to_fused (copy each token's row and scales to the rows
// pos[t, j], skipping pos < 0).  The page runs them as two kernels; every
// copy of a token casts identically, so here each token is read and cast once
// and its codes are written k times.
//
// Three forms, all with one 128-channel group per aligned 8-lane subgroup
// (lane l holds channels 16l..16l+15, two 16-byte loads; the group amax is a
// 3-step xor shuffle):
//   bulk (H <= 16384, H/128 % 4 == 0, 16-byte aligned out): one CTA per
//     token, the rows leave by TMA bulk copies;
//   row (other H <= 16384): whole tokens per CTA, 16-byte stores;
//   tile (H > 16384): one warp per 4 consecutive (token, group) units.
// HBM traffic is ~80% writes (k copies of 1 byte per channel plus scales,
// against 2 bytes per channel read once).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// One warp's view of a 4-unit tile: its token, group, x slice and the first
// 8 of the token's positions (slot l8 in lane l8 of each subgroup).
struct TileIn {
  uint4 a, b;
  int32_t pos0;
  uint32_t t;
  int g;
  bool active;
};

__device__ __forceinline__ void load_tile(const uint16_t* __restrict__ x,
                                          const int32_t* __restrict__ pos, uint32_t tile, int sub,
                                          int l8, uint32_t units, const FastDiv& fdG, int G, int H,
                                          int k, TileIn& in) {
  const uint32_t u = tile * 4 + sub;
  in.active = u < units;
  in.t = in.active ? fdG.div(u) : 0;
  in.g = in.active ? (int)(u - in.t * G) : 0;
  if (in.active) {
    const uint16_t* src = x + (int64_t)in.t * H + in.g * kGroup + l8 * 16;
    in.a = ld_stream_v4(src);
    in.b = ld_stream_v4(src + 8);
    in.pos0 = (l8 < k) ? __ldg(pos + (int64_t)in.t * k + l8) : -1;
  } else {
    in.a = make_uint4(0, 0, 0, 0);
    in.b = in.a;
    in.pos0 = -1;
  }
}

// G4: G % 4 == 0 (and out_sf 16-byte aligned), so a warp's 4 units are 4
// consecutive groups of one token and their 4 scales form one aligned 16-byte
// vector per destination row.
template <bool G4>
__global__ void __launch_bounds__(kThreads) expand_cast_kernel(
    const uint16_t* __restrict__ x, uint32_t units, int H, int k, const int32_t* __restrict__ pos,
    int64_t R, uint8_t* __restrict__ out, float* __restrict__ out_sf, FastDiv fdG,
    const int32_t* __restrict__ zsrc, SfOut sfo, unsigned* err) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;  // unit within the warp's tile
  const int l8 = lane & 7;    // 16-channel slice within the group
  const int G = H >> 7;
  const uint32_t tiles = (units + 3) >> 2;
  bool bad = false;
  // one tile per warp: the grid covers every tile (launch_g)
  const uint32_t tile = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tile < tiles) {
    TileIn cur;
    load_tile(x, pos, tile, sub, l8, units, fdG, G, H, k, cur);
    const uint4 a = cur.a, b = cur.b;
    const uint32_t t = cur.t;
    const int g = cur.g;
    const bool active = cur.active;
    int32_t mine = cur.pos0;
    const float amax = max8(absmax16_bf16(a, b));
    const float sf = group_scale_opts(amax, sfo.flags);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16_bf16(a, b, inv);
    float4 sf4;
    if (G4) {
      sf4.x = __shfl_sync(0xFFFFFFFFu, sf, 0);
      sf4.y = __shfl_sync(0xFFFFFFFFu, sf, 8);
      sf4.z = __shfl_sync(0xFFFFFFFFu, sf, 16);
      sf4.w = __shfl_sync(0xFFFFFFFFu, sf, 24);
    }
    uint8_t* qdst = out + g * kGroup + l8 * 16;
    float* sdst = out_sf + g;
    if (sfo.stage != nullptr && active && l8 == 0) store_stage(sfo.stage, sfo.flags, G, t, g, sf);
    for (int j0 = 0; j0 < k; j0 += 8) {
      if (j0 > 0)  // slots past the first 8 (k > 8)
        mine = (active && j0 + l8 < k) ? __ldg(pos + (int64_t)t * k + j0 + l8) : -1;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int32_t r = __shfl_sync(0xFFFFFFFFu, mine, (sub << 3) | jj);
        if (j0 + jj >= k || r < 0) continue;  // past k, or a dropped copy
        if (r >= R) {
          bad = true;
          continue;
        }
        st_stream_v4(qdst + (int64_t)r * H, q);
        if (sfo.flags != 0) {  // scale options: one lane per group stores its scale
          if (l8 == 0 && sfo.stage == nullptr) store_sf_opts(out_sf, sfo.flags, sfo.ld, G, r, g, sf);
        } else if (G4) {
          if (lane == 0) st_stream_v4(sdst + (int64_t)r * G, *reinterpret_cast<uint4*>(&sf4));
        } else if (l8 == 0) {
          st_stream_f32(sdst + (int64_t)r * G, sf);
        }
      }
    }
  }
  // warps numbered CTA-major, so consecutive 32-row groups (the all-padding
  // tail is one contiguous run) go to different CTAs instead of a few late ones
  if (zsrc != nullptr)
    zero_fill_rows(zsrc, R, H, H >> 7, out, out_sf,
                   (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x,
                   ((int64_t)gridDim.x * blockDim.x) >> 5, threadIdx.x & 31, sfo);
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

// Row form (H <= 16384): a CTA holds `tpc` whole tokens, H/16 threads per
// token, thread c of a token owning channels 16c..16c+15.  All k destination
// rows of a token are therefore written by one CTA at the same moment, which
// keeps fewer rows open across HBM at once than the tile form: on GB300 a
// scattered-row copy ran ~7% faster this way.
template <bool G4>
__global__ void __launch_bounds__(1024) expand_cast_rows_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int k, const int32_t* __restrict__ pos,
    int64_t R, uint8_t* __restrict__ out, float* __restrict__ out_sf, int tpc,
    const int32_t* __restrict__ zsrc, SfOut sfo, unsigned* err) {
  pdl_enter();
  const int P = H >> 4;  // threads per token
  const int G = H >> 7;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int tl = tid / P;  // token slot within the CTA (== tpc: padding threads)
  const int c = tid - tl * P;
  const int g = c >> 3;
  const int l8 = c & 7;
  const bool slot_ok = tl < tpc;
  const int64_t groups = (T + tpc - 1) / tpc;
  bool bad = false;
  // one token group per CTA: the grid covers every group (launch_rows)
  const int64_t grp = blockIdx.x;
  if (grp < groups) {
    const int64_t t = grp * tpc + tl;
    const bool active = slot_ok && t < T;
    uint4 ca = make_uint4(0, 0, 0, 0), cb = ca;
    int32_t mine = -1;
    if (active) {
      const uint16_t* src = x + t * H + c * 16;
      ca = ld_stream_v4(src);
      cb = ld_stream_v4(src + 8);
      mine = (l8 < k) ? __ldg(pos + t * k + l8) : -1;
    }
    const float amax = max8(absmax16_bf16(ca, cb));
    const float sf = group_scale_opts(amax, sfo.flags);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16_bf16(ca, cb, inv);
    float4 sf4;
    if (G4) {
      sf4.x = __shfl_sync(0xFFFFFFFFu, sf, 0);
      sf4.y = __shfl_sync(0xFFFFFFFFu, sf, 8);
      sf4.z = __shfl_sync(0xFFFFFFFFu, sf, 16);
      sf4.w = __shfl_sync(0xFFFFFFFFu, sf, 24);
    }
    uint8_t* qdst = out + c * 16;
    float* sdst = out_sf + g;
    if (sfo.stage != nullptr && active && l8 == 0) store_stage(sfo.stage, sfo.flags, G, t, g, sf);
    for (int j0 = 0; j0 < k; j0 += 8) {
      if (j0 > 0) mine = (active && j0 + l8 < k) ? __ldg(pos + t * k + j0 + l8) : -1;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int32_t r = __shfl_sync(0xFFFFFFFFu, mine, (lane & ~7) | jj);
        if (!active || j0 + jj >= k || r < 0) continue;
        if (r >= R) {
          bad = true;
          continue;
        }
        st_stream_v4(qdst + (int64_t)r * H, q);
        if (sfo.flags != 0) {  // scale options: one lane per group stores its scale
          if (l8 == 0 && sfo.stage == nullptr) store_sf_opts(out_sf, sfo.flags, sfo.ld, G, r, g, sf);
        } else if (G4) {
          if (lane == 0) st_stream_v4(sdst + (int64_t)r * G, *reinterpret_cast<uint4*>(&sf4));
        } else if (l8 == 0) {
          st_stream_f32(sdst + (int64_t)r * G, sf);
        }
      }
    }
  }
  // warps numbered CTA-major, so consecutive 32-row groups (the all-padding
  // tail is one contiguous run) go to different CTAs instead of a few late ones
  if (zsrc != nullptr)
    zero_fill_rows(zsrc, R, H, H >> 7, out, out_sf,
                   (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x,
                   ((int64_t)gridDim.x * blockDim.x) >> 5, threadIdx.x & 31, sfo);
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

// ---- bulk-store form --------------------------------------------------------
// Same thread layout as the row form (thread c of a token owns channels
// 16c..16c+15), one CTA per TOK consecutive tokens.  Every x load of the CTA's
// tokens is issued first; each token's codes and scales are then assembled in
// its own shared-memory slot and written by k TMA bulk copies (cp.async.bulk,
// shared -> global) issued by one thread, so no warp waits on k store
// instructions per slice.  The CTA retires once the copies have read shared
// memory (cp.async.bulk.wait_group.read).
// Needs G % 4 == 0 and a 16-byte aligned out, and for the bulk copy of
// row-major f32 scales a 16-byte aligned out_sf (bulk copies move multiples
// of 16 bytes between 16-byte aligned addresses); packed UE8M0 row-major
// scales take 8-, 4- or 1-byte stores by the alignment they find.
__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
               "r"(bytes)
               : "memory");
}

// The same copy with an L2 eviction policy.  With column-major or byte scale
// layouts, every scale store writes part of a 32-byte sector, and the sector
// is completed by other tokens' stores later; the token rows read and the code
// rows written are marked evict-first, so that the partly written scale lines
// stay in L2 until complete instead of going to HBM (and coming back) in
// pieces.
__device__ __forceinline__ void bulk_s2g_hint(void* gdst, uint32_t ssrc, uint32_t bytes,
                                              uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(gdst), "r"(ssrc), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// OPTS: scale options (sfo.flags != 0) are compiled in; ZF: the zero-fill of
// the padding rows (zsrc non-null) is.  The plain form (row-major f32 scales,
// copied in bulk with the codes; no padding) compiles neither.
// The chained form's prologue (warp 0, CHAIN): each of the CTA's copies is
// placed at offsets[e] + base[chunk][e] (the copies of expert e in earlier
// chunks) + its rank among its expert's copies in the chunk (held in pos on
// entry); pos and sorted_src are written and lane j of pv[i] gets the row of
// token t0 + i's copy j.
template <int TOK>
__device__ __forceinline__ void chain_place(const RouteChain& rc, int64_t t0, int64_t T, int k,
                                            int64_t R, int32_t* __restrict__ pos, int lane,
                                            int32_t (&pv)[TOK], bool& bad) {
  const int E = rc.E;
  int32_t e[TOK], lr[TOK];
#pragma unroll
  for (int i = 0; i < TOK; ++i) {  // the ids and ranks first: the other loads need the ids
    const int64_t t = t0 + i;
    const bool on = t < T && lane < k;
    e[i] = on ? __ldg(rc.idx + t * k + lane) : -1;
    lr[i] = on ? pos[t * k + lane] : 0;
  }
#pragma unroll
  for (int i = 0; i < TOK; ++i) {
    pv[i] = -1;
    const int64_t t = t0 + i;
    if (t >= T || lane >= k) continue;
    if ((unsigned)e[i] >= (unsigned)E) {  // never from the top-k kernel: flag, skip
      pos[t * k + lane] = -1;
      bad = true;
      continue;
    }
    const int32_t p = __ldg(rc.offsets + e[i]) +
                      __ldg(rc.base + (t >> rc.chunk_shift) * E + e[i]) + lr[i];
    if (p < 0 || (int64_t)p >= R) {
      pos[t * k + lane] = -1;
      bad = true;
      continue;
    }
    pos[t * k + lane] = p;
    rc.sorted_src[p] = (int32_t)(t * k + lane);
    pv[i] = p;
  }
}

// Held to 32 registers (no spills), so that 4 CTAs of 448 threads
// (H = 7168) fit an SM; with more registers only 3 or 2 do, and the bandwidth
// follows the tokens in flight.  Measured on GB300 at T = 65536 (H = 7168,
// k = 8, after an L2 flush) with packed UE8M0 column-major scales (staged,
// with the zero-fill): 0.765 ms at 56 registers and two tokens per CTA (2 CTAs
// per SM), 0.714 ms at 40 (3 CTAs per SM), 0.704 ms at 32 with one token per
// CTA; the padded layout 0.763 -> 0.738 ms between the last two.
template <int TOK, bool OPTS, bool ZF, bool CHAIN>
__global__ void __maxnreg__(32) expand_cast_bulk_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int k, const int32_t* __restrict__ pos,
    int64_t R, uint8_t* __restrict__ out, float* __restrict__ out_sf,
    const int32_t* __restrict__ zsrc, SfOut sfo, RouteChain rc, unsigned* err) {
  extern __shared__ __align__(128) uint8_t s_buf[];
  pdl_enter();
  const int P = H >> 4;  // threads per token
  const int G = H >> 7;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const bool act = tid < P;
  const int g = tid >> 3;
  const int l8 = tid & 7;
  const uint32_t stride = (uint32_t)((H + 4 * G + 127) / 128 * 128);  // bytes per token slot
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(s_buf);
  int32_t* spos_all = reinterpret_cast<int32_t*>(s_buf + (size_t)TOK * stride);  // [TOK][32]
  // the slots and the destination lists fit the launch's shared memory
  if (!MOE_DBG_OK((size_t)TOK * (stride + 128) <= dynamic_smem_bytes() && 16 * P <= (int)stride,
                  err))
    return;  // the same for every thread of the CTA
  bool bad = false;
  const int flags = OPTS ? sfo.flags : 0;
  // Scale layouts: row-major f32 (power-of-two rounded or not) leaves with the
  // codes by bulk copy; row-major UE8M0 bytes are assembled in shared memory
  // and written with wide stores by one warp (sf_wide: 8 or 4 bytes per
  // store, whichever the row length and out_sf's alignment allow); the rest
  // (column-major, direct or staged) is stored per group by one lane.
  const bool sf_bulk =
      !OPTS || ((flags & (MOE_SF_COLMAJOR | MOE_SF_UE8M0)) == 0 && sfo.stage == nullptr);
  const int sf_wide = (OPTS && (flags & MOE_SF_UE8M0) && !(flags & MOE_SF_COLMAJOR))
                          ? ue8m0_store_width(out_sf, G)
                          : 0;
  // only the column-major and byte scale layouts store partial lines
  const bool hint = OPTS && (flags & (MOE_SF_COLMAJOR | MOE_SF_UE8M0)) != 0 && sfo.stage == nullptr;
  const uint64_t policy = l2_evict_first_policy();
  const int64_t t0 = (int64_t)blockIdx.x * TOK;
  // every load of the CTA's tokens is issued before any of them is used
  uint4 a[TOK], b[TOK];
  int32_t pv[TOK];  // warp 0: lane j holds pos[t, j] (j < k <= 32)
#pragma unroll
  for (int i = 0; i < TOK; ++i) {
    const int64_t t = t0 + i;
    a[i] = make_uint4(0, 0, 0, 0);
    b[i] = a[i];
    pv[i] = -1;
    if (t < T) {
      if (act) {
        const uint16_t* src = x + t * H + tid * 16;
        if (hint) {
          a[i] = ld_stream_v4_hint(src, policy);
          b[i] = ld_stream_v4_hint(src + 8, policy);
        } else {
          a[i] = ld_stream_v4(src);
          b[i] = ld_stream_v4(src + 8);
        }
      }
      if (!CHAIN && tid < 32 && lane < k) pv[i] = __ldg(pos + t * k + lane);
    }
  }
  if (CHAIN && tid < 32)  // the x loads above are in flight meanwhile
    chain_place<TOK>(rc, t0, T, k, R, const_cast<int32_t*>(pos), lane, pv, bad);
  float sfv[TOK];
#pragma unroll
  for (int i = 0; i < TOK; ++i) {
    const float amax = max8(absmax16_bf16(a[i], b[i]));
    sfv[i] = group_scale_opts(amax, flags);
    const float inv = __fdiv_rn(1.0f, sfv[i]);
    const uint4 q = quant16_bf16(a[i], b[i], inv);
    uint8_t* sq = s_buf + (size_t)i * stride;
    if (act && t0 + i < T) {
      *reinterpret_cast<uint4*>(sq + tid * 16) = q;
      if (l8 == 0 && sf_bulk) *reinterpret_cast<float*>(sq + H + 4 * g) = sfv[i];
      if (l8 == 0 && sf_wide) sq[H + g] = (uint8_t)((__float_as_uint(sfv[i]) >> 23) & 0xFFu);
    }
    if (!sf_bulk && tid < 32) spos_all[i * 32 + tid] = pv[i];  // for every warp
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the copies
  __syncthreads();
  if (sf_wide) {
    // row-major UE8M0 by one warp (warp 1 where there is one, so that warp 0
    // issues its copies meanwhile)
    if ((tid >> 5) == (blockDim.x >= 64 ? 1 : 0)) {
#pragma unroll
      for (int i = 0; i < TOK; ++i)
        if (t0 + i < T)
          store_ue8m0_rows(reinterpret_cast<uint8_t*>(out_sf), s_buf + (size_t)i * stride + H,
                           spos_all + i * 32, k, G, R, sf_wide, lane, err);
    }
  } else if (!sf_bulk && act && l8 == 0) {  // scale options: per-group scale stores
#pragma unroll
    for (int i = 0; i < TOK; ++i) {
      const int64_t t = t0 + i;
      if (t >= T) continue;
      if (sfo.stage != nullptr) {
        store_stage(sfo.stage, flags, G, t, g, sfv[i]);
      } else {
        for (int j = 0; j < k; ++j) {
          const int32_t r = spos_all[i * 32 + j];
          if (r >= 0 && r < R) store_sf_opts(out_sf, flags, sfo.ld, G, r, g, sfv[i]);
        }
      }
    }
  }
  if (tid < 32) {
#pragma unroll
    for (int i = 0; i < TOK; ++i) {
      if (t0 + i >= T) continue;  // the same for the whole warp
      const uint32_t slot = sbase + (uint32_t)i * stride;
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xFFFFFFFFu, pv[i], j);
        if (tid == 0 && r >= 0) {
          if (r >= R) {
            bad = true;
          } else if (MOE_DBG_OK(bulk_copy_ok(out + (int64_t)r * H, slot, (uint32_t)H, sbase) &&
                                    (!sf_bulk || bulk_copy_ok(out_sf + (int64_t)r * G, slot + H,
                                                              (uint32_t)(4 * G), sbase)),
                                err)) {
            if (hint)
              bulk_s2g_hint(out + (int64_t)r * H, slot, (uint32_t)H, policy);
            else
              bulk_s2g(out + (int64_t)r * H, slot, (uint32_t)H);
            if (sf_bulk) bulk_s2g(out_sf + (int64_t)r * G, slot + H, (uint32_t)(4 * G));
          }
        }
      }
    }
    if (tid == 0) {
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // shared memory must stay valid until the copies have read it; their
      // global writes complete on their own after the CTA exits
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
  }
  // warps numbered CTA-major, so consecutive 32-row groups (the all-padding
  // tail is one contiguous run) go to different CTAs instead of a few late ones
  if (ZF && zsrc != nullptr)
    zero_fill_rows(zsrc, R, H, H >> 7, out, out_sf,
                   (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x,
                   ((int64_t)gridDim.x * blockDim.x) >> 5, threadIdx.x & 31, sfo);
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

// Tokens per CTA of the bulk form.  The grid is not persistent: one CTA per
// TOK consecutive tokens, retiring when its copies have read shared memory.
// Measured on GB300 (H = 7168, k = 8, after an L2 flush): 0.705 ms (1.01 of
// the measured copy peak) at T = 65536 and 94.8 us (0.94) at T = 8192, against
// 0.80 ms and 104 us for a persistent grid of 3 CTAs per SM that strode over
// the tokens with the next token's loads in flight.  The persistent grid kept
// the accesses in flight at any moment spread over the whole of x and q; here
// the CTAs in flight at once cover a compact run of consecutive tokens.  One
// token per CTA, at 32 registers, suits every form (with two, the option and
// zero-fill forms need more registers: see the kernel).
constexpr int kBulkTokensPerCta = 1;

template <int TOK, bool OPTS, bool ZF, bool CHAIN = false>
cudaError_t launch_bulk_t(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                        const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                        const int32_t* zsrc, SfOut sfo, const RouteChain& rc = RouteChain()) {
  const int P = H / 16;
  const int threads = (P + 31) / 32 * 32;
  const int G = H / kGroup;
  const size_t stride = (size_t)(H + 4 * G + 127) / 128 * 128;
  const size_t smem = (stride + 128) * TOK;  // per token: its slot and its 32 destinations
  const auto kern = expand_cast_bulk_kernel<TOK, OPTS, ZF, CHAIN>;
  if (smem > 48 * 1024) {
    cudaError_t st = allow_max_dynamic_smem(kern);
    if (st != cudaSuccess) return st;
  }
  int64_t blocks = (T + TOK - 1) / TOK;
  if (zsrc != nullptr) {  // enough warps for one 32-row group of the zero-fill each
    const int64_t zb = ((R + 31) / 32 + threads / 32 - 1) / (threads / 32);
    blocks = blocks > zb ? blocks : zb;
  }
  if (blocks < 1) blocks = 1;
  return launch_pdl(kern, (unsigned)blocks, threads, smem, c.stream,
                    static_cast<const uint16_t*>(x), T, H, k, pos, R, out, out_sf, zsrc, sfo, rc,
                    c.err);
}

cudaError_t launch_bulk(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                        const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                        const int32_t* zsrc, SfOut sfo) {
  constexpr int TK = kBulkTokensPerCta;
  if (sfo.flags != 0)
    return zsrc != nullptr
               ? launch_bulk_t<TK, true, true>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo)
               : launch_bulk_t<TK, true, false>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo);
  return zsrc != nullptr
             ? launch_bulk_t<TK, false, true>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo)
             : launch_bulk_t<TK, false, false>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo);
}

}  // namespace

cudaError_t launch_expand_cast_chain(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                                     int32_t* pos, uint8_t* out, float* out_sf,
                                     const RouteChain& rc) {
  return launch_bulk_t<kBulkTokensPerCta, false, false, true>(c, x, T, H, k, pos, T * k, out,
                                                              out_sf, nullptr, SfOut(), rc);
}

namespace {

// The fallback forms' grids cover all their work (one CTA per token group, one
// warp per tile) instead of a persistent grid of the resident CTAs striding
// over it, as the bulk form's: measured on GB300 (k = 8, after an L2 flush)
// the row form at H = 7296 (G = 57) ran at 0.84 of the measured copy peak
// against 0.73, at H = 640 at 0.63 against 0.42, and the tile form at
// H = 20480 at 0.96 against 0.82.  Each CTA or warp takes exactly its own
// group or tile (no loop, no prefetch of a next one), so the grid must cover
// them all; against the same grid with striding loops that prefetched the
// next item: row form 221.9 -> 215.7 us at T = 16384, H = 7296 and 86.7 ->
// 84.6 us at T = 65536, H = 640; tile form 269.0 -> 264.9 us at T = 8192,
// H = 20480 (output unchanged).
template <bool G4>
cudaError_t launch_rows(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                        const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                        const int32_t* zsrc, SfOut sfo) {
  const int P = H / 16;
  const int tpc = P >= 256 ? 1 : 256 / P;
  const int64_t groups = (T + tpc - 1) / tpc;
  const int blocks = (int)(groups > 0 ? groups : 1);  // >= 1: zero-fill
  const int threads = (P * tpc + 31) / 32 * 32;  // whole warps: the shuffles use full masks
  return launch_pdl(expand_cast_rows_kernel<G4>, blocks, threads, 0, c.stream,
                    static_cast<const uint16_t*>(x), T, H, k, pos, R, out, out_sf, tpc, zsrc, sfo,
                    c.err);
}

template <bool G4>
cudaError_t launch_g(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                     const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                     const int32_t* zsrc, SfOut sfo) {
  const int G = H / kGroup;
  const uint32_t units = (uint32_t)(T * G);  // < 2^31, checked by the caller
  const uint32_t tiles = (units + 3) / 4;
  const int64_t need = ((int64_t)tiles + (kThreads / 32) - 1) / (kThreads / 32);
  const int blocks = (int)(need > 0 ? need : 1);  // >= 1: zero-fill with T = 0
  return launch_pdl(expand_cast_kernel<G4>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, H, k, pos, R, out, out_sf,
                    FastDiv((uint32_t)G), zsrc, sfo, c.err);
}

// Column-major scales from the staged per-token rows: thread r writes row r
// of every column (f32 [G][ld], or packed UE8M0 words [ceil(G/4)][ld]) from
// the staged row of token sorted_src[r] / k (sorted_src holds copy indices
// t*k + j), or zeros where sorted_src[r] < 0 (padding rows, as the zero-fill
// writes them).  Consecutive threads write consecutive
// rows of a column, so each warp store is one whole 128-byte line; the staged
// rows are read back from L2 (T * G * 4 bytes at most, just written).
__global__ void __launch_bounds__(256) sf_gather_kernel(const uint8_t* __restrict__ stage,
                                                        const int32_t* __restrict__ src, int64_t R,
                                                        int64_t T, int k, int G, SfOut sfo,
                                                        void* __restrict__ out_sf, unsigned* err) {
  pdl_enter();
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int32_t s = __ldg(src + r);
  int64_t t = s < 0 ? -1 : s / k;
  if (t >= T) {
    flag_error(err, MOE_DEVERR_POS_RANGE);
    t = -1;  // unknown copy: zeros, never a read outside the staged rows
  }
  const int64_t tr = t >= 0 ? t : 0;  // row read only when t >= 0
  const int64_t ld = sfo.ld;
  if (sfo.flags & MOE_SF_UE8M0) {
    const int W = (G + 3) >> 2;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(stage) + tr * W;
    uint32_t* o = static_cast<uint32_t*>(out_sf) + r;
    const int full = G >> 2;  // words with 4 groups; a last partial word keeps its unused bytes
    for (int w = 0; w < full; ++w) o[w * ld] = t >= 0 ? row[w] : 0u;
    if (full < W) {
      const uint32_t v = t >= 0 ? row[full] : 0u;
      uint8_t* ob = reinterpret_cast<uint8_t*>(o + full * ld);
      for (int b = 0; b < (G & 3); ++b) ob[b] = (uint8_t)(v >> (8 * b));
    }
  } else {
    const float* row = reinterpret_cast<const float*>(stage) + tr * G;
    float* o = static_cast<float*>(out_sf) + r;
    int g = 0;
    if ((G & 3) == 0) {
      for (; g < G; g += 4) {
        const float4 v = t >= 0 ? *reinterpret_cast<const float4*>(row + g)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        o[(g + 0) * ld] = v.x;
        o[(g + 1) * ld] = v.y;
        o[(g + 2) * ld] = v.z;
        o[(g + 3) * ld] = v.w;
      }
    }
    for (; g < G; ++g) o[g * ld] = t >= 0 ? row[g] : 0.0f;
  }
}


cudaError_t launch_expand_cast_kernel(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                                      const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                                      const int32_t* zero_rows, SfOut sfo) {
  // the 16-byte scale store needs G % 4 == 0 and a 16-byte aligned out_sf
  const bool g4 = (H / kGroup) % 4 == 0 && (reinterpret_cast<uintptr_t>(out_sf) % 16) == 0;
  const bool aligned16 = (reinterpret_cast<uintptr_t>(out) % 16) == 0;
  // row-major f32 scales (flags 0 or power-of-two alone) leave by bulk copy
  const bool bulk_ok = (sfo.flags & (MOE_SF_COLMAJOR | MOE_SF_UE8M0)) != 0 || g4;
  if (H <= 16384 && bulk_ok && (H / kGroup) % 4 == 0 && aligned16)
    return launch_bulk(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo);
  if (H <= 16384)
    return g4 ? launch_rows<true>(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo)
              : launch_rows<false>(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo);
  return g4 ? launch_g<true>(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo)
            : launch_g<false>(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo);
}

}  // namespace

cudaError_t launch_sf_gather(const LaunchCtx& c, const int32_t* src, int64_t R, int64_t T, int k,
                             int G, SfOut sfo, void* out_sf) {
  if (R == 0) return cudaSuccess;
  const int64_t blocks = (R + 255) / 256;
  return launch_pdl(sf_gather_kernel, (int)blocks, 256, 0, c.stream,
                    static_cast<const uint8_t*>(sfo.stage), src, R, T, k, G, sfo, out_sf, c.err);
}

cudaError_t launch_expand_cast(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                               const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                               const int32_t* zero_rows, SfOut sfo) {
  cudaError_t e = launch_expand_cast_kernel(c, x, T, H, k, pos, R, out, out_sf, zero_rows, sfo);
  if (e != cudaSuccess || sfo.stage == nullptr) return e;
  return launch_sf_gather(c, zero_rows, R, T, k, H / kGroup, sfo, out_sf);
}

}  // namespace moe
