// swiglu_cast.cu -- SwiGLU fused with the per-group FP8 E4M3 cast.
//
// TileKernels article (itsolotime.com), section 3.3: in f32,
// val_l / (1 + exp(-val_l)) * val_r with val_l from the left (gate) half and
// val_r from the right (up) half of each row, then per-group absmax -> scale
// -> cast in the same kernel.  The section's variants (the clamp, the top-k
// weight, the clamp count) and the scale options are instances of the same
// kernels, one per option set (kOptW ... kOptK); the FP4 E2M1 output shares
// the loop (swiglu_cast_fp4_kernel).
//
// Work unit: one (row, 128-channel group) per aligned 8-lane subgroup; each
// lane reads 16 gate and 16 up values (four 16-byte loads) and writes one
// 16-byte code vector.  HBM traffic is ~80% reads.  Each warp takes one tile
// of 4 consecutive units, and the grid covers every tile (see kGridNote).  At
// ~1 GB per 0.15 ms the kernel
// must spend under ~12 instructions per element to stay memory-bound, which is
// why the activation uses the hardware exp2 and reciprocal.
#include <type_traits>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// The variants' options, fixed at compile time so that each instance carries
// only the code its options need: per-row weights (W), clamp (C), clamp count
// (K, only with C: without a clamp nothing is counted), and a scale option (S:
// POW2, UE8M0 or column-major).  OPT = 0 is the plain form of the page.
constexpr int kOptW = 1;
constexpr int kOptC = 2;
constexpr int kOptS = 4;
constexpr int kOptK = 8;

// Bit OPT set: that instance's grid is persistent (see kGridNote).
constexpr uint32_t kPersistentOpts = 0xCC00u;
__host__ __device__ constexpr bool ext_persistent(int opt) {
  return ((kPersistentOpts >> opt) & 1u) != 0;
}

// kGridNote: the grid is not persistent, except for the instances that count
// clamped values (K).  One warp per tile of units, so the CTAs in flight at
// any moment cover a compact run of consecutive rows.  Measured on GB300
// (65536 rows of 2 x 2048, after an L2 flush / back to back): E4M3 0.929 /
// 0.968 of the measured copy peak against 0.895 / 0.941 for a persistent grid
// of the resident CTAs striding over the tiles; E2M1 (group 32) 0.906 / 0.936
// against 0.870 / 0.898.  Writing the loop so that the compiler sees at most
// one tile per warp (its bound min(tiles, first + 1) instead of a stride)
// then gave, in one A/B: E4M3 0.929 -> 0.947 and 0.965 -> 0.992, E2M1 0.888
// -> 0.906 and 0.937 -> 0.957 (at 524288 rows E4M3 0.984 -> 1.006 single),
// output unchanged.  The K instances add one atomic per warp, which the
// persistent grid takes once per resident warp instead of once per tile:
// clamp and count 0.879 / 0.919 persistent against 0.848 / 0.882.  One
// instance per option set (W, C, K, S) against one instance for all options
// (48 registers, persistent), E4M3 single / back to back: weights 0.863 /
// 0.910 -> 0.929 / 0.985; scale options 0.859 / 0.912 -> 0.943 / 0.990;
// clamp 0.848 / 0.894 -> 0.895 / 0.940; clamp, weights, count and packed
// UE8M0 column-major scales 0.816 / 0.847 -> 0.830 / 0.863 (E2M1, group 32:
// weights 0.823 -> 0.888, clamp 0.808 -> 0.838, all four 0.751 -> 0.764),
// output unchanged.  The loops stride when persistent, so any grid size is
// correct for those instances.

__device__ __forceinline__ float swiglu(float g, float u) {
  // evaluated in the order written on the page, in f32, with the hardware
  // exp2 and reciprocal (__expf, __fdividef): a few ulps from the correctly
  // rounded value, which moves an E4M3 code only when v / sf lies within those
  // ulps of a rounding midpoint (about 1e-5 of elements).  For g < -88,
  // exp(-g) is +inf and g / inf gives a signed zero, as the IEEE division does.
  const float e = __expf(-g);
  return __fdividef(g, 1.0f + e) * u;
}

// min / max that return NaN when either operand is NaN (PTX min.NaN / max.NaN).
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Element i of 16 packed bf16 (two 16-byte words), as f32.
__device__ __forceinline__ float bf16_at(const uint4& a, const uint4& b, int i) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  return (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
}

// The clamp of the TileKernels article, section 3.3: gate min(g, c), up
// clamped to [-c, c].  NaN stays NaN, as min and max written as compares.
__device__ __forceinline__ void clamp_pair(float& g, float& u, float c) {
  g = min_nan(g, c);
  u = max_nan(min_nan(u, c), -c);
}

// The SwiGLU values from the packed words, optionally clamped and counted.
template <bool CLAMP, bool COUNT>
__device__ __forceinline__ void swiglu16(const uint4& ga, const uint4& gb, const uint4& ua,
                                         const uint4& ub, float c, unsigned& clamped,
                                         float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float g = bf16_at(ga, gb, i), u = bf16_at(ua, ub, i);
    if (COUNT) clamped += (g > c) + (fabsf(u) > c);
    if (CLAMP) clamp_pair(g, u, c);
    v[i] = swiglu(g, u);
  }
}

// The lane's 16 SwiGLU values of one (row, channel slice): the loaded gate and
// up words, the variants of the TileKernels article, section 3.3 (the
// clamp; the per-row top-k weight multiplied after silu(g) * u; clamp
// counting into `clamped`), then the activation.  Each path unpacks the words
// as it goes, so no unpacked copy of them stays live across a branch.  Every
// lane of the warp must call it (the count's fast-path vote).
template <int OPT>
__device__ __forceinline__ void lane_values(const uint4& ga, const uint4& gb, const uint4& ua,
                                            const uint4& ub, bool active, float wr,
                                            const SwigluExt& ext, unsigned& clamped,
                                            float (&v)[16]) {
  const float c = ext.clamp;
  if (OPT & kOptK) {
    // Fast path: nothing is clamped or counted unless some gate value or |up|
    // value of the warp exceeds c (max over 16 values: two min/max per
    // element, against seven for clamping and counting them all).
    float mg = bf16_at(ga, gb, 0), mu = fabsf(bf16_at(ua, ub, 0));
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      mg = fmaxf(mg, bf16_at(ga, gb, i));
      mu = fmaxf(mu, fabsf(bf16_at(ua, ub, i)));
    }
    if (__any_sync(0xFFFFFFFFu, active && (mg > c || mu > c))) {
      unsigned n = 0;
      swiglu16<true, true>(ga, gb, ua, ub, c, n, v);
      if (active) clamped += n;
    } else {
      swiglu16<false, false>(ga, gb, ua, ub, c, clamped, v);
    }
  } else if (OPT & kOptC) {
    // without a count, clamping every element costs less than the vote
    swiglu16<true, false>(ga, gb, ua, ub, c, clamped, v);
  } else {
    swiglu16<false, false>(ga, gb, ua, ub, c, clamped, v);
  }
  if (OPT & kOptW) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], wr);
  }
}

// One atomic per warp adds the warp's clamp count.
__device__ __forceinline__ void add_clamp_count(const SwigluExt& ext, unsigned clamped, int lane) {
  const unsigned total = __reduce_add_sync(0xFFFFFFFFu, clamped);
  if (lane == 0 && total) atomicAdd(ext.clamp_count, (unsigned long long)total);
}

// E4M3 output, with the options OPT (0: none of the variants).  The clamp
// count is kept per thread over its tiles and added once per warp.  The
// register caps keep 5 (count) or 6 CTAs of 256 threads resident per SM
// without spills (the count's instances spill at 6): each warp is
// latency-bound, so resident warps set the bandwidth.
template <int OPT>
__global__ void __launch_bounds__(kThreads, (OPT & kOptK) ? 5 : 6)
    swiglu_cast_kernel(const uint16_t* __restrict__ x, uint32_t units, int N,
                       uint8_t* __restrict__ out, float* __restrict__ out_sf, FastDiv fdG,
                       SwigluExt ext) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;
  const int l8 = lane & 7;
  const int G = N >> 7;
  const uint32_t tiles = (units + 3) >> 2;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  unsigned clamped = 0;
  // the grid covers every tile (each warp its own), or, persistent, strides
  // over them (see kGridNote)
  const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  constexpr bool strided = ext_persistent(OPT);
  const uint32_t t_step = strided ? warps : 1u;
  const uint32_t t_end = strided ? tiles : min(tiles, gw + 1);
  for (uint32_t tile = gw; tile < t_end; tile += t_step) {
    const uint32_t u = tile * 4 + sub;
    const bool active = u < units;
    const uint32_t r = active ? fdG.div(u) : 0;
    const int g = active ? (int)(u - r * G) : 0;
    const uint16_t* gate = x + (int64_t)r * 2 * N + g * kGroup + l8 * 16;
    const uint16_t* up = gate + N;
    uint4 ga = make_uint4(0, 0, 0, 0), gb = ga, ua = ga, ub = ga;
    float wr = 0.0f;
    if (active) {
      ga = ld_stream_v4(gate);
      gb = ld_stream_v4(gate + 8);
      ua = ld_stream_v4(up);
      ub = ld_stream_v4(up + 8);
      // issued with the row loads so that its latency overlaps theirs
      if (OPT & kOptW) wr = __ldg(ext.weights + r);
    }
    float v[16];
    lane_values<OPT>(ga, gb, ua, ub, active, wr, ext, clamped, v);
    const float amax = max8(absmax16(v));
    const float sf = (OPT & kOptS) ? group_scale_opts(amax, ext.sf.flags) : group_scale(amax);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16(v, inv);
    if (active) {
      st_stream_v4(out + (int64_t)r * N + g * kGroup + l8 * 16, q);
      if (l8 == 0) {
        if (OPT & kOptS)
          store_sf_opts(out_sf, ext.sf.flags, ext.sf.ld, G, r, g, sf);
        else
          st_stream_f32(out_sf + (int64_t)r * G + g, sf);
      }
    }
  }
  if (OPT & kOptK) add_clamp_count(ext, clamped, lane);
}

// FP4 E2M1 output (TileKernels article, 3.1's float4_e2m1fn: max 6,
// clamp_min 6 * 2^-126): groups of 16 L channels, L lanes per group, 32 / L
// groups per warp tile; 8 bytes of packed codes per lane.  Options, grid and
// register caps as the E4M3 kernel's.
template <int L, int OPT>
__global__ void __launch_bounds__(kThreads, (OPT & kOptK) ? 5 : 6)
    swiglu_cast_fp4_kernel(const uint16_t* __restrict__ x, uint32_t units, int N,
                           uint8_t* __restrict__ out, float* __restrict__ out_sf, FastDiv fdG,
                           SwigluExt ext) {
  pdl_enter();
  constexpr int U = 32 / L;  // groups per warp tile
  const int lane = threadIdx.x & 31;
  const int sub = lane / L;
  const int lg = lane % L;
  const int G = N / (16 * L);
  const uint32_t tiles = (units + U - 1) / U;
  const uint32_t warps = (gridDim.x * blockDim.x) >> 5;
  unsigned clamped = 0;
  const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  constexpr bool strided = ext_persistent(OPT);
  const uint32_t t_step = strided ? warps : 1u;
  const uint32_t t_end = strided ? tiles : min(tiles, gw + 1);
  for (uint32_t tile = gw; tile < t_end; tile += t_step) {
    const uint32_t u = tile * U + sub;
    const bool active = u < units;
    const uint32_t r = active ? fdG.div(u) : 0;
    const int g = active ? (int)(u - r * G) : 0;
    const uint16_t* gate = x + (int64_t)r * 2 * N + g * 16 * L + lg * 16;
    const uint16_t* up = gate + N;
    uint4 ga = make_uint4(0, 0, 0, 0), gb = ga, ua = ga, ub = ga;
    float wr = 0.0f;
    if (active) {
      ga = ld_stream_v4(gate);
      gb = ld_stream_v4(gate + 8);
      ua = ld_stream_v4(up);
      ub = ld_stream_v4(up + 8);
      if (OPT & kOptW) wr = __ldg(ext.weights + r);
    }
    float v[16];
    lane_values<OPT>(ga, gb, ua, ub, active, wr, ext, clamped, v);
    const float amax = maxL<L>(absmax16(v));
    const float sf = fp4_scale(amax, (OPT & kOptS) ? ext.sf.flags : 0);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint2 q = quant16_e2m1(v, inv);
    if (active) {
      st_stream_v2(out + (int64_t)r * (N >> 1) + g * 8 * L + lg * 8, q);
      if (lg == 0) {
        if (OPT & kOptS)
          store_sf_opts(out_sf, ext.sf.flags, ext.sf.ld, G, r, g, sf);
        else
          st_stream_f32(out_sf + (int64_t)r * G + g, sf);
      }
    }
  }
  if (OPT & kOptK) add_clamp_count(ext, clamped, lane);
}

// The option mask of a variant call: W, C, K and S as its arguments ask.
int opt_mask(const SwigluExt& ext) {
  const bool clamp = ext.has_clamp != 0;
  return (ext.weights != nullptr ? kOptW : 0) | (clamp ? kOptC : 0) |
         (clamp && ext.clamp_count != nullptr ? kOptK : 0) | (ext.sf.flags != 0 ? kOptS : 0);
}

// Calls launch<OPT>() for the instance of `opt`: OPT is one of the twelve
// masks opt_mask() gives (K only with C).
template <typename F>
cudaError_t dispatch_opt(int opt, F&& launch) {
  switch (opt) {
    case 0: return launch(std::integral_constant<int, 0>());
    case 1: return launch(std::integral_constant<int, 1>());
    case 2: return launch(std::integral_constant<int, 2>());
    case 3: return launch(std::integral_constant<int, 3>());
    case 4: return launch(std::integral_constant<int, 4>());
    case 5: return launch(std::integral_constant<int, 5>());
    case 6: return launch(std::integral_constant<int, 6>());
    case 7: return launch(std::integral_constant<int, 7>());
    case 10: return launch(std::integral_constant<int, 10>());
    case 11: return launch(std::integral_constant<int, 11>());
    case 14: return launch(std::integral_constant<int, 14>());
    case 15: return launch(std::integral_constant<int, 15>());
    default: return cudaErrorInvalidValue;
  }
}

// Blocks for `tiles` warp tiles: one warp each, or, for a persistent
// instance, at most the resident blocks of `kernel`.
template <typename K>
cudaError_t grid_for(const LaunchCtx& c, K kernel, bool persistent, uint32_t tiles, int* blocks) {
  const int64_t need = ((int64_t)tiles + (kThreads / 32) - 1) / (kThreads / 32);
  int64_t cap = need;
  if (persistent) {
    int per_sm = 0;
    cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (st != cudaSuccess) return st;
    cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  }
  *blocks = (int)(need < cap ? (need > 0 ? need : 1) : cap);
  return cudaSuccess;
}

template <int OPT>
cudaError_t launch_t(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                     float* out_sf, const SwigluExt& ext) {
  const int G = N / kGroup;
  const uint32_t units = (uint32_t)(M * G);  // < 2^31, checked by the caller
  int blocks = 0;
  cudaError_t st = grid_for(c, swiglu_cast_kernel<OPT>, ext_persistent(OPT), (units + 3) / 4,
                            &blocks);
  if (st != cudaSuccess) return st;
  return launch_pdl(swiglu_cast_kernel<OPT>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, N, out, out_sf, FastDiv((uint32_t)G),
                    ext);
}

template <int L, int OPT>
cudaError_t launch_fp4_t(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                         float* out_sf, const SwigluExt& ext) {
  constexpr int U = 32 / L;
  const int G = N / (16 * L);
  const uint32_t units = (uint32_t)(M * G);  // < 2^31, checked by the caller
  int blocks = 0;
  cudaError_t st = grid_for(c, swiglu_cast_fp4_kernel<L, OPT>, ext_persistent(OPT),
                            (units + U - 1) / U, &blocks);
  if (st != cudaSuccess) return st;
  return launch_pdl(swiglu_cast_fp4_kernel<L, OPT>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, N, out, out_sf, FastDiv((uint32_t)G),
                    ext);
}

template <int L>
cudaError_t launch_fp4(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                       float* out_sf, const SwigluExt& ext) {
  return dispatch_opt(opt_mask(ext), [&](auto opt) {
    return launch_fp4_t<L, decltype(opt)::value>(c, x, M, N, out, out_sf, ext);
  });
}

}  // namespace

cudaError_t launch_swiglu_cast_fp4(const LaunchCtx& c, const void* x, int64_t M, int N,
                                   uint8_t* out, void* out_sf, const SwigluExt& ext, int group) {
  float* sf = static_cast<float*>(out_sf);
  switch (group) {
    case 16: return launch_fp4<1>(c, x, M, N, out, sf, ext);
    case 32: return launch_fp4<2>(c, x, M, N, out, sf, ext);
    case 64: return launch_fp4<4>(c, x, M, N, out, sf, ext);
    case 128: return launch_fp4<8>(c, x, M, N, out, sf, ext);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_swiglu_cast(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                               float* out_sf) {
  return launch_t<0>(c, x, M, N, out, out_sf, SwigluExt());
}

cudaError_t launch_swiglu_cast_ex(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                                  void* out_sf, const SwigluExt& ext) {
  float* sf = static_cast<float*>(out_sf);
  return dispatch_opt(opt_mask(ext), [&](auto opt) {
    return launch_t<decltype(opt)::value>(c, x, M, N, out, sf, ext);
  });
}

}  // namespace moe
