// swiglu_cast.cu -- SwiGLU fused with the per-group FP8 E4M3 cast.
//
// TileKernels article (itsolotime.com), section 3.3: in f32,
// val_l / (1 + exp(-val_l)) * val_r with val_l from the left (gate) half and
// val_r from the right (up) half of each row, then per-group absmax -> scale
// -> cast in the same kernel (plain form: no clamp, no top-k weight).
//
// Work unit: one (row, 128-channel group) per aligned 8-lane subgroup; each
// lane reads 16 gate and 16 up values (four 16-byte loads) and writes one
// 16-byte code vector.  HBM traffic is ~80% reads.  Each warp takes one tile
// of 4 consecutive units, and the grid covers every tile (see kGridNote).  At
// ~1 GB per 0.15 ms the kernel
// must spend under ~12 instructions per element to stay memory-bound, which is
// why the activation uses the hardware exp2 and reciprocal.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr bool kExtPersistent = true;  // the variants' grid (see kGridNote)

// kGridNote: the plain forms' grid is not persistent.  One warp per tile of
// units, so the CTAs in flight at any moment cover a compact run of
// consecutive rows.  Measured on GB300 (65536 rows of 2 x 2048, after an L2
// flush / back to back): E4M3 0.929 / 0.968 of the measured copy peak against
// 0.895 / 0.941 for a persistent grid of the resident CTAs striding over the
// tiles; E2M1 (group 32) 0.906 / 0.936 against 0.870 / 0.898.  Writing the
// loop so that the compiler sees at most one tile per warp (its bound
// min(tiles, first + 1) instead of a stride) then gave, in one A/B: E4M3
// 0.929 -> 0.947 and 0.965 -> 0.992, E2M1 0.888 -> 0.906 and 0.937 -> 0.957
// (at 524288 rows E4M3 0.984 -> 1.006 single), output unchanged.  The variants (EXT) measured the other way round and keep the
// persistent grid (kExtPersistent): with per-row weights 0.86 / 0.90
// persistent against 0.82 / 0.85; with clamp, weights, count and packed UE8M0
// column-major scales 0.80 / 0.84 against 0.79 / 0.82 (E2M1 with clamp,
// weights and count 0.78 / 0.82 against 0.74 / 0.77).  The loops stride when
// persistent, so any grid size is correct for the variants.

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

// The lane's 16 SwiGLU values of one (row, channel slice): the loaded gate and
// up words, the EXT variants of the TileKernels article, section 3.3 (clamp:
// gate min(g, c), up clamped to [-c, c]; the per-row top-k weight multiplied
// after silu(g) * u; clamp counting into `clamped`), then the activation.
// Every lane of the warp must call it (the clamp's fast-path vote).
template <bool EXT>
__device__ __forceinline__ void lane_values(const uint4& ga, const uint4& gb, const uint4& ua,
                                            const uint4& ub, bool active, float wr,
                                            const SwigluExt& ext, unsigned& clamped,
                                            float (&v)[16]) {
  float gv[16], uv[16];
  unpack16(ga, gb, gv);
  unpack16(ua, ub, uv);
  if (EXT && ext.has_clamp) {
    // Fast path: the clamp changes nothing unless some gate value or |up|
    // value of the warp exceeds c (max over 16 values: two min/max per
    // element, against seven for clamping and counting them all).
    const float c = ext.clamp;
    float mg = gv[0], mu = fabsf(uv[0]);
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      mg = fmaxf(mg, gv[i]);
      mu = fmaxf(mu, fabsf(uv[i]));
    }
    if (__any_sync(0xFFFFFFFFu, active && (mg > c || mu > c))) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (active) clamped += (gv[i] > c) + (fabsf(uv[i]) > c);
        gv[i] = min_nan(gv[i], c);  // NaN stays NaN, as min written as a compare
        uv[i] = max_nan(min_nan(uv[i], c), -c);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = swiglu(gv[i], uv[i]);
  if (EXT && ext.weights != nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], wr);
  }
}

// One atomic per warp adds the warp's clamp count.
__device__ __forceinline__ void add_clamp_count(const SwigluExt& ext, unsigned clamped, int lane) {
  if (ext.clamp_count != nullptr) {
    const unsigned total = __reduce_add_sync(0xFFFFFFFFu, clamped);
    if (lane == 0 && total) atomicAdd(ext.clamp_count, (unsigned long long)total);
  }
}

// E4M3 output.  EXT = false compiles none of the variants.  The clamp count
// is kept per thread over its tiles and added once per warp.  The register
// caps keep 5 (EXT) or 6 CTAs of 256 threads resident per SM without spills:
// each warp is latency-bound, so resident warps set the bandwidth.
template <bool EXT>
__global__ void __launch_bounds__(kThreads, EXT ? 5 : 6)
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
  const bool strided = EXT && kExtPersistent;
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
      if (EXT && ext.weights != nullptr) wr = __ldg(ext.weights + r);
    }
    float v[16];
    lane_values<EXT>(ga, gb, ua, ub, active, wr, ext, clamped, v);
    const float amax = max8(absmax16(v));
    const float sf = EXT ? group_scale_opts(amax, ext.sf.flags) : group_scale(amax);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint4 q = quant16(v, inv);
    if (active) {
      st_stream_v4(out + (int64_t)r * N + g * kGroup + l8 * 16, q);
      if (l8 == 0) {
        if (EXT && ext.sf.flags != 0)
          store_sf_opts(out_sf, ext.sf.flags, ext.sf.ld, G, r, g, sf);
        else
          st_stream_f32(out_sf + (int64_t)r * G + g, sf);
      }
    }
  }
  if (EXT) add_clamp_count(ext, clamped, lane);
}

// FP4 E2M1 output (TileKernels article, 3.1's float4_e2m1fn: max 6,
// clamp_min 6 * 2^-126): groups of 16 L channels, L lanes per group, 32 / L
// groups per warp tile; 8 bytes of packed codes per lane.  EXT = false (no
// clamp, weight, count or scale option) compiles none of the variants and
// keeps 6 CTAs resident, as the E4M3 plain form.
template <int L, bool EXT>
__global__ void __launch_bounds__(kThreads, EXT ? 5 : 6)
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
  const bool strided = EXT && kExtPersistent;
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
      if (EXT && ext.weights != nullptr) wr = __ldg(ext.weights + r);
    }
    float v[16];
    lane_values<EXT>(ga, gb, ua, ub, active, wr, ext, clamped, v);
    const float amax = maxL<L>(absmax16(v));
    const float sf = fp4_scale(amax, EXT ? ext.sf.flags : 0);
    const float inv = __fdiv_rn(1.0f, sf);
    const uint2 q = quant16_e2m1(v, inv);
    if (active) {
      st_stream_v2(out + (int64_t)r * (N >> 1) + g * 8 * L + lg * 8, q);
      if (lg == 0) {
        if (EXT && ext.sf.flags != 0)
          store_sf_opts(out_sf, ext.sf.flags, ext.sf.ld, G, r, g, sf);
        else
          st_stream_f32(out_sf + (int64_t)r * G + g, sf);
      }
    }
  }
  if (EXT) add_clamp_count(ext, clamped, lane);
}

template <bool EXT>
cudaError_t launch_t(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                     float* out_sf, const SwigluExt& ext) {
  const int G = N / kGroup;
  const uint32_t units = (uint32_t)(M * G);  // < 2^31, checked by the caller
  const uint32_t tiles = (units + 3) / 4;
  const int64_t need = ((int64_t)tiles + (kThreads / 32) - 1) / (kThreads / 32);
  int64_t cap = need;
  if (EXT && kExtPersistent) {  // see kGridNote
    int per_sm = 0;
    cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, swiglu_cast_kernel<EXT>, kThreads, 0);
    if (st != cudaSuccess) return st;
    cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  }
  const int blocks = (int)(need < cap ? (need > 0 ? need : 1) : cap);
  return launch_pdl(swiglu_cast_kernel<EXT>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, N, out, out_sf, FastDiv((uint32_t)G),
                    ext);
}

template <int L, bool EXT>
cudaError_t launch_fp4_t(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                         float* out_sf, const SwigluExt& ext) {
  constexpr int U = 32 / L;
  const int G = N / (16 * L);
  const uint32_t units = (uint32_t)(M * G);  // < 2^31, checked by the caller
  const uint32_t tiles = (units + U - 1) / U;
  const int64_t need = ((int64_t)tiles + (kThreads / 32) - 1) / (kThreads / 32);
  int64_t cap = need;
  if (EXT && kExtPersistent) {  // see kGridNote
    int per_sm = 0;
    cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, swiglu_cast_fp4_kernel<L, EXT>, kThreads, 0);
    if (st != cudaSuccess) return st;
    cap = (int64_t)c.num_sms * (per_sm > 0 ? per_sm : 1);
  }
  const int blocks = (int)(need < cap ? (need > 0 ? need : 1) : cap);
  return launch_pdl(swiglu_cast_fp4_kernel<L, EXT>, blocks, kThreads, 0, c.stream,
                    static_cast<const uint16_t*>(x), units, N, out, out_sf, FastDiv((uint32_t)G),
                    ext);
}

template <int L>
cudaError_t launch_fp4(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                       float* out_sf, const SwigluExt& ext) {
  const bool plain = !ext.has_clamp && ext.weights == nullptr && ext.clamp_count == nullptr &&
                     ext.sf.flags == 0;
  return plain ? launch_fp4_t<L, false>(c, x, M, N, out, out_sf, ext)
               : launch_fp4_t<L, true>(c, x, M, N, out, out_sf, ext);
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
  return launch_t<false>(c, x, M, N, out, out_sf, SwigluExt());
}

cudaError_t launch_swiglu_cast_ex(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                                  void* out_sf, const SwigluExt& ext) {
  return launch_t<true>(c, x, M, N, out, static_cast<float*>(out_sf), ext);
}

}  // namespace moe
