// common.cuh -- device helpers shared by the kernels of the MoE routing + FP8
// path (sm_103a).  Nothing here is visible across the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <atomic>

#include "moe_route.h"

namespace moe {

// Scaling constants of the E4M3 per-group cast: the largest finite E4M3FN
// magnitude and the scale floor ("clamp_min_value" for E4M3 in the TileKernels
// article, section 3.1).
constexpr float kE4M3Max = 448.0f;
constexpr float kScaleFloor = 1e-4f;
constexpr int kGroup = 128;

// ------------------------------------------------------------ error flags

// Sets `bit` in the library's device error word (moe_get_device_status).
__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Debug-bounds build (compiled with MOE_DEBUG_BOUNDS defined): MOE_DBG_OK
// checks an index, size or alignment invariant that the kernel's
// construction guarantees, before the access it guards.  A false check sets
// MOE_DEVERR_BOUNDS and the caller skips the access; nothing traps.  In the
// normal build it is the constant true and the condition is not compiled.
#ifdef MOE_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_check(bool ok, unsigned* err) {
  if (!ok) flag_error(err, MOE_DEVERR_BOUNDS);
  return ok;
}
#define MOE_DBG_OK(cond, err) ::moe::dbg_check((cond), (err))
#else
#define MOE_DBG_OK(cond, err) true
#endif

// This launch's dynamic shared memory, in bytes.
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t n;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
  return n;
}

// The preconditions of a bulk shared -> global copy: the global and shared
// addresses and the size multiples of 16 bytes, the source inside this CTA's
// dynamic shared memory (which starts at the shared address sbase).
__device__ __forceinline__ bool bulk_copy_ok(const void* gdst, uint32_t ssrc, uint32_t bytes,
                                             uint32_t sbase) {
  return ((reinterpret_cast<uintptr_t>(gdst) | ssrc | bytes) & 15u) == 0 && ssrc >= sbase &&
         ssrc - sbase + bytes <= dynamic_smem_bytes();
}

// ---------------------------------------------------------------- memory ops

// 16-byte streaming load of data read exactly once: non-coherent path, no L1
// allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load through the normal cached path (data other CTAs re-read).
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte store of data nobody re-reads in this kernel (evict-first).
// The same load with an L2 eviction policy (a createpolicy result).
__device__ __forceinline__ uint4 ld_stream_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream_v2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream_f32(float* p, float v) {
  asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// ---------------------------------------------------------------- bf16 / fp8

// The two bf16 values packed in one 32-bit word, widened exactly to f32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two f32 values -> two E4M3FN codes (round to nearest even, saturate to
// +-448), `a` in the low byte.  This is the hardware conversion
// (cvt.rn.satfinite.e4m3x2.f32) reached through the CUDA header intrinsic.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Scale of one group from its absolute maximum (f32, IEEE rounding).
__device__ __forceinline__ float group_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, kScaleFloor), kE4M3Max);
}

// Scale options (MOE_SF_* in moe_route.h; TileKernels article, 3.1 round_sf /
// packed UE8M0 and 2.2 TMA-aligned column-major scales).  With POW2 (or
// UE8M0) the scale is the smallest power of two >= the plain scale: a
// positive normal f32 with a non-zero mantissa moves to the next exponent.
__device__ __forceinline__ float round_pow2_up(float s) {
  uint32_t b = __float_as_uint(s);
  if (b & 0x007FFFFFu) b = (b & 0xFF800000u) + 0x00800000u;
  return __uint_as_float(b);
}

__device__ __forceinline__ float group_scale_opts(float amax, int flags) {
  const float s = group_scale(amax);
  return (flags & (MOE_SF_POW2 | MOE_SF_UE8M0)) ? round_pow2_up(s) : s;
}

// Store scale `sf` of (row r, group g) in the flagged layout; UE8M0 stores
// the biased exponent byte of the (power-of-two) scale, packed four groups of
// a row per 32-bit word when column-major.  `zero` stores 0.0 / byte 0.
__device__ __forceinline__ void store_sf_opts(void* out_sf, int flags, int64_t ld, int G,
                                              int64_t r, int g, float sf, bool zero = false) {
  if (flags & MOE_SF_UE8M0) {
    const uint8_t byte = zero ? 0 : (uint8_t)((__float_as_uint(sf) >> 23) & 0xFFu);
    uint8_t* b = static_cast<uint8_t*>(out_sf);
    if (flags & MOE_SF_COLMAJOR)
      b[((int64_t)(g >> 2) * ld + r) * 4 + (g & 3)] = byte;
    else
      b[r * G + g] = byte;
  } else {
    float* f = static_cast<float*>(out_sf);
    const float v = zero ? 0.0f : sf;
    if (flags & MOE_SF_COLMAJOR)
      f[(int64_t)g * ld + r] = v;
    else
      f[r * G + g] = v;
  }
}

// Store token t's scale of group g into the row-major staging buffer.
__device__ __forceinline__ void store_stage(uint8_t* stage, int flags, int G, int64_t t, int g,
                                            float sf) {
  if (flags & MOE_SF_UE8M0)
    stage[t * (((G + 3) >> 2) << 2) + g] = (uint8_t)((__float_as_uint(sf) >> 23) & 0xFFu);
  else
    reinterpret_cast<float*>(stage)[t * G + g] = sf;
}

// Row-major UE8M0 scales with wide stores: the width (8 or 4 bytes) that
// out_sf's address and the row length G both allow, else 0 (byte stores).
__host__ __device__ __forceinline__ int ue8m0_store_width(const void* out_sf, int G) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(out_sf) | (uintptr_t)G;
  return (a & 7u) == 0 ? 8 : ((a & 3u) == 0 ? 4 : 0);
}

// One warp writes a token's G row-major UE8M0 scale bytes, held at `src` in
// shared memory (n-byte aligned), to each of its destination rows spos[j],
// j < k (skipped where negative or >= R), n = ue8m0_store_width bytes per
// store: G / n stores per row, spread over the lanes.
__device__ __forceinline__ void store_ue8m0_rows(uint8_t* out_sf, const uint8_t* src,
                                                 const int32_t* spos, int k, int G, int64_t R,
                                                 int n, int lane, unsigned* err) {
  const int per = G / n;
  for (int u = lane; u < k * per; u += 32) {
    const int j = u / per, c = u - j * per;
    const int32_t r = spos[j];
    if (r < 0 || r >= R) continue;
    uint8_t* dst = out_sf + (int64_t)r * G + c * n;
    if (!MOE_DBG_OK(((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) &
                     (uintptr_t)(n - 1)) == 0,
                    err))
      continue;
    if (n == 8)
      *reinterpret_cast<uint64_t*>(dst) = *reinterpret_cast<const uint64_t*>(src + c * n);
    else
      *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src + c * n);
  }
}

// Quantise 16 f32 values with multiplier `inv`, pack the 16 codes.
__device__ __forceinline__ uint4 quant16(const float (&v)[16], float inv) {
  uint4 q;
  q.x = e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
        (e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
  q.y = e4m3x2(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv)) |
        (e4m3x2(__fmul_rn(v[6], inv), __fmul_rn(v[7], inv)) << 16);
  q.z = e4m3x2(__fmul_rn(v[8], inv), __fmul_rn(v[9], inv)) |
        (e4m3x2(__fmul_rn(v[10], inv), __fmul_rn(v[11], inv)) << 16);
  q.w = e4m3x2(__fmul_rn(v[12], inv), __fmul_rn(v[13], inv)) |
        (e4m3x2(__fmul_rn(v[14], inv), __fmul_rn(v[15], inv)) << 16);
  return q;
}

// Unpack 16 bf16 (two 16-byte words) to f32.
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ float absmax16(const float (&v)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// The same two steps straight from 16 packed bf16 (two 16-byte words),
// unpacking on the fly so the caller keeps 8 registers instead of 16.
__device__ __forceinline__ float absmax16_bf16(const uint4& a, const uint4& b) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  return m;
}

__device__ __forceinline__ uint4 quant16_bf16(const uint4& a, const uint4& b, float inv) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
    c[i] = e4m3x2(__fmul_rn(bf16_lo(w0), inv), __fmul_rn(bf16_hi(w0), inv)) |
           (e4m3x2(__fmul_rn(bf16_lo(w1), inv), __fmul_rn(bf16_hi(w1), inv)) << 16);
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// ---------------------------------------------------------------- FP4 E2M1
// TileKernels article, 3.1: float4_e2m1fn's clamp_min_value is max_value *
// 2^-126 with max_value = 6.
// clamp_min_value of float4_e2m1fn: 6 * 2^-126 = 1.5 * 2^-124.
__device__ __forceinline__ float fp4_floor() { return __uint_as_float(0x01C00000u); }

__device__ __forceinline__ float fp4_scale(float amax, int flags) {
  const float s = __fdiv_rn(fmaxf(amax, fp4_floor()), 6.0f);
  return (flags & (MOE_SF_POW2 | MOE_SF_UE8M0)) ? round_pow2_up(s) : s;
}

// Two f32 values -> one byte of two E2M1 codes (round to nearest even,
// saturate to +-6), `lo` in the low nibble: the hardware conversion
// cvt.rn.satfinite.e2m1x2.f32, whose first source goes to the high nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// 16 f32 values times `inv` -> 8 bytes of packed E2M1 codes.
__device__ __forceinline__ uint2 quant16_e2m1(const float (&v)[16], float inv) {
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = e2m1x2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv));
    c[i >> 2] |= byte << (8 * (i & 3));
  }
  return make_uint2(c[0], c[1]);
}

// 16 bf16 values times `inv` -> 8 bytes of packed E2M1 codes.
__device__ __forceinline__ uint2 quant16_bf16_e2m1(const uint4& a, const uint4& b, float inv) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = e2m1x2(__fmul_rn(bf16_lo(w[i]), inv), __fmul_rn(bf16_hi(w[i]), inv));
    c[i >> 2] |= byte << (8 * (i & 3));
  }
  return make_uint2(c[0], c[1]);
}

// Max over the L lanes of an aligned L-lane subgroup.
template <int L>
__device__ __forceinline__ float maxL(float m) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

// Max over the 8 lanes of an aligned 8-lane subgroup.
__device__ __forceinline__ float max8(float m) {
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return m;
}

// Unsigned 32-bit division by a divisor fixed at launch, as one multiply-high
// and two shifts (Granlund and Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, round-up variant): for d with
// 2^(l-1) < d <= 2^l, m = floor(2^32 (2^l - d) / d) + 1 and
// n / d = (t + ((n - t) >> min(l,1))) >> max(l-1,0) with t = mulhi(n, m).
struct FastDiv {
  uint32_t d = 1, m = 1, s1 = 0, s2 = 0;
  FastDiv() = default;
  __host__ explicit FastDiv(uint32_t div) : d(div) {
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < div) ++l;
    m = (uint32_t)(((1ull << 32) * ((1ull << l) - div)) / div + 1);
    s1 = l < 1 ? l : 1;
    s2 = l > 0 ? l - 1 : 0;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(n, m);
    return (t + ((n - t) >> s1)) >> s2;
  }
};

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization and starts with pdl_enter(), which
// waits until the previous kernel on the stream has finished and its writes
// are visible, before any global memory access: stream order is unchanged for
// the data.  A kernel's CTAs release the next kernel as they exit (the
// implicit trigger), so the next launch is processed while the last CTAs
// drain instead of after the whole grid retires.  (Releasing it at kernel
// entry instead let waiting CTAs of the next kernel take SMs early and
// unbalanced the one-CTA-per-SM expand grid on GB300.)
__device__ __forceinline__ void pdl_enter() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace moe

// ------------------------------------------------------------- launch API
// Each kernel file exposes one host launcher; api.cu validates and calls it.
namespace moe {
struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  unsigned* err;  // device error word
};

// The device conversions on arbitrary f32 values, for tests (debug_cvt.cu).
cudaError_t launch_debug_cvt(const LaunchCtx& c, int fmt, const float* in, uint8_t* out,
                             int64_t n);

// Fused decode path (decode_fused.cu) and its test hooks.
extern std::atomic<int64_t> g_decode_timeout_ns;
extern std::atomic<int> g_decode_skip_signal;
size_t decode_fused_smem(int64_t T, int E, int k, int H, int num_sms, int* blocks, int* tpb);
cudaError_t launch_decode_fused(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                                const void* x, int H, int32_t* idx, float* w, int32_t* counts,
                                int32_t* offsets, int32_t* pos, int32_t* src, uint8_t* out,
                                float* out_sf, unsigned* ctl);

// Replicated-routing decode path (decode_replicated.cu): every block builds
// the route map of all T tokens itself (for small T also their selection),
// then writes its own tokens' rows.
constexpr int kDecodeReplicatedInlineTokens = 32;  // up to here the selection is repeated too
constexpr int kDecodeReplicatedMaxTokens = 2048;
bool decode_replicated_ok(int64_t T, int E, int k, int H);
cudaError_t launch_decode_replicated(const LaunchCtx& c, const float* scores, int64_t T, int E,
                                     int k, const void* x, int H, int32_t* idx, float* w,
                                     int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                                     uint8_t* out, float* out_sf);

// The route map alone in one launch for small T (the same kernel without the
// expand): every block builds it, then writes its own tokens' pos and
// sorted_src entries.
// Measured on GB300 (E = 256, k = 8): 6.8 against 10.9 us for the two-kernel
// map at T = 64 and 256, 8.9 against 10.9 at T = 1024, 12.9 against 10.9 at
// T = 2048.
constexpr int kRouteMapReplicatedMaxTokens = 1024;
bool route_map_replicated_ok(int64_t T, int E, int k);
cudaError_t launch_route_map_replicated(const LaunchCtx& c, const int32_t* idx, int64_t T, int E,
                                        int k, int32_t* counts, int32_t* offsets, int32_t* pos,
                                        int32_t* src);

cudaError_t launch_topk_gate(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                             int32_t* idx, float* w);
cudaError_t launch_route_map(const LaunchCtx& c, const int32_t* idx, int64_t T, int E, int k,
                             int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* sorted_src,
                             int32_t* ws, int64_t num_chunks);
cudaError_t launch_route_map_aligned(const LaunchCtx& c, const int32_t* idx, int64_t T, int E,
                                     int k, int align, int64_t num_rows, int32_t* counts,
                                     int32_t* offsets, int32_t* pos, int32_t* sorted_src,
                                     int32_t* ws, int64_t num_chunks);
// Scale output description for the cast kernels: flags 0 is the plain
// row-major f32 layout.
struct SfOut {
  int flags = 0;
  int64_t ld = 0;
  // Column-major layouts only: when non-null, the expand kernels write each
  // token's scales once, row-major, here ([T][G] f32, or [T][ceil(G/4)] packed
  // UE8M0 words), and launch_sf_gather then writes the column-major buffer
  // row by row from sorted_src with whole-line stores.
  uint8_t* stage = nullptr;
};

// Padded layouts (TileKernels article, section 2.2: expand_to_fused zero-fills
// the rows no token lands on in the same launch).  With zsrc non-null, every
// row r < num_rows whose zsrc[r] (the route map's sorted_src) is negative gets
// all-zero codes and scales.  Warp-granular: a warp reads 32 entries with one
// coalesced load and zeroes each marked row 512 bytes per store instruction.
// These rows are disjoint from every row a copy is written to.
__device__ __forceinline__ void zero_fill_rows(const int32_t* __restrict__ zsrc, int64_t num_rows,
                                               int row_bytes, int G, uint8_t* __restrict__ out,
                                               float* __restrict__ out_sf, int64_t gwarp,
                                               int64_t nwarps, int lane, SfOut sfo) {
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int64_t r0 = gwarp * 32; r0 < num_rows; r0 += nwarps * 32) {
    const int64_t r = r0 + lane;
    const bool z = r < num_rows && __ldg(zsrc + r) < 0;
    unsigned m = __ballot_sync(0xFFFFFFFFu, z);
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1;
      uint8_t* q = out + (r0 + i) * row_bytes;  // row_bytes: a multiple of 16
      for (int c = lane * 16; c < row_bytes; c += 512) st_stream_v4(q + c, zero);
      if (sfo.stage != nullptr) {
        // staged column-major scales: the gather writes these rows' zeros
      } else if (sfo.flags == 0) {
        float* sfr = out_sf + (r0 + i) * G;
        for (int g = lane; g < G; g += 32) st_stream_f32(sfr + g, 0.0f);
      } else {
        for (int g = lane; g < G; g += 32)
          store_sf_opts(out_sf, sfo.flags, sfo.ld, G, r0 + i, g, 0.0f, true);
      }
    }
  }
}

// Expand + FP4 E2M1 cast (expand_cast_fp4.cu): group 16, 32, 64 or 128.
cudaError_t launch_expand_cast_fp4(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                                   const int32_t* pos, int64_t R, uint8_t* out, void* out_sf,
                                   const int32_t* zero_rows, SfOut sfo, int group);

// Column-major scales from staged per-token rows (SfOut::stage), row by row
// from sorted_src; in expand_cast.cu.
cudaError_t launch_sf_gather(const LaunchCtx& c, const int32_t* src, int64_t R, int64_t T, int k,
                             int G, SfOut sfo, void* out_sf);

// The chained route + expand (route_chain.cu): the top-k kernel leaves, in
// pos, each copy's rank among its expert's copies within its chunk of
// consecutive tokens and writes one histogram row per chunk; a column scan
// turns the histogram into base[chunk][e], the copies of expert e in earlier
// chunks, and writes counts and offsets; the expand kernel then places every
// copy itself:
//   pos = offsets[e] + base[chunk][e] + rank in chunk,
// and writes pos and sorted_src before it stores the rows.
struct RouteChain {
  const int32_t* idx = nullptr;      // [T, k] experts of each token
  const int32_t* base = nullptr;     // [chunks, E]
  const int32_t* offsets = nullptr;  // [E + 1]
  int32_t* sorted_src = nullptr;     // [T * k], written
  int E = 0;
  int chunk_shift = 0;               // chunk = 1 << chunk_shift tokens
};
// The expand kernel's chained form (expand_cast.cu): plain E4M3 with f32
// row-major scales; needs H <= 16384, H / 128 % 4 == 0, 16-byte aligned out
// and out_sf, E <= 256.
cudaError_t launch_expand_cast_chain(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                                     int32_t* pos, uint8_t* out, float* out_sf,
                                     const RouteChain& rc);
// The whole chain (route_chain.cu); hist: (T >> chunk_shift rounded up) * E
// int32 of workspace (route_chain_workspace_bytes).
bool route_chain_ok(int64_t T, int E, int k, int H, const void* out, const void* out_sf);
size_t route_chain_workspace_bytes(int64_t T, int E);
// arrivals: a 32-bit counter that is zero before the call (left at zero).
cudaError_t launch_route_chain(const LaunchCtx& c, const float* scores, int64_t T, int E, int k,
                               const void* x, int H, int32_t* idx, float* w, int32_t* counts,
                               int32_t* offsets, int32_t* pos, int32_t* src, uint8_t* out,
                               float* out_sf, int32_t* hist, unsigned* arrivals);

cudaError_t launch_expand_cast(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                               const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                               const int32_t* zero_rows = nullptr, SfOut sfo = SfOut());
cudaError_t launch_swiglu_cast(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                               float* out_sf);
// SwiGLU variants: clamp (has_clamp), per-row weight (nullable), clamp count
// (nullable, added to), scale options.
struct SwigluExt {
  int has_clamp = 0;
  float clamp = 0.0f;
  const float* weights = nullptr;
  unsigned long long* clamp_count = nullptr;
  SfOut sf;
};
cudaError_t launch_swiglu_cast_fp4(const LaunchCtx& c, const void* x, int64_t M, int N,
                                   uint8_t* out, void* out_sf, const SwigluExt& ext, int group);
cudaError_t launch_swiglu_cast_ex(const LaunchCtx& c, const void* x, int64_t M, int N, uint8_t* out,
                                  void* out_sf, const SwigluExt& ext);
cudaError_t launch_combine(const LaunchCtx& c, const void* y, const float* w, const int32_t* pos,
                           int64_t T, int H, int k, int64_t R, void* out, bool out_f32);
cudaError_t launch_peak_copy(const LaunchCtx& c, const void* src, void* dst, size_t bytes);

// Route-map chunking: a chunk is a run of consecutive tokens, a multiple of
// 32 (one bitmap word per expert per 32 tokens) and at most
// kRouteMaxChunkTokens, aiming at about kRouteTargetChunks chunks (one wave
// of CTAs); one histogram row of E counters per chunk in the workspace.
constexpr int kRouteTargetChunks = 128;
constexpr int kRouteMaxChunkTokens = 512;
inline int64_t route_chunk_tokens(int64_t T) {
  int64_t c = (T + kRouteTargetChunks - 1) / kRouteTargetChunks;
  c = (c + 31) / 32 * 32;
  if (c > kRouteMaxChunkTokens) c = kRouteMaxChunkTokens;
  return c < 32 ? 32 : c;
}
inline int64_t route_num_chunks(int64_t T) {
  const int64_t c = route_chunk_tokens(T);
  return (T + c - 1) / c;
}

// Kernel launch counter (api.cu).
void count_launches(int n);

// api.cu: record a CUDA error for moe_last_cuda_error_string and return
// MOE_ERR_CUDA; and the current device's launch context (SM count, the address
// of the device error word), looked up once per device.  context() returns
// MOE_ERR_UNSUPPORTED for a device ordinal beyond the library's table.
moe_status_t cuda_fail(cudaError_t e);
moe_status_t context(void* stream, LaunchCtx* ctx);

// Let `kernel` take any dynamic shared memory a block can opt in to (the
// device's opt-in maximum minus the kernel's static shared memory; api.cu).
// Every call sets the same value for a kernel, so calls from several host
// threads cannot undo one another, as a per-call size could (a smaller value
// landing between another thread's set and its launch).  The cap does not
// change what a launch uses: that is the launch's own size.
cudaError_t allow_max_dynamic_smem(const void* kernel);
template <typename... KArgs>
inline cudaError_t allow_max_dynamic_smem(void (*kernel)(KArgs...)) {
  return allow_max_dynamic_smem(reinterpret_cast<const void*>(kernel));
}

// Launch `kernel` on `stream` with programmatic stream serialization (see
// pdl_enter) and count it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace moe
