// expand_cast_fp4.cu -- expand + per-group FP4 E2M1 cast.
//
// TileKernels article (itsolotime.com): section 3.1's CastOutputConfig names
// float4_e2m1fn as an output type with clamp_min_value = max_value * 2^-126
// (max_value = 6, so the scale stays a normal f32 and its inverse finite);
// section 3.2's per_token_cast takes the group absmax over num_per_channels
// channels, scale = max(amax, clamp_min) / max_value, and multiplies by the
// scale's inverse; section 2.2's expand_to_fused copies each token's codes and
// scales to the rows pos names.  Two codes per byte, element 2i in the low
// nibble.  Group sizes 16, 32, 64 and 128 (1, 2, 4 or 8 lanes of 16 channels).
//
// Same structure as the E4M3 bulk-store kernel: one CTA per token (see
// kFp4TokensPerCta), thread c owning channels 16c..16c+15; each token's packed
// codes (H/2 bytes) and, for row-major f32 scales with G % 4 == 0, its scales
// are staged in shared memory and leave with TMA bulk copies (cp.async.bulk)
// issued by one thread; row-major UE8M0 scales leave by one warp's wide
// stores; column-major scales are stored per group by one lane, or staged per
// token for the column-major gather.
#include "common.cuh"

namespace moe {
namespace {

// Tokens per CTA.  The grid is not persistent: one CTA per TOK consecutive
// tokens, retiring once its copies have read shared memory, so the CTAs in
// flight at any moment cover a compact run of tokens (the E4M3 bulk form's
// layout; there a persistent grid striding over the tokens ran at 0.89 of the
// measured copy peak against 1.01).  Each token writes fewer bytes here than
// in E4M3, and with the kernel's natural 55-59 registers (2 CTAs of 448
// threads per SM at H = 7168) more tokens per CTA paid: measured on GB300
// (H = 7168, k = 8, after an L2 flush) at T = 65536, group 32: 0.91 / 0.91 /
// 0.96 / 0.98 of the measured copy peak for 1 / 2 / 3 / 4 tokens per CTA.
// Held to 32 registers (no spills), 4 CTAs fit an SM and one token per CTA
// is best: group 32 at 1.01 (0.482 against 0.505 ms for 3 tokens per CTA
// unconstrained), group 16 at 1.00 (0.552 against 0.557 ms); at T = 8192
// 66 against 74 us (group 32).  40 registers with 1 or 2 tokens per CTA, and
// 48 with 2, were slower.
constexpr int kFp4TokensPerCta = 1;

__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
               "r"(bytes)
               : "memory");
}

// L = lanes per group (group = 16 L channels).  sf_bulk: row-major f32
// scales (power-of-two rounded or not) whose rows (4G bytes) are 16-byte
// multiples go out with the codes.  sf_wide: row-major UE8M0 bytes are
// assembled in shared memory and one warp writes them sf_wide (8 or 4) bytes
// per store.  Otherwise one lane per group stores its scale.  ZF: the
// zero-fill of the padding rows (zsrc non-null) is compiled in.
template <int L, int TOK, bool ZF>
__global__ void __maxnreg__(32) expand_cast_fp4_kernel(
    const uint16_t* __restrict__ x, int64_t T, int H, int k, const int32_t* __restrict__ pos,
    int64_t R, uint8_t* __restrict__ out, float* __restrict__ out_sf,
    const int32_t* __restrict__ zsrc, SfOut sfo, int sf_bulk, int sf_wide, unsigned* err) {
  extern __shared__ __align__(128) uint8_t s_buf[];
  pdl_enter();
  const int P = H >> 4;   // threads per token
  const int G = P / L;    // groups per token
  const int HB = H >> 1;  // code bytes per row
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const bool act = tid < P;
  const int g = tid / L;
  const bool lead = (tid % L) == 0;
  const uint32_t stride = (uint32_t)((HB + 4 * G + 127) / 128 * 128);  // bytes per token slot
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(s_buf);
  int32_t* spos_all = reinterpret_cast<int32_t*>(s_buf + (size_t)TOK * stride);  // [TOK][32]
  // the slots and the destination lists fit the launch's shared memory
  if (!MOE_DBG_OK((size_t)TOK * (stride + 128) <= dynamic_smem_bytes() && 8 * P <= (int)stride,
                  err))
    return;  // the same for every thread of the CTA
  bool bad = false;
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
        a[i] = ld_stream_v4(src);
        b[i] = ld_stream_v4(src + 8);
      }
      if (tid < 32 && lane < k) pv[i] = __ldg(pos + t * k + lane);
    }
  }
  float sfv[TOK];
#pragma unroll
  for (int i = 0; i < TOK; ++i) {
    const bool valid = t0 + i < T;
    const float amax = maxL<L>(absmax16_bf16(a[i], b[i]));
    sfv[i] = fp4_scale(amax, sfo.flags);
    const float inv = __fdiv_rn(1.0f, sfv[i]);
    const uint2 q = quant16_bf16_e2m1(a[i], b[i], inv);
    uint8_t* sq = s_buf + (size_t)i * stride;
    if (act && valid) {
      *reinterpret_cast<uint2*>(sq + tid * 8) = q;
      if (lead && sf_bulk) *reinterpret_cast<float*>(sq + HB + 4 * g) = sfv[i];
      if (lead && sf_wide) sq[HB + g] = (uint8_t)((__float_as_uint(sfv[i]) >> 23) & 0xFFu);
    }
    if (!sf_bulk && tid < 32) spos_all[i * 32 + tid] = valid ? pv[i] : -1;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the copies
  __syncthreads();
  if (sf_wide) {
    // by one warp (warp 1 where there is one, so that warp 0 issues its
    // copies meanwhile)
    if ((tid >> 5) == (blockDim.x >= 64 ? 1 : 0)) {
#pragma unroll
      for (int i = 0; i < TOK; ++i)
        if (t0 + i < T)
          store_ue8m0_rows(reinterpret_cast<uint8_t*>(out_sf), s_buf + (size_t)i * stride + HB,
                           spos_all + i * 32, k, G, R, sf_wide, lane, err);
    }
  } else if (!sf_bulk && act && lead) {  // one lane per group stores its scale
#pragma unroll
    for (int i = 0; i < TOK; ++i) {
      const int64_t t = t0 + i;
      if (t >= T) continue;
      if (sfo.stage != nullptr) {
        store_stage(sfo.stage, sfo.flags, G, t, g, sfv[i]);
      } else {
        const int32_t* spos = spos_all + i * 32;
        for (int j = 0; j < k; ++j) {
          const int32_t r = spos[j];
          if (r >= 0 && r < R) store_sf_opts(out_sf, sfo.flags, sfo.ld, G, r, g, sfv[i]);
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
          } else if (MOE_DBG_OK(bulk_copy_ok(out + (int64_t)r * HB, slot, (uint32_t)HB, sbase) &&
                                    (!sf_bulk || bulk_copy_ok(out_sf + (int64_t)r * G, slot + HB,
                                                              (uint32_t)(4 * G), sbase)),
                                err)) {
            bulk_s2g(out + (int64_t)r * HB, slot, (uint32_t)HB);
            if (sf_bulk) bulk_s2g(out_sf + (int64_t)r * G, slot + HB, (uint32_t)(4 * G));
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
  if (ZF && zsrc != nullptr)
    zero_fill_rows(zsrc, R, HB, G, out, out_sf,
                   (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x,
                   ((int64_t)gridDim.x * blockDim.x) >> 5, threadIdx.x & 31, sfo);
  if (bad) flag_error(err, MOE_DEVERR_POS_RANGE);
}

template <int L, bool ZF>
cudaError_t launch_lt(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                      const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                      const int32_t* zsrc, SfOut sfo) {
  constexpr int TOK = kFp4TokensPerCta;
  const int P = H / 16;
  const int threads = (P + 31) / 32 * 32;
  const int G = P / L;
  const size_t stride = (size_t)(H / 2 + 4 * G + 127) / 128 * 128;
  const size_t smem = (stride + sizeof(int32_t) * 32) * TOK;
  if (smem > 48 * 1024) {
    cudaError_t st = allow_max_dynamic_smem(expand_cast_fp4_kernel<L, TOK, ZF>);
    if (st != cudaSuccess) return st;
  }
  const bool rowmajor = !(sfo.flags & MOE_SF_COLMAJOR) && sfo.stage == nullptr;
  const int sf_bulk = (rowmajor && !(sfo.flags & MOE_SF_UE8M0) && G % 4 == 0 &&
                       reinterpret_cast<uintptr_t>(out_sf) % 16 == 0)
                          ? 1
                          : 0;
  const int sf_wide = rowmajor && (sfo.flags & MOE_SF_UE8M0) ? ue8m0_store_width(out_sf, G) : 0;
  int64_t blocks = (T + TOK - 1) / TOK;
  if (ZF) {  // enough warps for one 32-row group of the zero-fill each
    const int64_t zb = ((R + 31) / 32 + threads / 32 - 1) / (threads / 32);
    blocks = blocks > zb ? blocks : zb;
  }
  if (blocks < 1) blocks = 1;
  return launch_pdl(expand_cast_fp4_kernel<L, TOK, ZF>, (unsigned)blocks, threads, smem, c.stream,
                    static_cast<const uint16_t*>(x), T, H, k, pos, R, out, out_sf, zsrc, sfo,
                    sf_bulk, sf_wide, c.err);
}

template <int L>
cudaError_t launch_l(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                     const int32_t* pos, int64_t R, uint8_t* out, float* out_sf,
                     const int32_t* zsrc, SfOut sfo) {
  return zsrc != nullptr ? launch_lt<L, true>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo)
                         : launch_lt<L, false>(c, x, T, H, k, pos, R, out, out_sf, zsrc, sfo);
}

}  // namespace

cudaError_t launch_expand_cast_fp4(const LaunchCtx& c, const void* x, int64_t T, int H, int k,
                                   const int32_t* pos, int64_t R, uint8_t* out, void* out_sf,
                                   const int32_t* zero_rows, SfOut sfo, int group) {
  float* sf = static_cast<float*>(out_sf);
  cudaError_t e;
  switch (group) {
    case 16: e = launch_l<1>(c, x, T, H, k, pos, R, out, sf, zero_rows, sfo); break;
    case 32: e = launch_l<2>(c, x, T, H, k, pos, R, out, sf, zero_rows, sfo); break;
    case 64: e = launch_l<4>(c, x, T, H, k, pos, R, out, sf, zero_rows, sfo); break;
    case 128: e = launch_l<8>(c, x, T, H, k, pos, R, out, sf, zero_rows, sfo); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || sfo.stage == nullptr) return e;
  return launch_sf_gather(c, zero_rows, R, T, k, H / group, sfo, out_sf);
}

}  // namespace moe
