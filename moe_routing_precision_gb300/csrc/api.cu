// api.cu -- the extern "C" boundary declared in include/moe_route.h: host-side
// argument checks, per-device launch context, and status reporting.
//
// Every entry validates its arguments before touching the GPU; a rejected call
// launches nothing.  The only device state the library owns is one 32-bit
// error word per device (a __device__ variable, no allocation).
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;
struct DeviceState {
  std::once_flag once;
  cudaError_t init_status = cudaSuccess;
  int num_sms = 0;
  unsigned* err = nullptr;
};
DeviceState g_devices[kMaxDevices];
std::atomic<uint64_t> g_launches{0};
thread_local char g_last_cuda_error[256] = "no CUDA error";

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Control words of moe_route_expand_cast_fp8's workspace (its first 256
// bytes): words 0 and 1 belong to the fused decode launch, this one to the
// chained path's scan.
constexpr int kChainArrivalWord = 16;

bool experts_ok(int32_t E, int32_t k) {
  return E >= 1 && E <= MOE_MAX_EXPERTS && k >= 1 && k <= MOE_MAX_TOPK && k <= E;
}


}  // namespace

moe_status_t cuda_fail(cudaError_t e) {
  snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// Launch context of the current device: SM count and the address of the
// error word, looked up once per device.
moe_status_t context(void* stream, LaunchCtx* ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  DeviceState& d = g_devices[dev];
  std::call_once(d.once, [&d, dev]() {
    cudaError_t s = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (s == cudaSuccess) s = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_device_error);
    d.init_status = s;
  });
  if (d.init_status != cudaSuccess) return cuda_fail(d.init_status);
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->num_sms = d.num_sms;
  ctx->err = d.err;
  return MOE_OK;
}

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t allow_max_dynamic_smem(const void* kernel) {
  // the cap per kernel, computed once per process (every GPU here is the same part)
  static std::mutex mu;
  static const void* keys[64];
  static int caps[64];
  static int n = 0;
  int cap = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (keys[i] == kernel) cap = caps[i];
  }
  if (cap < 0) {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    cap = optin - (int)fa.sharedSizeBytes;
    std::lock_guard<std::mutex> lock(mu);
    if (n < 64) {
      keys[n] = kernel;
      caps[n] = cap;
      ++n;
    }
  }
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
}

#ifdef MOE_DEBUG_BOUNDS
namespace {
// The debug-bounds self-test: one check that is false by construction (a
// one-thread launch has no thread 1), guarding no memory access.
__global__ void debug_bounds_selftest_kernel(unsigned* err) {
  pdl_enter();
  (void)MOE_DBG_OK(threadIdx.x == 1, err);
}
}  // namespace
#endif

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ROUTE_ABI_VERSION; }

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

#ifdef MOE_DEBUG_BOUNDS
int32_t moe_debug_bounds_enabled(void) { return 1; }

moe_status_t moe_debug_bounds_selftest(void* stream) {
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_pdl(debug_bounds_selftest_kernel, 1, 1, 0, c.stream, c.err);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}
#else
int32_t moe_debug_bounds_enabled(void) { return 0; }

moe_status_t moe_debug_bounds_selftest(void*) { return MOE_ERR_UNSUPPORTED; }
#endif

const char* moe_last_cuda_error_string(void) { return g_last_cuda_error; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: bad pointer, size, alignment or range";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: valid request not implemented";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or launch failed";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: a kernel flagged out-of-range data or a timeout";
  }
  return "unknown moe_status_t";
}

moe_status_t moe_topk_gate(const float* scores, int64_t num_tokens, int32_t num_experts,
                           int32_t num_topk, int32_t* topk_idx, float* topk_weights,
                           int32_t weight_mode, void* stream) {
  if (num_tokens < 0 || !experts_ok(num_experts, num_topk)) return MOE_ERR_INVALID_ARG;
  if (weight_mode != MOE_WEIGHTS_NONE && weight_mode != MOE_WEIGHTS_SOFTMAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return MOE_OK;
  if (!scores || !topk_idx || !aligned(scores, 4) || !aligned(topk_idx, 4))
    return MOE_ERR_INVALID_ARG;
  if (weight_mode == MOE_WEIGHTS_SOFTMAX_TOPK && (!topk_weights || !aligned(topk_weights, 4)))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_topk_gate(c, scores, num_tokens, num_experts, num_topk, topk_idx,
                                   weight_mode == MOE_WEIGHTS_SOFTMAX_TOPK ? topk_weights : nullptr);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

size_t moe_route_map_workspace_bytes(int64_t num_tokens, int32_t num_experts, int32_t num_topk) {
  if (num_tokens <= 0 || num_experts < 1 || num_topk < 1 || num_topk > MOE_MAX_TOPK) return 0;
  const size_t bytes =
      (size_t)route_num_chunks(num_tokens) * (size_t)num_experts * sizeof(int32_t);
  return (bytes + 255) / 256 * 256;
}

moe_status_t moe_route_map(const int32_t* topk_idx, int64_t num_tokens, int32_t num_experts,
                           int32_t num_topk, int32_t* counts, int32_t* offsets, int32_t* pos,
                           int32_t* sorted_src, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (num_tokens < 0 || !experts_ok(num_experts, num_topk)) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (int64_t)num_topk >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0) {
    // nothing routed: counts and offsets are all zero
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * num_experts, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (num_experts + 1), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  if (!topk_idx || !pos || !sorted_src || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(pos, 4) ||
      !aligned(sorted_src, 4) || !aligned(workspace, 16))
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_route_map_workspace_bytes(num_tokens, num_experts, num_topk))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_route_map(c, topk_idx, num_tokens, num_experts, num_topk, counts, offsets,
                                   pos, sorted_src, static_cast<int32_t*>(workspace),
                                   route_num_chunks(num_tokens));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_route_map_aligned(const int32_t* topk_idx, int64_t num_tokens,
                                   int32_t num_experts, int32_t num_topk, int32_t align,
                                   int64_t num_rows, int32_t* counts, int32_t* offsets,
                                   int32_t* pos, int32_t* sorted_src, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (num_tokens < 0 || !experts_ok(num_experts, num_topk)) return MOE_ERR_INVALID_ARG;
  if (align < 1 || align > 4096 || num_rows < 0 || num_rows >= ((int64_t)1 << 31))
    return MOE_ERR_INVALID_ARG;
  if (num_tokens * (int64_t)num_topk + (int64_t)num_experts * (align - 1) >= ((int64_t)1 << 31))
    return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0) {
    if (num_rows > 0) return MOE_ERR_UNSUPPORTED;  // nothing to route: no padded rows either
    return moe_route_map(topk_idx, 0, num_experts, num_topk, counts, offsets, pos, sorted_src,
                         workspace, workspace_bytes, stream);
  }
  if (!topk_idx || !counts || !offsets || !pos || !sorted_src || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(pos, 4) ||
      !aligned(sorted_src, 4) || !aligned(workspace, 16))
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_route_map_workspace_bytes(num_tokens, num_experts, num_topk))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_route_map_aligned(c, topk_idx, num_tokens, num_experts, num_topk, align,
                                           num_rows, counts, offsets, pos, sorted_src,
                                           static_cast<int32_t*>(workspace),
                                           route_num_chunks(num_tokens));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_expand_cast_fp8_padded(const void* x, int64_t num_tokens, int32_t hidden,
                                        int32_t num_topk, const int32_t* pos,
                                        const int32_t* sorted_src, int64_t num_rows,
                                        uint8_t* out, float* out_sf, int32_t group,
                                        void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_rows < 0 || hidden < MOE_CAST_GROUP || hidden % MOE_CAST_GROUP != 0 ||
      num_topk < 1 || num_topk > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (num_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (hidden / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (num_tokens == 0 && num_rows == 0) return MOE_OK;
  if ((num_tokens > 0 && (!x || !pos)) || (num_rows > 0 && (!out || !out_sf || !sorted_src)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(pos, 4) || !aligned(sorted_src, 4) || !aligned(out, 16) ||
      !aligned(out_sf, 4))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  // with no tokens the kernels still run once over the rows to zero them
  cudaError_t e = launch_expand_cast(c, x, num_tokens, hidden, num_topk, pos, num_rows, out,
                                     out_sf, sorted_src);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_expand_cast_fp8(const void* x, int64_t num_tokens, int32_t hidden,
                                 int32_t num_topk, const int32_t* pos, int64_t num_rows,
                                 uint8_t* out, float* out_sf, int32_t group, void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_rows < 0 || hidden < MOE_CAST_GROUP || hidden % MOE_CAST_GROUP != 0 ||
      num_topk < 1 || num_topk > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (num_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (hidden / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MOE_OK;
  if (!x || !pos || (num_rows > 0 && (!out || !out_sf))) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(pos, 4) || !aligned(out, 16) || !aligned(out_sf, 4))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e =
      launch_expand_cast(c, x, num_tokens, hidden, num_topk, pos, num_rows, out, out_sf);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

}  // extern "C"

namespace moe {
namespace {
// Valid scale-option sets: UE8M0 needs POW2; column-major needs a leading
// dimension >= rows that keeps columns 16-byte aligned.
bool sf_opts_ok(uint32_t flags, int64_t ld, int64_t rows, const void* out_sf) {
  const uint32_t all = MOE_SF_COLMAJOR | MOE_SF_POW2 | MOE_SF_UE8M0;
  if (flags & ~all) return false;
  if ((flags & MOE_SF_UE8M0) && !(flags & MOE_SF_POW2)) return false;
  if (flags & MOE_SF_COLMAJOR) {
    if (ld < rows || ld % 4 != 0 || ld >= ((int64_t)1 << 31)) return false;
  }
  const bool bytes = (flags & MOE_SF_UE8M0) && !(flags & MOE_SF_COLMAJOR);
  return bytes || aligned(out_sf, 4);
}
}  // namespace
}  // namespace moe

extern "C" {

size_t moe_expand_cast_fp8_ex_workspace_bytes(int64_t num_tokens, int32_t hidden,
                                              uint32_t sf_flags) {
  if (num_tokens <= 0 || hidden < MOE_CAST_GROUP || !(sf_flags & MOE_SF_COLMAJOR)) return 0;
  const int64_t G = hidden / MOE_CAST_GROUP;
  const int64_t row = (sf_flags & MOE_SF_UE8M0) ? (G + 3) / 4 * 4 : G * 4;
  return (size_t)((num_tokens * row + 255) / 256 * 256);
}

moe_status_t moe_expand_cast_fp8_ex(const void* x, int64_t num_tokens, int32_t hidden,
                                    int32_t num_topk, const int32_t* pos,
                                    const int32_t* sorted_src, int64_t num_rows, uint8_t* out,
                                    void* out_sf, uint32_t sf_flags, int64_t sf_ld,
                                    void* workspace, size_t workspace_bytes, int32_t group,
                                    void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_rows < 0 || hidden < MOE_CAST_GROUP || hidden % MOE_CAST_GROUP != 0 ||
      num_topk < 1 || num_topk > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (num_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (hidden / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!sf_opts_ok(sf_flags, sf_ld, num_rows, out_sf)) return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0 && (num_rows == 0 || sorted_src == nullptr)) return MOE_OK;
  if ((num_tokens > 0 && (!x || !pos)) || (num_rows > 0 && (!out || !out_sf)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(pos, 4) || !aligned(sorted_src, 4) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  const size_t need = moe_expand_cast_fp8_ex_workspace_bytes(num_tokens, hidden, sf_flags);
  if (workspace != nullptr && (!aligned(workspace, 16) || workspace_bytes < need))
    return MOE_ERR_INVALID_ARG;
  const bool stage = need > 0 && workspace != nullptr && sorted_src != nullptr;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  SfOut sfo;
  sfo.flags = (int)sf_flags;
  sfo.ld = sf_ld;
  if (stage) sfo.stage = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_expand_cast(c, x, num_tokens, hidden, num_topk, pos, num_rows, out,
                                     static_cast<float*>(out_sf), sorted_src, sfo);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

size_t moe_expand_cast_fp4_workspace_bytes(int64_t num_tokens, int32_t hidden, int32_t group,
                                           uint32_t sf_flags) {
  if (num_tokens <= 0 || group <= 0 || hidden < group || !(sf_flags & MOE_SF_COLMAJOR)) return 0;
  const int64_t G = hidden / group;
  const int64_t row = (sf_flags & MOE_SF_UE8M0) ? (G + 3) / 4 * 4 : G * 4;
  return (size_t)((num_tokens * row + 255) / 256 * 256);
}

moe_status_t moe_expand_cast_fp4(const void* x, int64_t num_tokens, int32_t hidden,
                                 int32_t num_topk, const int32_t* pos, const int32_t* sorted_src,
                                 int64_t num_rows, uint8_t* out, void* out_sf, uint32_t sf_flags,
                                 int64_t sf_ld, void* workspace, size_t workspace_bytes,
                                 int32_t group, void* stream) {
  if (group != 16 && group != 32 && group != 64 && group != 128) return MOE_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_rows < 0 || hidden < 32 || hidden % 32 != 0 || hidden % group != 0 ||
      num_topk < 1 || num_topk > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (hidden > 16384) return MOE_ERR_UNSUPPORTED;
  if (num_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (!sf_opts_ok(sf_flags, sf_ld, num_rows, out_sf)) return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0 && (num_rows == 0 || sorted_src == nullptr)) return MOE_OK;
  if ((num_tokens > 0 && (!x || !pos)) || (num_rows > 0 && (!out || !out_sf)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(pos, 4) || !aligned(sorted_src, 4) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  const size_t need = moe_expand_cast_fp4_workspace_bytes(num_tokens, hidden, group, sf_flags);
  if (workspace != nullptr && (!aligned(workspace, 16) || workspace_bytes < need))
    return MOE_ERR_INVALID_ARG;
  const bool stage = need > 0 && workspace != nullptr && sorted_src != nullptr;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  SfOut sfo;
  sfo.flags = (int)sf_flags;
  sfo.ld = sf_ld;
  if (stage) sfo.stage = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_expand_cast_fp4(c, x, num_tokens, hidden, num_topk, pos, num_rows, out,
                                         out_sf, sorted_src, sfo, group);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t swiglu_cast_fp4(const void* x, int64_t num_rows, int32_t n, uint8_t* out,
                             void* out_sf, uint32_t sf_flags, int64_t sf_ld, int32_t has_clamp,
                             float clamp, const float* weights, uint64_t* clamp_count,
                             int32_t group, void* stream) {
  if (group != 16 && group != 32 && group != 64 && group != 128) return MOE_ERR_UNSUPPORTED;
  if (num_rows < 0 || n < 32 || n % 32 != 0 || n % group != 0) return MOE_ERR_INVALID_ARG;
  if (num_rows * (n / 16) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (has_clamp && !(clamp >= 0.0f && clamp <= 3.0e38f)) return MOE_ERR_INVALID_ARG;
  if (!sf_opts_ok(sf_flags, sf_ld, num_rows, out_sf)) return MOE_ERR_INVALID_ARG;
  if (num_rows == 0) return MOE_OK;
  if (!x || !out || !out_sf) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(weights, 4) || !aligned(clamp_count, 8))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  SwigluExt ext;
  ext.has_clamp = has_clamp ? 1 : 0;
  ext.clamp = clamp;
  ext.weights = weights;
  ext.clamp_count = reinterpret_cast<unsigned long long*>(clamp_count);
  ext.sf.flags = (int)sf_flags;
  ext.sf.ld = sf_ld;
  cudaError_t e = launch_swiglu_cast_fp4(c, x, num_rows, n, out, out_sf, ext, group);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t swiglu_cast_fp8_ex(const void* x, int64_t num_rows, int32_t n, uint8_t* out,
                                void* out_sf, uint32_t sf_flags, int64_t sf_ld, int32_t has_clamp,
                                float clamp, const float* weights, uint64_t* clamp_count,
                                int32_t group, void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (num_rows < 0 || n < MOE_CAST_GROUP || n % MOE_CAST_GROUP != 0) return MOE_ERR_INVALID_ARG;
  if (num_rows * (n / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (has_clamp && !(clamp >= 0.0f && clamp <= 3.0e38f)) return MOE_ERR_INVALID_ARG;
  if (!sf_opts_ok(sf_flags, sf_ld, num_rows, out_sf)) return MOE_ERR_INVALID_ARG;
  if (num_rows == 0) return MOE_OK;
  if (!x || !out || !out_sf) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(weights, 4) || !aligned(clamp_count, 8))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  SwigluExt ext;
  ext.has_clamp = has_clamp ? 1 : 0;
  ext.clamp = clamp;
  ext.weights = weights;
  ext.clamp_count = reinterpret_cast<unsigned long long*>(clamp_count);
  ext.sf.flags = (int)sf_flags;
  ext.sf.ld = sf_ld;
  cudaError_t e = launch_swiglu_cast_ex(c, x, num_rows, n, out, out_sf, ext);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t swiglu_cast_fp8(const void* x, int64_t num_rows, int32_t n, uint8_t* out,
                             float* out_sf, int32_t group, void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (num_rows < 0 || n < MOE_CAST_GROUP || n % MOE_CAST_GROUP != 0) return MOE_ERR_INVALID_ARG;
  if (num_rows * (n / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (num_rows == 0) return MOE_OK;
  if (!x || !out || !out_sf) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(out_sf, 4)) return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_swiglu_cast(c, x, num_rows, n, out, out_sf);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_combine(const void* y, const float* topk_weights, const int32_t* pos,
                         int64_t num_tokens, int32_t hidden, int32_t num_topk, int64_t num_rows,
                         void* out, int32_t out_dtype, void* stream) {
  if (num_tokens < 0 || num_rows < 0 || hidden < 8 || hidden % 8 != 0 || num_topk < 1 ||
      num_topk > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (out_dtype != MOE_OUT_BF16 && out_dtype != MOE_OUT_F32) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (hidden / 8) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MOE_OK;
  if (!topk_weights || !pos || !out || (num_rows > 0 && !y)) return MOE_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(topk_weights, 4) || !aligned(pos, 4) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_combine(c, y, topk_weights, pos, num_tokens, hidden, num_topk, num_rows,
                                 out, out_dtype == MOE_OUT_F32);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

size_t moe_route_expand_cast_fp8_workspace_bytes(int64_t num_tokens, int32_t num_experts,
                                                 int32_t num_topk) {
  const size_t route = moe_route_map_workspace_bytes(num_tokens, num_experts, num_topk);
  const size_t chain = route_chain_workspace_bytes(num_tokens, num_experts);
  return 256 + (route > chain ? route : chain);
}

moe_status_t moe_route_expand_cast_fp8(const float* scores, int64_t num_tokens,
                                       int32_t num_experts, int32_t num_topk, const void* x,
                                       int32_t hidden, int32_t* topk_idx, float* topk_weights,
                                       int32_t* counts, int32_t* offsets, int32_t* pos,
                                       int32_t* sorted_src, uint8_t* out, float* out_sf,
                                       void* workspace, size_t workspace_bytes, int32_t mode,
                                       int32_t group, void* stream) {
  if (group != MOE_CAST_GROUP) return MOE_ERR_UNSUPPORTED;
  if (mode != MOE_PATH_AUTO && mode != MOE_PATH_FUSED && mode != MOE_PATH_SEPARATE &&
      mode != MOE_PATH_REPLICATED && mode != MOE_PATH_CHAINED)
    return MOE_ERR_INVALID_ARG;
  if (num_tokens < 0 || !experts_ok(num_experts, num_topk)) return MOE_ERR_INVALID_ARG;
  if (hidden < MOE_CAST_GROUP || hidden % MOE_CAST_GROUP != 0) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (int64_t)num_topk >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (num_tokens * (hidden / MOE_CAST_GROUP) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4)) return MOE_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (!scores || !x || !topk_idx || !topk_weights || !pos || !sorted_src || !out || !out_sf ||
        !workspace)
      return MOE_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || !aligned(x, 16) || !aligned(topk_idx, 4) ||
        !aligned(topk_weights, 4) || !aligned(pos, 4) || !aligned(sorted_src, 4) ||
        !aligned(out, 16) || !aligned(out_sf, 4) || !aligned(workspace, 16))
      return MOE_ERR_INVALID_ARG;
    if (workspace_bytes <
        moe_route_expand_cast_fp8_workspace_bytes(num_tokens, num_experts, num_topk))
      return MOE_ERR_INVALID_ARG;
  }
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  const bool fused_ok =
      num_tokens > 0 &&
      decode_fused_smem(num_tokens, num_experts, num_topk, hidden, c.num_sms, nullptr, nullptr) > 0;
  const bool replicated_ok =
      num_tokens > 0 && decode_replicated_ok(num_tokens, num_experts, num_topk, hidden);
  const bool chained_ok =
      num_tokens > 0 && route_chain_ok(num_tokens, num_experts, num_topk, hidden, out, out_sf);
  if (mode == MOE_PATH_FUSED && !fused_ok && num_tokens > 0) return MOE_ERR_UNSUPPORTED;
  if (mode == MOE_PATH_REPLICATED && !replicated_ok && num_tokens > 0) return MOE_ERR_UNSUPPORTED;
  if (mode == MOE_PATH_CHAINED && !chained_ok && num_tokens > 0) return MOE_ERR_UNSUPPORTED;
  if (mode == MOE_PATH_AUTO && replicated_ok && num_tokens <= MOE_AUTO_REPLICATED_MAX_TOKENS)
    mode = MOE_PATH_REPLICATED;
  if (mode == MOE_PATH_CHAINED && chained_ok) {
    cudaError_t e = launch_route_chain(c, scores, num_tokens, num_experts, num_topk, x, hidden,
                                       topk_idx, topk_weights, counts, offsets, pos, sorted_src,
                                       out, out_sf,
                                       reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                                                  256),
                                       static_cast<unsigned*>(workspace) + kChainArrivalWord);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  if (mode == MOE_PATH_REPLICATED && replicated_ok) {
    cudaError_t e = launch_decode_replicated(c, scores, num_tokens, num_experts, num_topk, x,
                                             hidden, topk_idx, topk_weights, counts, offsets, pos,
                                             sorted_src, out, out_sf);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  if (mode == MOE_PATH_FUSED && fused_ok) {
    cudaError_t e = launch_decode_fused(c, scores, num_tokens, num_experts, num_topk, x, hidden,
                                        topk_idx, topk_weights, counts, offsets, pos, sorted_src,
                                        out, out_sf, static_cast<unsigned*>(workspace));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  moe_status_t r = moe_topk_gate(scores, num_tokens, num_experts, num_topk, topk_idx,
                                 topk_weights, MOE_WEIGHTS_SOFTMAX_TOPK, stream);
  if (r != MOE_OK) return r;
  void* route_ws = num_tokens > 0 ? static_cast<uint8_t*>(workspace) + 256 : nullptr;
  r = moe_route_map(topk_idx, num_tokens, num_experts, num_topk, counts, offsets, pos, sorted_src,
                    route_ws, num_tokens > 0 ? workspace_bytes - 256 : 0, stream);
  if (r != MOE_OK) return r;
  return moe_expand_cast_fp8(x, num_tokens, hidden, num_topk, pos, num_tokens * num_topk, out,
                             out_sf, group, stream);
}

moe_status_t moe_debug_set(int32_t key, int64_t value) {
  if (key == MOE_DEBUG_WAIT_TIMEOUT_NS) {
    if (value < 1000 || value > (int64_t)60 * 1000000000) return MOE_ERR_INVALID_ARG;
    g_decode_timeout_ns.store(value);
    return MOE_OK;
  }
  if (key == MOE_DEBUG_SKIP_ROUTE_SIGNAL) {
    g_decode_skip_signal.store(value != 0 ? 1 : 0);
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status_t moe_debug_cvt(int32_t format, const float* in, uint8_t* out, int64_t n,
                           void* stream) {
  if (format != MOE_DEBUG_CVT_E4M3 && format != MOE_DEBUG_CVT_E2M1) return MOE_ERR_INVALID_ARG;
  if (n < 0 || n % 4 != 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!in || !out || !aligned(in, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_debug_cvt(c, format, in, out, n);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_peak_copy(const void* src, void* dst, size_t bytes, void* stream) {
  if (bytes == 0) return MOE_OK;
  if (!src || !dst || bytes % 16 != 0 || !aligned(src, 16) || !aligned(dst, 16))
    return MOE_ERR_INVALID_ARG;
  LaunchCtx c;
  moe_status_t s = context(stream, &c);
  if (s != MOE_OK) return s;
  cudaError_t e = launch_peak_copy(c, src, dst, bytes);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

moe_status_t moe_get_device_status(void* stream, uint32_t* error_bits) {
  if (error_bits) *error_bits = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned bits = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&bits, g_device_error, sizeof bits);
  if (e == cudaSuccess && bits != 0) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e);
  if (error_bits) *error_bits = bits;
  return bits ? MOE_ERR_DEVICE : MOE_OK;
}

}  // extern "C"
