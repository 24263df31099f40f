// route_map_noalloc.cu -- moe_route_map for callers that cannot allocate
// device memory.
//
// Some callers own every byte of device memory themselves and may not call
// cudaMalloc (or any allocator) while they run: inference-engine plugins whose
// host framework hands out all buffers from its own arena, and runtimes that
// fix their memory budget at start-up.  Such a caller can pass inputs and
// outputs but has no way to provide moe_route_map's workspace.  This entry
// point runs the same route-map kernels with their per-chunk histogram in a
// fixed file-scope device array instead.
//
// The array is a __device__ variable, so every GPU that loads this library
// holds it (kRouteScratchBytes) until the process exits, whether or not the
// entry point is ever called.  Host code must not hand the array's name to a
// kernel: on the host that name is only a stand-in, not a device address.  The
// device address is looked up with cudaGetSymbolAddress once per device, on
// the first call made while that device is current.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

// 1 MiB: the histogram is one row of E int32 per chunk, and there are at most
// 128 chunks until a chunk reaches 512 tokens, so every problem with
// T <= 65536 fits (any E), and larger ones while ceil(T/512) * E <= 2^18.
constexpr size_t kRouteScratchBytes = MOE_ROUTE_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  void* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_map_noalloc(const int32_t* topk_idx, int64_t num_tokens,
                                               int32_t num_experts, int32_t num_topk,
                                               int32_t* counts, int32_t* offsets, int32_t* pos,
                                               int32_t* sorted_src, void* stream) {
  if (num_tokens < 0 || num_experts < 1 || num_experts > MOE_MAX_EXPERTS || num_topk < 1 ||
      num_topk > MOE_MAX_TOPK || num_topk > num_experts)
    return MOE_ERR_INVALID_ARG;
  if (num_tokens * (int64_t)num_topk >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return moe_route_map(topk_idx, 0, num_experts, num_topk, counts, offsets,
                                            pos, sorted_src, nullptr, 0, stream);
  if (!topk_idx || !counts || !offsets || !pos || !sorted_src) return MOE_ERR_INVALID_ARG;
  // the same alignment rule as moe_route_map: every array is int32
  const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
  if (misaligned(topk_idx) || misaligned(counts) || misaligned(offsets) || misaligned(pos) ||
      misaligned(sorted_src))
    return MOE_ERR_INVALID_ARG;
  if (moe_route_map_workspace_bytes(num_tokens, num_experts, num_topk) > kRouteScratchBytes)
    return MOE_ERR_UNSUPPORTED;  // beyond the static scratch: use moe_route_map

  // the library's launch context: SM count and the device error word (itself
  // a __device__ variable, so nothing is allocated here either)
  LaunchCtx c;
  moe_status_t st = context(stream, &c);
  if (st != MOE_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  ScratchSlot& s = g_slots[dev];
  std::call_once(s.once, [&s]() {
    // runs with `dev` current: this is that device's address of the array
    s.status = cudaGetSymbolAddress(&s.ptr, g_route_scratch);
  });
  if (s.status != cudaSuccess) return cuda_fail(s.status);
  if (s.ptr == nullptr) return MOE_ERR_CUDA;

  const int64_t chunks = route_num_chunks(num_tokens);
  // every histogram entry the kernels read is written first in the same call,
  // so the scratch needs no clearing between calls
  e = launch_route_map(c, topk_idx, num_tokens, num_experts, num_topk, counts, offsets, pos,
                       sorted_src, static_cast<int32_t*>(s.ptr), chunks);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}
