// route_noalloc.cu -- moe_route_noalloc: the routing step for callers that
// cannot allocate device memory.
//
// moe_route needs a caller-provided workspace (the per-chunk expert
// histograms of the counting sort). Some callers have no way to provide one:
// a plugin inside a host framework that owns all device memory and exposes no
// allocator to it, or a latency-critical loop where cudaMalloc is forbidden
// because it can synchronise the whole device. For them this entry point keeps
// the scratch in a fixed array compiled into the library, so a call needs only
// the inputs and outputs.
//
// The array is 4 MiB (1,048,576 int32), and every GPU that loads the library
// holds it until the process exits. It is enough for ceil(T/8) * E <= 1,048,576
// (e.g. T = 65536 tokens at E = 128, or T = 32768 at E = 256); larger shapes are
// rejected with MOE_ERR_WORKSPACE before anything is launched.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kRouteScratchInts = size_t(1) << 20;

// Routing scratch shared by every moe_route_noalloc call on a device. The
// kernels overwrite every element they read before reading it (each chunk's
// histogram row is written in full, zeros included), so nothing has to be
// cleared between calls.
__device__ __align__(256) int32_t g_route_scratch[kRouteScratchInts];

// In host code g_route_scratch names a host-side stand-in, not device memory.
// The device address is looked up on every call, for the device current on
// the calling thread: a cached address would go stale if the device were
// reset (or its primary context recreated) while the library stays loaded,
// and a per-call lookup needs no shared state between host threads. The
// first lookup on a device also loads the library's device code there.
moe_status route_scratch(int32_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
  *out = static_cast<int32_t*>(p);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const void* x, const void* w_router, const float* bias, int dtype,
                                        int T, int d, int E, int k, float* logits, int flags,
                                        int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
                                        int32_t* dest_row, int32_t* src_row, void* stream) {
  if (T < 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (moe::route_workspace_bytes(T, E) > moe::kRouteScratchInts * sizeof(int32_t)) return MOE_ERR_WORKSPACE;
  int32_t* scratch = nullptr;
  const moe_status st = moe::route_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe_route(x, w_router, bias, dtype, T, d, E, k, logits, flags, topk_idx, gates, counts, offsets,
                   dest_row, src_row, scratch, moe::kRouteScratchInts * sizeof(int32_t), stream);
}
