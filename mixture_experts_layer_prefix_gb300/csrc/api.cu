// api.cu -- the extern "C" entry points of libmoe declared in include/moe.h:
// argument validation, workspace carving and dispatch to the kernels.
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "mxfp8_common.cuh"

namespace moe {

__device__ int g_moe_error_word;

// The error word's device address, cached per device ordinal (host threads
// may race to fill a slot; they store the same value, so relaxed atomics
// suffice). A device reset while the library stays loaded reloads its module:
// callers that reset a device must not keep launching through this library.
int* device_error_word() {
  static std::atomic<int*> ptrs[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  int* q = ptrs[dev].load(std::memory_order_relaxed);
  if (!q) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_error_word) != cudaSuccess) return nullptr;
    q = static_cast<int*>(p);
    ptrs[dev].store(q, std::memory_order_relaxed);
  }
  return q;
}

static std::atomic<unsigned long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

// Launch-timing recorder (instrumentation): while armed, each launch records
// one event on its stream just before it; moe_timing_finish records the
// closing event. Event i to event i+1 then brackets launch i when the
// launches ran in order on one stream.
namespace {
constexpr int kMaxTimed = 256;
struct LaunchTimer {
  std::mutex mu;
  std::atomic<int> armed{0};  // launches still to record
  int n = 0;                  // launches recorded
  int dev = -1;               // device the events belong to
  bool closed = false;
  cudaEvent_t ev[kMaxTimed + 1] = {};
  const char* names[kMaxTimed] = {};
};
LaunchTimer& launch_timer() {
  static LaunchTimer t;
  return t;
}
}  // namespace

void mark_launch(cudaStream_t st, const char* name) {
  LaunchTimer& t = launch_timer();
  if (t.armed.load(std::memory_order_relaxed) <= 0) return;
  std::lock_guard<std::mutex> g(t.mu);
  if (t.armed.load(std::memory_order_relaxed) <= 0 || t.n >= kMaxTimed) return;
  if (cudaEventRecord(t.ev[t.n], st) != cudaSuccess) return;
  t.names[t.n++] = name;
  t.armed.fetch_sub(1, std::memory_order_relaxed);
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }
inline size_t elem_bytes(int dtype) { return dtype == MOE_F32 ? 4 : 2; }
inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

moe_status check_dims(int T, int d, int E, int k) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (k > 8 || E > 1024 || d % 64 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_dtype(int dtype) {
  return (dtype == MOE_F32 || dtype == MOE_BF16 || dtype == MOE_MXFP8) ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// Activations and weights are bf16 in memory on the MXFP8 path too; only the
// expert GEMMs quantise their operands.
inline int storage(int dtype) { return dtype == MOE_MXFP8 ? MOE_BF16 : dtype; }

#define MOE_TRY(expr)                    \
  do {                                   \
    moe_status s_ = (expr);              \
    if (s_ != MOE_OK) return s_;         \
  } while (0)

#define MOE_NEED(p)                                   \
  do {                                                \
    if ((p) == nullptr) return MOE_ERR_INVALID_ARG;   \
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;      \
  } while (0)

// Workspace of the backward GEMM chain: dh [R][2f], plus dA [R][f] on the
// fp32 path (the bf16 path fuses the SwiGLU backward into the dA GEMM), or the
// weight gradients' expert order [E] after dh on the bf16 path.
size_t mlp_bwd_ws(long R, int E, int f, int dtype) {
  const size_t dh = align256((size_t)R * 2 * f * elem_bytes(dtype));
  return dtype == MOE_F32 ? align256((size_t)R * f * elem_bytes(dtype)) + dh : dh + align256((size_t)E * 4);
}

template <typename T>
moe_status mlp_fwd_simt(const void* x_perm, const void* wg, const void* wu, const void* wd,
                        const int32_t* offsets, int R, int E, int d, int f, void* h, void* a,
                        void* y, cudaStream_t st) {
  SimtGemm g{};
  g.A = x_perm; g.sAm = d; g.sAk = 1;
  g.B0 = wg; g.B1 = wu; g.sBk = f; g.sBn = 1; g.sBe = (long)d * f; g.kSplit = d; g.nSplit = f;
  g.C0 = h; g.C1 = h; g.sCm = 2L * f; g.sCn = 1; g.cSplit = 2 * f;
  g.offsets = offsets; g.E = E; g.M = R; g.N = 2 * f; g.K = d;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g, st)));
  MOE_CUDA_TRY(launch_swiglu_fwd<T>(h, R, f, a, st));
  SimtGemm g2{};
  g2.A = a; g2.sAm = f; g2.sAk = 1;
  g2.B0 = wd; g2.B1 = wd; g2.sBk = d; g2.sBn = 1; g2.sBe = (long)f * d; g2.kSplit = f; g2.nSplit = d;
  g2.C0 = y; g2.C1 = y; g2.sCm = d; g2.sCn = 1; g2.cSplit = d;
  g2.offsets = offsets; g2.E = E; g2.M = R; g2.N = d; g2.K = f;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g2, st)));
  return MOE_OK;
}

template <typename T>
moe_status mlp_bwd_simt(const void* dy_perm, const void* x_perm, const void* h, const void* a,
                        const void* wg, const void* wu, const void* wd, const int32_t* offsets,
                        int R, int E, int d, int f, void* dx_perm, void* dwg, void* dwu, void* dwd,
                        void* ws, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  void* da = w;
  void* dh = w + align256((size_t)R * f * sizeof(T));
  // dA = dY . Wd^T
  SimtGemm g{};
  g.A = dy_perm; g.sAm = d; g.sAk = 1;
  g.B0 = wd; g.B1 = wd; g.sBk = 1; g.sBn = d; g.sBe = (long)f * d; g.kSplit = d; g.nSplit = f;
  g.C0 = da; g.C1 = da; g.sCm = f; g.sCn = 1; g.cSplit = f;
  g.offsets = offsets; g.E = E; g.M = R; g.N = f; g.K = d;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g, st)));
  MOE_CUDA_TRY(launch_swiglu_bwd<T>(da, h, R, f, dh, st));
  // dx_perm = dh_g . Wg^T + dh_u . Wu^T
  SimtGemm g2{};
  g2.A = dh; g2.sAm = 2L * f; g2.sAk = 1;
  g2.B0 = wg; g2.B1 = wu; g2.sBk = 1; g2.sBn = f; g2.sBe = (long)d * f; g2.kSplit = f; g2.nSplit = d;
  g2.C0 = dx_perm; g2.C1 = dx_perm; g2.sCm = d; g2.sCn = 1; g2.cSplit = d;
  g2.offsets = offsets; g2.E = E; g2.M = R; g2.N = d; g2.K = 2 * f;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g2, st)));
  // dWd[e] = A_e^T dY_e
  SimtGemm g3{};
  g3.A = a; g3.sAm = 1; g3.sAk = f;
  g3.B0 = dy_perm; g3.B1 = dy_perm; g3.sBk = d; g3.sBn = 1; g3.sBe = 0; g3.kSplit = 1 << 30; g3.nSplit = d;
  g3.C0 = dwd; g3.C1 = dwd; g3.sCe = (long)f * d; g3.sCm = d; g3.sCn = 1; g3.cSplit = d;
  g3.offsets = offsets; g3.E = E; g3.M = f; g3.N = d; g3.kragged = 1;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g3, st)));
  // [dWg | dWu][e] = x_perm_e^T dh_e
  SimtGemm g4{};
  g4.A = x_perm; g4.sAm = 1; g4.sAk = d;
  g4.B0 = dh; g4.B1 = dh; g4.sBk = 2L * f; g4.sBn = 1; g4.sBe = 0; g4.kSplit = 1 << 30; g4.nSplit = 2 * f;
  g4.C0 = dwg; g4.C1 = dwu; g4.sCe = (long)d * f; g4.sCm = f; g4.sCn = 1; g4.cSplit = f;
  g4.offsets = offsets; g4.E = E; g4.M = d; g4.N = 2 * f; g4.kragged = 1;
  MOE_CUDA_TRY((launch_simt_gemm<T, T, T>(g4, st)));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(int T, int d, int E, int k, int f, int dtype) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || f <= 0) return 0;
  const long R = (long)T * k;
  size_t route = align256(route_workspace_bytes(T, E));
  size_t bwd = mlp_bwd_ws(R, E, f, dtype == MOE_F32 ? MOE_F32 : MOE_BF16);
  size_t ws = route > bwd ? route : bwd;
  const size_t stats = align256(route_stats_workspace_bytes(T, E));
  ws = ws > stats ? ws : stats;
  if (dtype == MOE_MXFP8) {
    const size_t mf = mx_fwd_workspace(R, E, d, f), mb = mx_bwd_workspace(R, E, d, f);
    ws = ws > mf ? ws : mf;
    ws = ws > mb ? ws : mb;
  }
  return ws;
}

moe_status moe_route(const void* x, const void* w_router, const float* bias, int dtype, int T, int d,
                     int E, int k, float* logits, int flags, int32_t* topk_idx, float* gates,
                     int32_t* counts, int32_t* offsets, int32_t* dest_row, int32_t* src_row,
                     void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  MOE_NEED(counts); MOE_NEED(offsets);
  if (T > 0) {
    MOE_NEED(logits); MOE_NEED(topk_idx); MOE_NEED(gates); MOE_NEED(dest_row); MOE_NEED(src_row);
  }
  if (workspace_bytes < route_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
  if (route_workspace_bytes(T, E) > 0) MOE_NEED(workspace);
  cudaStream_t st = S(stream);
  if (!(flags & MOE_ROUTE_LOGITS_IN) && T > 0) {
    MOE_NEED(x); MOE_NEED(w_router);
    if (bias && !aligned16(bias)) return MOE_ERR_ALIGNMENT;
    SimtGemm g{};
    g.A = x; g.sAm = d; g.sAk = 1;
    g.B0 = w_router; g.B1 = w_router; g.sBk = 1; g.sBn = d; g.sBe = 0; g.kSplit = d; g.nSplit = E;
    g.C0 = logits; g.C1 = logits; g.sCm = E; g.sCn = 1; g.cSplit = E;
    g.col_bias = bias; g.offsets = nullptr; g.E = 1; g.M = T; g.N = E; g.K = d;
    if (dtype == MOE_F32) MOE_CUDA_TRY((launch_simt_gemm<float, float, float>(g, st)));
    else MOE_CUDA_TRY(tc_router_logits(x, w_router, bias, T, d, E, logits, st));
  }
  MOE_CUDA_TRY(launch_route_meta(logits, T, E, k, topk_idx, gates, counts, offsets, dest_row, src_row,
                                 static_cast<int32_t*>(workspace), st));
  return MOE_OK;
}

moe_status moe_permute(const void* x, int dtype, int T, int d, int k, const int32_t* dest_row,
                       void* x_perm, void* stream) {
  MOE_TRY(check_dims(T, d, k, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  if (T == 0) return MOE_OK;
  MOE_NEED(x); MOE_NEED(dest_row); MOE_NEED(x_perm);
  if (dtype == MOE_F32) MOE_CUDA_TRY(launch_permute<float>(x, T, d, k, dest_row, x_perm, S(stream)));
  else MOE_CUDA_TRY(launch_permute<__nv_bfloat16>(x, T, d, k, dest_row, x_perm, S(stream)));
  return MOE_OK;
}

moe_status moe_permute_bwd(const void* dx_perm, int dtype, int T, int d, int E, int k,
                           const int32_t* dest_row, const int32_t* topk_idx, const float* dlogits,
                           const void* w_router, void* dx, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  if (T == 0) return MOE_OK;
  const int given = (topk_idx != nullptr) + (dlogits != nullptr) + (w_router != nullptr);
  if (given != 0 && given != 3) return MOE_ERR_INVALID_ARG;
  MOE_NEED(dx_perm); MOE_NEED(dest_row); MOE_NEED(dx);
  if (given == 3) { MOE_NEED(topk_idx); MOE_NEED(dlogits); MOE_NEED(w_router); }
  if (dtype == MOE_F32)
    MOE_CUDA_TRY(launch_permute_bwd<float>(dx_perm, T, d, E, k, dest_row, topk_idx, dlogits, w_router,
                                           dx, S(stream)));
  else
    MOE_CUDA_TRY(launch_permute_bwd<__nv_bfloat16>(dx_perm, T, d, E, k, dest_row, topk_idx, dlogits,
                                                   w_router, dx, S(stream)));
  return MOE_OK;
}

moe_status moe_combine_fwd(const void* y_perm, const float* gates, const int32_t* dest_row, int dtype,
                           int T, int d, int k, void* y, void* stream) {
  MOE_TRY(check_dims(T, d, k, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  if (T == 0) return MOE_OK;
  MOE_NEED(y_perm); MOE_NEED(gates); MOE_NEED(dest_row); MOE_NEED(y);
  if (dtype == MOE_F32)
    MOE_CUDA_TRY(launch_combine_fwd<float>(y_perm, gates, dest_row, T, d, k, y, S(stream)));
  else
    MOE_CUDA_TRY(launch_combine_fwd<__nv_bfloat16>(y_perm, gates, dest_row, T, d, k, y, S(stream)));
  return MOE_OK;
}

moe_status moe_combine_bwd(const void* dy, const void* y_perm, const float* gates,
                           const int32_t* dest_row, int dtype, int T, int d, int k, void* dy_perm,
                           float* dgates, void* stream) {
  MOE_TRY(check_dims(T, d, k, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  if (T == 0) return MOE_OK;
  MOE_NEED(dy); MOE_NEED(y_perm); MOE_NEED(gates); MOE_NEED(dest_row); MOE_NEED(dy_perm);
  MOE_NEED(dgates);
  if (dtype == MOE_F32)
    MOE_CUDA_TRY(launch_combine_bwd<float>(dy, y_perm, gates, dest_row, T, d, k, dy_perm, dgates,
                                           S(stream)));
  else
    MOE_CUDA_TRY(launch_combine_bwd<__nv_bfloat16>(dy, y_perm, gates, dest_row, T, d, k, dy_perm,
                                                   dgates, S(stream)));
  return MOE_OK;
}

moe_status moe_route_bwd(const float* dgates, const float* gates, const int32_t* topk_idx,
                         const int32_t* offsets, const int32_t* src_row, const void* x,
                         int dtype, int T, int d, int E, int k, float* dlogits, float* dw_router,
                         void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  MOE_TRY(check_dtype(dtype));
  dtype = storage(dtype);
  MOE_NEED(offsets); MOE_NEED(dw_router);
  if (T > 0) {
    MOE_NEED(dgates); MOE_NEED(gates); MOE_NEED(topk_idx); MOE_NEED(src_row); MOE_NEED(x);
    MOE_NEED(dlogits);
  }
  if (dtype == MOE_F32)
    MOE_CUDA_TRY(launch_route_bwd<float>(dgates, gates, topk_idx, offsets, src_row, x, T, d, E, k,
                                         dlogits, dw_router, S(stream)));
  else
    MOE_CUDA_TRY(launch_route_bwd<__nv_bfloat16>(dgates, gates, topk_idx, offsets, src_row, x, T,
                                                 d, E, k, dlogits, dw_router, S(stream)));
  return MOE_OK;
}

moe_status moe_grouped_mlp_fwd(const void* x_perm, const void* w_gate, const void* w_up,
                               const void* w_down, int dtype, const int32_t* offsets, int R, int E,
                               int d, int f, void* h_save, void* a_save, void* y_perm,
                               void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(check_dims(R, d, E, 1));
  MOE_TRY(check_dtype(dtype));
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (f % 64 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_gate); MOE_NEED(w_up); MOE_NEED(w_down); MOE_NEED(offsets);
  if (R == 0) return MOE_OK;
  MOE_NEED(x_perm); MOE_NEED(h_save); MOE_NEED(a_save); MOE_NEED(y_perm);
  if (dtype == MOE_MXFP8) {
    if (d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < mx_fwd_workspace(R, E, d, f)) return MOE_ERR_WORKSPACE;
    MOE_NEED(workspace);
    MOE_CUDA_TRY(mx_mlp_fwd(x_perm, w_gate, w_up, w_down, offsets, R, E, d, f, h_save, a_save, y_perm,
                            workspace, S(stream)));
    return MOE_OK;
  }
  if (dtype == MOE_F32)
    return mlp_fwd_simt<float>(x_perm, w_gate, w_up, w_down, offsets, R, E, d, f, h_save, a_save, y_perm,
                               S(stream));
  MOE_CUDA_TRY(tc_mlp_fwd(x_perm, w_gate, w_up, w_down, offsets, R, E, d, f, h_save, a_save, y_perm,
                          S(stream)));
  return MOE_OK;
}

moe_status moe_grouped_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h_save,
                               const void* a_save, const void* w_gate, const void* w_up,
                               const void* w_down, int dtype, const int32_t* offsets, int R, int E,
                               int d, int f, void* dx_perm, void* dw_gate, void* dw_up,
                               void* dw_down, void* workspace, size_t workspace_bytes,
                               void* stream) {
  MOE_TRY(check_dims(R, d, E, 1));
  MOE_TRY(check_dtype(dtype));
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (f % 64 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_gate); MOE_NEED(w_up); MOE_NEED(w_down); MOE_NEED(offsets);
  MOE_NEED(dw_gate); MOE_NEED(dw_up); MOE_NEED(dw_down);
  if (dtype == MOE_MXFP8) {
    if (d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < mx_bwd_workspace(R, E, d, f)) return MOE_ERR_WORKSPACE;
    if (R > 0) {
      MOE_NEED(dy_perm); MOE_NEED(x_perm); MOE_NEED(h_save); MOE_NEED(a_save); MOE_NEED(dx_perm);
    }
    MOE_NEED(workspace);
    MOE_CUDA_TRY(mx_mlp_bwd(dy_perm, x_perm, h_save, a_save, w_gate, w_up, w_down, offsets, R, E, d, f,
                            dx_perm, dw_gate, dw_up, dw_down, workspace, S(stream)));
    return MOE_OK;
  }
  if (workspace_bytes < mlp_bwd_ws(R, E, f, dtype)) return MOE_ERR_WORKSPACE;
  if (R > 0) {
    MOE_NEED(dy_perm); MOE_NEED(x_perm); MOE_NEED(h_save); MOE_NEED(a_save); MOE_NEED(dx_perm);
  }
  if (R > 0 || dtype != MOE_F32) MOE_NEED(workspace);  // bf16: the expert order table lives there
  if (dtype == MOE_F32)
    return mlp_bwd_simt<float>(dy_perm, x_perm, h_save, a_save, w_gate, w_up, w_down, offsets, R, E, d,
                               f, dx_perm, dw_gate, dw_up, dw_down, workspace, S(stream));
  MOE_CUDA_TRY(tc_mlp_bwd(dy_perm, x_perm, h_save, a_save, w_gate, w_up, w_down, offsets, R, E, d, f,
                          dx_perm, dw_gate, dw_up, dw_down, workspace, S(stream)));
  return MOE_OK;
}

moe_status moe_permute_mxfp8(const void* x, int T, int d, int k, int E, const int32_t* dest_row,
                             const int32_t* topk_idx, const int32_t* offsets, uint8_t* x_codes, uint8_t* x_scales,
                             void* x_perm, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  if (d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_NEED(x); MOE_NEED(dest_row); MOE_NEED(topk_idx); MOE_NEED(offsets); MOE_NEED(x_codes); MOE_NEED(x_scales);
  if (x_perm && !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
  MOE_CUDA_TRY(launch_permute_quant(x, T, d, k, E, dest_row, topk_idx, offsets, x_codes, x_scales, x_perm,
                                    S(stream)));
  return MOE_OK;
}

moe_status moe_combine_bwd_mxfp8(const void* dy, const void* y_perm, const float* gates, const int32_t* dest_row,
                                 const int32_t* topk_idx, const int32_t* offsets, int T, int d, int k, int E,
                                 uint8_t* dy_codes, uint8_t* dy_scales, void* dy_perm, float* dgates, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  if (d % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  MOE_NEED(dy); MOE_NEED(y_perm); MOE_NEED(gates); MOE_NEED(dest_row); MOE_NEED(topk_idx); MOE_NEED(offsets);
  MOE_NEED(dy_codes); MOE_NEED(dy_scales); MOE_NEED(dgates);
  if (dy_perm && !aligned16(dy_perm)) return MOE_ERR_ALIGNMENT;
  MOE_CUDA_TRY(launch_combine_bwd_quant(dy, y_perm, gates, dest_row, topk_idx, offsets, T, d, k, E, dy_codes,
                                        dy_scales, dy_perm, dgates, S(stream)));
  return MOE_OK;
}

size_t moe_mxfp8_row_scales_size(int R, int E, int K) {
  if (R < 0 || E <= 0 || K <= 0 || K % 128 != 0) return 0;
  return (size_t)mx_row_tiles(R, E) * 4 * K;
}

size_t moe_mxfp8_weights_size(int E, int d, int f) {
  if (E <= 0 || d <= 0 || f <= 0) return 0;
  return mx_weights_bytes(E, d, f);
}

moe_status moe_mxfp8_prepare_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int d, int f,
                                     void* wq, size_t wq_bytes, void* stream) {
  if (E <= 0 || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_gate); MOE_NEED(w_up); MOE_NEED(w_down); MOE_NEED(wq);
  if (wq_bytes < mx_weights_bytes(E, d, f)) return MOE_ERR_WORKSPACE;
  MOE_CUDA_TRY(mx_prepare_weights(w_gate, w_up, w_down, E, d, f, wq, S(stream)));
  return MOE_OK;
}

moe_status moe_use_cta_pairs(int enable) {
  set_cta_pairs(enable);
  set_mx_cta_pairs(enable);
  return MOE_OK;
}

size_t moe_mxfp8_col_operand_size(int R, int E, int K) {
  if (R < 0 || E <= 0 || K <= 0 || K % 128 != 0) return 0;
  return mx_col_operand_bytes(R, E, K);
}

moe_status moe_mxfp8_mlp_fwd(const uint8_t* x_codes, const uint8_t* x_scales, const void* wq, const int32_t* offsets,
                             int R, int E, int d, int f, void* h_save, void* a_save, void* y_perm, uint8_t* a_cols,
                             void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(check_dims(R, d, E, 1));
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(wq); MOE_NEED(offsets);
  if (R == 0) return MOE_OK;
  MOE_NEED(x_codes); MOE_NEED(x_scales); MOE_NEED(h_save); MOE_NEED(a_save); MOE_NEED(y_perm);
  if (workspace_bytes < mx_fwd_workspace(R, E, d, f)) return MOE_ERR_WORKSPACE;
  MOE_NEED(workspace);
  if (a_cols && !aligned16(a_cols)) return MOE_ERR_ALIGNMENT;
  MOE_CUDA_TRY(mx_mlp_fwd(nullptr, nullptr, nullptr, nullptr, offsets, R, E, d, f, h_save, a_save, y_perm, workspace,
                          S(stream), x_codes, x_scales, wq, a_cols));
  return MOE_OK;
}

moe_status moe_mxfp8_mlp_bwd(const uint8_t* dy_codes, const uint8_t* dy_scales, const void* dy_perm,
                             const void* x_perm, const void* h_save, const void* a_save, const uint8_t* a_cols,
                             const void* wq, const int32_t* offsets, int R, int E, int d, int f, void* dx_perm,
                             void* dw_gate, void* dw_up, void* dw_down, void* workspace, size_t workspace_bytes,
                             void* stream) {
  MOE_TRY(check_dims(R, d, E, 1));
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(wq); MOE_NEED(offsets);
  MOE_NEED(dw_gate); MOE_NEED(dw_up); MOE_NEED(dw_down);
  if (workspace_bytes < mx_bwd_workspace(R, E, d, f)) return MOE_ERR_WORKSPACE;
  MOE_NEED(workspace);
  if (R > 0) {
    MOE_NEED(dy_codes); MOE_NEED(dy_scales); MOE_NEED(dy_perm); MOE_NEED(x_perm); MOE_NEED(h_save);
    MOE_NEED(a_save); MOE_NEED(dx_perm);
  }
  if (a_cols && !aligned16(a_cols)) return MOE_ERR_ALIGNMENT;
  MOE_CUDA_TRY(mx_mlp_bwd(dy_perm, x_perm, h_save, a_save, nullptr, nullptr, nullptr, offsets, R, E, d, f, dx_perm,
                          dw_gate, dw_up, dw_down, workspace, S(stream), dy_codes, dy_scales, wq, a_cols));
  return MOE_OK;
}

moe_status moe_route_stats(const float* logits, const int32_t* counts, int T, int E, int k, float* probs_mean,
                           float* stats, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(counts); MOE_NEED(probs_mean); MOE_NEED(stats);
  const size_t need = route_stats_workspace_bytes(T, E);
  if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
  if (T > 0) {
    MOE_NEED(logits); MOE_NEED(workspace);
  }
  MOE_CUDA_TRY(launch_route_stats(logits, counts, T, E, k, probs_mean, stats, static_cast<float*>(workspace),
                                  S(stream)));
  return MOE_OK;
}

moe_status moe_dispatch_mlp_fwd(const void* x, const int32_t* src_row, int T, int k, const void* w_gate,
                                const void* w_up, const void* w_down, int dtype, const int32_t* offsets, int E,
                                int d, int f, void* h_save, void* a_save, void* y_perm, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  MOE_TRY(check_dtype(dtype));
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (f % 64 != 0 || (long)T * k > 0x7FFFFFFFL) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_gate); MOE_NEED(w_up); MOE_NEED(w_down); MOE_NEED(offsets);
  if (T == 0) return MOE_OK;
  MOE_NEED(x); MOE_NEED(src_row); MOE_NEED(h_save); MOE_NEED(a_save); MOE_NEED(y_perm);
  MOE_CUDA_TRY(tc_mlp_fwd(x, w_gate, w_up, w_down, offsets, T * k, E, d, f, h_save, a_save, y_perm, S(stream),
                          src_row, k, T));
  return MOE_OK;
}

moe_status moe_dispatch_mlp_bwd(const void* dy_perm, const void* x, const int32_t* src_row, int T, int k,
                                const void* h_save, const void* a_save, const void* w_gate, const void* w_up,
                                const void* w_down, int dtype, const int32_t* offsets, int E, int d, int f,
                                void* dx_perm, void* dw_gate, void* dw_up, void* dw_down, void* workspace,
                                size_t workspace_bytes, void* stream) {
  MOE_TRY(check_dims(T, d, E, k));
  MOE_TRY(check_dtype(dtype));
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (f <= 0) return MOE_ERR_INVALID_ARG;
  if (f % 64 != 0 || (long)T * k > 0x7FFFFFFFL) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_gate); MOE_NEED(w_up); MOE_NEED(w_down); MOE_NEED(offsets);
  MOE_NEED(dw_gate); MOE_NEED(dw_up); MOE_NEED(dw_down);
  const int R = T * k;
  if (workspace_bytes < mlp_bwd_ws(R, E, f, dtype)) return MOE_ERR_WORKSPACE;
  MOE_NEED(workspace);  // the expert order table lives there even when R = 0
  if (R > 0) {
    MOE_NEED(dy_perm); MOE_NEED(x); MOE_NEED(src_row); MOE_NEED(h_save); MOE_NEED(a_save);
    MOE_NEED(dx_perm);
  }
  MOE_CUDA_TRY(tc_mlp_bwd(dy_perm, x, h_save, a_save, w_gate, w_up, w_down, offsets, R, E, d, f, dx_perm,
                          dw_gate, dw_up, dw_down, workspace, S(stream), src_row, k, T));
  return MOE_OK;
}

moe_status mxfp8_quantize(const void* src, int rows, int K, int axis, const int32_t* seg_offsets,
                          int nseg, uint8_t* dst_e4m3, uint8_t* dst_e8m0, void* stream) {
  if (rows < 0 || K <= 0 || (axis != 0 && axis != 1)) return MOE_ERR_INVALID_ARG;
  if (axis == 0 && K % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if (axis == 1 && (K % 8 != 0 || (seg_offsets && (nseg <= 0 || nseg > 4096)))) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_NEED(src); MOE_NEED(dst_e4m3); MOE_NEED(dst_e8m0);
  if (seg_offsets) MOE_NEED(seg_offsets);
  if (axis == 0)
    MOE_CUDA_TRY(launch_mxfp8_quant_rows(src, rows, K, dst_e4m3, dst_e8m0, S(stream)));
  else
    MOE_CUDA_TRY(launch_mxfp8_quant_cols(src, rows, K, seg_offsets, nseg, dst_e4m3, dst_e8m0, S(stream)));
  return MOE_OK;
}

moe_status moe_get_device_error(void* stream) {
  MOE_CUDA_TRY(cudaStreamSynchronize(S(stream)));
  int v = 0;
  MOE_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_moe_error_word, sizeof(int)));
  if (v != 0) {
    const int zero = 0;
    MOE_CUDA_TRY(cudaMemcpyToSymbol(g_moe_error_word, &zero, sizeof(int)));
  }
  return static_cast<moe_status>(v);
}

uint64_t moe_launch_count(void) { return (uint64_t)g_launches.load(std::memory_order_relaxed); }

moe_status moe_timing_arm(int n) {
  if (n <= 0 || n > kMaxTimed) return MOE_ERR_INVALID_ARG;
  LaunchTimer& t = launch_timer();
  std::lock_guard<std::mutex> g(t.mu);
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (t.dev != dev) {  // events are created on (and belong to) the current device
    if (t.dev >= 0) {
      int cur = dev;
      cudaSetDevice(t.dev);
      for (auto& e : t.ev) cudaEventDestroy(e);
      cudaSetDevice(cur);
    }
    t.dev = -1;
    for (auto& e : t.ev) MOE_CUDA_TRY(cudaEventCreate(&e));
    t.dev = dev;
  }
  t.n = 0;
  t.closed = false;
  t.armed.store(n, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status moe_timing_finish(void* stream) {
  LaunchTimer& t = launch_timer();
  std::lock_guard<std::mutex> g(t.mu);
  t.armed.store(0, std::memory_order_relaxed);
  if (t.dev < 0) return MOE_ERR_INVALID_ARG;
  MOE_CUDA_TRY(cudaEventRecord(t.ev[t.n], S(stream)));
  t.closed = true;
  return MOE_OK;
}

int moe_timing_read(float* ms, const char** names, int cap) {
  LaunchTimer& t = launch_timer();
  std::lock_guard<std::mutex> g(t.mu);
  if (!t.closed || ms == nullptr || cap < 0) return -1;
  if (cudaEventSynchronize(t.ev[t.n]) != cudaSuccess) return -1;
  const int n = t.n < cap ? t.n : cap;
  for (int i = 0; i < n; ++i) {
    if (cudaEventElapsedTime(&ms[i], t.ev[i], t.ev[i + 1]) != cudaSuccess) return -1;
    if (names) names[i] = t.names[i];
  }
  return n;
}

int moe_sm_count(void) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // extern "C"
