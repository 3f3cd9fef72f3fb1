// kernels.h -- internal host-side launchers of libmoe (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

namespace tc {
int sm_count();  // SMs of the current device (cached on first use)
}

// ------------------------------------------------------------- routing
constexpr int kTokensPerChunk = 8;  // tokens per routing chunk (one warp)
int route_num_chunks(int T);
size_t route_workspace_bytes(int T, int E);
cudaError_t launch_route_meta(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* gates, int32_t* counts, int32_t* offsets, int32_t* dest_row,
                              int32_t* src_row, int32_t* hist, cudaStream_t st);

// combine backward writing the MXFP8 row quantisation of dy_perm (bf16 only;
// scales as scale chunks grouped by per-expert 128-row tiles)
cudaError_t launch_combine_bwd_quant(const void* dy, const void* y_perm, const float* gates,
                                     const int32_t* dest_row, const int32_t* topk_idx, const int32_t* offsets,
                                     int Tn, int d, int k, int E, uint8_t* q, uint8_t* qsc, void* dy_perm,
                                     float* dgates, cudaStream_t st);

// ------------------------------------------------------ routing statistics
size_t route_stats_workspace_bytes(int T, int E);
cudaError_t launch_route_stats(const float* logits, const int32_t* counts, int T, int E, int k, float* probs_mean,
                               float* stats, float* partial, cudaStream_t st);

// ------------------------------------------------ permute / combine / router bwd
template <typename T>
cudaError_t launch_permute(const void* x, int Tn, int d, int k, const int32_t* dest_row, void* x_perm,
                           cudaStream_t st);
template <typename T>
cudaError_t launch_combine_fwd(const void* y_perm, const float* gates, const int32_t* dest_row, int Tn,
                               int d, int k, void* y, cudaStream_t st);
template <typename T>
cudaError_t launch_combine_bwd(const void* dy, const void* y_perm, const float* gates,
                               const int32_t* dest_row, int Tn, int d, int k, void* dy_perm,
                               float* dgates, cudaStream_t st);
template <typename T>
cudaError_t launch_permute_bwd(const void* dx_perm, int Tn, int d, int E, int k,
                               const int32_t* dest_row, const int32_t* topk_idx, const float* dlogits,
                               const void* w_r, void* dx, cudaStream_t st);
template <typename T>
cudaError_t launch_route_bwd(const float* dgates, const float* gates, const int32_t* topk_idx,
                             const int32_t* offsets, const int32_t* src_row, const void* x,
                             int Tn, int d, int E, int k, float* dlogits, float* dw_r,
                             cudaStream_t st);

// ------------------------------------------------------ CUDA-core grouped GEMM
struct SimtGemm {
  const void* A;
  long sAm, sAk;
  const void* B0;
  const void* B1;
  long sBk, sBn, sBe;
  int kSplit, nSplit;
  void* C0;
  void* C1;
  long sCm, sCn, sCe;
  int cSplit;
  const float* col_bias;
  const int32_t* offsets;  // nullptr: one group of M rows (row-ragged mode only)
  int E;
  int M, N, K;
  int kragged;
};
template <typename TA, typename TB, typename TC>
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t st);
template <typename T>
cudaError_t launch_swiglu_fwd(const void* h, long rows, int f, void* a, cudaStream_t st);
template <typename T>
cudaError_t launch_swiglu_bwd(const void* da, const void* h, long rows, int f, void* dh, cudaStream_t st);

// ------------------------------------------- tcgen05 grouped GEMMs (bf16)
// src_row (optional): the dispatch is fused into GEMM1 and its wgrad; x_perm
// then points at x [T][d] and row r of the dispatched matrix is x[src_row[r] / gk].
cudaError_t tc_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd,
                       const int32_t* offsets, int R, int E, int d, int f, void* h, void* a, void* y,
                       cudaStream_t st, const int32_t* src_row = nullptr, int gk = 1, int T = 0);
cudaError_t tc_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* dh, cudaStream_t st,
                       const int32_t* src_row = nullptr, int gk = 1, int T = 0);

// ------------------------------------------------------------------ MXFP8
// Where a row quantiser puts the scale byte of block b of row r:
//   kScalesPlain  sc[r][K/32] (public layout)
//   kScalesChunk  scale chunks (mxfp8_common.cuh), group r / 128 (weights)
//   kScalesTiles  scale chunks, group = the row's per-expert 128-row tile
//                 (offsets: [E+1] expert offsets; GEMM row operands)
enum ScaleLayout { kScalesPlain = 0, kScalesChunk = 1, kScalesTiles = 2 };
cudaError_t launch_mxfp8_quant_rows(const void* src, long rows, long K, uint8_t* q, uint8_t* sc, cudaStream_t st,
                                    int layout = kScalesPlain, const int32_t* offsets = nullptr, int E = 0);
// packed: scales as scale chunks (GEMM operand layout); otherwise one byte per
// block, [blocks][C] (public layout).
cudaError_t launch_mxfp8_quant_cols(const void* src, int rows, int C, const int32_t* seg, int nseg,
                                    uint8_t* q, uint8_t* sc, cudaStream_t st, bool packed = false);
// A weight [rows][C] (rows and C multiples of 128) quantised along its
// columns (qc, sc_c: the packed quant_cols layout) and along its rows (qr,
// sc_r: kScalesChunk) from one read.
cudaError_t launch_mxfp8_quant_dual(const void* src, long rows, int C, uint8_t* qc, uint8_t* sc_c, uint8_t* qr,
                                    uint8_t* sc_r, cudaStream_t st);
// Dispatch with the row quantisation fused: q [T*k][d], sc as scale chunks
// grouped by per-expert 128-row tiles; the bf16 x_perm too when given.
cudaError_t launch_permute_quant(const void* x, int T, int d, int k, int E, const int32_t* dest_row,
                                 const int32_t* topk_idx, const int32_t* offsets, uint8_t* q, uint8_t* sc,
                                 void* x_perm, cudaStream_t st);

// Experts by row count, largest first (ties by index), into order [E]; E <= 1024.
// Weight-gradient kernel choice: 0 single-CTA tiles, 1 CTA pairs (process-wide).
void set_cta_pairs(int on);
void set_mx_cta_pairs(int on);
cudaError_t launch_expert_order(const int32_t* offsets, int E, int32_t* order, cudaStream_t st);

cudaError_t tc_router_logits(const void* x, const void* w_r, const float* bias, int T, int d, int E,
                             float* logits, cudaStream_t st);

// ------------------------------------------- MXFP8 grouped GEMMs (bf16 in/out)
size_t mx_fwd_workspace(long R, int E, int d, int f);
size_t mx_bwd_workspace(long R, int E, int d, int f);
// a_cols (optional): GEMM1's epilogue also writes A quantised along the
// experts' rows (codes [R][f], then the scale chunks; mx_col_operand_bytes).
size_t mx_col_operand_bytes(long R, int E, int K);
cudaError_t mx_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd, const int32_t* offsets,
                       int R, int E, int d, int f, void* h, void* a, void* y, void* ws, cudaStream_t st,
                       const uint8_t* xq_codes = nullptr, const uint8_t* xq_scales = nullptr,
                       const void* wq = nullptr, uint8_t* a_cols = nullptr);
// dyq_codes/dyq_scales (optional): dy_perm's rows already quantised by the
// combine backward.
cudaError_t mx_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* ws, cudaStream_t st,
                       const uint8_t* dyq_codes = nullptr, const uint8_t* dyq_scales = nullptr,
                       const void* wq = nullptr, const uint8_t* a_cols = nullptr);
// The weights quantised once per update in both K layouts (wq: mx_weights_bytes).
size_t mx_weights_bytes(int E, int d, int f);
cudaError_t mx_prepare_weights(const void* wg, const void* wu, const void* wd, int E, int d, int f, void* wq,
                               cudaStream_t st);

}  // namespace moe
