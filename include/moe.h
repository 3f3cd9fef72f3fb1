/*
 * moe.h -- C ABI of libmoe, the single-GPU Mixture-of-Experts layer
 * (forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * The operations follow "Introducing Olmo-core 3: open, scalable training
 * infrastructure for large MoE models" (page 1), section "Scaling and
 * optimizing MoE training": routing metadata is computed and kept on the GPU
 * so the host can enqueue work without waiting for a copy back; routed rows
 * are written directly into each expert's input buffer; one grouped GEMM runs
 * all experts' feed-forward computations; MXFP8 is supported for the expert
 * GEMMs. The layer math (softmax over E router logits, top-k, gates
 * renormalised to sum 1, SwiGLU experts, E4M3 elements with one E8M0 scale
 * per 32 along K) is the definition of the 8/128-expert top-4 benchmark
 * layer of that page's introduction.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Notation: T tokens, d hidden size, E experts, k experts per token,
 *    f expert FFN width, R = T*k routed rows.
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise. The
 *    caller owns and allocates every buffer, including the workspace; the
 *    library never allocates or frees memory and keeps no state besides one
 *    error word per device.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream): no host synchronisation, no
 *    device-to-host copy. Counts and offsets never leave the device.
 *  - Layouts are row-major: x [T][d]; w_router [E][d] (row e is expert e's
 *    router vector); w_gate, w_up [E][d][f]; w_down [E][f][d].
 *  - dtype: MOE_F32 (everything fp32) or MOE_BF16 (activations and weights
 *    bf16; router logits, gates and all accumulation fp32). MXFP8 expert
 *    GEMMs are requested with MOE_MXFP8 where a call says so.
 *  - Argument, shape and alignment errors are returned synchronously and
 *    nothing is launched. Requirements: T >= 0, 1 <= k <= 8, k <= E <= 1024,
 *    d and f multiples of 64, pointers 16-byte aligned.
 *  - Errors found on the device (an index out of range, a bounded wait that
 *    ran out) set the device error word; kernels then exit cleanly and never
 *    trap. moe_get_device_error() reads and clears it.
 *  - Identical inputs give bit-identical outputs (no floating-point atomics).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, k > E, ...        */
  MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported set (see above)    */
  MOE_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned               */
  MOE_ERR_WORKSPACE = 4,     /* workspace smaller than moe_workspace_size()    */
  MOE_ERR_CUDA = 5,          /* a CUDA runtime call failed                     */
  MOE_ERR_DEVICE_INDEX = 6,  /* device error word: index out of range          */
  MOE_ERR_TIMEOUT = 7,       /* device error word: a bounded wait ran out      */
  MOE_ERR_DEVICE_PAIR = 8    /* device error word: the two CTAs of a pair got
                                different TMEM columns (their GEMM is skipped) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_MXFP8 = 2 } moe_dtype;

/* Flags of moe_route. */
#define MOE_ROUTE_LOGITS_IN 1 /* skip the router GEMM: `logits` is an input */

/* Bytes of workspace that the calls below need for this shape (the maximum
   over all calls). A sizing helper: the pages have no counterpart. */
size_t moe_workspace_size(int T, int d, int E, int k, int f, int dtype);

/* Routing: router GEMM, softmax + top-k gates, per-expert counts, offsets and
   the row placement ("Scaling and optimizing MoE training": on-GPU routing
   metadata; rows placed directly into expert input buffers).
     logits[t][e] = bias[e] + sum_c x[t][c] * w_router[e][c]     (fp32 accum)
     topk_idx[t][0..k) = the k largest logits, ties to the smaller index,
                         ordered by (logit desc, index asc)
     gates[t][j]  = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max)
     counts[e]    = number of (t, j) with topk_idx[t][j] == e
     offsets[e]   = sum_{e' < e} counts[e'], offsets[E] = T*k  (unpadded)
     dest_row[t][j] = offsets[e] + #{t' < t routed to e}   (rows of one expert
                      in token order); src_row[dest_row[t][j]] = t*k + j
   x: [T][d] dtype; w_router: [E][d] dtype; bias: [E] fp32 or NULL (a constant
   per-expert logit bias, no gradient); logits: [T][E] fp32, written, or read
   when flags & MOE_ROUTE_LOGITS_IN (then x/w_router/bias are unused);
   topk_idx, dest_row: [T][k] int32; gates [T][k] fp32; counts [E];
   offsets [E+1]; src_row [T*k] int32. */
moe_status moe_route(const void* x, const void* w_router, const float* bias, int dtype, int T,
                     int d, int E, int k, float* logits, int flags, int32_t* topk_idx, float* gates,
                     int32_t* counts, int32_t* offsets, int32_t* dest_row, int32_t* src_row,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Dispatch ("Scaling and optimizing MoE training": row-wise expert
   parallelism writes the routed rows straight into the experts' input
   buffers; on one GPU those buffers are the contiguous expert segments of
   x_perm):  x_perm[dest_row[t][j]] = x[t]  (an exact copy).
   x: [T][d]; x_perm: [T*k][d]; both dtype. */
moe_status moe_permute(const void* x, int dtype, int T, int d, int k, const int32_t* dest_row,
                       void* x_perm, void* stream);

/* Backward of the dispatch above (same section), plus the router's share
   of dx when dlogits is given (the benchmark layer's backward -- page 1
   introduction, 8/128-expert top-4 study -- carries the gate gradient into
   the router and on to x):  dx[t] = sum_j dx_perm[dest_row[t][j]]
                 + sum_j dlogits[t][topk_idx[t][j]] * w_router[topk_idx[t][j]]
   (fp32 sums in j order, one rounding to dtype). topk_idx, dlogits and
   w_router are either all NULL (no router term) or all given. */
moe_status moe_permute_bwd(const void* dx_perm, int dtype, int T, int d, int E, int k,
                           const int32_t* dest_row, const int32_t* topk_idx, const float* dlogits,
                           const void* w_router, void* dx, void* stream);

/* Combine: the inverse of the dispatch ("Scaling and optimizing MoE
   training": each routed row's expert output returns from its expert's buffer
   to its token), weighted by the renormalised gates of the benchmark layer
   (page 1 introduction):
     y[t] = sum_j gates[t][j] * y_perm[dest_row[t][j]]
   (fp32 sum in j order, rounded once to dtype). y_perm [T*k][d]; y [T][d]. */
moe_status moe_combine_fwd(const void* y_perm, const float* gates, const int32_t* dest_row,
                           int dtype, int T, int d, int k, void* y, void* stream);

/* Backward of the combine (same section and layer definition as
   moe_combine_fwd):
     dy_perm[dest_row[t][j]] = gates[t][j] * dy[t]            (dtype)
     dgates[t][j] = sum_c dy[t][c] * y_perm[dest_row[t][j]][c] (fp32) */
moe_status moe_combine_bwd(const void* dy, const void* y_perm, const float* gates,
                           const int32_t* dest_row, int dtype, int T, int d, int k, void* dy_perm,
                           float* dgates, void* stream);

/* Router backward: the gradient through moe_route's gates (softmax over
   the selected logits, the benchmark layer's renormalised top-k gates, page 1
   introduction) and its router GEMM ("Scaling and optimizing MoE training":
   routing tokens to experts). The router's share of dx is added by
   moe_permute_bwd, which writes dx once.
     dlogits[t][i] = g_i * (dg_i - sum_j g_j dg_j) for i in top-k, 0 otherwise
     dw_router[e][c] = sum over rows r of expert e of dlogits[t(r)][e] * x[t(r)][c]
   with t(r) = src_row[r] / k (fp32 sum in row order, i.e. ascending token).
   dlogits [T][E] fp32; dw_router [E][d] fp32; x [T][d] dtype, the layer's
   input (each token's row is read once per selected expert, from L2 after
   the first). */
moe_status moe_route_bwd(const float* dgates, const float* gates, const int32_t* topk_idx,
                         const int32_t* offsets, const int32_t* src_row, const void* x,
                         int dtype, int T, int d, int E, int k, float* dlogits, float* dw_router,
                         void* stream);

/* Routing load statistics, kept alongside the routing metadata (the pages
   name an unbalanced token distribution as the risk of expert routing but
   give no formula; these are the plainest statistics):
     probs_mean[e] = (1/T) sum_t softmax(logits[t])_e   (softmax over all E)
     stats[0] = E * sum_e (counts[e] / (T k)) * probs_mean[e]   (1 if balanced)
     stats[1] = max_e counts[e] * E / (T k)   (largest load over the mean)
     stats[2] = number of experts with counts[e] == 0
     stats[3] = population std of counts / mean count
   logits [T][E] fp32 and counts [E] int32 as moe_route left them; probs_mean
   [E] and stats [4] fp32, written on the device (no host sync). Every sum runs
   in a fixed order (bit-reproducible). workspace: at least
   ceil(T / 256) * E * 4 bytes (moe_workspace_size is always enough). E <= 1024. */
moe_status moe_route_stats(const float* logits, const int32_t* counts, int T, int E, int k, float* probs_mean,
                           float* stats, void* workspace, size_t workspace_bytes, void* stream);

/* Grouped SwiGLU expert MLP, forward, all experts in one launch per GEMM
   ("Scaling and optimizing MoE training": grouped GEMM). For every expert e
   and row r in [offsets[e], offsets[e+1]):
     h_g = x_perm[r] . w_gate[e],  h_u = x_perm[r] . w_up[e]   (fp32 accum)
     a   = silu(h_g) * h_u,  y_perm[r] = a . w_down[e]
   Outputs, saved for the backward: h_save [R][2f] = (h_g | h_u) and
   a_save [R][f], plus y_perm [R][d]; all dtype. offsets: [E+1] device
   int32 from moe_route; R = T*k is the row count the caller allocated. */
moe_status moe_grouped_mlp_fwd(const void* x_perm, const void* w_gate, const void* w_up,
                               const void* w_down, int dtype, const int32_t* offsets, int R, int E,
                               int d, int f, void* h_save, void* a_save, void* y_perm,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Grouped SwiGLU expert MLP, backward, again one launch per GEMM for all
   experts ("Scaling and optimizing MoE training": grouped GEMM). With
   dh = (dh_g | dh_u):
     da = dy_perm[r] . w_down[e]^T;  dh_g = da * h_u * silu'(h_g);
     dh_u = da * silu(h_g);  dx_perm[r] = dh_g . w_gate[e]^T + dh_u . w_up[e]^T
     dw_down[e] = sum_r a_save[r]^T dy_perm[r];
     dw_gate[e] = sum_r x_perm[r]^T dh_g[r];  dw_up[e] = sum_r x_perm[r]^T dh_u[r]
   (sums over the rows of expert e; experts with no rows get zero
   gradients). dw_* are written (not accumulated), dtype. dh lives in the
   workspace, and so does the order in which the weight-gradient GEMMs walk
   the experts (most rows first, which balances their ragged cost across the
   SMs); the workspace is needed even when R = 0 (bf16, MXFP8). */
moe_status moe_grouped_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h_save,
                               const void* a_save, const void* w_gate, const void* w_up,
                               const void* w_down, int dtype, const int32_t* offsets, int R, int E,
                               int d, int f, void* dx_perm, void* dw_gate, void* dw_up,
                               void* dw_down, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Selects the kernel of the weight-gradient GEMMs: the bf16 ones of
   moe_grouped_mlp_bwd and the GEMM2 one of moe_dispatch_mlp_bwd (its GEMM1
   weight gradient gathers rows and keeps one CTA per SM), and the MXFP8 ones
   of moe_mxfp8_mlp_bwd. Process-wide, for launches issued after the call
   ("Scaling and optimizing MoE training": grouped GEMM; the kernel choice
   itself has no counterpart in the pages). 0 (the default): one CTA per SM,
   bf16 256x256 gradient tiles (two fp32 accumulators fill TMEM), MXFP8
   128x256 tiles (the block scales take the rest of TMEM). 1: CTA pairs
   (2-CTA clusters) with tcgen05.mma.cta_group::2 (M=256 across both SMs):
   bf16 256x256 tiles, each SM holding a 128x256 half twice over so that the
   epilogue overlaps the next tile's MMAs; MXFP8 256x256 tiles, each SM
   holding its 128x256 half and the block scales. Both give the same results
   up to fp32 summation order. Returns MOE_OK. */
moe_status moe_use_cta_pairs(int enable);

/* The dispatch fused into the grouped MLP ("Scaling and optimizing MoE
   training": routed rows go straight into the experts' inputs, and the layer
   avoids reshuffling data). bf16 only (MOE_ERR_UNSUPPORTED otherwise).

   moe_dispatch_mlp_fwd computes exactly moe_permute followed by
   moe_grouped_mlp_fwd (same outputs, bit for bit) without writing x_perm:
   GEMM1 reads row r of its A operand from x[src_row[r] / k] (x [T][d],
   src_row [T*k] device int32 from moe_route), four rows per TMA gather.
   R = T*k must fit an int.

   moe_dispatch_mlp_bwd computes exactly moe_grouped_mlp_bwd on that x_perm,
   with the GEMM1 weight gradient gathering its x rows the same way; it needs
   the same workspace as moe_grouped_mlp_bwd.

   Cost: every GEMM1 output-column tile gathers its rows again, and one row
   gather moves 4 x 128 bytes; on GB300 these calls are slower than
   moe_permute followed by the grouped MLP (which reads whole TMA boxes). */
moe_status moe_dispatch_mlp_fwd(const void* x, const int32_t* src_row, int T, int k, const void* w_gate,
                                const void* w_up, const void* w_down, int dtype, const int32_t* offsets, int E,
                                int d, int f, void* h_save, void* a_save, void* y_perm, void* stream);
moe_status moe_dispatch_mlp_bwd(const void* dy_perm, const void* x, const int32_t* src_row, int T, int k,
                                const void* h_save, const void* a_save, const void* w_gate, const void* w_up,
                                const void* w_down, int dtype, const int32_t* offsets, int E, int d, int f,
                                void* dx_perm, void* dw_gate, void* dw_up, void* dw_down, void* workspace,
                                size_t workspace_bytes, void* stream);

/* MXFP8 with the row quantisation of the dispatched activations moved into
   the kernels that produce them ("Scaling and optimizing MoE training": the
   MXFP8 gains come from the expert feed-forward and from moving expert data;
   the savings must exceed the cost of the format conversion):

   The expert GEMMs read E8M0 scales as "scale chunks": 512 bytes per (group
   of 128 rows of an operand, K stage of 128 elements), in the order the
   tensor-memory scale copy takes them. A row operand ([R][K], rows in expert
   segments given by offsets) is grouped by per-expert 128-row tiles: row r of
   expert e (offsets[e] <= r < offsets[e+1]) is index t = (r - offsets[e]) % 128
   of group G = (offsets[e] + 127 e) / 128 + (r - offsets[e]) / 128, and the
   scale of its block b (elements 32b..32b+31) is byte
       512 (G K/128 + b/4) + 16 (t % 32) + 4 ((t / 32) % 4) + b % 4.
   Bytes of indices past an expert's last row are not written (the GEMMs do
   not store those rows). Such an operand's scales take
   moe_mxfp8_row_scales_size(R, E, K) bytes (0 unless K % 128 == 0).

   moe_permute_mxfp8: the dispatch of x as E4M3 codes x_codes [T*k][d] and
   E8M0 scale chunks x_scales (moe_mxfp8_row_scales_size(T*k, E, d) bytes);
   row dest_row[t][j] holds x[t] quantised along d in blocks of 32 (the codes
   and scale values mxfp8_quantize gives for moe_permute's bf16 x_perm).
   x bf16 [T][d]; topk_idx, offsets as moe_route returned them (they place
   each row in its expert's tiles). x_perm (optional, may be NULL) receives
   the bf16 dispatch as well (the weight gradient quantises it along its
   rows). d % 128 == 0, else MOE_ERR_UNSUPPORTED.

   moe_combine_bwd_mxfp8: moe_combine_bwd that also writes the row
   quantisation (dy_codes [T*k][d], scale chunks dy_scales of
   moe_mxfp8_row_scales_size(T*k, E, d) bytes) of the bf16-rounded values
   gates[t][j] * dy[t]; dy_perm (optional, may be NULL) receives the bf16
   values; dgates as moe_combine_bwd. d % 128 == 0.

   moe_mxfp8_prepare_weights: quantises w_gate, w_up and w_down once per
   weight update into both layouts the expert GEMMs read -- along the weight's
   rows in blocks of 32 (GEMM1 and GEMM2 forward: K = d, f) and along its
   columns in blocks of 32 (the dgrads: K = f, d) -- into wq
   (moe_mxfp8_weights_size(E, d, f) bytes, caller-owned, device). Call it
   after every weight update; moe_mxfp8_mlp_fwd/bwd read the weights only
   from wq. d and f multiples of 128.

   moe_mxfp8_mlp_fwd: moe_grouped_mlp_fwd(MOE_MXFP8) with GEMM1 reading
   x_codes/x_scales and the weights read from wq (no quantisation pass of its
   own). Same outputs, same workspace. a_cols (optional, may be NULL; device,
   moe_mxfp8_col_operand_size(R, E, f) bytes, 16-byte aligned): GEMM1's
   epilogue also writes A = silu(h_g) * h_u quantised along the experts' rows
   (blocks of 32 rows from each expert's first row, the tail block
   zero-padded) -- the GEMM2 weight gradient's A operand -- so that the
   backward need not quantise a_save again.

   moe_mxfp8_mlp_bwd: moe_grouped_mlp_bwd(MOE_MXFP8) with the GEMM2 dgrad
   reading dy_codes/dy_scales and the weights read from wq; dy_perm and
   x_perm (bf16) feed the expert-segment quantisations of the weight
   gradients, and a_save that of A unless a_cols (what moe_mxfp8_mlp_fwd wrote
   there for the same step, or NULL) is given. Same outputs (bit for bit with
   or without a_cols), same workspace. d and f multiples of 128.

   moe_mxfp8_col_operand_size: bytes of an operand of R rows and K columns
   quantised along the experts' rows: E4M3 codes [R][K] (padded to 256 bytes)
   followed by its scale chunks (0 unless K % 128 == 0). */
size_t moe_mxfp8_weights_size(int E, int d, int f);
moe_status moe_mxfp8_prepare_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int d, int f,
                                     void* wq, size_t wq_bytes, void* stream);
size_t moe_mxfp8_row_scales_size(int R, int E, int K);
moe_status moe_permute_mxfp8(const void* x, int T, int d, int k, int E, const int32_t* dest_row,
                             const int32_t* topk_idx, const int32_t* offsets, uint8_t* x_codes, uint8_t* x_scales,
                             void* x_perm, void* stream);
moe_status moe_combine_bwd_mxfp8(const void* dy, const void* y_perm, const float* gates, const int32_t* dest_row,
                                 const int32_t* topk_idx, const int32_t* offsets, int T, int d, int k, int E,
                                 uint8_t* dy_codes, uint8_t* dy_scales, void* dy_perm, float* dgates, void* stream);
size_t moe_mxfp8_col_operand_size(int R, int E, int K);
moe_status moe_mxfp8_mlp_fwd(const uint8_t* x_codes, const uint8_t* x_scales, const void* wq, const int32_t* offsets,
                             int R, int E, int d, int f, void* h_save, void* a_save, void* y_perm, uint8_t* a_cols,
                             void* workspace, size_t workspace_bytes, void* stream);
moe_status moe_mxfp8_mlp_bwd(const uint8_t* dy_codes, const uint8_t* dy_scales, const void* dy_perm,
                             const void* x_perm, const void* h_save, const void* a_save, const uint8_t* a_cols,
                             const void* wq, const int32_t* offsets, int R, int E, int d, int f, void* dx_perm,
                             void* dw_gate, void* dw_up, void* dw_down, void* workspace, size_t workspace_bytes,
                             void* stream);

/* MXFP8 block quantisation ("Scaling and optimizing MoE training": MXFP8):
   E4M3 codes with one E8M0 scale per 32 consecutive elements.
     axis 0: src [rows][K] bf16, blocks of 32 along K inside a row;
             dst_e4m3 [rows][K], dst_e8m0 [rows][K/32]. K % 32 == 0.
     axis 1: blocks of 32 consecutive rows of one column; with seg_offsets
             ([nseg+1] device int32, NULL for one segment of all rows) blocks
             start at each segment's first row and a segment's last block is
             zero-padded; dst_e4m3 [rows][K]; dst_e8m0 [nblk][K] where segment
             g owns block rows from sum_{h<g} ceil(len_h/32) -- the caller
             sizes dst_e8m0 for ceil(rows/32) + nseg block rows.
   Scale exponent s = ceil(log2(amax / 448)) clamped to [-127, 127]
   (s = -127 for an all-zero block), byte s + 127; elements are
   round-to-nearest-even of v * 2^-s, saturated to +-448. */
moe_status mxfp8_quantize(const void* src, int rows, int K, int axis, const int32_t* seg_offsets,
                          int nseg, uint8_t* dst_e4m3, uint8_t* dst_e8m0, void* stream);

/* moe_route for callers that cannot allocate device memory (the pages have no
   counterpart to this call). It computes exactly what moe_route computes, with
   the same arguments minus the workspace: its scratch lives in a 4 MiB array
   compiled into the library, which every GPU that loads the library keeps
   until the process exits. Shapes with ceil(T/8) * E > 1,048,576 return
   MOE_ERR_WORKSPACE without launching anything. Every call looks up the
   array's device address on the calling thread's current device (so a device
   reset leaves no stale address behind); the first call on a device also loads
   the library's device code there, so make it before any stream capture. The
   call allocates nothing. All calls on a device share the one array, so calls
   that may overlap on the GPU (different streams, or different host threads)
   race with each other and must be ordered by the caller. */
moe_status moe_route_noalloc(const void* x, const void* w_router, const float* bias, int dtype, int T,
                             int d, int E, int k, float* logits, int flags, int32_t* topk_idx,
                             float* gates, int32_t* counts, int32_t* offsets, int32_t* dest_row,
                             int32_t* src_row, void* stream);

/* Self-test of the bounded waits (failure detection; the pages have no
   counterpart). Launches one 64-thread block on `stream` in which warp 0 waits
   on an mbarrier that nothing arrives on, for at most `cycles` SM clock cycles
   (1 <= cycles <= 4e9, about 2 s at 2 GHz), while warp 1 waits on another one
   with the GEMMs' own limit (~2 s). Warp 0's wait expires: it sets the device
   error word to MOE_ERR_TIMEOUT and raises the block's abort flag, which ends
   warp 1's wait as well; the kernel then returns normally (no trap). out: [2]
   int32 device buffer, 16-byte aligned; out[w] = 1 if warp w's wait completed,
   0 if it gave up (so {0, 0} after a correct run). The caller reads the error
   word with moe_get_device_error(); the context stays usable. */
moe_status moe_selftest_wait_timeout(long long cycles, int32_t* out, void* stream);

/* Synchronises `stream`, then returns and clears this device's error word
   (MOE_OK if no kernel reported an error). Error reporting of this library:
   the pages have no counterpart. */
moe_status moe_get_device_error(void* stream);

/* Number of SMs the kernels size their persistent grids for (0 on error).
   Instrumentation: the pages have no counterpart. */
int moe_sm_count(void);

/* Number of kernels this process has launched through libmoe so far (a host
   counter, bumped once per successful launch; for instrumentation; the
   pages have no counterpart). */
uint64_t moe_launch_count(void);

/* Launch timing, for measurement (instrumentation: the pages have no
   counterpart). moe_timing_arm(n) arms a process-wide recorder: each of the
   next n kernel launches made through the library (1 <= n <= 256) records a
   CUDA event on its own stream just before it starts. moe_timing_finish(stream)
   records a closing event on `stream` and disarms the recorder.
   moe_timing_read(ms, names, cap) waits for the closing event and, for the
   first min(recorded, cap) launches, writes ms[i] = time from launch i's event
   to the next event (launch i+1's, or the closing one) and names[i] = a static
   string naming the kernel (names may be NULL); it returns that count, or -1
   if nothing was finished. When the launches ran back to back on one stream,
   ms[i] is launch i's device duration (plus any idle gap before the next
   launch, so the host should run ahead of the GPU). Arming creates CUDA events
   (not device memory) on the current device the first time. Not meant for
   concurrent use by several threads. */
moe_status moe_timing_arm(int n);
moe_status moe_timing_finish(void* stream);
int moe_timing_read(float* ms, const char** names, int cap);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
