// permute.cu -- dispatch (permute), combine, their backward passes and the
// router backward. All are HBM-bound row gathers/scatters: one warp per token
// row, 16-byte vector loads and stores, fp32 arithmetic, one rounding per
// output element. ("Introducing Olmo-core 3", section "Scaling and optimizing
// MoE training": routed rows are placed directly into the experts' input
// buffers; the combine is the gate-weighted return to token order.)
#include "common.cuh"
#include "kernels.h"
#include "mxfp8_common.cuh"

namespace moe {

namespace {

constexpr int kRowWarps = 8;

// 16 loaded bytes as floats: 8 bf16 or 4 fp32 elements (the load of Vec16
// split in two, so the bytes can be requested well before they are used).
__device__ __forceinline__ void unpack16(const uint4& q, float* v, const __nv_bfloat16*) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void unpack16(const uint4& q, float* v, const float*) {
  v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
  v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
}

// x_perm[dest_row[t][j]] = x[t]
template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
permute_kernel(const T* __restrict__ x, int Tn, int d, int k, const int32_t* __restrict__ dest_row,
               T* __restrict__ x_perm, int* err) {
  using V = Vec16<T>;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  int dest = lane < k ? dest_row[(size_t)t * k + lane] : 0;
  const unsigned ok = usable_pairs(dest, 0, lane, k, (long)Tn * k, 0, err);
  const T* src = x + (size_t)t * d;
  for (int c = lane * V::N; c < d; c += 32 * V::N) {
    const uint4 q = *reinterpret_cast<const uint4*>(src + c);
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, dest, j);
      if (!((ok >> j) & 1u)) continue;
      *reinterpret_cast<uint4*>(x_perm + (size_t)r * d + c) = q;
    }
  }
}

// y[t] = sum_j g[t][j] * y_perm[dest_row[t][j]]   (fp32, j ascending)
// KMAX: the largest k the instance handles; each column step requests its k
// rows before adding any.
template <typename T, int KMAX>
__global__ void __launch_bounds__(kRowWarps * 32)
combine_fwd_kernel(const T* __restrict__ y_perm, const float* __restrict__ gates,
                   const int32_t* __restrict__ dest_row, int Tn, int d, int k, T* __restrict__ y, int* err) {
  using V = Vec16<T>;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  const int my_dest = lane < k ? dest_row[(size_t)t * k + lane] : 0;
  const float my_g = lane < k ? gates[(size_t)t * k + lane] : 0.0f;
  const unsigned ok = usable_pairs(my_dest, 0, lane, k, (long)Tn * k, 0, err);
  int dest[KMAX];
  float g[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    dest[j] = __shfl_sync(0xffffffffu, my_dest, j);
    g[j] = __shfl_sync(0xffffffffu, my_g, j);
  }
  for (int c = lane * V::N; c < d; c += 32 * V::N) {
    uint4 yv[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && ((ok >> j) & 1u)) yv[j] = *reinterpret_cast<const uint4*>(y_perm + (size_t)dest[j] * d + c);
    float acc[V::N];
#pragma unroll
    for (int i = 0; i < V::N; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k && ((ok >> j) & 1u)) {
        float v[V::N];
        unpack16(yv[j], v, y_perm);
#pragma unroll
        for (int i = 0; i < V::N; ++i) acc[i] = fmaf(g[j], v[i], acc[i]);
      }
    }
    V::store(y + (size_t)t * d + c, acc);
  }
}

// dy_perm[dest] = g * dy[t];  dgates[t][j] = <dy[t], y_perm[dest]>
// KMAX: the largest k the instance handles (arrays of per-slot state).
// QUANT (bf16 only): also write dy_perm's MXFP8 row quantisation (q [T*k][d]
// E4M3; qsc E8M0 as the GEMM's scale chunks, grouped by per-expert 128-row
// tiles found from topk_idx and offs) of the bf16-rounded g * dy values -- the
// codes and scales mxfp8_quantize(dy_perm, rows) gives -- and dy_perm itself
// only when given.
template <typename T, int KMAX, bool QUANT = false>
__global__ void __launch_bounds__(kRowWarps * 32)
combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ y_perm,
                   const float* __restrict__ gates, const int32_t* __restrict__ dest_row, int Tn,
                   int d, int k, T* __restrict__ dy_perm, float* __restrict__ dgates, int* err,
                   uint8_t* __restrict__ q = nullptr, uint8_t* __restrict__ qsc = nullptr,
                   const int32_t* __restrict__ topk_idx = nullptr, const int32_t* __restrict__ offs = nullptr,
                   int E = 0) {
  using V = Vec16<T>;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  const int my_dest = lane < k ? dest_row[(size_t)t * k + lane] : 0;
  const float my_g = lane < k ? gates[(size_t)t * k + lane] : 0.0f;
  // QUANT: the pair's expert must hold its row (the scale chunk is found from it)
  int my_e = 0;
  if (QUANT && lane < k) {
    my_e = topk_idx[(size_t)t * k + lane];
    if (my_e >= 0 && my_e < E && (my_dest < offs[my_e] || my_dest >= offs[my_e + 1])) my_e = -1;
  }
  const unsigned ok = usable_pairs(my_dest, my_e, lane, k, (long)Tn * k, QUANT ? E : 0, err);
  int dest[KMAX];
  float g[KMAX], dot[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    dest[j] = __shfl_sync(0xffffffffu, my_dest, j);
    g[j] = __shfl_sync(0xffffffffu, my_g, j);
    dot[j] = 0.0f;
  }
  // QUANT: the scale chunk row of each dispatched row (its per-expert 128-row
  // tile and its index in the tile)
  size_t sbase[QUANT ? KMAX : 1];
  if constexpr (QUANT) {
    int my_grp = 0, my_t = 0;
    if (lane < k && ((ok >> lane) & 1u)) {
      const int e = my_e, o = offs[e];
      my_grp = static_cast<int>(mx_row_tile_base(o, e)) + ((my_dest - o) >> 7);
      my_t = (my_dest - o) & 127;
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      sbase[j] = ((size_t)__shfl_sync(0xffffffffu, my_grp, j) * (d / 128) << 9) +
                 mx_chunk_lane(__shfl_sync(0xffffffffu, my_t, j));
  }
  // warp-uniform loop (the quantising variant shuffles inside it); lanes past d
  // contribute zeros and store nothing
  for (int cb = 0; cb < d; cb += 32 * V::N) {
    const int c = cb + lane * V::N;
    const bool act = c < d;
    // every row of the step is requested before any is used
    uint4 uq = make_uint4(0, 0, 0, 0), yq[KMAX];
    if (act) uq = *reinterpret_cast<const uint4*>(dy + (size_t)t * d + c);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      yq[j] = make_uint4(0, 0, 0, 0);
      if (act && j < k && ((ok >> j) & 1u)) yq[j] = *reinterpret_cast<const uint4*>(y_perm + (size_t)dest[j] * d + c);
    }
    float u[V::N];
    unpack16(uq, u, dy);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k && ((ok >> j) & 1u)) {
        float v[V::N], w[V::N];
        unpack16(yq[j], v, y_perm);
#pragma unroll
        for (int i = 0; i < V::N; ++i) {
          dot[j] = fmaf(u[i], v[i], dot[j]);
          w[i] = g[j] * u[i];
        }
        if constexpr (QUANT) {
          static_assert(V::N == 8, "a 32-element block is 4 lanes of 8 bf16");
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < V::N; ++i) {
            w[i] = __bfloat162float(__float2bfloat16_rn(w[i]));
            amax = fmaxf(amax, fabsf(w[i]));
          }
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          const int sx = mx_e8m0_exponent(amax);
          const float m = mx_pow2_neg(sx);
          const uint32_t lo = mx_e4m3x2(w[0] * m, w[1] * m) | mx_e4m3x2(w[2] * m, w[3] * m) << 16;
          const uint32_t hi = mx_e4m3x2(w[4] * m, w[5] * m) | mx_e4m3x2(w[6] * m, w[7] * m) << 16;
          if (act) {
            *reinterpret_cast<uint2*>(q + (size_t)dest[j] * d + c) = make_uint2(lo, hi);
            const int b = c / 32;
            if ((lane & 3) == 0) qsc[sbase[j] + ((size_t)(b / 4) << 9) + (b & 3)] = static_cast<uint8_t>(sx + 127);
            if (dy_perm) V::store(dy_perm + (size_t)dest[j] * d + c, w);
          }
        } else if (act) {
          V::store(dy_perm + (size_t)dest[j] * d + c, w);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < k) {
      const float s = warp_sum(dot[j]);
      if (lane == 0) dgates[(size_t)t * k + j] = s;
    }
  }
}

// dx[t] = sum_j dx_perm[dest[t][j]] (+ sum_j dl[t][e_j] * w_r[e_j])
// KMAX: the largest k the instance handles. ROUTER: the router term is added
// (dlogits and w_r given). Each column step first requests all of its rows --
// the k rows of dx_perm and, with ROUTER, the k rows of w_r -- and only then
// adds them, so the two sets of loads wait on memory together.
template <typename T, int KMAX, bool ROUTER>
__global__ void __launch_bounds__(kRowWarps * 32)
permute_bwd_kernel(const T* __restrict__ dx_perm, int Tn, int d, int E, int k,
                   const int32_t* __restrict__ dest_row, const int32_t* __restrict__ topk_idx,
                   const float* __restrict__ dlogits, const T* __restrict__ w_r,
                   T* __restrict__ dx, int* err) {
  using V = Vec16<T>;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  const int my_dest = lane < k ? dest_row[(size_t)t * k + lane] : 0;
  int my_e = 0;
  if (ROUTER && lane < k) my_e = topk_idx[(size_t)t * k + lane];
  const unsigned ok = usable_pairs(my_dest, my_e, lane, k, (long)Tn * k, ROUTER ? E : 0, err);
  float my_dl = 0.0f;
  if (ROUTER && lane < k && ((ok >> lane) & 1u)) my_dl = dlogits[(size_t)t * E + my_e];
  int dest[KMAX], ex[KMAX];
  float dl[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    dest[j] = __shfl_sync(0xffffffffu, my_dest, j);
    ex[j] = __shfl_sync(0xffffffffu, my_e, j);
    dl[j] = __shfl_sync(0xffffffffu, my_dl, j);
  }
  for (int c = lane * V::N; c < d; c += 32 * V::N) {
    uint4 xv[KMAX], wv[ROUTER ? KMAX : 1];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k && ((ok >> j) & 1u)) xv[j] = *reinterpret_cast<const uint4*>(dx_perm + (size_t)dest[j] * d + c);
    if constexpr (ROUTER) {
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && ((ok >> j) & 1u)) wv[j] = *reinterpret_cast<const uint4*>(w_r + (size_t)ex[j] * d + c);
    }
    float acc[V::N];
#pragma unroll
    for (int i = 0; i < V::N; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k && ((ok >> j) & 1u)) {
        float v[V::N];
        unpack16(xv[j], v, dx_perm);
#pragma unroll
        for (int i = 0; i < V::N; ++i) acc[i] += v[i];
      }
    }
    if constexpr (ROUTER) {
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && ((ok >> j) & 1u)) {
          float w[V::N];
          unpack16(wv[j], w, w_r);
#pragma unroll
          for (int i = 0; i < V::N; ++i) acc[i] = fmaf(dl[j], w[i], acc[i]);
        }
      }
    }
    V::store(dx + (size_t)t * d + c, acc);
  }
}

// dlogits[t][i] = g_i (dg_i - sum_j g_j dg_j) on the selected experts, else 0.
__global__ void __launch_bounds__(kRowWarps * 32)
router_dlogits_kernel(const float* __restrict__ dgates, const float* __restrict__ gates,
                      const int32_t* __restrict__ topk_idx, int Tn, int E, int k,
                      float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  if (t >= Tn) return;
  float g = 0.0f, dg = 0.0f;
  int e = -1;
  if (lane < k) {
    g = gates[(size_t)t * k + lane];
    dg = dgates[(size_t)t * k + lane];
    e = topk_idx[(size_t)t * k + lane];
  }
  const float s = warp_sum(g * dg);
  const float dl = g * (dg - s);
  int ej[8];
  float dlj[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ej[j] = __shfl_sync(0xffffffffu, e, j);
    dlj[j] = __shfl_sync(0xffffffffu, dl, j);
  }
  for (int c = lane; c < E; c += 32) {
    float v = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && ej[j] == c) v = dlj[j];
    dlogits[(size_t)t * E + c] = v;
  }
}

// dw_r[e][c] = sum over rows r of expert e of dlogits[t(r)][e] * x[t(r)][c],
// t(r) = src_row[r] / k. The token rows are gathered from x (T rows, which
// stay in L2 across the k experts that read each) rather than from the
// k-times larger x_perm. Grid (E, d / 64): a CTA owns 64 columns of one
// expert, so a heavily loaded expert's rows spread over d / 64 CTAs. A warp
// reads RPW rows at once (LPR lanes of 16 bytes per row); the row groups of a
// warp are added by a fixed shuffle tree and the 8 warps in fixed order
// through shared memory, so the result is bit-reproducible.
template <typename T>
__global__ void __launch_bounds__(256)
router_dw_kernel(const float* __restrict__ dlogits, const int32_t* __restrict__ offsets,
                 const int32_t* __restrict__ src_row, const T* __restrict__ x, int d, int E,
                 int k, float* __restrict__ dw_r) {
  constexpr int VN = Vec16<T>::N;   // elements per 16 bytes
  constexpr int COLS = 64;          // columns per CTA
  constexpr int LPR = COLS / VN;    // lanes per row
  constexpr int RPW = 32 / LPR;     // rows a warp reads at once
  constexpr int STEP = 8 * RPW;     // rows the CTA reads at once
  __shared__ float part[8][COLS];
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int c = blockIdx.y * COLS + sub * VN;  // d % 64 == 0: always inside the row
  const int r0 = offsets[e], r1 = offsets[e + 1];
  float acc[VN];
#pragma unroll
  for (int i = 0; i < VN; ++i) acc[i] = 0.0f;
  int r = r0 + warp * RPW + grp;
  for (; r + 3 * STEP < r1; r += 4 * STEP) {
    float v[4][VN], w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = src_row[r + u * STEP] / k;
      w[u] = dlogits[(size_t)t * E + e];
      Vec16<T>::load(x + (size_t)t * d + c, v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = fmaf(w[u], v[u][i], acc[i]);
  }
  for (; r < r1; r += STEP) {
    float v[VN];
    const int t = src_row[r] / k;
    const float w = dlogits[(size_t)t * E + e];
    Vec16<T>::load(x + (size_t)t * d + c, v);
#pragma unroll
    for (int i = 0; i < VN; ++i) acc[i] = fmaf(w, v[i], acc[i]);
  }
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < VN; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  if (grp == 0) {
#pragma unroll
    for (int i = 0; i < VN; ++i) part[warp][sub * VN + i] = acc[i];
  }
  __syncthreads();
  if (threadIdx.x < COLS) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][threadIdx.x];
    dw_r[(size_t)e * d + blockIdx.y * COLS + threadIdx.x] = s;
  }
}

template <typename T> inline int row_grid(int Tn) { return (Tn + kRowWarps - 1) / kRowWarps; }

}  // namespace

template <typename T>
cudaError_t launch_permute(const void* x, int Tn, int d, int k, const int32_t* dest_row, void* x_perm,
                           cudaStream_t st) {
  if (Tn == 0) return cudaSuccess;
  MOE_COUNTED_AS("permute", st) permute_kernel<T><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(
      static_cast<const T*>(x), Tn, d, k, dest_row, static_cast<T*>(x_perm), device_error_word());
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine_fwd(const void* y_perm, const float* gates, const int32_t* dest_row, int Tn,
                               int d, int k, void* y, cudaStream_t st) {
  if (Tn == 0) return cudaSuccess;
  if (k <= 4)
    MOE_COUNTED_AS("combine_fwd", st) combine_fwd_kernel<T, 4><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const T*>(y_perm), gates, dest_row, Tn, d, k, static_cast<T*>(y), device_error_word());
  else
    MOE_COUNTED_AS("combine_fwd", st) combine_fwd_kernel<T, 8><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const T*>(y_perm), gates, dest_row, Tn, d, k, static_cast<T*>(y), device_error_word());
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_combine_bwd(const void* dy, const void* y_perm, const float* gates,
                               const int32_t* dest_row, int Tn, int d, int k, void* dy_perm,
                               float* dgates, cudaStream_t st) {
  if (Tn == 0) return cudaSuccess;
  if (k <= 4)
    MOE_COUNTED_AS("combine_bwd", st) combine_bwd_kernel<T, 4><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const T*>(dy), static_cast<const T*>(y_perm), gates, dest_row, Tn, d, k,
        static_cast<T*>(dy_perm), dgates, device_error_word());
  else
    MOE_COUNTED_AS("combine_bwd", st) combine_bwd_kernel<T, 8><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const T*>(dy), static_cast<const T*>(y_perm), gates, dest_row, Tn, d, k,
        static_cast<T*>(dy_perm), dgates, device_error_word());
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd_quant(const void* dy, const void* y_perm, const float* gates,
                                     const int32_t* dest_row, const int32_t* topk_idx, const int32_t* offsets,
                                     int Tn, int d, int k, int E, uint8_t* q, uint8_t* qsc, void* dy_perm,
                                     float* dgates, cudaStream_t st) {
  using B = __nv_bfloat16;
  if (Tn == 0) return cudaSuccess;
  if (k <= 4)
    MOE_COUNTED_AS("combine_bwd", st) combine_bwd_kernel<B, 4, true><<<row_grid<B>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const B*>(dy), static_cast<const B*>(y_perm), gates, dest_row, Tn, d, k, static_cast<B*>(dy_perm),
        dgates, device_error_word(), q, qsc, topk_idx, offsets, E);
  else
    MOE_COUNTED_AS("combine_bwd", st) combine_bwd_kernel<B, 8, true><<<row_grid<B>(Tn), kRowWarps * 32, 0, st>>>(
        static_cast<const B*>(dy), static_cast<const B*>(y_perm), gates, dest_row, Tn, d, k, static_cast<B*>(dy_perm),
        dgates, device_error_word(), q, qsc, topk_idx, offsets, E);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_permute_bwd(const void* dx_perm, int Tn, int d, int E, int k,
                               const int32_t* dest_row, const int32_t* topk_idx, const float* dlogits,
                               const void* w_r, void* dx, cudaStream_t st) {
  if (Tn == 0) return cudaSuccess;
#define MOE_PBWD(KM, RT)                                                                               \
  MOE_COUNTED_AS("permute_bwd", st) permute_bwd_kernel<T, KM, RT><<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>( \
      static_cast<const T*>(dx_perm), Tn, d, E, k, dest_row, topk_idx, dlogits, static_cast<const T*>(w_r),     \
      static_cast<T*>(dx), device_error_word())
  const bool router = dlogits != nullptr;
  if (k <= 4) {
    if (router) MOE_PBWD(4, true); else MOE_PBWD(4, false);
  } else {
    if (router) MOE_PBWD(8, true); else MOE_PBWD(8, false);
  }
#undef MOE_PBWD
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_route_bwd(const float* dgates, const float* gates, const int32_t* topk_idx,
                             const int32_t* offsets, const int32_t* src_row, const void* x,
                             int Tn, int d, int E, int k, float* dlogits, float* dw_r,
                             cudaStream_t st) {
  if (Tn > 0)
    MOE_COUNTED_AS("router_dlogits", st) router_dlogits_kernel<<<row_grid<T>(Tn), kRowWarps * 32, 0, st>>>(dgates, gates, topk_idx, Tn,
                                                                       E, k, dlogits);
  dim3 grid(E, d / 64);
  MOE_COUNTED_AS("router_dw", st) router_dw_kernel<T><<<grid, 256, 0, st>>>(dlogits, offsets, src_row, static_cast<const T*>(x),
                                            d, E, k, dw_r);
  return cudaGetLastError();
}

#define MOE_INST(T)                                                                              \
  template cudaError_t launch_permute<T>(const void*, int, int, int, const int32_t*, void*,      \
                                         cudaStream_t);                                          \
  template cudaError_t launch_combine_fwd<T>(const void*, const float*, const int32_t*, int, int, \
                                             int, void*, cudaStream_t);                          \
  template cudaError_t launch_combine_bwd<T>(const void*, const void*, const float*,             \
                                             const int32_t*, int, int, int, void*, float*,       \
                                             cudaStream_t);                                      \
  template cudaError_t launch_permute_bwd<T>(const void*, int, int, int, int, const int32_t*,    \
                                             const int32_t*, const float*, const void*, void*,   \
                                             cudaStream_t);                                      \
  template cudaError_t launch_route_bwd<T>(const float*, const float*, const int32_t*,           \
                                           const int32_t*, const int32_t*, const void*, int, int, \
                                           int, int, float*, float*, cudaStream_t);
MOE_INST(float)
MOE_INST(__nv_bfloat16)
#undef MOE_INST

}  // namespace moe
