// gemm_simt.cu -- CUDA-core grouped GEMM over ragged expert segments, for the
// fp32 layer (a tiny layer whose operands tensor cores would round) and for
// the fp32-output router GEMM. The bf16 expert GEMMs run on tcgen05
// (gemm_tc.cu).
//
//   C(m, n) = sum_k A(m, k) * B(k, n)  (+ col_bias[n]),   fp32 accumulation
//
// Row-ragged mode (forward / dgrad): rows of A and C are the routed rows;
// rows [offsets[e], offsets[e+1]) use expert e's B. K-ragged mode (wgrad):
// the reduction runs over the rows of expert e and C_e is expert e's [M][N]
// gradient; an expert with no rows gets zeros.
//
// B(k, n) comes from B0 when k < kSplit and n < nSplit, else from B1 at
// (k - kSplit or k, n - nSplit or n): this stitches the gate and up weights
// into one operand. C(m, n) goes to C0 when n < cSplit, else to C1.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ int s_e, s_m0, s_mend;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const TA* A = static_cast<const TA*>(g.A);

  int e, m0, m_end, k0, k_end;
  if (!g.kragged) {
    if (tid == 0) {
      int ee = -1, mm0 = 0, mend = 0;
      if (g.offsets == nullptr) {
        ee = 0; mm0 = blockIdx.x * BM; mend = g.M;
        if (mm0 >= mend) ee = -1;
      } else {
        int acc = 0;
        for (int q = 0; q < g.E; ++q) {
          const int lo = g.offsets[q], hi = g.offsets[q + 1];
          const int tiles = (hi - lo + BM - 1) / BM;
          if ((int)blockIdx.x < acc + tiles) {
            ee = q; mm0 = lo + ((int)blockIdx.x - acc) * BM; mend = hi;
            break;
          }
          acc += tiles;
        }
      }
      s_e = ee; s_m0 = mm0; s_mend = mend;
    }
    __syncthreads();
    e = s_e; m0 = s_m0; m_end = s_mend;
    if (e < 0) return;
    k0 = 0; k_end = g.K;
  } else {
    e = blockIdx.z;
    m0 = blockIdx.x * BM; m_end = g.M;
    k0 = g.offsets[e]; k_end = g.offsets[e + 1];
  }
  const int n0 = blockIdx.y * BN;
  const size_t b_e = g.kragged ? 0 : (size_t)e * g.sBe;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int kb = k0; kb < k_end; kb += BK) {
    // A tile: BM x BK (1024 elements, 4 per thread)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * 256, mm = idx / BK, kk = idx % BK;
      const int m = m0 + mm, kq = kb + kk;
      float v = 0.0f;
      if (m < m_end && kq < k_end) v = to_f32(A[(size_t)m * g.sAm + (size_t)kq * g.sAk]);
      As[kk][mm] = v;
    }
    // B tile: BK x BN
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * 256, kk = idx / BN, nn = idx % BN;
      const int n = n0 + nn, kq = kb + kk;
      float v = 0.0f;
      if (n < g.N && kq < k_end) {
        const bool lo = kq < g.kSplit && n < g.nSplit;
        const TB* B = static_cast<const TB*>(lo ? g.B0 : g.B1);
        const int kb2 = kq < g.kSplit ? kq : kq - g.kSplit;
        const int nb2 = n < g.nSplit ? n : n - g.nSplit;
        v = to_f32(B[b_e + (size_t)kb2 * g.sBk + (size_t)nb2 * g.sBn]);
      }
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  const size_t c_e = g.kragged ? (size_t)e * g.sCe : 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= m_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      if (g.col_bias) v += g.col_bias[n];
      TC* C = static_cast<TC*>(n < g.cSplit ? g.C0 : g.C1);
      const int nc = n < g.cSplit ? n : n - g.cSplit;
      C[c_e + (size_t)m * g.sCm + (size_t)nc * g.sCn] = from_f32<TC>(v);
    }
  }
}

// a = silu(hg) * hu with h = (hg | hu) rows of width 2f.
template <typename T>
__global__ void swiglu_fwd_kernel(const T* __restrict__ h, long rows, int f, T* __restrict__ a) {
  const long n = rows * f;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long r = i / f, c = i % f;
    const float hg = to_f32(h[r * 2 * f + c]), hu = to_f32(h[r * 2 * f + f + c]);
    a[i] = from_f32<T>(silu_f(hg) * hu);
  }
}

// dh_g = da * hu * silu'(hg), dh_u = da * silu(hg)
template <typename T>
__global__ void swiglu_bwd_kernel(const T* __restrict__ da, const T* __restrict__ h, long rows, int f,
                                  T* __restrict__ dh) {
  const long n = rows * f;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long r = i / f, c = i % f;
    const float hg = to_f32(h[r * 2 * f + c]), hu = to_f32(h[r * 2 * f + f + c]);
    const float g = to_f32(da[i]);
    const float s = sigmoid_f(hg);
    dh[r * 2 * f + c] = from_f32<T>(g * hu * s * (1.0f + hg * (1.0f - s)));
    dh[r * 2 * f + f + c] = from_f32<T>(g * hg * s);
  }
}

}  // namespace

template <typename TA, typename TB, typename TC>
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t st) {
  dim3 grid;
  if (!g.kragged) {
    const int mt = g.offsets ? (g.M + BM - 1) / BM + g.E : (g.M + BM - 1) / BM;
    if (mt == 0) return cudaSuccess;
    grid = dim3(mt, (g.N + BN - 1) / BN, 1);
  } else {
    grid = dim3((g.M + BM - 1) / BM, (g.N + BN - 1) / BN, g.E);
  }
  MOE_COUNTED_AS("simt_gemm", st) simt_gemm_kernel<TA, TB, TC><<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_swiglu_fwd(const void* h, long rows, int f, void* a, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  MOE_COUNTED_AS("swiglu_fwd", st) swiglu_fwd_kernel<T><<<1024, 256, 0, st>>>(static_cast<const T*>(h), rows, f, static_cast<T*>(a));
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_swiglu_bwd(const void* da, const void* h, long rows, int f, void* dh, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  MOE_COUNTED_AS("swiglu_bwd", st) swiglu_bwd_kernel<T><<<1024, 256, 0, st>>>(static_cast<const T*>(da), static_cast<const T*>(h), rows,
                                             f, static_cast<T*>(dh));
  return cudaGetLastError();
}

template cudaError_t launch_simt_gemm<float, float, float>(const SimtGemm&, cudaStream_t);
template cudaError_t launch_simt_gemm<__nv_bfloat16, __nv_bfloat16, float>(const SimtGemm&, cudaStream_t);
template cudaError_t launch_simt_gemm<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(const SimtGemm&,
                                                                                  cudaStream_t);
template cudaError_t launch_swiglu_fwd<float>(const void*, long, int, void*, cudaStream_t);
template cudaError_t launch_swiglu_fwd<__nv_bfloat16>(const void*, long, int, void*, cudaStream_t);
template cudaError_t launch_swiglu_bwd<float>(const void*, const void*, long, int, void*, cudaStream_t);
template cudaError_t launch_swiglu_bwd<__nv_bfloat16>(const void*, const void*, long, int, void*,
                                                      cudaStream_t);

}  // namespace moe
