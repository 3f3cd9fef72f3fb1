// gemm_tc.cu -- the six grouped expert GEMMs of the SwiGLU MoE layer on the
// 5th-generation tensor cores ("Introducing Olmo-core 3", section "Scaling and
// optimizing MoE training": a grouped GEMM combines the many small per-expert
// computations into one efficient one).
//
// One persistent kernel per GEMM, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//               128-byte swizzled, filled by cp.async.bulk.tensor.
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma M=128 N=256 K=16 into
//               one of two 256-column fp32 accumulators (512 TMEM columns),
//               so the epilogue of tile i overlaps the MMAs of tile i+1.
//   warps 2..9  epilogue: tcgen05.ld of the accumulator, fused SwiGLU (fwd or
//               bwd) math, bf16 (or fp32 router logits) stores with row/column
//               masks; two warps per TMEM lane quadrant, each half the columns.
// Tiles are enumerated on the device from the expert offsets (the host never
// sees the per-expert counts): forward/dgrad tiles cover 128 routed rows of
// one expert (rows past the expert's end are computed and not stored);
// wgrad tiles cover a 128x256 block of one expert's weight gradient and
// reduce over that expert's rows (a ragged K; the rows past its end are
// zeroed in shared memory before the MMA; an expert with no rows gets zeros).
// Every wait is bounded; on a timeout the CTA sets the device error word,
// drains what it started and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * 64 * 2;  // one 64 (MN) x 64 (K) MN-major box
constexpr int NUM_EPI_WARPS = 8;  // two warps per TMEM lane quadrant, each half the columns
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz

enum Kind { FPROP1 = 0, FPROP2 = 1, DGRAD2 = 2, DGRAD1 = 3, WGRAD2 = 4, WGRAD1 = 5, ROUTER = 6 };

struct Params {
  const int32_t* offsets;  // nullptr: one dense group of R rows (router GEMM)
  const float* bias;       // router: per-column bias (or nullptr)
  int E, R, d, f;
  int N;        // output columns of the GEMM
  int M;        // wgrad: output rows
  int n_tiles, m_tiles;
  void* out0;
  void* out1;
  const void* aux;
  int* err;
};

template <int KIND> struct Traits;
// H = x_perm . [Wg | Wu]   (A K-major [R][d]; B MN-major Wg/Wu[e][d][f])
template <> struct Traits<FPROP1> { static constexpr bool kragged = false, a_mn = false, b_mn = true; };
// y_perm = A . Wd          (A K-major [R][f]; B MN-major Wd[e][f][d])
template <> struct Traits<FPROP2> { static constexpr bool kragged = false, a_mn = false, b_mn = true; };
// dA = dy_perm . Wd^T      (A K-major [R][d]; B K-major Wd[e][f][d])
template <> struct Traits<DGRAD2> { static constexpr bool kragged = false, a_mn = false, b_mn = false; };
// dx_perm = dh . [Wg|Wu]^T (A K-major [R][2f]; B K-major Wg/Wu[e][d][f])
template <> struct Traits<DGRAD1> { static constexpr bool kragged = false, a_mn = false, b_mn = false; };
// dWd[e] = A_e^T dy_perm_e (A MN-major [R][f]; B MN-major [R][d])
template <> struct Traits<WGRAD2> { static constexpr bool kragged = true, a_mn = true, b_mn = true; };
// [dWg|dWu][e] = x_perm_e^T dh_e (A MN-major [R][d]; B MN-major [R][2f])
template <> struct Traits<WGRAD1> { static constexpr bool kragged = true, a_mn = true, b_mn = true; };
// logits = x . W_r^T + bias, fp32 out (A K-major [T][d]; B K-major W_r[E][d])
template <> struct Traits<ROUTER> { static constexpr bool kragged = false, a_mn = false, b_mn = false; };

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Smem* sm, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sm->abort_flag)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      set_error(err, MOE_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sm->abort_flag) = 1;
      return false;
    }
  }
}

struct Tile {
  int e, m0, row_end, n_idx, m_idx, nkb, k_row0;
};

// Decode linear tile t. Row-ragged: expert e owns tstart[e]..tstart[e+1]
// (m-tiles x n-tiles, n fastest). K-ragged: every expert owns m_tiles x n_tiles.
template <int KIND>
__device__ __forceinline__ Tile decode(int t, const Params& p, const int* offs, const int* tstart) {
  Tile tl;
  if (!Traits<KIND>::kragged) {
    int lo = 0, hi = p.E;  // find e with tstart[e] <= t < tstart[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tstart[mid] <= t) lo = mid; else hi = mid;
    }
    const int e = lo, local = t - tstart[e];
    tl.e = e;
    tl.m_idx = local / p.n_tiles;
    tl.n_idx = local % p.n_tiles;
    tl.m0 = offs[e] + tl.m_idx * BM;
    tl.row_end = offs[e + 1];
    const int K = (KIND == FPROP1 || KIND == DGRAD2 || KIND == ROUTER) ? p.d : (KIND == FPROP2 ? p.f : 2 * p.f);
    tl.nkb = K / BK;
    tl.k_row0 = 0;
  } else {
    const int per = p.m_tiles * p.n_tiles;
    tl.e = t / per;
    const int local = t % per;
    tl.m_idx = local / p.n_tiles;
    tl.n_idx = local % p.n_tiles;
    tl.m0 = tl.m_idx * BM;
    tl.row_end = offs[tl.e + 1];
    tl.k_row0 = offs[tl.e];
    tl.nkb = (tl.row_end - tl.k_row0 + BK - 1) / BK;
  }
  return tl;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * i + 2 * j], v[8 * i + 2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    d[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = s[i];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const Params p) {
  using Tr = Traits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem* sm = reinterpret_cast<Smem*>(smem + STAGES * STAGE_BYTES);
  int* offs = reinterpret_cast<int*>(sm + 1);
  int* tstart = offs + (p.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- prologue: offsets and the tile table in shared memory
  if (p.offsets) {
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) offs[i] = p.offsets[i];
  } else if (threadIdx.x == 0) {
    offs[0] = 0;
    offs[1] = p.R;
  }
  __syncthreads();
  int total;
  if (!Tr::kragged) {
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        const int cnt = e < p.E ? offs[e + 1] - offs[e] : 0;
        int v = ((cnt + BM - 1) / BM) * p.n_tiles, incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int nb = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += nb;
        }
        if (e < p.E) tstart[e] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) tstart[p.E] = carry;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm->full[s], 1);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm->tfull[b], 1);
      ptx::mbar_init(&sm->tempty[b], NUM_EPI_WARPS);
    }
    ptx::mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  total = Tr::kragged ? p.E * p.m_tiles * p.n_tiles : tstart[p.E];
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ===================================================== TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB0);
      ptx::prefetch_tmap(&tmB1);
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode<KIND>(t, p, offs, tstart);
        for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!wait_bar(&sm->empty[s], ph ^ 1u, sm, p.err)) { ok = false; break; }
          uint8_t* a = smem + s * STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          uint64_t* fb = &sm->full[s];
          ptx::mbar_expect_tx(fb, STAGE_BYTES);
          const int k0 = kb * BK;
          if (KIND == FPROP1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * 128;
            ptx::tma_load_3d(b + 0 * BOX_BYTES, &tmB0, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + 1 * BOX_BYTES, &tmB0, fb, n0 + 64, k0, tl.e);
            ptx::tma_load_3d(b + 2 * BOX_BYTES, &tmB1, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + 3 * BOX_BYTES, &tmB1, fb, n0 + 64, k0, tl.e);
          } else if (KIND == FPROP2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * BN;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_3d(b + j * BOX_BYTES, &tmB0, fb, n0 + 64 * j, k0, tl.e);
          } else if (KIND == DGRAD2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
          } else if (KIND == ROUTER) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            ptx::tma_load_2d(b, &tmB0, fb, k0, tl.n_idx * BN);
          } else if (KIND == DGRAD1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            if (k0 < p.f) ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
            else ptx::tma_load_3d(b, &tmB1, fb, k0 - p.f, tl.n_idx * BN, tl.e);
          } else {  // WGRAD2 / WGRAD1: K runs over the expert's rows
            const int row = tl.k_row0 + k0;
            ptx::tma_load_2d(a + 0 * BOX_BYTES, &tmA, fb, tl.m0, row);
            ptx::tma_load_2d(a + 1 * BOX_BYTES, &tmA, fb, tl.m0 + 64, row);
            const int n0 = tl.n_idx * BN;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_2d(b + j * BOX_BYTES, &tmB0, fb, n0 + 64 * j, row);
          }
        }
      }
      if (!ok) {
        // drain: wait (bounded) for loads already issued into stages the MMA will not consume
        for (int s = 0; s < STAGES; ++s) {
          const long long t0 = clock64();
          while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                 !ptx::mbar_try_wait(&sm->full[s], 1)) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ========================================================= MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, Tr::a_mn ? 1 : 0, Tr::b_mn ? 1 : 0);
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode<KIND>(t, p, offs, tstart);
      if (tl.nkb == 0) continue;
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!wait_bar(&sm->tempty[buf], aph ^ 1u, sm, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        if (!wait_bar(&sm->full[s], ph, sm, p.err)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * STAGE_BYTES;
        if (Tr::kragged) {
          const int valid = tl.row_end - (tl.k_row0 + kb * BK);
          if (valid < BK) {
            // rows past the expert's end belong to the next expert: zero them in A
            const int nrow = BK - valid, per_box = nrow * 8;
            for (int i = lane; i < 2 * per_box; i += 32) {
              const int box = i / per_box, rem = i % per_box;
              const int row = valid + rem / 8, chunk = rem % 8;
              *reinterpret_cast<uint4*>(a + box * BOX_BYTES + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = Tr::a_mn ? ptx::smem_desc_sw128(a_addr + ks * 2048, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = Tr::b_mn ? ptx::smem_desc_sw128(b_addr + ks * 2048, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            ptx::mma_f16(d_tmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&sm->empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(&sm->tfull[buf]);
      __syncwarp();
      ++acc_it;
    }
    if (!ok && lane == 0) {
      // let issued MMAs finish before TMEM is released
      ptx::mma_commit(&sm->drain);
      const long long t0 = clock64();
      while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->drain, 0)) {
      }
    }
  } else {
    // ============================================================ epilogue
    // Warp w reads TMEM lanes 32*(w%4)..+31 (rows of the tile); the two warps
    // of a quadrant split the tile's columns in halves.
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    const int row_in_tile = q * 32 + lane;
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND>(t, p, offs, tstart);
      if (Tr::kragged) {
        const int m = tl.m0 + row_in_tile;
        const int n0 = tl.n_idx * BN;
        const bool row_ok = m < p.M;
        const bool empty_k = tl.nkb == 0;
        int buf = 0;
        if (!empty_k) {
          buf = acc_it & 1;
          const uint32_t aph = (acc_it >> 1) & 1u;
          if (!wait_bar(&sm->tfull[buf], aph, sm, p.err)) break;
          ptx::tc_fence_after();
        }
        const uint32_t tbase = tmem + static_cast<uint32_t>(buf * BN) + (static_cast<uint32_t>(q * 32) << 16);
        for (int c = half * 4; c < half * 4 + 4; ++c) {
          float v[32];
          if (!empty_k) {
            uint32_t r[32];
            ptx::tmem_ld32(tbase + c * 32, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          const int n = n0 + c * 32;
          if (!row_ok || n >= p.N) continue;
          __nv_bfloat16* dst;
          if (KIND == WGRAD2) dst = static_cast<__nv_bfloat16*>(p.out0) + ((size_t)tl.e * p.M + m) * p.N + n;
          else dst = n < p.f ? static_cast<__nv_bfloat16*>(p.out0) + ((size_t)tl.e * p.d + m) * p.f + n
                             : static_cast<__nv_bfloat16*>(p.out1) + ((size_t)tl.e * p.d + m) * p.f + (n - p.f);
          store_bf16x32(dst, v);
        }
        if (!empty_k) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm->tempty[buf]);
          ++acc_it;
        }
        continue;
      }
      // row-ragged epilogues
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      const int row = tl.m0 + row_in_tile;
      const bool row_ok = row < tl.row_end;
      if (!wait_bar(&sm->tfull[buf], aph, sm, p.err)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + static_cast<uint32_t>(buf * BN) + (static_cast<uint32_t>(q * 32) << 16);
      if (KIND == FPROP1) {
        const int n0 = tl.n_idx * 128;
        for (int c = half * 2; c < half * 2 + 2; ++c) {
          uint32_t rg[32], ru[32];
          ptx::tmem_ld32(tbase + c * 32, rg);
          ptx::tmem_ld32(tbase + 128 + c * 32, ru);
          ptx::tmem_wait_ld();
          const int n = n0 + c * 32;
          if (!row_ok || n >= p.f) continue;
          float hg[32], hu[32], av[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            hg[i] = __uint_as_float(rg[i]);
            hu[i] = __uint_as_float(ru[i]);
            av[i] = silu_f(hg[i]) * hu[i];
          }
          __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out0) + (size_t)row * 2 * p.f;
          store_bf16x32(h + n, hg);
          store_bf16x32(h + p.f + n, hu);
          store_bf16x32(static_cast<__nv_bfloat16*>(p.out1) + (size_t)row * p.f + n, av);
        }
      } else if (KIND == DGRAD2) {
        // dh_g = da * h_u * silu'(h_g), dh_u = da * silu(h_g); h is loaded before the
        // accumulator so the global latency overlaps the TMEM read
        const int n0 = tl.n_idx * BN;
        const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(p.aux) + (size_t)row * 2 * p.f;
        __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(p.out0) + (size_t)row * 2 * p.f;
        for (int c = half * 4; c < half * 4 + 4; ++c) {
          const int n = n0 + c * 32;
          const bool ok = row_ok && n < p.N;
          float hg[32], hu[32];
          if (ok) {
            load_bf16x32(h + n, hg);
            load_bf16x32(h + p.f + n, hu);
          }
          uint32_t r[32];
          ptx::tmem_ld32(tbase + c * 32, r);
          ptx::tmem_wait_ld();
          if (!ok) continue;
          float dg[32], du[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float da = __uint_as_float(r[i]);
            const float s = sigmoid_f(hg[i]);
            dg[i] = da * hu[i] * s * (1.0f + hg[i] * (1.0f - s));
            du[i] = da * hg[i] * s;
          }
          store_bf16x32(dh + n, dg);
          store_bf16x32(dh + p.f + n, du);
        }
      } else if (KIND == ROUTER) {
        const int n0 = tl.n_idx * BN;
        float* out = static_cast<float*>(p.out0) + (size_t)row * p.N;
        for (int c = half * 4; c < half * 4 + 4; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(tbase + c * 32, r);
          ptx::tmem_wait_ld();
          const int n = n0 + c * 32;
          if (!row_ok || n >= p.N) continue;
          if (n + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 o;
              o.x = __uint_as_float(r[i]) + (p.bias ? p.bias[n + i] : 0.0f);
              o.y = __uint_as_float(r[i + 1]) + (p.bias ? p.bias[n + i + 1] : 0.0f);
              o.z = __uint_as_float(r[i + 2]) + (p.bias ? p.bias[n + i + 2] : 0.0f);
              o.w = __uint_as_float(r[i + 3]) + (p.bias ? p.bias[n + i + 3] : 0.0f);
              *reinterpret_cast<float4*>(out + n + i) = o;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (n + i < p.N) out[n + i] = __uint_as_float(r[i]) + (p.bias ? p.bias[n + i] : 0.0f);
          }
        }
      } else {  // FPROP2, DGRAD1: plain bf16 store
        const int n0 = tl.n_idx * BN;
        for (int c = half * 4; c < half * 4 + 4; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(tbase + c * 32, r);
          ptx::tmem_wait_ld();
          const int n = n0 + c * 32;
          if (!row_ok || n >= p.N) continue;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          store_bf16x32(static_cast<__nv_bfloat16*>(p.out0) + (size_t)row * p.N + n, v);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm->tempty[buf]);
      ++acc_it;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 [rows][inner] row-major, box (box_inner, box_rows), 128-byte swizzle
bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
            uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, rows > 0 ? rows : 1};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [E][rows][inner], box (box_inner, box_rows, 1)
bool map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t E, uint32_t box_inner,
            uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, E};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t smem_bytes(int E) { return 1024 + STAGES * STAGE_BYTES + sizeof(Smem) + 2 * (E + 1) * sizeof(int) + 64; }

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  }
  return n;
}

template <int KIND>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const Params& p,
                   long max_tiles, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = smem_bytes(p.E);
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
  MOE_COUNTED tc_gemm_kernel<KIND><<<grid, NUM_THREADS, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

}  // namespace tc

using namespace tc;

cudaError_t tc_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd,
                       const int32_t* offsets, int R, int E, int d, int f, void* h, void* a, void* y,
                       cudaStream_t st) {
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  // GEMM1 + SwiGLU: tiles of 128 f-columns (gate 128 | up 128 in one N=256 MMA)
  if (!map_2d(&mA, x_perm, d, R, 64, BM) || !map_3d(&mB0, wg, f, d, E, 64, 64) ||
      !map_3d(&mB1, wu, f, d, E, 64, 64))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + 127) / 128; p.out0 = h; p.out1 = a;
  cudaError_t e = launch<FPROP1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
  if (e != cudaSuccess) return e;
  // GEMM2
  if (!map_2d(&mA, a, f, R, 64, BM) || !map_3d(&mB0, wd, d, f, E, 64, 64)) return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = y; p.out1 = nullptr;
  return launch<FPROP2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
}

cudaError_t tc_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* dh, cudaStream_t st) {
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  cudaError_t e;
  // dA = dy . Wd^T with the SwiGLU backward fused: writes dh
  if (!map_2d(&mA, dy_perm, d, R, 64, BM) || !map_3d(&mB0, wd, d, f, E, 64, BN)) return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + BN - 1) / BN; p.out0 = dh; p.aux = h;
  e = launch<DGRAD2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
  if (e != cudaSuccess) return e;
  // dWd[e] = A_e^T dy_e
  if (!map_2d(&mA, a, f, R, 64, 64) || !map_2d(&mB0, dy_perm, d, R, 64, 64)) return cudaErrorInvalidValue;
  p.M = f; p.N = d; p.m_tiles = (f + BM - 1) / BM; p.n_tiles = (d + BN - 1) / BN; p.out0 = dwd;
  e = launch<WGRAD2>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st);
  if (e != cudaSuccess) return e;
  // dx_perm = dh_g . Wg^T + dh_u . Wu^T
  if (!map_2d(&mA, dh, 2L * f, R, 64, BM) || !map_3d(&mB0, wg, f, d, E, 64, BN) ||
      !map_3d(&mB1, wu, f, d, E, 64, BN))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = dx_perm; p.aux = nullptr;
  e = launch<DGRAD1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
  if (e != cudaSuccess) return e;
  // [dWg | dWu][e] = x_perm_e^T dh_e
  if (!map_2d(&mA, x_perm, d, R, 64, 64) || !map_2d(&mB0, dh, 2L * f, R, 64, 64)) return cudaErrorInvalidValue;
  p.M = d; p.N = 2 * f; p.m_tiles = (d + BM - 1) / BM; p.n_tiles = (2 * f + BN - 1) / BN;
  p.out0 = dwg; p.out1 = dwu;
  return launch<WGRAD1>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st);
}

cudaError_t tc_router_logits(const void* x, const void* w_r, const float* bias, int T, int d, int E,
                             float* logits, cudaStream_t st) {
  CUtensorMap mA, mB;
  Params p{};
  p.offsets = nullptr; p.bias = bias; p.E = 1; p.R = T; p.d = d; p.f = 0; p.err = device_error_word();
  if (!map_2d(&mA, x, d, T, 64, BM) || !map_2d(&mB, w_r, d, E, 64, BN)) return cudaErrorInvalidValue;
  p.N = E; p.n_tiles = (E + BN - 1) / BN; p.out0 = logits;
  return launch<ROUTER>(mA, mB, mB, p, (long)((T + BM - 1) / BM) * p.n_tiles, st);
}

}  // namespace moe
