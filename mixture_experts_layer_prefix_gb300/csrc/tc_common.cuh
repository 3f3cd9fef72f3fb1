// tc_common.cuh -- pieces shared by the bf16 and the MXFP8 grouped GEMMs:
// the GEMM kinds, kernel parameters, the device-side ragged tile decoder, the
// bounded mbarrier wait and the fused epilogues (TMEM accumulator -> bf16 or
// fp32 outputs, with the SwiGLU forward/backward math).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "mxfp8_common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BN = 256, STAGES = 4;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz

// The six grouped expert GEMMs of the SwiGLU layer and the router GEMM.
enum Kind { FPROP1 = 0, FPROP2 = 1, DGRAD2 = 2, DGRAD1 = 3, WGRAD2 = 4, WGRAD1 = 5, ROUTER = 6 };

struct Params {
  const int32_t* offsets;  // [E+1] device offsets; nullptr: one dense group of R rows
  const float* bias;       // router: per-column bias (or nullptr)
  int E, R, d, f;
  int N;                   // output columns of the GEMM
  int M;                   // wgrad: output rows
  int n_tiles, m_tiles;
  void* out0;
  void* out1;
  const void* aux;         // DGRAD2: h_save
  const uint8_t* sfa;      // MXFP8: scale bytes of A (layout per kind)
  const uint8_t* sfb0;     // MXFP8: scale bytes of B (gate / the only B)
  const uint8_t* sfb1;     // MXFP8: scale bytes of the second B (up)
  uint8_t* qout;           // optional: the epilogue also writes its bf16 output
  uint8_t* qsc;            //   quantised along rows (E4M3 codes, E8M0 per 32)
  uint8_t* qcol;           // optional (GEMM2 dgrad): ... and along the expert's
  uint8_t* qcsc;           //   rows in blocks of 32 (weight-gradient operand)
  // Dispatch fused into the A operand (GEMM1 forward and wgrad): row r of A is
  // row src_row[r] / gk of x [T][d] (A's tensor map); nullptr: A is x_perm.
  const int32_t* src_row;
  int gk, T;
  // Weight-gradient kinds: experts in the order their tiles are walked
  // (largest row count first, from expert_order_kernel); nullptr: 0..E-1.
  const int32_t* order;
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

// Bounded wait on an mbarrier phase, at most `limit` SM cycles. On expiry:
// set the device error word and the CTA's abort flag (so the other roles stop
// too) and return false; a wait that sees the abort flag returns false too.
__device__ __forceinline__ bool wait_bar_for(uint64_t* bar, uint32_t parity, int* abort_flag, int* err,
                                             long long limit) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (clock64() - t0 > limit) {
      set_error(err, MOE_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int* abort_flag, int* err) {
  return wait_bar_for(bar, parity, abort_flag, err, kWaitLimitCycles);
}

struct Tile {
  int e, m0, row_end, n_idx, m_idx, nkb, k_row0;
};

// Tile index of this CTA's r-th tile. Row-tile kinds stride over the tile list
// (tile cost is the same K for every tile). Weight-gradient tiles cost their
// expert's row count, and their list runs from the largest expert down (the
// expert order table): those are walked in a snake over the CTAs (even rounds
// CTA b takes slot b, odd rounds slot G-1-b), so a falling cost spreads evenly.
template <bool KRAGGED>
__device__ __forceinline__ int sched_tile(int r) {
  const int g = gridDim.x, b = blockIdx.x;
  return KRAGGED ? r * g + ((r & 1) ? g - 1 - b : b) : b + r * g;
}

template <int KIND>
__device__ __forceinline__ int gemm_k(const Params& p) {
  return (KIND == FPROP1 || KIND == DGRAD2 || KIND == ROUTER) ? p.d : (KIND == FPROP2 ? p.f : 2 * p.f);
}

// Decode linear tile t. Row-ragged: expert e owns tstart[e]..tstart[e+1]
// (m-tiles x n-tiles, n fastest). K-ragged: every expert owns m_tiles x
// n_tiles tiles and its K loop runs over its rows, BK rows per stage.
template <int KIND, int BK, int TBM = BM>
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
    tl.m0 = offs[e] + tl.m_idx * TBM;
    tl.row_end = offs[e + 1];
    tl.nkb = gemm_k<KIND>(p) / BK;
    tl.k_row0 = 0;
  } else {
    const int per = p.m_tiles * p.n_tiles;
    tl.e = p.order ? __ldg(p.order + t / per) : t / per;
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

// Offsets into shared memory and (row-ragged kinds) the per-expert tile
// prefix table; called by all threads of the CTA, ends with __syncthreads.
template <int KIND, int NTHREADS, int TBM = BM>
__device__ __forceinline__ void build_tile_table(const Params& p, int* offs, int* tstart) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.offsets) {
    for (int i = threadIdx.x; i <= p.E; i += NTHREADS) offs[i] = p.offsets[i];
  } else if (threadIdx.x == 0) {
    offs[0] = 0;
    offs[1] = p.R;
  }
  __syncthreads();
  if (!Traits<KIND>::kragged && warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int cnt = e < p.E ? offs[e + 1] - offs[e] : 0;
      const int v = ((cnt + TBM - 1) / TBM) * p.n_tiles;
      int incl = v;
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
  __syncthreads();
}


// Row-segment traffic through a per-warp staging buffer. An epilogue thread
// owns one output row (its TMEM lane), so a direct store instruction of a
// warp touches 32 rows with 16 bytes each. Staged in shared memory (32 rows x
// 64 bytes, 16-byte granules XOR-swizzled by row pair so that the row-wise and
// the column-wise accesses are both free of bank conflicts), each global
// instruction moves 8 rows x 64 contiguous bytes.
constexpr int STG_BYTES = 32 * 64;
__device__ __forceinline__ int stg_off(int r, int g) { return r * 64 + ((g ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void pack_bf16x32(const float* v, uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// Lane r holds w = row r's 64 bytes; dst is row 0 of the warp's 32 rows
// (leading dimension ld bytes). Rows >= nrows are not written.
__device__ __forceinline__ void warp_store_rows_b(uint8_t* stg, const uint32_t (&w)[16], uint8_t* dst,
                                                  size_t ld, int nrows, int lane) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    *reinterpret_cast<uint4*>(stg + stg_off(lane, g)) = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
  __syncwarp();
  const int g = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4*>(stg + stg_off(r, g));
    if (r < nrows) *reinterpret_cast<uint4*>(dst + (size_t)r * ld + 16 * g) = v;
  }
  __syncwarp();
}
// The same for 32 bf16 values per row (ld in elements).
__device__ __forceinline__ void warp_store_rows(uint8_t* stg, const uint32_t (&w)[16], __nv_bfloat16* dst,
                                                size_t ld, int nrows, int lane) {
  warp_store_rows_b(stg, w, reinterpret_cast<uint8_t*>(dst), 2 * ld, nrows, lane);
}
// 32-byte rows (32 E4M3 codes per row): 2 granules per row, XOR-swizzled by
// row quad; each global instruction moves 16 rows x 32 bytes.
__device__ __forceinline__ int stg32_off(int r, int g) { return r * 32 + ((g ^ ((r >> 2) & 1)) << 4); }
__device__ __forceinline__ void warp_store_rows32(uint8_t* stg, const uint32_t (&w)[8], uint8_t* dst, size_t ld,
                                                  int nrows, int lane) {
#pragma unroll
  for (int g = 0; g < 2; ++g)
    *reinterpret_cast<uint4*>(stg + stg32_off(lane, g)) = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
  __syncwarp();
  const int g = lane & 1;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 16 * i + (lane >> 1);
    const uint4 v = *reinterpret_cast<const uint4*>(stg + stg32_off(r, g));
    if (r < nrows) *reinterpret_cast<uint4*>(dst + (size_t)r * ld + 16 * g) = v;
  }
  __syncwarp();
}
// Scale chunk row of row q * 32 + lane of a row tile, in the per-expert
// 128-row tile layout of an operand with K = ld (see mxfp8_common.cuh).
__device__ __forceinline__ size_t tile_scale_row(const Tile& tl, int q, int lane, int ld) {
  const long grp = mx_row_tile_base(tl.m0 - tl.m_idx * BM, tl.e) + tl.m_idx;
  return ((size_t)grp * (ld / 128) << 9) + mx_chunk_lane(q * 32 + lane);
}
// MXFP8 row quantisation of a 32-column chunk held as packed bf16 pairs (the
// stored values): codes to qout[row][col..col+32) through the staging buffer
// ([rows][ld] matrix), the scale byte of each valid row into its scale chunk
// (srow: the lane's tile_scale_row).
__device__ __forceinline__ void quant_rows_staged(const Params& p, uint8_t* stg, const uint32_t (&w)[16], int wrow,
                                                  int nrows, int ld, int col, int lane, size_t srow) {
  const float amax = absmax_bf16x32(w);
  const int sx = mx_e8m0_exponent(amax);
  const float m = mx_pow2_neg(sx);
  uint32_t cw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    cw[i] = mx_e4m3x2(__uint_as_float(w[2 * i] << 16) * m, __uint_as_float(w[2 * i] & 0xFFFF0000u) * m) |
            (mx_e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * m, __uint_as_float(w[2 * i + 1] & 0xFFFF0000u) * m) << 16);
  const uint8_t sb = static_cast<uint8_t>(sx + 127);
  if (lane < nrows) p.qsc[srow + ((size_t)(col >> 7) << 9) + ((col >> 5) & 3)] = sb;
  warp_store_rows32(stg, cw, p.qout + (size_t)wrow * ld + col, ld, nrows, lane);
}

// MXFP8 quantisation of the same chunk along its rows, in blocks of 32 rows:
// the warp's rows are one such block of the expert segment (rows >= nrows are
// past the segment's end and count as zero). Codes to qcol[row][col..col+32)
// ([rows][ld] matrix), the scale of column col + lane into its scale chunk
// (K stage `stage`, the block q within it; a block wholly past the end gets
// 127). The column maxima come from a butterfly over the lanes on bf16 pairs
// (16 shuffles: lane l ends with column l's), the 32 scale factors return to every lane
// through 128 bytes of the warp's staging buffer, and each lane encodes its own
// row, which leaves as 16 rows x 32 B per store.
__device__ __forceinline__ void quant_cols_staged(const Params& p, uint8_t* stg, const uint32_t (&w)[16], int wrow,
                                                  int nrows, int ld, int col, int lane, long stage, int q) {
  const uint32_t live = lane < nrows ? 0x7FFF7FFFu : 0u;  // magnitudes; rows past the end count as zero
  uint32_t a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = w[i] & live;
  colmax_step<8>(a, lane);
  colmax_step<4>(a, lane);
  colmax_step<2>(a, lane);
  colmax_step<1>(a, lane);
  a[0] = bf16x2_max(a[0], __shfl_xor_sync(0xffffffffu, a[0], 1));
  const int sx = mx_e8m0_exponent((lane & 1) ? bf16_hi(a[0]) : bf16_lo(a[0]));  // column col + lane
  float* ms = reinterpret_cast<float*>(stg);
  ms[lane] = mx_pow2_neg(sx);
  __syncwarp();
  float m[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = reinterpret_cast<const float4*>(ms)[i];
    m[4 * i] = v.x; m[4 * i + 1] = v.y; m[4 * i + 2] = v.z; m[4 * i + 3] = v.w;
  }
  __syncwarp();  // the buffer is reused for the codes below
  uint32_t cw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    cw[i] = mx_e4m3x2(bf16_lo(w[2 * i]) * m[4 * i], bf16_hi(w[2 * i]) * m[4 * i + 1]) |
            (mx_e4m3x2(bf16_lo(w[2 * i + 1]) * m[4 * i + 2], bf16_hi(w[2 * i + 1]) * m[4 * i + 3]) << 16);
  warp_store_rows32(stg, cw, p.qcol + (size_t)wrow * ld + col, ld, nrows, lane);
  const int c = col + lane;
  p.qcsc[((stage * (ld / 128) + c / 128) << 9) + mx_chunk_lane(c & 127) + q] =
      static_cast<uint8_t>(nrows > 0 ? sx + 127 : 127);
}

// The reverse, in two halves so that the global latency can overlap other
// work: issue reads the warp's 32 rows x 32 bf16 from src coalesced (rows >=
// nrows read as zero); finish hands lane r row r (16 packed bf16 pairs).
__device__ __forceinline__ void warp_load_rows_issue(uint4 (&t)[4], const __nv_bfloat16* src, size_t ld, int nrows,
                                                     int lane) {
  const int g = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    t[i] = r < nrows ? *reinterpret_cast<const uint4*>(src + (size_t)r * ld + 8 * g) : make_uint4(0, 0, 0, 0);
  }
}
__device__ __forceinline__ void warp_load_rows_finish(uint8_t* stg, const uint4 (&t)[4], uint32_t (&w)[16],
                                                      int lane) {
  const int g0 = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(stg + stg_off(8 * i + (lane >> 2), g0)) = t[i];
  __syncwarp();
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint4 q = *reinterpret_cast<const uint4*>(stg + stg_off(lane, g));
    w[4 * g] = q.x;
    w[4 * g + 1] = q.y;
    w[4 * g + 2] = q.z;
    w[4 * g + 3] = q.w;
  }
  __syncwarp();
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Staged form of the row-tile epilogue (see warp_store_rows): every lane of
// the warp takes part; stg is the warp's STG_BYTES buffer. Row-tile kinds
// FPROP1, FPROP2, DGRAD1, DGRAD2 without quantisation.
template <int KIND, int TBN = BN, bool QUANT = false>
__device__ __forceinline__ void epilogue_tile_staged(const Params& p, const Tile& tl, uint32_t tbase, int q, int lane,
                                                     int c_beg, int c_end, uint8_t* stg) {
  static_assert(KIND == FPROP1 || KIND == FPROP2 || KIND == DGRAD1 || KIND == DGRAD2, "row-tile kinds");
  const int wrow = tl.m0 + q * 32;  // the warp's first row
  const int nrows = max(0, min(32, tl.row_end - wrow));
  uint32_t w[16];
  if (KIND == FPROP1) {
    const int n0 = tl.n_idx * 128;
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * 2 * p.f;
    __nv_bfloat16* a = static_cast<__nv_bfloat16*>(p.out1) + (size_t)wrow * p.f;
    for (int c = c_beg; c < c_end; ++c) {
      uint32_t rg[32], ru[32];
      ptx::tmem_ld32(tbase + c * 32, rg);
      ptx::tmem_ld32(tbase + 128 + c * 32, ru);
      ptx::tmem_wait_ld();
      const int n = n0 + c * 32;
      if (n >= p.f) continue;
      uint32_t wa[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float g0 = __uint_as_float(rg[2 * i]), g1 = __uint_as_float(rg[2 * i + 1]);
        const float u0 = __uint_as_float(ru[2 * i]), u1 = __uint_as_float(ru[2 * i + 1]);
        wa[i] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
        w[i] = pack_bf16x2(g0, g1);
      }
      warp_store_rows(stg, w, h + n, 2 * (size_t)p.f, nrows, lane);
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(ru[2 * i]), __uint_as_float(ru[2 * i + 1]));
      warp_store_rows(stg, w, h + p.f + n, 2 * (size_t)p.f, nrows, lane);
      warp_store_rows(stg, wa, a + n, p.f, nrows, lane);
      if (QUANT && p.qout) quant_rows_staged(p, stg, wa, wrow, nrows, p.f, n, lane, tile_scale_row(tl, q, lane, p.f));
    }
  } else if (KIND == DGRAD2) {
    // dh_g = da * h_u * silu'(h_g), dh_u = da * silu(h_g); the reads of h are
    // issued before the accumulator load so their latency overlaps it
    const int n0 = tl.n_idx * TBN;
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(p.aux) + (size_t)wrow * 2 * p.f;
    __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * 2 * p.f;
    for (int c = c_beg; c < c_end; ++c) {
      const int n = n0 + c * 32;
      const bool nok = n < p.N;
      uint4 tg[4], tu[4];
      if (nok) {
        warp_load_rows_issue(tg, h + n, 2 * (size_t)p.f, nrows, lane);
        warp_load_rows_issue(tu, h + p.f + n, 2 * (size_t)p.f, nrows, lane);
      }
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c * 32, r);
      ptx::tmem_wait_ld();
      if (!nok) continue;
      uint32_t hg[16], hu[16], wu[16];
      warp_load_rows_finish(stg, tg, hg, lane);
      warp_load_rows_finish(stg, tu, hu, lane);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float dg2[2], du2[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float g = j ? bf16_hi(hg[i]) : bf16_lo(hg[i]);
          const float u = j ? bf16_hi(hu[i]) : bf16_lo(hu[i]);
          const float da = __uint_as_float(r[2 * i + j]);
          const float s = sigmoid_f(g);
          dg2[j] = da * u * s * (1.0f + g * (1.0f - s));
          du2[j] = da * g * s;
        }
        w[i] = pack_bf16x2(dg2[0], dg2[1]);
        wu[i] = pack_bf16x2(du2[0], du2[1]);
      }
      if (!QUANT || p.out0) {
        warp_store_rows(stg, w, dh + n, 2 * (size_t)p.f, nrows, lane);
        warp_store_rows(stg, wu, dh + p.f + n, 2 * (size_t)p.f, nrows, lane);
      }
      if (QUANT && p.qout) {
        const size_t srow = tile_scale_row(tl, q, lane, 2 * p.f);
        quant_rows_staged(p, stg, w, wrow, nrows, 2 * p.f, n, lane, srow);
        quant_rows_staged(p, stg, wu, wrow, nrows, 2 * p.f, p.f + n, lane, srow);
      }
      if (QUANT && p.qcol) {
        const long stage = mx_row_tile_base(tl.m0 - tl.m_idx * BM, tl.e) + tl.m_idx;
        quant_cols_staged(p, stg, w, wrow, nrows, 2 * p.f, n, lane, stage, q);
        quant_cols_staged(p, stg, wu, wrow, nrows, 2 * p.f, p.f + n, lane, stage, q);
      }
    }
  } else {  // FPROP2, DGRAD1: plain bf16 store
    const int n0 = tl.n_idx * TBN;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * p.N;
    for (int c = c_beg; c < c_end; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(tbase + c * 32, r);
      ptx::tmem_wait_ld();
      const int n = n0 + c * 32;
      if (n >= p.N) continue;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      pack_bf16x32(v, w);
      warp_store_rows(stg, w, out + n, p.N, nrows, lane);
    }
  }
}

// Epilogue of a router-logits tile for the rows of one TMEM lane quadrant
// (lane = row): fp32 logits plus the optional bias, accumulator chunks
// [c_beg, c_end) of 32 columns.
template <int TBN = BN>
__device__ __forceinline__ void epilogue_router(const Params& p, const Tile& tl, uint32_t tbase, int row_in_tile,
                                                int c_beg, int c_end) {
  const int row = tl.m0 + row_in_tile;
  const bool row_ok = row < tl.row_end;
  const int n0 = tl.n_idx * TBN;
  float* out = static_cast<float*>(p.out0) + (size_t)row * p.N;
  for (int c = c_beg; c < c_end; ++c) {
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
}

// Number of 32-column accumulator chunks an epilogue covers (FPROP1 pairs).
template <int KIND>
__host__ __device__ constexpr int epi_chunks() { return KIND == FPROP1 ? 4 : BN / 32; }

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encoder();
// [rows][inner] row-major, box (box_inner, box_rows), 128-byte swizzle
bool map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
            uint64_t rows, uint32_t box_inner, uint32_t box_rows);
// [E][rows][inner], box (box_inner, box_rows, 1)
bool map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
            uint64_t rows, uint64_t E, uint32_t box_inner, uint32_t box_rows);
int sm_count();

}  // namespace tc
}  // namespace moe
