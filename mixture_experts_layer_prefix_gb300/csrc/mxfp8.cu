// mxfp8.cu -- MXFP8 block quantisation ("Introducing Olmo-core 3", section
// "Scaling and optimizing MoE training": MXFP8, a lower-precision format whose
// savings must exceed the cost of converting between formats).
//
// A block is 32 consecutive elements along the GEMM's K. Its E8M0 byte is
// s + 127 with s = ceil(log2(amax / 448)) clamped to [-127, 127] (the
// smallest power of two that needs no saturation; an all-zero block gets
// s = -127); elements are round-to-nearest-even of v * 2^-s, saturated to
// +-448, through CUDA's fp8 conversion.
//
//   rows kernel: blocks along the contiguous axis of [rows][K]; one thread per
//                block (64 B in, 32 B + 1 B out), coalesced across threads.
//   cols kernel: blocks of 32 consecutive rows of one column, starting at each
//                segment's first row (segments = per-expert row ranges from
//                the device offsets); a segment's last block is zero-padded.
//                Each thread owns 2 columns and keeps the block's 32 rows in
//                registers between the maxima and the conversion.
//   dual kernel: a weight tile read once and written quantised both ways.
//   dispatch:    the permute with each token's row quantised once (below).
// The GEMM operands' scales are written as scale chunks (mxfp8_common.cuh);
// mxfp8_quantize's public layouts are the plain ones.
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "mxfp8_common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int e8m0_exponent(float amax) { return mx_e8m0_exponent(amax); }
__device__ __forceinline__ float pow2_neg(int s) { return mx_pow2_neg(s); }

// MODE (ScaleLayout): where the scale byte of block b of row r goes.
template <int MODE>
__global__ void __launch_bounds__(256)
quant_rows_kernel(const __nv_bfloat16* __restrict__ src, long nblocks, int kblocks, uint8_t* __restrict__ q,
                  uint8_t* __restrict__ sc, const int32_t* __restrict__ offs, int E) {
  const long blk = blockIdx.x * (long)blockDim.x + threadIdx.x;
  if (blk >= nblocks) return;
  float v[32];
  const __nv_bfloat16* p = src + blk * 32;
#pragma unroll
  for (int i = 0; i < 4; ++i) Vec16<__nv_bfloat16>::load(p + 8 * i, v + 8 * i);
  uint32_t w[8];
  const uint8_t s = mx_quant_block32_regs(v, w);
  uint4* out = reinterpret_cast<uint4*>(q + blk * 32);
  out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  out[1] = make_uint4(w[4], w[5], w[6], w[7]);
  if (MODE == kScalesPlain) {
    sc[blk] = s;
    return;
  }
  const long row = blk / kblocks;
  const int b = static_cast<int>(blk % kblocks);
  long grp;
  int t;
  if (MODE == kScalesChunk) {
    grp = row >> 7;
    t = static_cast<int>(row & 127);
  } else {
    int lo = 0, hi = E;  // the expert holding the row: offs[lo] <= row < offs[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(offs + mid) <= row) lo = mid; else hi = mid;
    }
    const long local = row - __ldg(offs + lo);
    grp = mx_row_tile_base(__ldg(offs + lo), lo) + (local >> 7);
    t = static_cast<int>(local & 127);
  }
  sc[((grp * (kblocks / 4) + b / 4) << 9) + mx_chunk_lane(t) + (b & 3)] = s;
}

// Block-row table: segment g owns block rows [bstart[g], bstart[g+1]).
// PACKED: scales go to scale chunks (GEMM operand layout): K stage w (four
// block rows of a segment; the stages of segment g are numbered from
// mx_row_tile_base(seg[g], g), like the segment's 128-row tiles) and column
// group c / 128 form chunk w * (C / 128) + c / 128, and block j of the stage
// of column c is byte mx_chunk_lane(c % 128) + j of it; bytes past a
// segment's last block are 127.
// A CTA handles kColBlockRows block rows of 256 columns; each thread owns 2
// consecutive columns (a warp reads 128 contiguous bytes of a row) and holds
// its 32 x 2 block in registers, so every input byte is read from memory
// once (block maxima, then conversion) at an occupancy that keeps enough
// loads in flight.
constexpr int kColBlockRows = 4;

template <bool PACKED>
__global__ void __launch_bounds__(128, 6)
quant_cols_kernel(const __nv_bfloat16* __restrict__ src, int rows, int C, const int32_t* __restrict__ seg,
                  int nseg, uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  extern __shared__ int bstart[];  // nseg + 1 block-row starts
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base < nseg; base += 32) {
      const int g = base + lane;
      int len = 0;
      if (g < nseg) len = seg ? seg[g + 1] - seg[g] : rows;
      const int v = (len + 31) / 32;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      if (g < nseg) bstart[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) bstart[nseg] = carry;
  }
  __syncthreads();
  __shared__ __align__(16) uint8_t cbuf[32 * 256];  // the block row's codes, [row][256 columns]
  const int c = (blockIdx.x * 128 + tid) * 2;  // x: column slices, so CTAs in flight share rows
  const bool act = c < C;  // C % 8 == 0: the 8- or 16-byte pieces below are all in or all out
  const int ngroups = (bstart[nseg] + kColBlockRows - 1) / kColBlockRows;
  for (int grp = blockIdx.y; grp < ngroups; grp += gridDim.y)
  for (int brow = grp * kColBlockRows; brow < (grp + 1) * kColBlockRows; ++brow) {
    if (brow >= bstart[nseg]) break;
    int lo = 0, hi = nseg;  // bstart[lo] <= brow < bstart[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (bstart[mid] <= brow) lo = mid; else hi = mid;
    }
    const int g0 = seg ? seg[lo] : 0, g1 = seg ? seg[lo + 1] : rows;
    const int local = brow - bstart[lo];
    const int r0 = g0 + local * 32, nr = min(32, g1 - r0);
    uint32_t blk[32];
    const uint32_t* sp = reinterpret_cast<const uint32_t*>(src + (size_t)r0 * C + (act ? c : 0));
    const int cw = C / 2;  // row stride in 32-bit words
#pragma unroll
    for (int i = 0; i < 32; ++i) blk[i] = (act && i < nr) ? __ldg(sp + i * cw) : 0u;
    float amax0 = 0.0f, amax1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      amax0 = fmaxf(amax0, fabsf(__uint_as_float(blk[i] << 16)));
      amax1 = fmaxf(amax1, fabsf(__uint_as_float(blk[i] & 0xFFFF0000u)));
    }
    int sx[2];
    sx[0] = e8m0_exponent(amax0);
    sx[1] = e8m0_exponent(amax1);
    const float m0 = pow2_neg(sx[0]), m1 = pow2_neg(sx[1]);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t b = mx_e4m3x2(__uint_as_float(blk[i] << 16) * m0, __uint_as_float(blk[i] & 0xFFFF0000u) * m1);
      *reinterpret_cast<uint16_t*>(cbuf + i * 256 + 2 * tid) = static_cast<uint16_t>(b);
    }
    __syncthreads();
    if ((C & 15) == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 16 threads per row, 16 bytes each
        const int id = tid + 128 * j, r = id >> 4, g = id & 15;
        const int cc = blockIdx.x * 256 + 16 * g;
        if (r < nr && cc < C)
          *reinterpret_cast<uint4*>(q + (size_t)(r0 + r) * C + cc) = *reinterpret_cast<const uint4*>(cbuf + r * 256 + 16 * g);
      }
    } else {  // C % 16 == 8: rows start 8-byte aligned only
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // 32 threads per row, 8 bytes each
        const int id = tid + 128 * j, r = id >> 5, g = id & 31;
        const int cc = blockIdx.x * 256 + 8 * g;
        if (r < nr && cc < C)
          *reinterpret_cast<uint2*>(q + (size_t)(r0 + r) * C + cc) = *reinterpret_cast<const uint2*>(cbuf + r * 256 + 8 * g);
      }
    }
    __syncthreads();
    if (!act) continue;
    if (!PACKED) {
      const uint32_t b = static_cast<uint32_t>(sx[0] + 127) | static_cast<uint32_t>(sx[1] + 127) << 8;
      *reinterpret_cast<uint16_t*>(sc + (size_t)brow * C + c) = static_cast<uint16_t>(b);
    } else {
      const long word = mx_row_tile_base(g0, lo) + local / 4;
      const int byte = local % 4;
      const bool last = brow == bstart[lo + 1] - 1;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint8_t* w = sc + (((size_t)word * (C / 128) + (c + j) / 128) << 9) + mx_chunk_lane(c + j);
        w[byte] = static_cast<uint8_t>(sx[j] + 127);
        if (last)
          for (int b = byte + 1; b < 4; ++b) w[b] = 127;
      }
    }
  }
}

// Weight preparation: each 32x128 tile of a weight [rows][C] is read once
// (cp.async, two tiles in flight per block) and written quantised along its
// columns (blocks of 32 rows: the forward GEMMs' K) and along its rows (blocks
// of 32 columns: the dgrads' K), both as [rows][C] codes plus scale chunks.
// Warp w takes the tile's columns 32w..32w+31 with one row per lane: the
// lane's 32 values are its row block; the 32 column maxima come from a
// butterfly over the lanes on bf16 pairs (16 shuffles), and their scales
// return to every lane through 128 bytes of shared memory. The bytes equal
// those of the separate column and row quantisers. rows and C are multiples
// of 128, so no block crosses a weight matrix; blocks stride over the tiles
// (those of one 32-row band are consecutive, so W is read in order).
constexpr int kDualCols = 128, kDualPitch = kDualCols + 8;  // bf16 per staged row (16-byte pad)
constexpr int kDualTile = 32 * kDualPitch;
constexpr int kDualCodePitch = kDualCols + 16;  // bytes per staged code row (conflict-free 16-byte stores)
__global__ void __launch_bounds__(128, 8)
quant_dual_kernel(const __nv_bfloat16* __restrict__ src, int C, long ntiles, uint8_t* __restrict__ qc,
                  uint8_t* __restrict__ sc_c, uint8_t* __restrict__ qr, uint8_t* __restrict__ sc_r) {
  __shared__ __align__(16) __nv_bfloat16 tile[2 * kDualTile];
  __shared__ __align__(16) float col_mul[4][32];
  __shared__ __align__(16) uint8_t codes[2][32 * kDualCodePitch];  // the tile's row codes, column codes
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cg = C / kDualCols;
  auto issue = [&](long t, int buf) {  // a half-warp copies one 256-byte row segment per step
    const long row0 = t / cg * 32;
    const int c0 = static_cast<int>(t % cg) * kDualCols;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int id = tid + 128 * i, r = id >> 4, g = id & 15;
      const __nv_bfloat16* gp = src + (row0 + r) * C + c0 + 8 * g;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                       __cvta_generic_to_shared(tile + buf * kDualTile + r * kDualPitch + 8 * g))),
                   "l"(gp)
                   : "memory");
    }
  };
  long t = blockIdx.x;
  if (t < ntiles) issue(t, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int it = 0; t < ntiles; t += gridDim.x, ++it) {
    if (t + gridDim.x < ntiles) issue(t + gridDim.x, (it + 1) & 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile's copies have landed
    __syncthreads();
    const long row0 = t / cg * 32, row = row0 + lane;  // this lane's row
    const int c0 = static_cast<int>(t % cg) * kDualCols, cl = 32 * warp;  // this warp's columns c0 + cl ..
    uint32_t w[16];  // the lane's row, columns cl..cl+31, as bf16 pairs
    {
      const __nv_bfloat16* tl = tile + (it & 1) * kDualTile + lane * kDualPitch + cl;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = *reinterpret_cast<const uint4*>(tl + 8 * i);
        w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
      }
    }
    {  // along the row: the lane's 32 values are one block
      const int sx = e8m0_exponent(absmax_bf16x32(w));
      const float m = pow2_neg(sx);
      uint32_t cw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        cw[i] = mx_e4m3x2(bf16_lo(w[2 * i]) * m, bf16_hi(w[2 * i]) * m) |
                (mx_e4m3x2(bf16_lo(w[2 * i + 1]) * m, bf16_hi(w[2 * i + 1]) * m) << 16);
      uint4* out = reinterpret_cast<uint4*>(codes[0] + lane * kDualCodePitch + cl);
      out[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      out[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      sc_r[(((row >> 7) * cg + c0 / 128) << 9) + mx_chunk_lane(static_cast<int>(row & 127)) + warp] =
          static_cast<uint8_t>(sx + 127);
    }
    {  // along the columns: lane l ends with column cl + l's maximum over the 32 rows
      uint32_t a[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = w[i] & 0x7FFF7FFFu;
      colmax_step<8>(a, lane);
      colmax_step<4>(a, lane);
      colmax_step<2>(a, lane);
      colmax_step<1>(a, lane);
      a[0] = bf16x2_max(a[0], __shfl_xor_sync(0xffffffffu, a[0], 1));
      const int sx = e8m0_exponent((lane & 1) ? bf16_hi(a[0]) : bf16_lo(a[0]));
      col_mul[warp][lane] = pow2_neg(sx);
      sc_c[(((row0 >> 7) * cg + c0 / 128) << 9) + mx_chunk_lane(cl + lane) + ((row0 >> 5) & 3)] =
          static_cast<uint8_t>(sx + 127);
      __syncwarp();
      float m[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = reinterpret_cast<const float4*>(col_mul[warp])[i];
        m[4 * i] = v.x; m[4 * i + 1] = v.y; m[4 * i + 2] = v.z; m[4 * i + 3] = v.w;
      }
      uint32_t cw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        cw[i] = mx_e4m3x2(bf16_lo(w[2 * i]) * m[4 * i], bf16_hi(w[2 * i]) * m[4 * i + 1]) |
                (mx_e4m3x2(bf16_lo(w[2 * i + 1]) * m[4 * i + 2], bf16_hi(w[2 * i + 1]) * m[4 * i + 3]) << 16);
      uint4* out = reinterpret_cast<uint4*>(codes[1] + lane * kDualCodePitch + cl);
      out[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      out[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    }
    __syncthreads();  // both code tiles are staged
    // each instruction stores four rows' 128-byte segments of one layout
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int id = tid + 128 * i, lay = id >> 8, r = (id >> 3) & 31, g = id & 7;
      uint8_t* dst = (lay == 0 ? qr : qc) + (row0 + r) * C + c0 + 16 * g;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(codes[lay] + r * kDualCodePitch + 16 * g);
    }
    __syncthreads();  // the tile buffer is refilled next iteration; col_mul and codes are reused
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Quantise before dispatch: each token's row of x is quantised once along d
// (blocks of 32; lane L owns elements 8L + 256i, so a block is 4 lanes) and
// the codes and scale bytes are written to the token's k dispatched rows
// (with x_perm given, the bf16 row too). The codes and scale values equal
// mxfp8_quantize(x_perm, rows) of the bf16 dispatch; the scales are stored as
// the GEMM's scale chunks, grouped by per-expert 128-row tiles.
constexpr int kPermWarps = 8;
__global__ void __launch_bounds__(kPermWarps * 32)
permute_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int d, int k, int E,
                     const int32_t* __restrict__ dest_row, const int32_t* __restrict__ topk_idx,
                     const int32_t* __restrict__ offs, uint8_t* __restrict__ q, uint8_t* __restrict__ sc,
                     __nv_bfloat16* __restrict__ x_perm, int* err) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kPermWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  int dest = 0, grp = 0, tt = 0, e = 0;  // lane j < k: dispatched row j, its scale group and index in it
  if (lane < k) {
    dest = dest_row[(size_t)t * k + lane];
    e = topk_idx[(size_t)t * k + lane];
    // the pair's expert must hold its row (the scale chunk is found from it)
    if (e >= 0 && e < E && (dest < offs[e] || dest >= offs[e + 1])) e = -1;
  }
  const unsigned ok = usable_pairs(dest, e, lane, k, (long)T * k, E, err);
  if (lane < k && ((ok >> lane) & 1u)) {
    const int o = offs[e];
    grp = static_cast<int>(mx_row_tile_base(o, e)) + ((dest - o) >> 7);
    tt = (dest - o) & 127;
  }
  const int stages = d / 128;
  for (int cb = 0; cb < d; cb += 256) {  // warp-uniform: every lane reaches the shuffles
    const int c = cb + lane * 8;
    const bool act = c < d;  // d % 32 == 0: a 4-lane block is all in or all out
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (act) {
      raw = *reinterpret_cast<const uint4*>(x + (size_t)t * d + c);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int sx = e8m0_exponent(amax);
    const float m = pow2_neg(sx);
    const uint32_t lo = mx_e4m3x2(v[0] * m, v[1] * m) | mx_e4m3x2(v[2] * m, v[3] * m) << 16;
    const uint32_t hi = mx_e4m3x2(v[4] * m, v[5] * m) | mx_e4m3x2(v[6] * m, v[7] * m) << 16;
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, dest, j);
      const int g = __shfl_sync(0xffffffffu, grp, j), ti = __shfl_sync(0xffffffffu, tt, j);
      if (!act || !((ok >> j) & 1u)) continue;
      *reinterpret_cast<uint2*>(q + (size_t)r * d + c) = make_uint2(lo, hi);
      if (x_perm) *reinterpret_cast<uint4*>(x_perm + (size_t)r * d + c) = raw;
      const int b = c / 32;
      if ((lane & 3) == 0)
        sc[(((size_t)g * stages + b / 4) << 9) + mx_chunk_lane(ti) + (b & 3)] = static_cast<uint8_t>(sx + 127);
    }
  }
}

}  // namespace

cudaError_t launch_permute_quant(const void* x, int T, int d, int k, int E, const int32_t* dest_row,
                                 const int32_t* topk_idx, const int32_t* offsets, uint8_t* q, uint8_t* sc,
                                 void* x_perm, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  MOE_COUNTED_AS("permute_quant", st) permute_quant_kernel<<<(T + kPermWarps - 1) / kPermWarps, kPermWarps * 32, 0, st>>>(
      static_cast<const __nv_bfloat16*>(x), T, d, k, E, dest_row, topk_idx, offsets, q, sc,
      static_cast<__nv_bfloat16*>(x_perm), device_error_word());
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quant_rows(const void* src, long rows, long K, uint8_t* q, uint8_t* sc, cudaStream_t st,
                                    int layout, const int32_t* offsets, int E) {
  const long nblocks = rows * (K / 32);
  if (nblocks == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((nblocks + 255) / 256);
  const auto* s = static_cast<const __nv_bfloat16*>(src);
  const int kb = static_cast<int>(K / 32);
  if (layout == kScalesPlain)
    MOE_COUNTED_AS("quant_rows", st) quant_rows_kernel<kScalesPlain><<<grid, 256, 0, st>>>(s, nblocks, kb, q, sc, offsets, E);
  else if (layout == kScalesChunk)
    MOE_COUNTED_AS("quant_rows", st) quant_rows_kernel<kScalesChunk><<<grid, 256, 0, st>>>(s, nblocks, kb, q, sc, offsets, E);
  else
    MOE_COUNTED_AS("quant_rows", st) quant_rows_kernel<kScalesTiles><<<grid, 256, 0, st>>>(s, nblocks, kb, q, sc, offsets, E);
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quant_dual(const void* src, long rows, int C, uint8_t* qc, uint8_t* sc_c, uint8_t* qr,
                                    uint8_t* sc_r, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const long ntiles = rows / 32 * (C / kDualCols);
  static std::atomic<int> cached{0};  // resident blocks per SM, computed once
  int per_sm = cached.load(std::memory_order_relaxed);
  if (per_sm <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_dual_kernel, 128, 0) != cudaSuccess || per_sm <= 0)
      per_sm = 8;
    cached.store(per_sm, std::memory_order_relaxed);
  }
  const long grid = std::min<long>(ntiles, (long)tc::sm_count() * per_sm);
  MOE_COUNTED_AS("quant_dual", st) quant_dual_kernel<<<static_cast<unsigned>(grid), 128, 0, st>>>(static_cast<const __nv_bfloat16*>(src), C,
                                                                           ntiles, qc, sc_c, qr, sc_r);
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quant_cols(const void* src, int rows, int C, const int32_t* seg, int nseg,
                                    uint8_t* q, uint8_t* sc, cudaStream_t st, bool packed) {
  const int nseg_eff = seg ? nseg : 1;
  const long max_brows = (rows + 31) / 32 + nseg_eff;
  if (rows == 0) return cudaSuccess;
  const long groups = (max_brows + kColBlockRows - 1) / kColBlockRows;
  dim3 grid(static_cast<unsigned>((C + 255) / 256), static_cast<unsigned>(groups < 65535 ? groups : 65535));
  const size_t smem = (nseg_eff + 1) * sizeof(int);
  if (packed)
    MOE_COUNTED_AS("quant_cols", st) quant_cols_kernel<true><<<grid, 128, smem, st>>>(static_cast<const __nv_bfloat16*>(src), rows, C,
                                                                 seg, nseg_eff, q, sc);
  else
    MOE_COUNTED_AS("quant_cols", st) quant_cols_kernel<false><<<grid, 128, smem, st>>>(static_cast<const __nv_bfloat16*>(src), rows, C,
                                                                  seg, nseg_eff, q, sc);
  return cudaGetLastError();
}

}  // namespace moe
