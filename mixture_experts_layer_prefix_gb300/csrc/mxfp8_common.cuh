// mxfp8_common.cuh -- device helpers of the MXFP8 block format shared by the
// quantisers and the GEMM epilogues that quantise their own outputs: E8M0
// exponent of a block maximum, exact power-of-two scaling, E4M3 conversion.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// E8M0 exponent s = ceil(log2(amax / 448)) clamped to [-127, 127], from the
// fp32 bits of amax (amax >= 0, finite); zero or subnormal amax gives -127.
__device__ __forceinline__ int mx_e8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xFFu);
  if (ef == 0) return -127;                  // zero or subnormal: 2^e <= 2^-127
  int s = (ef - 127) - 8;                    // amax in [2^e, 2^(e+1)), 448 = 1.75 * 2^8
  if ((b & 0x7FFFFFu) > 0x600000u) s += 1;   // mantissa above 1.75: 2^(e-8) * 448 < amax
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s as an exact fp32 (s in [-127, 127]; 2^-127 is subnormal).
__device__ __forceinline__ float mx_pow2_neg(int s) {
  const int ef = 127 - s;
  return ef >= 1 ? __uint_as_float(static_cast<uint32_t>(ef) << 23) : __uint_as_float(1u << 22);
}

// Scale chunks: the block-scaled GEMMs fetch their E8M0 scales as 512-byte
// chunks, one per (group of 128 rows or columns of an operand, K stage of 128
// elements), each already in the order the tensor-memory scale copy takes:
// the scale of index t of the group (t < 128) for block b of the stage
// (b < 4) is byte mx_chunk_lane(t) + b. Chunk c starts at byte 512 c.
__host__ __device__ __forceinline__ uint32_t mx_chunk_lane(int t) {
  return static_cast<uint32_t>((t & 31) * 16 + ((t >> 5) & 3) * 4);
}
// Row operands of the grouped GEMMs are tiled per expert: the m-th 128-row
// tile of expert e (rows from offs_e) is group mx_row_tile_base(offs_e, e) + m.
// With base (offs_e + 127 e) / 128 the groups of consecutive experts never
// overlap (base[e+1] - base[e] >= ceil(rows_e / 128)) and no prefix over the
// experts is needed.
__host__ __device__ __forceinline__ long mx_row_tile_base(long offs_e, int e) { return (offs_e + 127L * e) >> 7; }
// Groups spanned by a row operand of R rows over E experts.
__host__ __device__ __forceinline__ long mx_row_tiles(long R, int E) { return (R + 127L * E) / 128 + 1; }

// bf16 pairs held in 32-bit words: element 0 in the low half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Element-wise maximum of two bf16 pairs.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Largest magnitude among 32 bf16 values held as 16 pairs (exact).
__device__ __forceinline__ float absmax_bf16x32(const uint32_t (&w)[16]) {
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = bf16x2_max(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = bf16x2_max(m[2 * i], m[2 * i + 1]);
  m[0] = bf16x2_max(m[0], m[1]);
  m[2] = bf16x2_max(m[2], m[3]);
  m[0] = bf16x2_max(m[0], m[2]);
  return fmaxf(bf16_lo(m[0]), bf16_hi(m[0]));
}

// One step of a butterfly reduce-scatter of per-column maxima over the warp,
// on bf16 pairs (word i = columns 2i, 2i+1): with 2H words per lane, the lane
// keeps the H words picked by lane bit 2H and takes the max with its partner's
// copy of them (lane ^ 2H; the partner keeps the other H). After the steps
// H = 8, 4, 2, 1, word 0 of lane l holds columns 2(l/2), 2(l/2)+1, maxed over
// the 16 lanes that agree with l in bit 0.
template <int H>
__device__ __forceinline__ void colmax_step(uint32_t (&a)[16], int lane) {
  const bool up = (lane & (2 * H)) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const uint32_t keep = up ? a[H + i] : a[i];
    const uint32_t give = up ? a[i] : a[H + i];
    a[i] = bf16x2_max(keep, __shfl_xor_sync(0xffffffffu, give, 2 * H));
  }
}

// Round-to-nearest-even E4M3 codes of v0 (low byte) and v1 (high byte),
// saturated to +-448, from one paired conversion.
__device__ __forceinline__ uint32_t mx_e4m3x2(float v0, float v1) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3));
}

// Quantise one block of 32 values into 32 E4M3 codes (w, little-endian
// bytes in element order); returns the E8M0 byte.
__device__ __forceinline__ uint8_t mx_quant_block32_regs(const float* v, uint32_t (&w)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_e8m0_exponent(amax);
  const float m = mx_pow2_neg(s);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = mx_e4m3x2(v[4 * i] * m, v[4 * i + 1] * m) | (mx_e4m3x2(v[4 * i + 2] * m, v[4 * i + 3] * m) << 16);
  return static_cast<uint8_t>(s + 127);
}

// Quantise one block of 32 values: 32 E4M3 codes (16-byte aligned
// destination) and one E8M0 byte.
__device__ __forceinline__ void mx_quant_block32(const float* v, uint8_t* codes, uint8_t* scale) {
  uint32_t w[8];
  *scale = mx_quant_block32_regs(v, w);
  uint4* out = reinterpret_cast<uint4*>(codes);
  out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  out[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace moe
