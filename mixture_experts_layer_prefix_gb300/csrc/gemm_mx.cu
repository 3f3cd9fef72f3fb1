// gemm_mx.cu -- the six grouped expert GEMMs in MXFP8 ("Introducing Olmo-core
// 3", section "Scaling and optimizing MoE training": MXFP8 for the expert
// feed-forward, where most of its gain came from). Every operand is E4M3 with
// one E8M0 scale per 32 elements along that GEMM's K; accumulation is fp32;
// outputs are bf16, with the same fused SwiGLU epilogues as the bf16 GEMMs.
//
// One persistent kernel per GEMM, one CTA per SM:
//   warp 0      TMA producer: 4-stage ring of (A 128x128, B 256x128) E4M3
//               tiles (128 B rows, 128-byte swizzle).
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::mxf8f6f4
//               block_scale (M=128, N=256, K=32; 4 per stage, scale id = K step).
//   warps 2..5  scale loaders (one per TMEM lane quadrant): read the stage's
//               E8M0 bytes of A (one 32-bit word per row) and B (eight words
//               per lane, one per 32 output columns, written in every
//               quadrant) and store them into a TMEM scale ring with
//               tcgen05.st, then arrive on the stage's scale barrier.
//   warps 6..9  epilogue (one per quadrant), as in the bf16 kernel.
// TMEM: accumulator columns [0,256) (one buffer: the scale ring needs the
// rest of the columns a second buffer would use), A scales at 256 + 4s, B
// scales at 272 + 8s for stage s.
#include "kernels.h"
#include "tc_common.cuh"

namespace moe {
namespace tc {
namespace mx {
namespace {

constexpr int BK = 128;  // E4M3 elements (bytes) per stage along K
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 128 * 128;  // one 128 (MN) x 128 (K) box
constexpr int NUM_THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SFA_COL = 256, SFB_COL = 272;

struct Smem {
  uint64_t full[STAGES];
  uint64_t sfull[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Four scale bytes of consecutive 32-blocks along K for MN index `col` from a
// [block rows][ncols] table, or 1.0 (127) where the block is past `nblk`.
__device__ __forceinline__ uint32_t gather4(const uint8_t* tab, long blk0, int nblk_avail, long ncols, long col) {
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t b = j < nblk_avail ? tab[(blk0 + j) * ncols + col] : 127u;
    w |= b << (8 * j);
  }
  return w;
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const Params p) {
  using Tr = Traits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem* sm = reinterpret_cast<Smem*>(smem + STAGES * STAGE_BYTES);
  int* offs = reinterpret_cast<int*>(sm + 1);
  int* tstart = offs + (p.E + 1);
  int* bstart = tstart + (p.E + 1);  // wgrad: first 32-row scale block of each expert segment
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  build_tile_table<KIND, NUM_THREADS>(p, offs, tstart);
  if (Tr::kragged && warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int v = e < p.E ? (offs[e + 1] - offs[e] + 31) / 32 : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      if (e < p.E) bstart[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm->full[s], 1);
      ptx::mbar_init(&sm->sfull[s], 4);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    ptx::mbar_init(&sm->tfull, 1);
    ptx::mbar_init(&sm->tempty, 4);
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
  const int total = Tr::kragged ? p.E * p.m_tiles * p.n_tiles : tstart[p.E];
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
        const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
        for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
          uint8_t* a = smem + s * STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          uint64_t* fb = &sm->full[s];
          ptx::mbar_expect_tx(fb, STAGE_BYTES);
          const int k0 = kb * BK;
          if (KIND == FPROP1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * 128;
            ptx::tma_load_3d(b, &tmB0, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + BOX_BYTES, &tmB1, fb, n0, k0, tl.e);
          } else if (KIND == FPROP2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * BN;
            ptx::tma_load_3d(b, &tmB0, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + BOX_BYTES, &tmB0, fb, n0 + 128, k0, tl.e);
          } else if (KIND == DGRAD2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
          } else if (KIND == DGRAD1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            if (k0 < p.f) ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
            else ptx::tma_load_3d(b, &tmB1, fb, k0 - p.f, tl.n_idx * BN, tl.e);
          } else {  // WGRAD2 / WGRAD1: K runs over the expert's rows
            const int row = tl.k_row0 + k0;
            ptx::tma_load_2d(a, &tmA, fb, tl.m0, row);
            const int n0 = tl.n_idx * BN;
            ptx::tma_load_2d(b, &tmB0, fb, n0, row);
            ptx::tma_load_2d(b + BOX_BYTES, &tmB0, fb, n0 + 128, row);
          }
        }
      }
      if (!ok) {
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
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      if (tl.nkb == 0) continue;
      if (!wait_bar(&sm->tempty, (acc_it & 1u) ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        if (!wait_bar(&sm->full[s], ph, &sm->abort_flag, p.err) ||
            !wait_bar(&sm->sfull[s], ph, &sm->abort_flag, p.err)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * STAGE_BYTES;
        if (Tr::kragged) {
          const int valid = tl.row_end - (tl.k_row0 + kb * BK);
          if (valid < BK) {
            // rows past the expert's end belong to the next expert: zero them in A
            for (int i = valid * 8 + lane; i < BK * 8; i += 32)
              *reinterpret_cast<uint4*>(a + i * 16) = make_uint4(0, 0, 0, 0);
            ptx::fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int ks = 0; ks < BK / 32; ++ks) {
            const uint64_t ad = Tr::a_mn ? ptx::smem_desc_sw128(a_addr + ks * 4096, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = Tr::b_mn ? ptx::smem_desc_sw128(b_addr + ks * 4096, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            const uint32_t idesc = ptx::idesc_mxf8_f32(BM, BN, Tr::a_mn ? 1 : 0, Tr::b_mn ? 1 : 0, ks, ks);
            ptx::mma_mxf8(tmem, ad, bd, idesc, tmem + SFA_COL + 4 * s, tmem + SFB_COL + 8 * s,
                          (kb > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&sm->empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(&sm->tfull);
      __syncwarp();
      ++acc_it;
    }
    if (!ok && lane == 0) {
      ptx::mma_commit(&sm->drain);
      const long long t0 = clock64();
      while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->drain, 0)) {
      }
    }
  } else if (warp < 6) {
    // ====================================================== scale loaders
    const int q = warp & 3;
    const int r_tile = q * 32 + lane;
    uint32_t it = 0;
    const long Kd = gemm_k<KIND>(p);
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      bool ok = true;
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        const int k0 = kb * BK;
        uint32_t wa, wb[8];
        if (!Tr::kragged) {
          // A: rows quantised along K, table [R][K/32]
          const int row = tl.m0 + r_tile;
          wa = row < p.R ? ld_u32(p.sfa + (size_t)row * (Kd / 32) + k0 / 32) : 0x7F7F7F7Fu;
        } else {
          // A: columns quantised along the expert's rows, table [blocks][M]
          const int m = tl.m0 + r_tile;
          const int nblk = (tl.row_end - tl.k_row0 + 31) / 32;
          wa = m < p.M ? gather4(p.sfa, bstart[tl.e] + 4 * kb, nblk - 4 * kb, p.M, m) : 0x7F7F7F7Fu;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w = 0x7F7F7F7Fu;
          if (KIND == FPROP1) {
            const int n = tl.n_idx * 128 + lane + 32 * (c & 3);
            const uint8_t* tab = c < 4 ? p.sfb0 : p.sfb1;  // [E*d/32][f]
            if (n < p.f) w = gather4(tab, ((long)tl.e * p.d + k0) / 32, 4, p.f, n);
          } else if (KIND == FPROP2) {
            const int n = tl.n_idx * BN + lane + 32 * c;  // [E*f/32][d]
            if (n < p.d) w = gather4(p.sfb0, ((long)tl.e * p.f + k0) / 32, 4, p.d, n);
          } else if (KIND == DGRAD2) {
            const int n = tl.n_idx * BN + lane + 32 * c;  // [E*f][d/32]
            if (n < p.f) w = ld_u32(p.sfb0 + ((size_t)tl.e * p.f + n) * (p.d / 32) + k0 / 32);
          } else if (KIND == DGRAD1) {
            const int n = tl.n_idx * BN + lane + 32 * c;  // [E*d][f/32]
            if (n < p.d) {
              const uint8_t* tab = k0 < p.f ? p.sfb0 : p.sfb1;
              const int kk = k0 < p.f ? k0 : k0 - p.f;
              w = ld_u32(tab + ((size_t)tl.e * p.d + n) * (p.f / 32) + kk / 32);
            }
          } else {  // WGRAD: B columns quantised along the expert's rows, table [blocks][N]
            const int n = tl.n_idx * BN + lane + 32 * c;
            const int nblk = (tl.row_end - tl.k_row0 + 31) / 32;
            if (n < p.N) w = gather4(p.sfb0, bstart[tl.e] + 4 * kb, nblk - 4 * kb, p.N, n);
          }
          wb[c] = w;
        }
        if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        ptx::tmem_st4(tmem + lane_base + SFA_COL + 4 * s, wa, wa, wa, wa);
        ptx::tmem_st8(tmem + lane_base + SFB_COL + 8 * s, wb);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm->sfull[s]);
      }
      if (!ok) break;
    }
  } else {
    // ============================================================ epilogue
    const int q = warp & 3;
    constexpr int NC = epi_chunks<KIND>();
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      const bool empty_k = tl.nkb == 0;
      if (!empty_k) {
        if (!wait_bar(&sm->tfull, acc_it & 1u, &sm->abort_flag, p.err)) break;
        ptx::tc_fence_after();
      }
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
      epilogue_tile<KIND>(p, tl, tbase, q * 32 + lane, 0, NC, empty_k);
      if (!empty_k) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm->tempty);
        ++acc_it;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

size_t smem_bytes(int E) { return 1024 + STAGES * STAGE_BYTES + sizeof(Smem) + 3 * (E + 1) * sizeof(int) + 64; }

template <int KIND>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const Params& p,
                   long max_tiles, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = smem_bytes(p.E);
  cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
  MOE_COUNTED mx_gemm_kernel<KIND><<<grid, NUM_THREADS, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

constexpr CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

inline size_t al(size_t b) { return (b + 255) & ~size_t(255); }

// One quantised operand in the workspace: E4M3 codes and E8M0 scales.
struct QBuf {
  uint8_t* q;
  uint8_t* s;
};

struct Carver {
  char* p;
  size_t used = 0;
  QBuf take(size_t codes, size_t scales) {
    QBuf b{reinterpret_cast<uint8_t*>(p + used), nullptr};
    used += al(codes);
    b.s = reinterpret_cast<uint8_t*>(p + used);
    used += al(scales);
    return b;
  }
  void* raw(size_t bytes) {
    void* r = p + used;
    used += al(bytes);
    return r;
  }
};

// Scale-block rows of a [rows][C] operand quantised along rows in E segments.
inline size_t seg_blocks(long rows, int E) { return (size_t)(rows + 31) / 32 + E + 1; }

}  // namespace

size_t fwd_workspace(long R, int E, int d, int f) {
  const size_t Ed = (size_t)E * d;
  return al(R * (size_t)d) + al(R * (size_t)d / 32) + al(R * (size_t)f) + al(R * (size_t)f / 32) +
         2 * (al(Ed * f) + al(Ed / 32 * f)) + al((size_t)E * f * d) + al((size_t)E * f / 32 * d);
}

size_t bwd_workspace(long R, int E, int d, int f) {
  const size_t Ed = (size_t)E * d, Ef = (size_t)E * f;
  return al(R * 2 * (size_t)f * 2)                                         // dh (bf16)
         + al(R * (size_t)d) + al(R * (size_t)d / 32)                      // dy rows
         + al(R * (size_t)d) + al(seg_blocks(R, E) * d)                    // dy segment columns
         + al(R * (size_t)f) + al(seg_blocks(R, E) * f)                    // a segment columns
         + al(Ef * d) + al(Ef * d / 32)                                    // w_down rows
         + al(R * 2 * (size_t)f) + al(R * 2 * (size_t)f / 32)              // dh rows
         + al(R * 2 * (size_t)f) + al(seg_blocks(R, E) * 2 * f)            // dh segment columns
         + 2 * (al(Ed * f) + al(Ed * f / 32))                              // w_gate, w_up rows
         + al(R * (size_t)d) + al(seg_blocks(R, E) * d);                   // x segment columns
}

}  // namespace mx
}  // namespace tc

using namespace tc;

cudaError_t mx_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd, const int32_t* offsets,
                       int R, int E, int d, int f, void* h, void* a, void* y, void* ws, cudaStream_t st) {
  using namespace mx;
  Carver cv{static_cast<char*>(ws)};
  const long Ed = (long)E * d, Ef = (long)E * f;
  QBuf xq = cv.take((size_t)R * d, (size_t)R * d / 32);
  QBuf aq = cv.take((size_t)R * f, (size_t)R * f / 32);
  QBuf wgq = cv.take((size_t)Ed * f, (size_t)Ed / 32 * f);
  QBuf wuq = cv.take((size_t)Ed * f, (size_t)Ed / 32 * f);
  QBuf wdq = cv.take((size_t)Ef * d, (size_t)Ef / 32 * d);
  cudaError_t e;
  // operands of GEMM1 along d: x rows, w_gate / w_up columns (32-row blocks never cross experts)
  if ((e = launch_mxfp8_quant_rows(x_perm, R, d, xq.q, xq.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_cols(wg, (int)Ed, f, nullptr, 1, wgq.q, wgq.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_cols(wu, (int)Ed, f, nullptr, 1, wuq.q, wuq.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_cols(wd, (int)Ef, d, nullptr, 1, wdq.q, wdq.s, st)) != cudaSuccess) return e;

  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  if (!map_2d(&mA, xq.q, U8, 1, d, R, 128, BM) || !map_3d(&mB0, wgq.q, U8, 1, f, d, E, 128, 128) ||
      !map_3d(&mB1, wuq.q, U8, 1, f, d, E, 128, 128))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + 127) / 128; p.out0 = h; p.out1 = a;
  p.sfa = xq.s; p.sfb0 = wgq.s; p.sfb1 = wuq.s;
  if ((e = launch<FPROP1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess) return e;
  // GEMM2 along f: A rows, w_down columns
  if ((e = launch_mxfp8_quant_rows(a, R, f, aq.q, aq.s, st)) != cudaSuccess) return e;
  if (!map_2d(&mA, aq.q, U8, 1, f, R, 128, BM) || !map_3d(&mB0, wdq.q, U8, 1, d, f, E, 128, 128))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = y; p.out1 = nullptr;
  p.sfa = aq.s; p.sfb0 = wdq.s; p.sfb1 = nullptr;
  return launch<FPROP2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
}

cudaError_t mx_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* ws, cudaStream_t st) {
  using namespace mx;
  Carver cv{static_cast<char*>(ws)};
  const long Ed = (long)E * d, Ef = (long)E * f;
  void* dh = cv.raw((size_t)R * 2 * f * 2);
  QBuf dyr = cv.take((size_t)R * d, (size_t)R * d / 32);
  QBuf dyc = cv.take((size_t)R * d, seg_blocks(R, E) * d);
  QBuf ac = cv.take((size_t)R * f, seg_blocks(R, E) * f);
  QBuf wdr = cv.take((size_t)Ef * d, (size_t)Ef * d / 32);
  QBuf dhr = cv.take((size_t)R * 2 * f, (size_t)R * 2 * f / 32);
  QBuf dhc = cv.take((size_t)R * 2 * f, seg_blocks(R, E) * 2 * f);
  QBuf wgr = cv.take((size_t)Ed * f, (size_t)Ed * f / 32);
  QBuf wur = cv.take((size_t)Ed * f, (size_t)Ed * f / 32);
  QBuf xc = cv.take((size_t)R * d, seg_blocks(R, E) * d);
  cudaError_t e;
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();

  // dA = dy . Wd^T (K = d): dy rows, w_down rows; SwiGLU backward fused -> dh
  if ((e = launch_mxfp8_quant_rows(dy_perm, R, d, dyr.q, dyr.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_rows(wd, Ef, d, wdr.q, wdr.s, st)) != cudaSuccess) return e;
  if (!map_2d(&mA, dyr.q, U8, 1, d, R, 128, BM) || !map_3d(&mB0, wdr.q, U8, 1, d, f, E, 128, BN))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + BN - 1) / BN; p.out0 = dh; p.aux = h;
  p.sfa = dyr.s; p.sfb0 = wdr.s;
  if ((e = launch<DGRAD2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess) return e;

  // dWd[e] = A_e^T dy_e (K = the expert's rows): A and dy quantised along rows per expert
  if ((e = launch_mxfp8_quant_cols(a, R, f, offsets, E, ac.q, ac.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_cols(dy_perm, R, d, offsets, E, dyc.q, dyc.s, st)) != cudaSuccess) return e;
  if (!map_2d(&mA, ac.q, U8, 1, f, R, 128, 128) || !map_2d(&mB0, dyc.q, U8, 1, d, R, 128, 128))
    return cudaErrorInvalidValue;
  p.M = f; p.N = d; p.m_tiles = (f + BM - 1) / BM; p.n_tiles = (d + BN - 1) / BN; p.out0 = dwd; p.aux = nullptr;
  p.sfa = ac.s; p.sfb0 = dyc.s;
  if ((e = launch<WGRAD2>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st)) != cudaSuccess) return e;

  // dx_perm = dh . [Wg | Wu]^T (K = 2f): dh rows, w_gate / w_up rows
  if ((e = launch_mxfp8_quant_rows(dh, R, 2L * f, dhr.q, dhr.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_rows(wg, Ed, f, wgr.q, wgr.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_rows(wu, Ed, f, wur.q, wur.s, st)) != cudaSuccess) return e;
  if (!map_2d(&mA, dhr.q, U8, 1, 2L * f, R, 128, BM) || !map_3d(&mB0, wgr.q, U8, 1, f, d, E, 128, BN) ||
      !map_3d(&mB1, wur.q, U8, 1, f, d, E, 128, BN))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = dx_perm;
  p.sfa = dhr.s; p.sfb0 = wgr.s; p.sfb1 = wur.s;
  if ((e = launch<DGRAD1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess) return e;

  // [dWg | dWu][e] = x_e^T dh_e (K = the expert's rows)
  if ((e = launch_mxfp8_quant_cols(x_perm, R, d, offsets, E, xc.q, xc.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_cols(dh, R, 2 * f, offsets, E, dhc.q, dhc.s, st)) != cudaSuccess) return e;
  if (!map_2d(&mA, xc.q, U8, 1, d, R, 128, 128) || !map_2d(&mB0, dhc.q, U8, 1, 2L * f, R, 128, 128))
    return cudaErrorInvalidValue;
  p.M = d; p.N = 2 * f; p.m_tiles = (d + BM - 1) / BM; p.n_tiles = (2 * f + BN - 1) / BN;
  p.out0 = dwg; p.out1 = dwu; p.sfa = xc.s; p.sfb0 = dhc.s; p.sfb1 = nullptr;
  return launch<WGRAD1>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st);
}

size_t mx_fwd_workspace(long R, int E, int d, int f) { return tc::mx::fwd_workspace(R, E, d, f); }
size_t mx_bwd_workspace(long R, int E, int d, int f) { return tc::mx::bwd_workspace(R, E, d, f); }

}  // namespace moe
