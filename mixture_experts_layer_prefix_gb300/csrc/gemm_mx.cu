// gemm_mx.cu -- the six grouped expert GEMMs in MXFP8 ("Introducing Olmo-core
// 3", section "Scaling and optimizing MoE training": MXFP8 for the expert
// feed-forward, where most of its gain came from). Every operand is E4M3 with
// one E8M0 scale per 32 elements along that GEMM's K; accumulation is fp32;
// outputs are bf16, with the same fused SwiGLU epilogues as the bf16 GEMMs.
//
// One persistent kernel per GEMM, one CTA per SM:
//   warp 0      producer. Lane 0 issues TMA for a 4-stage ring of
//               (A 128x128, B 256x128) E4M3 tiles (128 B rows, 128-byte
//               swizzle) and bulk copies of the stage's E8M0 scale chunks
//               (512 B per 128 rows or columns, stored by the quantisers in
//               the order the tensor-memory copy takes) into a small shared
//               staging area, all tracked by the same stage barrier.
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp moves the
//               scales from shared memory into a TMEM ring (32x128b copies
//               replicated to all four lane quadrants), then four
//               tcgen05.mma kind::mxf8f6f4 block_scale (M=128, N=256, K=32,
//               scale-factor id = K step).
//   warps 2..9  epilogue, two warps per TMEM lane quadrant.
// Output tiles are 128 rows by TBN columns. With TBN = 128 two accumulators
// fit next to the scale ring and alternate, as in the bf16 GEMMs. GEMM1
// (TBN = 256: 128 gate + 128 up columns) has one accumulator, so each warp
// first copies its 128 columns into registers and releases it, then computes
// and stores while the next tile's MMAs run.
// TMEM: accumulators in columns [0,256); scales of stage s: A at 256 + 4s,
// B at 272 + (TBN/32)s. Shared scale staging of a stage: A 512 B (row r of the
// copy = tile rows r, 32+r, 64+r, 96+r), then B TBN/128 x 512 B (copy h row r
// = tile columns 128h + r, +32, +64, +96).
// The two weight gradients can also run on CTA pairs (mx_wgrad_pair_kernel,
// below, selected with moe_use_cta_pairs): 256 x 256 tiles with
// tcgen05.mma.cta_group::2.
#include <atomic>

#include "kernels.h"
#include "tc_common.cuh"

namespace moe {
namespace tc {
namespace mx {
namespace {

constexpr int BK = 128;  // E4M3 elements (bytes) per stage along K
constexpr int A_BYTES = BM * BK;
constexpr int BOX_BYTES = 128 * 128;  // one 128 (MN) x 128 (K) box
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;

// Tile geometry for a tile width TBN (columns of B / of the output tile):
// TBN = 256 uses one accumulator (the scale ring needs the columns a second
// one would take); TBN = 128 fits two and double-buffers like the bf16 GEMMs.
template <int TBN> struct Geo {
  static constexpr int B_BYTES = TBN * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SCB = TBN / 128;             // 32x128b copies of B scales per stage
  static constexpr int SC_BYTES = 512 + 512 * SCB;  // scale staging per stage
  static constexpr int ACC = TBN == 128 ? 2 : 1;    // accumulator buffers
  static constexpr uint32_t SFA_COL = 256;          // after the accumulators
  static constexpr uint32_t SFB_COL = SFA_COL + 4 * STAGES;
  static constexpr uint32_t SFB_STRIDE = TBN / 32;  // TMEM columns of B scales per stage
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Non-swizzled shared-memory descriptor of a [rows][16 B] source of tcgen05.cp
// (8-row groups 128 B apart).
__device__ __forceinline__ uint64_t cp_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(16 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// bf16 store of one 32-column chunk of a plain or wgrad output: the warp's
// 32 rows (lane = row), packed bf16 pairs, through the warp's staging buffer.
template <int KIND, int TBN>
__device__ __forceinline__ void store_chunk(const Params& p, const Tile& tl, int q, int lane, int c,
                                            const uint32_t (&w)[16], uint8_t* stg) {
  const int n = tl.n_idx * TBN + c * 32;
  if (n >= p.N) return;
  if (Traits<KIND>::kragged) {
    const int m = tl.m0 + q * 32;
    const int nrows = max(0, min(32, p.M - m));
    __nv_bfloat16* dst;
    size_t ld;
    if (KIND == WGRAD2) {
      dst = static_cast<__nv_bfloat16*>(p.out0) + ((size_t)tl.e * p.M + m) * p.N + n;
      ld = p.N;
    } else {
      dst = n < p.f ? static_cast<__nv_bfloat16*>(p.out0) + ((size_t)tl.e * p.d + m) * p.f + n
                    : static_cast<__nv_bfloat16*>(p.out1) + ((size_t)tl.e * p.d + m) * p.f + (n - p.f);
      ld = p.f;
    }
    warp_store_rows(stg, w, dst, ld, nrows, lane);
  } else {
    const int wrow = tl.m0 + q * 32;
    const int nrows = max(0, min(32, tl.row_end - wrow));
    warp_store_rows(stg, w, static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * p.N + n, p.N, nrows, lane);
  }
}

// GEMM2 dgrad: the h rows (gate and up halves) of a warp's two 32-column
// chunks are copied into the warp's shared buffer with cp.async when the tile
// starts, so they land while its MMAs run (H_WARP bytes per warp: chunk j at
// 4096 j, gate then up, each [32 rows][64 B] in the staging swizzle; rows past
// the expert's end read as zeros).
constexpr int H_WARP = 2 * 4096;
__device__ __forceinline__ void h_prefetch(const Params& p, const Tile& tl, int q, int lane, int c_beg, int c_end,
                                           int tbn, uint8_t* hbuf) {
  const int wrow = tl.m0 + q * 32;
  const int nrows = max(0, min(32, tl.row_end - wrow));
  const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(p.aux);
  for (int c = c_beg; c < c_end; ++c) {
    const int n = tl.n_idx * tbn + c * 32;
    if (n >= p.N) continue;
#pragma unroll
    for (int part = 0; part < 2; ++part) {  // gate columns n.., up columns f + n..
      uint8_t* dst = hbuf + (c - c_beg) * 4096 + part * 2048;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int id = lane + 32 * i, r = id >> 2, g = id & 3;
        const bool ok = r < nrows;
        const __nv_bfloat16* src = h + (ok ? (size_t)(wrow + r) * 2 * p.f + part * p.f + n + 8 * g : 0);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(dst + stg_off(r, g))),
                     "l"(src), "r"(ok ? 16 : 0)
                     : "memory");
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// GEMM2 dgrad epilogue with h taken from the warp's prefetched buffer: dh_g =
// da * h_u * silu'(h_g), dh_u = da * silu(h_g), quantised along 2f and along
// the expert's rows (dh itself is stored only when p.out0 is set).
__device__ __forceinline__ void epilogue_dgrad2_mx(const Params& p, const Tile& tl, uint32_t tbase, int q, int lane,
                                                   int c_beg, int c_end, int tbn, uint8_t* stg, const uint8_t* hbuf) {
  const int wrow = tl.m0 + q * 32;
  const int nrows = max(0, min(32, tl.row_end - wrow));
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();
  __nv_bfloat16* dh = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * 2 * p.f;
  const size_t srow = tile_scale_row(tl, q, lane, 2 * p.f);
  const long stage = mx_row_tile_base(tl.m0 - tl.m_idx * BM, tl.e) + tl.m_idx;
  for (int c = c_beg; c < c_end; ++c) {
    const int n = tl.n_idx * tbn + c * 32;
    uint32_t r[32];
    ptx::tmem_ld32(tbase + c * 32, r);
    ptx::tmem_wait_ld();
    if (n >= p.N) continue;
    const uint8_t* hb = hbuf + (c - c_beg) * 4096;
    uint32_t hg[16], hu[16], w[16], wu[16];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 a = *reinterpret_cast<const uint4*>(hb + stg_off(lane, g));
      const uint4 b = *reinterpret_cast<const uint4*>(hb + 2048 + stg_off(lane, g));
      hg[4 * g] = a.x; hg[4 * g + 1] = a.y; hg[4 * g + 2] = a.z; hg[4 * g + 3] = a.w;
      hu[4 * g] = b.x; hu[4 * g + 1] = b.y; hu[4 * g + 2] = b.z; hu[4 * g + 3] = b.w;
    }
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
    if (p.out0) {
      warp_store_rows(stg, w, dh + n, 2 * (size_t)p.f, nrows, lane);
      warp_store_rows(stg, wu, dh + p.f + n, 2 * (size_t)p.f, nrows, lane);
    }
    if (p.qout) {
      quant_rows_staged(p, stg, w, wrow, nrows, 2 * p.f, n, lane, srow);
      quant_rows_staged(p, stg, wu, wrow, nrows, 2 * p.f, p.f + n, lane, srow);
    }
    if (p.qcol) {
      quant_cols_staged(p, stg, w, wrow, nrows, 2 * p.f, n, lane, stage, q);
      quant_cols_staged(p, stg, wu, wrow, nrows, 2 * p.f, p.f + n, lane, stage, q);
    }
  }
  __syncwarp();  // the buffer is refilled for the next tile
}

template <int KIND, int TBN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const Params p) {
  using Tr = Traits<KIND>;
  using G = Geo<TBN>;
  static_assert(KIND != FPROP1 || TBN == 256, "GEMM1 tiles pair 128 gate with 128 up columns");
  static_assert(!(Tr::kragged && Geo<TBN>::ACC == 2), "weight-gradient tiles use the single 256-column accumulator");
  static_assert(KIND != DGRAD2 || TBN == 128, "the h buffer holds a warp's two 32-column chunks");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sc_area = smem + STAGES * G::STAGE_BYTES;
  uint8_t* stg_area = sc_area + STAGES * G::SC_BYTES;  // epilogue staging, STG_BYTES per warp
  uint8_t* h_area = stg_area + NUM_EPI_WARPS * STG_BYTES;  // GEMM2 dgrad: h rows, H_WARP per warp
  constexpr int H_BYTES = KIND == DGRAD2 ? NUM_EPI_WARPS * H_WARP : 0;
  Smem* sm = reinterpret_cast<Smem*>(h_area + H_BYTES);
  int* offs = reinterpret_cast<int*>(sm + 1);
  int* tstart = offs + (p.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  build_tile_table<KIND, NUM_THREADS>(p, offs, tstart);
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
  const int total = Tr::kragged ? p.E * p.m_tiles * p.n_tiles : tstart[p.E];
  const uint32_t tmem = sm->tmem_base;
  const long Kd = gemm_k<KIND>(p);

  if (warp == 0) {
    // ===================================================== producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB0);
      ptx::prefetch_tmap(&tmB1);
    }
    uint32_t it = 0;
    bool ok = true;
    for (int r = 0, t = sched_tile<Tr::kragged>(0); t < total && ok; t = sched_tile<Tr::kragged>(++r)) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
        uint64_t* fb = &sm->full[s];
        const int k0 = kb * BK;
        if (lane == 0) {
          uint8_t* a = smem + s * G::STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          // B column groups of 128 that exist (N need not be a multiple of
          // the tile width): only their scale chunks are fetched
          const int nb = KIND == FPROP1 ? 2 : min(G::SCB, (p.N - tl.n_idx * TBN + 127) / 128);
          ptx::mbar_expect_tx(fb, G::STAGE_BYTES + 512 + 512 * nb);
          // ---- E8M0 scale chunks (512 B per 128 rows or columns and K stage):
          // A's, then one per 128 columns of B
          uint8_t* sa = sc_area + s * G::SC_BYTES;
          uint8_t* sb = sa + 512;
          if (!Tr::kragged) {  // rows in per-expert 128-row tiles, K = Kd
            const long grp = mx_row_tile_base(offs[tl.e], tl.e) + tl.m_idx;
            ptx::bulk_load(sa, p.sfa + ((grp * (Kd / 128) + kb) << 9), 512, fb);
          } else {  // features m0.. at K stage kb of the expert's per-expert 128-row tiles
            const long w = mx_row_tile_base(offs[tl.e], tl.e) + kb;
            ptx::bulk_load(sa, p.sfa + ((w * (p.M / 128) + tl.m_idx) << 9), 512, fb);
          }
          if (KIND == FPROP1) {  // w_gate | w_up columns: K stage e d/128 + kb, column group n_idx
            const long c = ((long)tl.e * (p.d / 128) + kb) * (p.f / 128) + tl.n_idx;
            ptx::bulk_load(sb, p.sfb0 + (c << 9), 512, fb);
            ptx::bulk_load(sb + 512, p.sfb1 + (c << 9), 512, fb);
          } else if (KIND == FPROP2) {  // w_down columns: K stage e f/128 + kb
            const long c = ((long)tl.e * (p.f / 128) + kb) * (p.d / 128) + (long)tl.n_idx * G::SCB;
            ptx::bulk_load(sb, p.sfb0 + (c << 9), 512 * nb, fb);
          } else if (KIND == DGRAD2) {  // w_down rows (f) along d
#pragma unroll
            for (int j = 0; j < G::SCB; ++j) {
              if (j >= nb) break;
              const long grp = (long)tl.e * (p.f / 128) + (long)tl.n_idx * G::SCB + j;
              ptx::bulk_load(sb + 512 * j, p.sfb0 + ((grp * (p.d / 128) + kb) << 9), 512, fb);
            }
          } else if (KIND == DGRAD1) {  // w_gate rows (d) along f for K < f, then w_up's
            const int kfs = p.f / 128;
            const uint8_t* src = kb < kfs ? p.sfb0 : p.sfb1;
            const int kk = kb < kfs ? kb : kb - kfs;
#pragma unroll
            for (int j = 0; j < G::SCB; ++j) {
              if (j >= nb) break;
              const long grp = (long)tl.e * (p.d / 128) + (long)tl.n_idx * G::SCB + j;
              ptx::bulk_load(sb + 512 * j, src + ((grp * kfs + kk) << 9), 512, fb);
            }
          } else {  // wgrad: B features at the expert's K stage
            const long c = (mx_row_tile_base(offs[tl.e], tl.e) + kb) * (p.N / 128) + (long)tl.n_idx * G::SCB;
            ptx::bulk_load(sb, p.sfb0 + (c << 9), 512 * nb, fb);
          }
          // ---- E4M3 tiles
          if (KIND == FPROP1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * 128;
            ptx::tma_load_3d(b, &tmB0, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + BOX_BYTES, &tmB1, fb, n0, k0, tl.e);
          } else if (KIND == FPROP2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            const int n0 = tl.n_idx * TBN;
#pragma unroll
            for (int j = 0; j < G::SCB; ++j) ptx::tma_load_3d(b + j * BOX_BYTES, &tmB0, fb, n0 + 128 * j, k0, tl.e);
          } else if (KIND == DGRAD2) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * TBN, tl.e);
          } else if (KIND == DGRAD1) {
            ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
            if (k0 < p.f) ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * TBN, tl.e);
            else ptx::tma_load_3d(b, &tmB1, fb, k0 - p.f, tl.n_idx * TBN, tl.e);
          } else {  // WGRAD2 / WGRAD1: K runs over the expert's rows
            const int row = tl.k_row0 + k0;
            ptx::tma_load_2d(a, &tmA, fb, tl.m0, row);
            const int n0 = tl.n_idx * TBN;
#pragma unroll
            for (int j = 0; j < G::SCB; ++j) ptx::tma_load_2d(b + j * BOX_BYTES, &tmB0, fb, n0 + 128 * j, row);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        const long long t0 = clock64();
        while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
               !ptx::mbar_try_wait(&sm->full[s], 1)) {
        }
      }
    }
  } else if (warp == 1) {
    // ========================================================= MMA issuer
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int r = 0, t = sched_tile<Tr::kragged>(0); t < total && ok; t = sched_tile<Tr::kragged>(++r)) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      if (tl.nkb == 0) continue;
      const int buf = G::ACC == 2 ? (acc_it & 1) : 0;
      const uint32_t aph = (G::ACC == 2 ? (acc_it >> 1) : acc_it) & 1u;
      if (!wait_bar(&sm->tempty[buf], aph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * TBN);
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1u;
        if (!wait_bar(&sm->full[s], ph, &sm->abort_flag, p.err)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * G::STAGE_BYTES;
        int nks = BK / 32;
        if (Tr::kragged) {
          const int valid = tl.row_end - (tl.k_row0 + kb * BK);
          if (valid < BK) {
            // skip K steps made only of rows past the expert's end; zero the
            // rest of the last partial step in A (one 128-row box), which the
            // async proxy then reads
            nks = (valid + 31) / 32;
            for (int i = valid * 8 + lane; i < nks * 32 * 8; i += 32)
              *reinterpret_cast<uint4*>(a + i * 16) = make_uint4(0, 0, 0, 0);
            ptx::fence_proxy_async_smem();
          }
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t sa = ptx::smem_u32(sc_area + s * G::SC_BYTES);
          const uint32_t sfa = tmem + G::SFA_COL + 4 * s, sfb = tmem + G::SFB_COL + G::SFB_STRIDE * s;
          tmem_cp_32x128b_x4(sfa, cp_desc(sa));
#pragma unroll
          for (int j = 0; j < G::SCB; ++j) tmem_cp_32x128b_x4(sfb + 4 * j, cp_desc(sa + 512 + 512 * j));
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + A_BYTES;
          for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ad = Tr::a_mn ? ptx::smem_desc_sw128(a_addr + ks * 4096, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = Tr::b_mn ? ptx::smem_desc_sw128(b_addr + ks * 4096, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            const uint32_t idesc = ptx::idesc_mxf8_f32(BM, TBN, Tr::a_mn ? 1 : 0, Tr::b_mn ? 1 : 0, ks, ks);
            ptx::mma_mxf8(d_tmem, ad, bd, idesc, sfa, sfb, (kb > 0 || ks > 0) ? 1u : 0u);
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
      ptx::mma_commit(&sm->drain);
      const long long t0 = clock64();
      while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->drain, 0)) {
      }
    }
  } else {
    // ============================================================ epilogue
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    uint8_t* stg = stg_area + ew * STG_BYTES;
    constexpr int NC = KIND == FPROP1 ? 4 : TBN / 32;  // chunks of the tile (FPROP1: gate/up pairs)
    uint32_t acc_it = 0;
    for (int r = 0, t = sched_tile<Tr::kragged>(0); t < total; t = sched_tile<Tr::kragged>(++r)) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      if (tl.nkb == 0) {  // wgrad of an expert without rows: dW_e = 0
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
        for (int c = half * NC / 2; c < (half + 1) * NC / 2; ++c) store_chunk<KIND, TBN>(p, tl, q, lane, c, z, stg);
        continue;
      }
      if (KIND == DGRAD2)  // this tile's h rows land in shared memory while its MMAs run
        h_prefetch(p, tl, q, lane, half * NC / 2, (half + 1) * NC / 2, TBN, h_area + ew * H_WARP);
      const int buf = G::ACC == 2 ? (acc_it & 1) : 0;
      const uint32_t aph = (G::ACC == 2 ? (acc_it >> 1) : acc_it) & 1u;
      if (!wait_bar(&sm->tfull[buf], aph, &sm->abort_flag, p.err)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + static_cast<uint32_t>(buf * TBN) + (static_cast<uint32_t>(q * 32) << 16);
      if (G::ACC == 2 || KIND == DGRAD2) {
        // double-buffered (or too many registers to drain first): epilogue straight from TMEM
        if constexpr (KIND == DGRAD2)
          epilogue_dgrad2_mx(p, tl, tbase, q, lane, half * NC / 2, (half + 1) * NC / 2, TBN, stg, h_area + ew * H_WARP);
        else if constexpr (!Tr::kragged)
          epilogue_tile_staged<KIND, TBN, true>(p, tl, tbase, q, lane, half * NC / 2, (half + 1) * NC / 2, stg);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm->tempty[buf]);
      } else {
        // single accumulator: copy this warp's 128 columns out as packed bf16,
        // release it, then store
        if constexpr (KIND == FPROP1) {
          // the raw fp32 gate/up values leave TMEM first (the shortest hold of
          // the accumulator); the SwiGLU math runs after its release
          uint32_t rg[2][32], ru[2][32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            ptx::tmem_ld32(tbase + (2 * half + cc) * 32, rg[cc]);
            ptx::tmem_ld32(tbase + 128 + (2 * half + cc) * 32, ru[cc]);
          }
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm->tempty[buf]);
          const int wrow = tl.m0 + q * 32;
          const int nrows = max(0, min(32, tl.row_end - wrow));
          __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * 2 * p.f;
          __nv_bfloat16* ao = static_cast<__nv_bfloat16*>(p.out1) + (size_t)wrow * p.f;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int n = tl.n_idx * 128 + (2 * half + cc) * 32;
            if (n >= p.f) continue;
            uint32_t w[16], wa[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(rg[cc][2 * i]), g1 = __uint_as_float(rg[cc][2 * i + 1]);
              const float u0 = __uint_as_float(ru[cc][2 * i]), u1 = __uint_as_float(ru[cc][2 * i + 1]);
              w[i] = pack_bf16x2(g0, g1);
              wa[i] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
            }
            warp_store_rows(stg, w, h + n, 2 * (size_t)p.f, nrows, lane);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(ru[cc][2 * i]), __uint_as_float(ru[cc][2 * i + 1]));
            warp_store_rows(stg, w, h + p.f + n, 2 * (size_t)p.f, nrows, lane);
            warp_store_rows(stg, wa, ao + n, p.f, nrows, lane);
            if (p.qout) quant_rows_staged(p, stg, wa, wrow, nrows, p.f, n, lane, tile_scale_row(tl, q, lane, p.f));
            if (p.qcol)  // A along the expert's rows too (the GEMM2 weight gradient's A operand)
              quant_cols_staged(p, stg, wa, wrow, nrows, p.f, n, lane,
                                mx_row_tile_base(tl.m0 - tl.m_idx * BM, tl.e) + tl.m_idx, q);
          }
        } else {
          uint32_t w[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            ptx::tmem_ld32(tbase + (4 * half + c) * 32, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) w[c][i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm->tempty[buf]);
#pragma unroll
          for (int c = 0; c < 4; ++c) store_chunk<KIND, TBN>(p, tl, q, lane, 4 * half + c, w[c], stg);
        }
      }
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

template <int KIND, int TBN>
size_t smem_bytes(int E) {
  return 1024 + STAGES * Geo<TBN>::STAGE_BYTES + STAGES * Geo<TBN>::SC_BYTES + NUM_EPI_WARPS * STG_BYTES +
         (KIND == DGRAD2 ? NUM_EPI_WARPS * H_WARP : 0) + sizeof(Smem) + 2 * (E + 1) * sizeof(int) + 64;
}

template <int KIND, int TBN>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const Params& p,
                   long max_tiles, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = smem_bytes<KIND, TBN>(p.E);
  cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<KIND, TBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
  MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, true), st) mx_gemm_kernel<KIND, TBN><<<grid, NUM_THREADS, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// MXFP8 weight gradients on CTA pairs (2-CTA clusters,
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale). A single CTA's tile
// stops at 128 x 256 here: the block scales take the TMEM columns a second
// 256-column accumulator would need, so its operands cost 48 KB per 128-row K
// stage. A pair computes a 256 x 256 block of one expert's gradient: each CTA
// loads its own 128 features of A and its own 128 columns of B per stage
// (32 KB for the same MMA work per SM), its own A scale chunk and both B
// scale chunks. In a pair MMA each CTA's TMEM must hold the B scales of all
// 256 columns and the A scales of its own rows; tcgen05.cp.cta_group::2,
// issued by the even CTA, copies each CTA's staged chunks into its own TMEM.
// Each CTA's TMEM receives its 128 rows x 256 columns of the accumulator (one
// buffer, drained into registers and released before the stores).
//   warp 0      both CTAs: producer of its own half of each stage.
//   warp 1      even CTA: scale copies and MMA issue; each stage's release
//               and each finished accumulator are committed to both CTAs.
//               odd CTA: relay; zeroes its A rows past the expert's end once
//               its half has landed, then arrives on the even CTA's `full`.
//   warps 2..9  both CTAs: epilogue of its own 128 rows.
// All 32 lanes of a warp poll each barrier; every wait is bounded, and a CTA
// that gives up raises both CTAs' abort flags.
constexpr int PX_NS = 6;
constexpr int PX_A = 128 * BK;                                 // own 128 features x 128 K rows
constexpr int PX_STAGE = 2 * PX_A;                             // + own 128 columns of B
constexpr int PX_SC = 512 + 1024;                              // A chunk, then both B chunks
constexpr uint32_t PX_SFA = 256, PX_SFB = 288;  // TMEM scale rings (B scales 32-column aligned)
static_assert(PX_SFA + 4 * PX_NS <= PX_SFB && PX_SFB + 8 * PX_NS <= TMEM_COLS, "scale rings fit next to the accumulator");

struct PxSmem {
  uint64_t full[PX_NS];
  uint64_t empty[PX_NS];
  uint64_t tfull, tempty, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void tmem_cp_pair_32x128b_x4(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Bounded wait on a local mbarrier whose arrivals may come from the other CTA
// of the pair; on expiry it sets the error word and both CTAs' abort flags.
__device__ __forceinline__ bool px_wait(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t peer_abort,
                                        int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      set_error(err, MOE_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      ptx::st_cluster_u32(peer_abort, 1u);
      return false;
    }
  }
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mx_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Params p) {
  static_assert(KIND == WGRAD1 || KIND == WGRAD2, "weight-gradient kinds");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sc_area = smem + PX_NS * PX_STAGE;
  uint8_t* stg_area = sc_area + PX_NS * PX_SC;
  PxSmem* sm = reinterpret_cast<PxSmem*>(stg_area + NUM_EPI_WARPS * STG_BYTES);
  const int* __restrict__ offs = p.offsets;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank(), peer = rank ^ 1u;
  const int cid = static_cast<int>(ptx::cluster_id_x()), ncl = static_cast<int>(ptx::n_clusters_x());
  auto in_cta = [&](const void* x, uint32_t r) { return ptx::mapa(ptx::smem_u32(x), r); };
  const uint32_t peer_abort = in_cta(&sm->abort_flag, peer);

  if (threadIdx.x == 0) {
    for (int s = 0; s < PX_NS; ++s) {
      ptx::mbar_init(&sm->full[s], rank == 0 ? 2 : 1);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    ptx::mbar_init(&sm->tfull, 1);
    ptx::mbar_init(&sm->tempty, 2 * NUM_EPI_WARPS);
    ptx::mbar_init(&sm->drain, 1);
    sm->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&sm->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  if (threadIdx.x == 0 && ptx::ld_cluster_u32(in_cta(&sm->tmem_base, peer)) != tmem) {
    set_error(p.err, MOE_ERR_DEVICE_PAIR);
    sm->abort_flag = 1;
  }
  __syncthreads();
  const bool run = sm->abort_flag == 0;

  const int per = p.m_tiles * p.n_tiles;  // m_tiles: blocks of 256 features
  const int total = p.E * per;
  // the pair's r-th tile: experts largest first, a snake over the pairs
  auto tile_of = [&](int r) { return r * ncl + ((r & 1) ? ncl - 1 - cid : cid); };
  struct WT {
    int e, m0, n_idx, r0, r1, nkb;
    long kst0;  // the expert's first K stage in the scale chunks
  };
  auto decode_w = [&](int t) {
    WT w;
    w.e = p.order ? __ldg(p.order + t / per) : t / per;
    const int local = t % per;
    w.m0 = (local / p.n_tiles) * 256;
    w.n_idx = local % p.n_tiles;
    w.r0 = __ldg(offs + w.e);
    w.r1 = __ldg(offs + w.e + 1);
    w.nkb = (w.r1 - w.r0 + BK - 1) / BK;
    w.kst0 = mx_row_tile_base(w.r0, w.e);
    return w;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    const bool ok = px_wait(bar, parity, &sm->abort_flag, peer_abort, p.err);
    return __all_sync(0xffffffffu, ok) != 0;
  };
  // rows past the expert's end belong to the next expert: zero them in this
  // CTA's A box (K steps made only of them are skipped); returns the K steps
  auto zero_tail = [&](uint8_t* a, int valid) {
    const int nks = (valid + 31) / 32;
    for (int i = valid * 8 + lane; i < nks * 32 * 8; i += 32)
      *reinterpret_cast<uint4*>(a + i * 16) = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    return nks;
  };

  if (warp == 0) {
    // ===================================================== producer
    if (run) {
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
      }
      uint32_t it = 0;
      bool ok = true;
      for (int r = 0, t = tile_of(0); t < total && ok; t = tile_of(++r)) {
        const WT w = decode_w(t);
        for (int kb = 0; kb < w.nkb; ++kb, ++it) {
          const int s = it % PX_NS;
          if (!warp_wait(&sm->empty[s], ((it / PX_NS) & 1u) ^ 1u)) { ok = false; break; }
          if (lane == 0) {
            uint8_t* a = smem + s * PX_STAGE;
            uint8_t* b = a + PX_A;
            uint8_t* sa = sc_area + s * PX_SC;
            uint64_t* fb = &sm->full[s];
            const int n0 = w.n_idx * 256;
            const int nb = min(2, (p.N - n0 + 127) / 128);  // B column groups that exist
            ptx::mbar_expect_tx(fb, PX_STAGE + 512 + 512 * nb);
            const int row = w.r0 + kb * BK;
            ptx::tma_load_2d(a, &tmA, fb, w.m0 + 128 * static_cast<int>(rank), row);
            ptx::tma_load_2d(b, &tmB, fb, n0 + 128 * static_cast<int>(rank), row);
            // scale chunks of K stage kst: this CTA's 128 features (clamped:
            // a block past M computes rows that are not stored), all of B's
            const long kst = w.kst0 + kb;
            const int ga = min(w.m0 / 128 + static_cast<int>(rank), p.M / 128 - 1);
            ptx::bulk_load(sa, p.sfa + ((kst * (p.M / 128) + ga) << 9), 512, fb);
            ptx::bulk_load(sa + 512, p.sfb0 + ((kst * (p.N / 128) + n0 / 128) << 9), 512 * nb, fb);
          }
          __syncwarp();
        }
      }
      // the even CTA's commits release these stages: wait for the last ones
      // before the CTA may finish
      for (int k = 0; k < PX_NS && ok; ++k, ++it) ok = warp_wait(&sm->empty[it % PX_NS], ((it / PX_NS) & 1u) ^ 1u);
      if (!ok && lane == 0) {
        for (int s = 0; s < PX_NS; ++s) {
          const long long t0 = clock64();
          while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                 !ptx::mbar_try_wait(&sm->full[s], 1)) {
          }
        }
      }
    }
  } else if (warp == 1 && rank == 1) {
    // ============================================ relay (odd CTA of the pair)
    const uint32_t leader_full0 = in_cta(&sm->full[0], 0);
    uint32_t it = 0;
    bool ok = run;
    for (int r = 0, t = tile_of(0); t < total && ok; t = tile_of(++r)) {
      const WT w = decode_w(t);
      for (int kb = 0; kb < w.nkb; ++kb, ++it) {
        const int s = it % PX_NS;
        if (!warp_wait(&sm->full[s], (it / PX_NS) & 1u)) { ok = false; break; }
        const int valid = w.r1 - (w.r0 + kb * BK);
        if (valid < BK) zero_tail(smem + s * PX_STAGE, valid);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(leader_full0 + 8u * s);
      }
    }
  } else if (warp == 1) {
    // ============================================ MMA issuer (even CTA)
    const uint32_t peer_empty0 = in_cta(&sm->empty[0], 1), peer_tfull = in_cta(&sm->tfull, 1);
    uint32_t it = 0, acc_it = 0;
    bool ok = run;
    for (int r = 0, t = tile_of(0); t < total && ok; t = tile_of(++r)) {
      const WT w = decode_w(t);
      if (w.nkb == 0) continue;
      if (!warp_wait(&sm->tempty, (acc_it & 1u) ^ 1u)) { ok = false; break; }
      ptx::tc_fence_after();
      for (int kb = 0; kb < w.nkb; ++kb, ++it) {
        const int s = it % PX_NS;
        if (!warp_wait(&sm->full[s], (it / PX_NS) & 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * PX_STAGE;
        const int valid = w.r1 - (w.r0 + kb * BK);
        const int nks = valid < BK ? zero_tail(a, valid) : BK / 32;
        __syncwarp();
        if (lane == 0) {
          const uint32_t sa = ptx::smem_u32(sc_area + s * PX_SC);
          const uint32_t sfa = tmem + PX_SFA + 4 * s, sfb = tmem + PX_SFB + 8 * s;
          tmem_cp_pair_32x128b_x4(sfa, cp_desc(sa));
          tmem_cp_pair_32x128b_x4(sfb, cp_desc(sa + 512));
          tmem_cp_pair_32x128b_x4(sfb + 4, cp_desc(sa + 1024));
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + PX_A;
          for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + ks * 4096, BOX_BYTES, 1024);
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 4096, BOX_BYTES, 1024);
            mma_mxf8_pair(tmem, ad, bd, ptx::idesc_mxf8_f32(2 * BM, 256, 1, 1, ks, ks), sfa, sfb,
                          (kb > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit_pair(ptx::smem_u32(&sm->empty[s]));
          ptx::mma_commit_pair(peer_empty0 + 8u * s);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        ptx::mma_commit_pair(ptx::smem_u32(&sm->tfull));
        ptx::mma_commit_pair(peer_tfull);
      }
      __syncwarp();
      ++acc_it;
    }
    if (!ok && run && lane == 0) {
      ptx::mma_commit_pair(ptx::smem_u32(&sm->drain));
      const long long t0 = clock64();
      while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->drain, 0)) {
      }
    }
  } else {
    // ============================================================ epilogue
    // warp (q, half): TMEM lanes 32q..32q+31 (this CTA's rows), columns
    // 128 half .. +127, moved into registers as packed bf16 and released to
    // the even CTA's `tempty` before the stores.
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    uint8_t* stg = stg_area + ew * STG_BYTES;
    const uint32_t leader_tempty = in_cta(&sm->tempty, 0);
    uint32_t acc_it = 0;
    for (int r = 0, t = tile_of(0); t < total && run; t = tile_of(++r)) {
      const WT w = decode_w(t);
      Tile tl{};
      tl.e = w.e;
      tl.m0 = w.m0 + 128 * static_cast<int>(rank);
      tl.n_idx = w.n_idx;
      uint32_t v[4][16];
      if (w.nkb == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) v[c][i] = 0u;  // expert with no rows: dW_e = 0
      } else {
        if (!warp_wait(&sm->tfull, acc_it & 1u)) break;
        ptx::tc_fence_after();
        const uint32_t tbase = tmem + static_cast<uint32_t>(half * 128) + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          ptx::tmem_ld32(tbase + c * 32, rr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[c][i] = pack_bf16x2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(leader_tempty);
        ++acc_it;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) store_chunk<KIND, 256>(p, tl, q, lane, 4 * half + c, v[c], stg);
    }
  }

  // No CTA of the pair leaves while the other may still reach its shared
  // memory or TMEM; then both free the pair's TMEM together.
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <int KIND>
cudaError_t launch_wgrad_pair(const CUtensorMap& a, const CUtensorMap& b, const Params& p, cudaStream_t st) {
  const long tiles = (long)p.E * p.m_tiles * p.n_tiles;
  if (tiles <= 0) return cudaSuccess;
  const size_t smem = 1024 + PX_NS * (PX_STAGE + PX_SC) + NUM_EPI_WARPS * STG_BYTES + sizeof(PxSmem) + 64;
  cudaError_t e = cudaFuncSetAttribute(mx_wgrad_pair_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // pairs resident at once (a pair needs two SMs of one GPC); computed once
  static std::atomic<int> cached_pairs{0};
  int max_pairs = cached_pairs.load(std::memory_order_relaxed);
  if (max_pairs <= 0) {
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    e = cudaOccupancyMaxActiveClusters(&max_pairs, mx_wgrad_pair_kernel<KIND>, &cfg);
    if (e != cudaSuccess) return e;
    if (max_pairs <= 0) return cudaErrorLaunchOutOfResources;
    cached_pairs.store(max_pairs, std::memory_order_relaxed);
  }
  const long pairs = tiles < max_pairs ? tiles : max_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  return MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, true), st)
      cudaLaunchKernelEx(&cfg, mx_wgrad_pair_kernel<KIND>, a, b, p);
}


// Output tile widths (measured choice): 256 with one accumulator released
// early, except the GEMM2 dgrad, whose SwiGLU-backward epilogue reads h and
// gains more from a double-buffered accumulator than it loses to the narrower
// tile (the wgrads and GEMM2 re-read A twice as often at 128 and got slower).
constexpr int kN_FPROP1 = 256, kN_FPROP2 = 256, kN_DGRAD2 = 128, kN_DGRAD1 = 256, kN_WGRAD = 256;
// The weight gradients run on CTA pairs (256 x 256 tiles, mx_wgrad_pair_kernel)
// when selected with moe_use_cta_pairs(1); one CTA per SM by default.
std::atomic<int> g_wgrad_pairs{0};

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
};

// The prepared weights: each of w_gate, w_up, w_down quantised along both of
// the K axes the expert GEMMs use (columns: blocks of 32 rows; rows: blocks of
// 32 columns; scales as scale chunks), carved from one caller buffer.
struct MxWeights {
  QBuf wg_c, wu_c, wd_c, wd_r, wg_r, wu_r;
};
inline MxWeights carve_weights(void* base, int E, int d, int f) {
  Carver cv{static_cast<char*>(base)};
  const size_t Ed = (size_t)E * d, Ef = (size_t)E * f;
  MxWeights w;
  w.wg_c = cv.take(Ed * f, Ed / 32 * f);
  w.wu_c = cv.take(Ed * f, Ed / 32 * f);
  w.wd_c = cv.take(Ef * d, Ef / 32 * d);
  w.wd_r = cv.take(Ef * d, Ef * d / 32);
  w.wg_r = cv.take(Ed * f, Ed * f / 32);
  w.wu_r = cv.take(Ed * f, Ed * f / 32);
  return w;
}

// Bytes of the scale chunks of a [rows][C] operand quantised along rows in E
// segments (K stages of 4 blocks; a segment's stages start anew).
inline size_t seg_words_bytes(long rows, int E, long C) { return ((size_t)(rows + 127) / 128 + E + 1) * C * 4; }

}  // namespace

// Bytes of the scale chunks of a row operand with K columns, grouped by
// per-expert 128-row tiles.
inline size_t tile_scale_bytes(long R, int E, long K) { return (size_t)mx_row_tiles(R, E) * 4 * K; }

size_t fwd_workspace(long R, int E, int d, int f) {
  const size_t Ed = (size_t)E * d;
  return al(R * (size_t)d) + al(tile_scale_bytes(R, E, d)) + al(R * (size_t)f) + al(tile_scale_bytes(R, E, f)) +
         2 * (al(Ed * f) + al(Ed / 32 * f)) + al((size_t)E * f * d) + al((size_t)E * f / 32 * d);
}

size_t bwd_workspace(long R, int E, int d, int f) {
  const size_t Ed = (size_t)E * d, Ef = (size_t)E * f;
  return al(R * (size_t)d) + al(tile_scale_bytes(R, E, d))                 // dy rows
         + al(R * (size_t)d) + al(seg_words_bytes(R, E, d))                    // dy segment columns
         + al(R * (size_t)f) + al(seg_words_bytes(R, E, f))                    // a segment columns
         + al(Ef * d) + al(Ef * d / 32)                                    // w_down rows
         + al(R * 2 * (size_t)f) + al(tile_scale_bytes(R, E, 2L * f))      // dh rows
         + al(R * 2 * (size_t)f) + al(seg_words_bytes(R, E, 2L * f))            // dh segment columns
         + 2 * (al(Ed * f) + al(Ed * f / 32))                              // w_gate, w_up rows
         + al(R * (size_t)d) + al(seg_words_bytes(R, E, d))                    // x segment columns
         + al((size_t)E * 4);                                              // expert order
}

}  // namespace mx
}  // namespace tc

using namespace tc;

size_t mx_col_operand_bytes(long R, int E, int K) { return mx::al((size_t)R * K) + mx::al(mx::seg_words_bytes(R, E, K)); }

cudaError_t mx_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd, const int32_t* offsets,
                       int R, int E, int d, int f, void* h, void* a, void* y, void* ws, cudaStream_t st,
                       const uint8_t* xq_codes, const uint8_t* xq_scales, const void* wq, uint8_t* a_cols) {
  using namespace mx;
  Carver cv{static_cast<char*>(ws)};
  const long Ed = (long)E * d, Ef = (long)E * f;
  QBuf xq = cv.take((size_t)R * d, tile_scale_bytes(R, E, d));
  QBuf aq = cv.take((size_t)R * f, tile_scale_bytes(R, E, f));
  QBuf wgq = cv.take((size_t)Ed * f, (size_t)Ed / 32 * f);
  QBuf wuq = cv.take((size_t)Ed * f, (size_t)Ed / 32 * f);
  QBuf wdq = cv.take((size_t)Ef * d, (size_t)Ef / 32 * d);
  cudaError_t e;
  // operands of GEMM1 along d: x rows (already quantised when the dispatch did
  // it), w_gate / w_up columns (32-row blocks never cross experts)
  if (xq_codes) {
    xq.q = const_cast<uint8_t*>(xq_codes);
    xq.s = const_cast<uint8_t*>(xq_scales);
  } else if ((e = launch_mxfp8_quant_rows(x_perm, R, d, xq.q, xq.s, st, kScalesTiles, offsets, E)) != cudaSuccess) {
    return e;
  }
  if (wq) {  // prepared once per weight update
    const MxWeights w = carve_weights(const_cast<void*>(wq), E, d, f);
    wgq = w.wg_c;
    wuq = w.wu_c;
    wdq = w.wd_c;
  } else {
    if ((e = launch_mxfp8_quant_cols(wg, (int)Ed, f, nullptr, 1, wgq.q, wgq.s, st, true)) != cudaSuccess) return e;
    if ((e = launch_mxfp8_quant_cols(wu, (int)Ed, f, nullptr, 1, wuq.q, wuq.s, st, true)) != cudaSuccess) return e;
    if ((e = launch_mxfp8_quant_cols(wd, (int)Ef, d, nullptr, 1, wdq.q, wdq.s, st, true)) != cudaSuccess) return e;
  }

  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  if (!map_2d(&mA, xq.q, U8, 1, d, R, 128, BM) || !map_3d(&mB0, wgq.q, U8, 1, f, d, E, 128, 128) ||
      !map_3d(&mB1, wuq.q, U8, 1, f, d, E, 128, 128))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + 127) / 128; p.out0 = h; p.out1 = a;
  p.sfa = xq.s; p.sfb0 = wgq.s; p.sfb1 = wuq.s;
  p.qout = aq.q; p.qsc = aq.s;  // the epilogue also quantises A along f for GEMM2
  if (a_cols) {                  // ... and along the experts' rows for the GEMM2 weight gradient
    p.qcol = a_cols;
    p.qcsc = a_cols + al((size_t)R * f);
  }
  if ((e = launch<FPROP1, kN_FPROP1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess)
    return e;
  p.qout = nullptr; p.qsc = nullptr; p.qcol = nullptr; p.qcsc = nullptr;
  // GEMM2 along f: A rows (written by GEMM1's epilogue), w_down columns
  if (!map_2d(&mA, aq.q, U8, 1, f, R, 128, BM) || !map_3d(&mB0, wdq.q, U8, 1, d, f, E, 128, 128))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + kN_FPROP2 - 1) / kN_FPROP2; p.out0 = y; p.out1 = nullptr;
  p.sfa = aq.s; p.sfb0 = wdq.s; p.sfb1 = nullptr;
  return launch<FPROP2, kN_FPROP2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
}

cudaError_t mx_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* ws, cudaStream_t st,
                       const uint8_t* dyq_codes, const uint8_t* dyq_scales, const void* wq, const uint8_t* a_cols) {
  using namespace mx;
  Carver cv{static_cast<char*>(ws)};
  const long Ed = (long)E * d, Ef = (long)E * f;
  QBuf dyr = cv.take((size_t)R * d, tile_scale_bytes(R, E, d));
  QBuf dyc = cv.take((size_t)R * d, seg_words_bytes(R, E, d));
  QBuf ac = cv.take((size_t)R * f, seg_words_bytes(R, E, f));
  QBuf wdr = cv.take((size_t)Ef * d, (size_t)Ef * d / 32);
  QBuf dhr = cv.take((size_t)R * 2 * f, tile_scale_bytes(R, E, 2L * f));
  QBuf dhc = cv.take((size_t)R * 2 * f, seg_words_bytes(R, E, 2L * f));
  QBuf wgr = cv.take((size_t)Ed * f, (size_t)Ed * f / 32);
  QBuf wur = cv.take((size_t)Ed * f, (size_t)Ed * f / 32);
  QBuf xc = cv.take((size_t)R * d, seg_words_bytes(R, E, d));
  int32_t* order = reinterpret_cast<int32_t*>(cv.p + cv.used);
  cudaError_t e;
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  // the weight gradients walk their experts largest first
  if ((e = launch_expert_order(offsets, E, order, st)) != cudaSuccess) return e;

  // dA = dy . Wd^T (K = d): dy rows (already quantised when the combine
  // backward did it), w_down rows; SwiGLU backward fused -> dh
  if (dyq_codes) {
    dyr.q = const_cast<uint8_t*>(dyq_codes);
    dyr.s = const_cast<uint8_t*>(dyq_scales);
  } else if ((e = launch_mxfp8_quant_rows(dy_perm, R, d, dyr.q, dyr.s, st, kScalesTiles, offsets, E)) !=
             cudaSuccess) {
    return e;
  }
  MxWeights w{};
  if (wq) {
    w = carve_weights(const_cast<void*>(wq), E, d, f);
    wdr = w.wd_r;
  } else if ((e = launch_mxfp8_quant_rows(wd, Ef, d, wdr.q, wdr.s, st, kScalesChunk)) != cudaSuccess) {
    return e;
  }
  if (!map_2d(&mA, dyr.q, U8, 1, d, R, 128, BM) || !map_3d(&mB0, wdr.q, U8, 1, d, f, E, 128, kN_DGRAD2))
    return cudaErrorInvalidValue;
  // dh itself is never stored: the epilogue quantises it along 2f (the GEMM1
  // dgrad's A) and along the expert's rows (the GEMM1 wgrad's B)
  p.N = f; p.n_tiles = (f + kN_DGRAD2 - 1) / kN_DGRAD2; p.out0 = nullptr; p.aux = h;
  p.sfa = dyr.s; p.sfb0 = wdr.s;
  p.qout = dhr.q; p.qsc = dhr.s;
  p.qcol = dhc.q; p.qcsc = dhc.s;
  if ((e = launch<DGRAD2, kN_DGRAD2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess)
    return e;
  p.qout = nullptr; p.qsc = nullptr; p.qcol = nullptr; p.qcsc = nullptr;

  // dWd[e] = A_e^T dy_e (K = the expert's rows): A and dy quantised along rows per expert
  // (A already, when the forward's GEMM1 epilogue wrote it)
  if (a_cols) {
    ac.q = const_cast<uint8_t*>(a_cols);
    ac.s = const_cast<uint8_t*>(a_cols) + al((size_t)R * f);
  } else if ((e = launch_mxfp8_quant_cols(a, R, f, offsets, E, ac.q, ac.s, st, true)) != cudaSuccess) {
    return e;
  }
  if ((e = launch_mxfp8_quant_cols(dy_perm, R, d, offsets, E, dyc.q, dyc.s, st, true)) != cudaSuccess) return e;
  if (!map_2d(&mA, ac.q, U8, 1, f, R, 128, 128) || !map_2d(&mB0, dyc.q, U8, 1, d, R, 128, 128))
    return cudaErrorInvalidValue;
  p.M = f; p.N = d; p.n_tiles = (d + kN_WGRAD - 1) / kN_WGRAD; p.out0 = dwd;
  p.aux = nullptr;
  p.sfa = ac.s; p.sfb0 = dyc.s;
  p.order = order;
  const bool pairs = g_wgrad_pairs.load(std::memory_order_relaxed) != 0;
  if (pairs) {
    p.m_tiles = (f + 255) / 256;
    e = launch_wgrad_pair<WGRAD2>(mA, mB0, p, st);
  } else {
    p.m_tiles = (f + BM - 1) / BM;
    e = launch<WGRAD2, kN_WGRAD>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st);
  }
  if (e != cudaSuccess) return e;
  p.order = nullptr;

  // dx_perm = dh . [Wg | Wu]^T (K = 2f): dh rows, w_gate / w_up rows
  if (wq) {
    wgr = w.wg_r;
    wur = w.wu_r;
  } else {
    if ((e = launch_mxfp8_quant_rows(wg, Ed, f, wgr.q, wgr.s, st, kScalesChunk)) != cudaSuccess) return e;
    if ((e = launch_mxfp8_quant_rows(wu, Ed, f, wur.q, wur.s, st, kScalesChunk)) != cudaSuccess) return e;
  }
  if (!map_2d(&mA, dhr.q, U8, 1, 2L * f, R, 128, BM) || !map_3d(&mB0, wgr.q, U8, 1, f, d, E, 128, kN_DGRAD1) ||
      !map_3d(&mB1, wur.q, U8, 1, f, d, E, 128, kN_DGRAD1))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + kN_DGRAD1 - 1) / kN_DGRAD1; p.out0 = dx_perm;
  p.sfa = dhr.s; p.sfb0 = wgr.s; p.sfb1 = wur.s;
  if ((e = launch<DGRAD1, kN_DGRAD1>(mA, mB0, mB1, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st)) != cudaSuccess)
    return e;

  // [dWg | dWu][e] = x_e^T dh_e (K = the expert's rows)
  if ((e = launch_mxfp8_quant_cols(x_perm, R, d, offsets, E, xc.q, xc.s, st, true)) != cudaSuccess) return e;
  if (!map_2d(&mA, xc.q, U8, 1, d, R, 128, 128) || !map_2d(&mB0, dhc.q, U8, 1, 2L * f, R, 128, 128))
    return cudaErrorInvalidValue;
  p.M = d; p.N = 2 * f; p.n_tiles = (2 * f + kN_WGRAD - 1) / kN_WGRAD;
  p.out0 = dwg; p.out1 = dwu; p.sfa = xc.s; p.sfb0 = dhc.s; p.sfb1 = nullptr;
  p.order = order;
  if (pairs) {
    p.m_tiles = (d + 255) / 256;
    return launch_wgrad_pair<WGRAD1>(mA, mB0, p, st);
  }
  p.m_tiles = (d + BM - 1) / BM;
  return launch<WGRAD1, kN_WGRAD>(mA, mB0, mB0, p, (long)E * p.m_tiles * p.n_tiles, st);
}

size_t mx_fwd_workspace(long R, int E, int d, int f) { return tc::mx::fwd_workspace(R, E, d, f); }

size_t mx_weights_bytes(int E, int d, int f) {  // the carve_weights layout
  using tc::mx::al;
  const size_t Ed = (size_t)E * d, Ef = (size_t)E * f;
  return 2 * (al(Ed * f) + al(Ed / 32 * f)) + (al(Ef * d) + al(Ef / 32 * d)) + (al(Ef * d) + al(Ef * d / 32)) +
         2 * (al(Ed * f) + al(Ed * f / 32));
}

cudaError_t mx_prepare_weights(const void* wg, const void* wu, const void* wd, int E, int d, int f, void* wq,
                               cudaStream_t st) {
  const tc::mx::MxWeights w = tc::mx::carve_weights(wq, E, d, f);
  const int Ed = E * d, Ef = E * f;
  cudaError_t e;
  // one read per weight: columns (blocks of 32 rows; K stages never cross
  // experts as d, f are multiples of 128) and rows (blocks of 32 columns)
  if ((e = launch_mxfp8_quant_dual(wg, Ed, f, w.wg_c.q, w.wg_c.s, w.wg_r.q, w.wg_r.s, st)) != cudaSuccess) return e;
  if ((e = launch_mxfp8_quant_dual(wu, Ed, f, w.wu_c.q, w.wu_c.s, w.wu_r.q, w.wu_r.s, st)) != cudaSuccess) return e;
  return launch_mxfp8_quant_dual(wd, Ef, d, w.wd_c.q, w.wd_c.s, w.wd_r.q, w.wd_r.s, st);
}
size_t mx_bwd_workspace(long R, int E, int d, int f) { return tc::mx::bwd_workspace(R, E, d, f); }
void set_mx_cta_pairs(int on) { tc::mx::g_wgrad_pairs.store(on ? 1 : 0, std::memory_order_relaxed); }

}  // namespace moe
