// gemm_tc.cu -- the six bf16 grouped expert GEMMs of the SwiGLU MoE layer and
// the router GEMM on the 5th-generation tensor cores ("Introducing Olmo-core
// 3", section "Scaling and optimizing MoE training": a grouped GEMM combines
// the many small per-expert computations into one efficient one).
//
// One persistent kernel per GEMM, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: 4-stage ring of (A 128x64, B 256x64) bf16 tiles,
//               128-byte swizzled, filled by cp.async.bulk.tensor (the router
//               GEMM, N = E: 6 stages of (A 128x64, B 128x64)).
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma M=128 N=256 K=16 into
//               one of two 256-column fp32 accumulators (512 TMEM columns),
//               so the epilogue of tile i overlaps the MMAs of tile i+1
//               (router: N=128 into two 128-column accumulators).
//   warps 2..9  epilogue: tcgen05.ld of the accumulator, fused SwiGLU (fwd or
//               bwd) math, bf16 (or fp32 router logits) stores with row/column
//               masks; two warps per TMEM lane quadrant, each half the columns.
// Tiles are enumerated on the device from the expert offsets (the host never
// sees the per-expert counts): forward/dgrad tiles cover 128 routed rows of
// one expert -- 256 for GEMM2 and the GEMM1 dgrad (tc_row256_kernel) -- and
// rows past the expert's end are computed and not stored;
// wgrad tiles cover a 128x256 block of one expert's weight gradient and
// reduce over that expert's rows (a ragged K; the rows past its end are
// zeroed in shared memory before the MMA; an expert with no rows gets zeros).
// Every wait is bounded; on a timeout the CTA sets the device error word,
// drains what it started and returns.
#include <atomic>

#include "kernels.h"
#include "tc_common.cuh"

namespace moe {
namespace tc {
namespace {

constexpr int BK = 64;  // bf16 elements per stage along K (128 bytes)
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * 64 * 2;  // one 64 (MN) x 64 (K) MN-major box
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int OUT_STG_BYTES = NUM_EPI_WARPS * STG_BYTES;  // epilogue staging, one buffer per warp

constexpr int MAX_STAGES = 6;  // the deepest ring of the kernels below

struct Smem {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Stages of the row-tile ring for a tile width TBN: 48 KB stages at the full
// width, 32 KB stages (and more of them) for the 128-column router tiles.
template <int TBN> constexpr int row_stages() { return TBN == BN ? STAGES : MAX_STAGES; }
template <int TBN> constexpr int row_stage_bytes() { return A_BYTES + TBN * BK * 2; }

// GATHER: the dispatch is fused into GEMM1 (FPROP1 only; p.src_row set).
// TBN: output columns per tile (256; 128 for the router logits, N = E).
template <int KIND, bool GATHER = false, int TBN = BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const Params p) {
  using Tr = Traits<KIND>;
  static_assert(!Tr::kragged, "weight gradients run in tc_wgrad_kernel");
  static_assert(TBN == BN || (KIND == ROUTER && TBN == 128), "narrow tiles for the router only");
  constexpr int NS = row_stages<TBN>();
  constexpr int STAGE_BYTES = row_stage_bytes<TBN>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + NS * STAGE_BYTES;  // epilogue staging
  Smem* sm = reinterpret_cast<Smem*>(out_stage + OUT_STG_BYTES);
  int* offs = reinterpret_cast<int*>(sm + 1);
  int* tstart = offs + (p.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  build_tile_table<KIND, NUM_THREADS>(p, offs, tstart);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
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
  const int total = tstart[p.E];
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ===================================================== TMA producer
    if constexpr (!GATHER) {
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB0);
        ptx::prefetch_tmap(&tmB1);
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
          const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
          for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
            const int s = it % NS;
            const uint32_t ph = (it / NS) & 1u;
            if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
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
              ptx::tma_load_2d(b, &tmB0, fb, k0, tl.n_idx * TBN);
            } else {  // DGRAD1
              ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
              if (k0 < p.f) ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
              else ptx::tma_load_3d(b, &tmB1, fb, k0 - p.f, tl.n_idx * BN, tl.e);
            }
          }
        }
        if (!ok) {
          // drain: wait (bounded) for loads already issued into stages the MMA will not consume
          for (int s = 0; s < NS; ++s) {
            const long long t0 = clock64();
            while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                   !ptx::mbar_try_wait(&sm->full[s], 1)) {
            }
          }
        }
      }
    } else {
      // GEMM1 with the dispatch fused: lane 0 waits for free stages and
      // issues the B loads; lane L gathers A rows 4L..4L+3 of the tile
      // straight from x (row src_row[r] / gk; rows past R read zeros) with
      // one TMA row gather per stage.
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB0);
        ptx::prefetch_tmap(&tmB1);
      }
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
        int tok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = tl.m0 + 4 * lane + i;
          tok[i] = r < p.R ? __ldg(p.src_row + r) / p.gk : p.T;
        }
        for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
          const int s = it % NS;
          const uint32_t ph = (it / NS) & 1u;
          bool free_stage = true;
          if (lane == 0) free_stage = wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, free_stage, 0)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + s * STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          uint64_t* fb = &sm->full[s];
          const int k0 = kb * BK;
          if (lane == 0) ptx::mbar_expect_tx(fb, STAGE_BYTES);
          __syncwarp();
          ptx::tma_gather4(a + lane * 512, &tmA, fb, k0, tok[0], tok[1], tok[2], tok[3]);
          if (lane == 0) {
            const int n0 = tl.n_idx * 128;
            ptx::tma_load_3d(b + 0 * BOX_BYTES, &tmB0, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + 1 * BOX_BYTES, &tmB0, fb, n0 + 64, k0, tl.e);
            ptx::tma_load_3d(b + 2 * BOX_BYTES, &tmB1, fb, n0, k0, tl.e);
            ptx::tma_load_3d(b + 3 * BOX_BYTES, &tmB1, fb, n0 + 64, k0, tl.e);
          }
        }
      }
      if (!ok && lane == 0) {
        for (int s = 0; s < NS; ++s) {
          const long long t0 = clock64();
          while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                 !ptx::mbar_try_wait(&sm->full[s], 1)) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ========================================================= MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, TBN, Tr::a_mn ? 1 : 0, Tr::b_mn ? 1 : 0);
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      if (tl.nkb == 0) continue;
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!wait_bar(&sm->tempty[buf], aph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * TBN);
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % NS;
        const uint32_t ph = (it / NS) & 1u;
        if (!wait_bar(&sm->full[s], ph, &sm->abort_flag, p.err)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * STAGE_BYTES;
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + A_BYTES;
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
    const int ew = warp - 2, q = warp & 3, half = ew >> 2;
    constexpr int NC = KIND == ROUTER ? TBN / 32 : epi_chunks<KIND>();
    uint8_t* stg = out_stage + ew * STG_BYTES;
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND, BK>(t, p, offs, tstart);
      if (tl.nkb == 0) continue;
      const int buf = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1u;
      if (!wait_bar(&sm->tfull[buf], aph, &sm->abort_flag, p.err)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + static_cast<uint32_t>(buf * TBN) + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (KIND == ROUTER)
        epilogue_router<TBN>(p, tl, tbase, q * 32 + lane, half * NC / 2, (half + 1) * NC / 2);
      else
        epilogue_tile_staged<KIND>(p, tl, tbase, q, lane, half * NC / 2, (half + 1) * NC / 2, stg);
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

template <int KIND, int TBN = BN>
size_t smem_bytes(int E) {
  return 1024 + row_stages<TBN>() * row_stage_bytes<TBN>() + OUT_STG_BYTES + sizeof(Smem) +
         2 * (E + 1) * sizeof(int) + 64;
}

template <int KIND, bool GATHER = false, int TBN = BN>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const Params& p,
                   long max_tiles, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  const size_t smem = smem_bytes<KIND, TBN>(p.E);
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<KIND, GATHER, TBN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
  MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, false), st)
      tc_gemm_kernel<KIND, GATHER, TBN><<<grid, NUM_THREADS, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// GEMM2 forward and the GEMM1 dgrad (plain bf16 epilogues) in 256-row tiles.
// The row-tile GEMMs are bound by the operand stream from L2, not by the
// tensor pipe: a 128x256 tile moves 48 KB per 4.2 MFLOP. Here two 128-row
// halves of A share each B stage (64 KB per 8.4 MFLOP, 1.5x less traffic per
// FLOP); both 256-column fp32 accumulators fill TMEM, so the epilogue drains
// them into registers as packed bf16 and releases TMEM before it stores,
// while the producer already streams the next tile. A tile whose second half
// holds no rows of its expert loads one A box and issues half the MMAs, so
// the padding per expert stays below 128 rows.
constexpr int RBM = 256;
constexpr int R_A_BYTES = RBM * BK * 2;       // two 128-row K-major boxes
constexpr int R_STAGE = R_A_BYTES + B_BYTES;  // 64 KB
constexpr int R_NS = 3;

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_row256_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                 const __grid_constant__ CUtensorMap tmB1, const Params p) {
  static_assert(KIND == FPROP2 || KIND == DGRAD1, "plain-store row kinds");
  using Tr = Traits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + R_NS * R_STAGE;
  Smem* sm = reinterpret_cast<Smem*>(out_stage + OUT_STG_BYTES);
  int* offs = reinterpret_cast<int*>(sm + 1);
  int* tstart = offs + (p.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  build_tile_table<KIND, NUM_THREADS, RBM>(p, offs, tstart);
  if (threadIdx.x == 0) {
    for (int s = 0; s < R_NS; ++s) {
      ptx::mbar_init(&sm->full[s], 1);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    ptx::mbar_init(&sm->tfull[0], 1);
    ptx::mbar_init(&sm->tempty[0], NUM_EPI_WARPS);
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
  const int total = tstart[p.E];
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
        const Tile tl = decode<KIND, BK, RBM>(t, p, offs, tstart);
        const bool two = tl.m0 + BM < tl.row_end;  // the second 128-row half holds rows
        for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
          const int s = it % R_NS;
          const uint32_t ph = (it / R_NS) & 1u;
          if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
          uint8_t* a = smem + s * R_STAGE;
          uint8_t* b = a + R_A_BYTES;
          uint64_t* fb = &sm->full[s];
          ptx::mbar_expect_tx(fb, (two ? R_A_BYTES : A_BYTES) + B_BYTES);
          const int k0 = kb * BK;
          ptx::tma_load_2d(a, &tmA, fb, k0, tl.m0);
          if (two) ptx::tma_load_2d(a + A_BYTES, &tmA, fb, k0, tl.m0 + BM);
          if (KIND == FPROP2) {
            const int n0 = tl.n_idx * BN;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_3d(b + j * BOX_BYTES, &tmB0, fb, n0 + 64 * j, k0, tl.e);
          } else {  // DGRAD1: w_gate rows for K < f, then w_up's
            if (k0 < p.f) ptx::tma_load_3d(b, &tmB0, fb, k0, tl.n_idx * BN, tl.e);
            else ptx::tma_load_3d(b, &tmB1, fb, k0 - p.f, tl.n_idx * BN, tl.e);
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < R_NS; ++s) {
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
      const Tile tl = decode<KIND, BK, RBM>(t, p, offs, tstart);
      const int halves = tl.m0 + BM < tl.row_end ? 2 : 1;
      if (!wait_bar(&sm->tempty[0], (acc_it & 1u) ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      for (int kb = 0; kb < tl.nkb; ++kb, ++it) {
        const int s = it % R_NS;
        const uint32_t ph = (it / R_NS) & 1u;
        if (!wait_bar(&sm->full[s], ph, &sm->abort_flag, p.err)) { ok = false; break; }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(smem + s * R_STAGE), b_addr = a_addr + R_A_BYTES;
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t bd = Tr::b_mn ? ptx::smem_desc_sw128(b_addr + ks * 2048, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            for (int h = 0; h < halves; ++h) {
              const uint64_t ad = ptx::smem_desc_sw128(a_addr + h * A_BYTES + ks * 32, 16, 1024);
              ptx::mma_f16(tmem + h * BN, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(&sm->empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(&sm->tfull[0]);
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
    // warps 2..5 take rows 0..127 of the tile (accumulator 0), warps 6..9 rows
    // 128..255 (accumulator 1); lane = row. Each thread moves its 256-column
    // row into registers as packed bf16, TMEM is handed back, then the rows go
    // out 32 columns at a time through the warp's staging buffer.
    const int ew = warp - 2, q = warp & 3, mh = ew >> 2;
    uint8_t* stg = out_stage + ew * STG_BYTES;
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode<KIND, BK, RBM>(t, p, offs, tstart);
      const bool mine = mh == 0 || tl.m0 + BM < tl.row_end;
      if (!wait_bar(&sm->tfull[0], acc_it & 1u, &sm->abort_flag, p.err)) break;
      ptx::tc_fence_after();
      uint32_t hold[BN / 32][16];
      if (mine) {
        const uint32_t tbase = tmem + static_cast<uint32_t>(mh * BN) + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {  // 16 columns at a time keeps the drain within the register budget
          uint32_t r[16];
          ptx::tmem_ld16(tbase + c * 16, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            hold[c >> 1][(c & 1) * 8 + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm->tempty[0]);
      ++acc_it;
      if (!mine) continue;
      const int wrow = tl.m0 + mh * BM + q * 32;
      const int nrows = max(0, min(32, tl.row_end - wrow));
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out0) + (size_t)wrow * p.N + tl.n_idx * BN;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        if (tl.n_idx * BN + c * 32 < p.N) warp_store_rows(stg, hold[c], out + c * 32, p.N, nrows, lane);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int KIND>
cudaError_t launch_row256(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const Params& p,
                          int R, cudaStream_t st) {
  const long max_tiles = ((long)(R + RBM - 1) / RBM + p.E) * p.n_tiles;
  if (R <= 0 || max_tiles <= 0) return cudaSuccess;
  const size_t smem = 1024 + R_NS * R_STAGE + OUT_STG_BYTES + sizeof(Smem) + 2 * (p.E + 1) * sizeof(int) + 64;
  cudaError_t e = cudaFuncSetAttribute(tc_row256_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(max_tiles < sm_count() ? max_tiles : sm_count());
  MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, false), st) tc_row256_kernel<KIND><<<grid, NUM_THREADS, smem, st>>>(a, b0, b1, p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Weight gradients: dW_e = X_e^T Y_e over the rows of expert e. These tiles
// leave the tensor cores idle: they are bound by the operand traffic from L2,
// so they use 256x256 output tiles (two 128-row halves of M sharing one B
// tile; both 256-column fp32 accumulators fill TMEM) to cut that traffic per
// FLOP by 1.5x against 128x256 tiles. Single-buffered accumulator, drained
// into registers at once so the stores overlap the next tile's MMAs; the
// producer keeps loading the next tile's stages meanwhile.
constexpr int WBM = 256;
constexpr int W_A_BYTES = WBM * BK * 2;  // 4 boxes of 64 (M) x 64 (K rows)
constexpr int W_B_BYTES = BN * BK * 2;   // 4 boxes of 64 (N) x 64 (K rows)
constexpr int W_STAGE = W_A_BYTES + W_B_BYTES;
constexpr int W_NS = 3;
constexpr int W_STG = 32 * 128;  // per epilogue warp: 32 rows x 64 bf16, 16-byte granules XOR-swizzled by row

// GATHER: the dispatch is fused into the GEMM1 wgrad (WGRAD1 only; p.src_row set).
template <int KIND, bool GATHER = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
  static_assert(Traits<KIND>::kragged, "weight-gradient kinds only");
  static_assert(!GATHER || KIND == WGRAD1, "the row gather feeds the GEMM1 wgrad only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem* sm = reinterpret_cast<Smem*>(smem + W_NS * W_STAGE + NUM_EPI_WARPS * W_STG);
  const int* __restrict__ offs = p.offsets;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < W_NS; ++s) {
      ptx::mbar_init(&sm->full[s], 1);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    ptx::mbar_init(&sm->tfull[0], 1);
    ptx::mbar_init(&sm->tempty[0], NUM_EPI_WARPS);
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
  const int per = p.m_tiles * p.n_tiles;
  const int total = p.E * per;
  const uint32_t tmem = sm->tmem_base;
  auto decode_w = [&](int t, int& e, int& m0, int& n0, int& r0, int& r1, int& nkb) {
    e = p.order ? __ldg(p.order + t / per) : t / per;
    const int local = t % per;
    m0 = (local / p.n_tiles) * WBM;
    n0 = (local % p.n_tiles) * BN;
    r0 = __ldg(offs + e);
    r1 = __ldg(offs + e + 1);
    nkb = (r1 - r0 + BK - 1) / BK;
  };

  if (warp == 0) {
    // ===================================================== TMA producer
    if constexpr (!GATHER) {
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        uint32_t it = 0;
        bool ok = true;
        for (int r = 0, t = sched_tile<true>(0); t < total && ok; t = sched_tile<true>(++r)) {
          int e, m0, n0, r0, r1, nkb;
          decode_w(t, e, m0, n0, r0, r1, nkb);
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const int s = it % W_NS;
            const uint32_t ph = (it / W_NS) & 1u;
            if (!wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
            uint8_t* a = smem + s * W_STAGE;
            uint8_t* b = a + W_A_BYTES;
            uint64_t* fb = &sm->full[s];
            ptx::mbar_expect_tx(fb, W_STAGE);
            const int row = r0 + kb * BK;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_2d(a + j * BOX_BYTES, &tmA, fb, m0 + 64 * j, row);
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_2d(b + j * BOX_BYTES, &tmB, fb, n0 + 64 * j, row);
          }
        }
        if (!ok) {
          for (int s = 0; s < W_NS; ++s) {
            const long long t0 = clock64();
            while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                   !ptx::mbar_try_wait(&sm->full[s], 1)) {
            }
          }
        }
      }
    } else {
      // GEMM1 wgrad with the dispatch fused: lane 0 waits for free stages and
      // issues the B loads; lane L gathers K rows 4(L%16)..+3 of the stage for
      // A boxes 2(L/16) and 2(L/16)+1 straight from x with TMA row gathers,
      // the next stage's token indices loading while this stage waits. Rows
      // past the expert's end (and columns past d) read zeros.
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
      }
      const int grp = lane & 15, jb = (lane >> 4) * 2;
      uint32_t it = 0;
      bool ok = true;
      for (int r = 0, t = sched_tile<true>(0); t < total && ok; t = sched_tile<true>(++r)) {
        int e, m0, n0, r0, r1, nkb;
        decode_w(t, e, m0, n0, r0, r1, nkb);
        auto tokens = [&](int kb, int (&tk)[4]) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = r0 + kb * BK + 4 * grp + i;
            tk[i] = r < r1 ? __ldg(p.src_row + r) / p.gk : p.T;
          }
        };
        int nxt[4] = {0, 0, 0, 0};
        if (nkb > 0) tokens(0, nxt);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int cur[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
          if (kb + 1 < nkb) tokens(kb + 1, nxt);
          const int s = it % W_NS;
          const uint32_t ph = (it / W_NS) & 1u;
          bool free_stage = true;
          if (lane == 0) free_stage = wait_bar(&sm->empty[s], ph ^ 1u, &sm->abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, free_stage, 0)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + s * W_STAGE;
          uint8_t* b = a + W_A_BYTES;
          uint64_t* fb = &sm->full[s];
          if (lane == 0) ptx::mbar_expect_tx(fb, W_STAGE);
          __syncwarp();
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
            ptx::tma_gather4(a + (jb + jj) * BOX_BYTES + grp * 512, &tmA, fb, m0 + 64 * (jb + jj), cur[0], cur[1],
                             cur[2], cur[3]);
          if (lane == 0) {
            const int row = r0 + kb * BK;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_2d(b + j * BOX_BYTES, &tmB, fb, n0 + 64 * j, row);
          }
        }
      }
      if (!ok && lane == 0) {
        for (int s = 0; s < W_NS; ++s) {
          const long long t0 = clock64();
          while (clock64() - t0 < kWaitLimitCycles / 8 && !ptx::mbar_try_wait(&sm->full[s], 0) &&
                 !ptx::mbar_try_wait(&sm->full[s], 1)) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ========================================================= MMA issuer
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, 1, 1);
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int r = 0, t = sched_tile<true>(0); t < total && ok; t = sched_tile<true>(++r)) {
      int e, m0, n0, r0, r1, nkb;
      decode_w(t, e, m0, n0, r0, r1, nkb);
      if (nkb == 0) continue;
      if (!wait_bar(&sm->tempty[0], (acc_it & 1u) ^ 1u, &sm->abort_flag, p.err)) { ok = false; break; }
      ptx::tc_fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % W_NS;
        const uint32_t ph = (it / W_NS) & 1u;
        if (!wait_bar(&sm->full[s], ph, &sm->abort_flag, p.err)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * W_STAGE;
        int nks = BK / 16;
        const int valid = r1 - (r0 + kb * BK);
        if (valid < BK) {
          // rows past the expert's end belong to the next expert: skip K steps made
          // only of them and zero the rest of the last partial step in the four A boxes
          nks = (valid + 15) / 16;
          const int nrow = nks * 16 - valid, per_box = nrow * 8;
          for (int i = lane; i < 4 * per_box; i += 32) {
            const int box = i / per_box, rem = i % per_box;
            const int rr = valid + rem / 8, chunk = rem % 8;
            *reinterpret_cast<uint4*>(a + box * BOX_BYTES + rr * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
          }
          if (nrow > 0) ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + W_A_BYTES;
          for (int ks = 0; ks < nks; ++ks) {
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 2048, BOX_BYTES, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t ad = ptx::smem_desc_sw128(a_addr + h * 2 * BOX_BYTES + ks * 2048, BOX_BYTES, 1024);
              ptx::mma_f16(tmem + h * BN, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(&sm->empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(&sm->tfull[0]);
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
    // warps 2..5 take M half 0, warps 6..9 M half 1; lanes are rows. Each
    // thread first moves its whole 256-column row of the accumulator into
    // registers as packed bf16 pairs (128 words) and hands TMEM back, so the
    // next tile's MMAs start while this tile's stores go out.
    const int ew = warp - 2, q = warp & 3, mh = ew >> 2;
    uint32_t acc_it = 0;
    for (int r = 0, t = sched_tile<true>(0); t < total; t = sched_tile<true>(++r)) {
      int e, m0, n0, r0, r1, nkb;
      decode_w(t, e, m0, n0, r0, r1, nkb);
      uint32_t hold[BN / 2];
      if (nkb > 0) {
        if (!wait_bar(&sm->tfull[0], acc_it & 1u, &sm->abort_flag, p.err)) break;
        ptx::tc_fence_after();
        const uint32_t tbase = tmem + static_cast<uint32_t>(mh * BN) + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          uint32_t r[16];
          ptx::tmem_ld16(tbase + c * 16, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            hold[c * 8 + i] = *reinterpret_cast<uint32_t*>(&h2);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm->tempty[0]);
        ++acc_it;
      } else {
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) hold[i] = 0u;  // expert with no rows: dW_e = 0
      }
      // Stores go out 64 columns at a time through this warp's staging
      // buffer: each lane writes its row, then each instruction stores four
      // rows' 128-byte segments (8 lanes per row), so every request covers
      // whole lines.
      const int mb = m0 + mh * 128 + q * 32;
      uint8_t* stg = smem + W_NS * W_STAGE + ew * W_STG;
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        const int n = n0 + c * 64;
        if (n >= p.N) break;
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((g ^ (lane & 7)) << 4)) =
              make_uint4(hold[c * 32 + 4 * g], hold[c * 32 + 4 * g + 1], hold[c * 32 + 4 * g + 2],
                         hold[c * 32 + 4 * g + 3]);
        __syncwarp();
        const int g = lane & 7;
        __nv_bfloat16* base;
        size_t ld;
        if (KIND == WGRAD2) {
          base = static_cast<__nv_bfloat16*>(p.out0) + ((size_t)e * p.M + mb) * p.N + n;
          ld = p.N;
        } else {
          base = n < p.f ? static_cast<__nv_bfloat16*>(p.out0) + ((size_t)e * p.d + mb) * p.f + n
                         : static_cast<__nv_bfloat16*>(p.out1) + ((size_t)e * p.d + mb) * p.f + (n - p.f);
          ld = p.f;
        }
        base += 8 * g;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3);
          const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 128 + ((g ^ (r & 7)) << 4));
          if (mb + r < p.M) *reinterpret_cast<uint4*>(base + r * ld) = v;
        }
        __syncwarp();
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

template <int KIND, bool GATHER = false>
cudaError_t launch_wgrad(const CUtensorMap& a, const CUtensorMap& b, const Params& p, cudaStream_t st) {
  const long tiles = (long)p.E * p.m_tiles * p.n_tiles;
  if (tiles <= 0) return cudaSuccess;
  const size_t smem = 1024 + W_NS * W_STAGE + NUM_EPI_WARPS * W_STG + sizeof(Smem) + 64;
  cudaError_t e = cudaFuncSetAttribute(tc_wgrad_kernel<KIND, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, false), st) tc_wgrad_kernel<KIND, GATHER><<<grid, NUM_THREADS, smem, st>>>(a, b, p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Weight gradients on CTA pairs (2-CTA clusters, tcgen05.mma.cta_group::2),
// selected with moe_use_cta_pairs(1). A pair computes a 256x256 block of one
// expert's gradient: each CTA loads its own 128 rows of M (A boxes) and its own
// 128 of the N columns (B boxes), 64 KB per 128-row K stage, and the even CTA
// issues one M=256 N=256 MMA per K step that reads both CTAs' shared memory.
// Each CTA's TMEM receives its 128 rows x 256 columns, so the 512 columns hold
// two accumulators: the next tile's MMAs run while the epilogue drains the
// previous one. Operand bytes per FLOP are those of the single-CTA 256x256
// tile, whose accumulators fill TMEM instead.
//   warp 0      both CTAs: TMA producer of its own half of each stage.
//   warp 1      even CTA: MMA issuer; it commits each stage's release to both
//               CTAs' `empty` barriers and each finished accumulator to both
//               CTAs' `tfull` barriers.
//               odd CTA: relay; waits for its half of a stage to land, zeroes
//               the rows past the expert's end in its A boxes, then arrives on
//               the even CTA's `full` barrier (two arrivals per phase there:
//               its producer's and the relay's).
//   warps 2..9  both CTAs: epilogue of its own 128 rows; they arrive on the even
//               CTA's `tempty` barrier when the accumulator has been read.
// All 32 lanes of a warp poll each barrier: a warp whose other lanes sit at a
// warp barrier while one lane polls resumes late after the phase completes.
// Every wait is bounded; a CTA that gives up raises both CTAs' abort flags.
constexpr int PBK = 128;              // K rows per stage
constexpr int P_BOX = 64 * PBK * 2;   // one 64 (M or N) x 128 (K rows) box
constexpr int P_A_BYTES = 2 * P_BOX;  // this CTA's 128 rows of M
constexpr int P_STAGE = 4 * P_BOX;    // + its 128 columns of N
constexpr int P_NS = 3;

struct PairSmem {
  uint64_t full[P_NS];
  uint64_t empty[P_NS];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Bounded wait on a local mbarrier whose arrivals may come from the other CTA
// of the pair. On expiry it sets the error word and both CTAs' abort flags.
__device__ __forceinline__ bool wait_pair(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t peer_abort,
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
tc_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Params p) {
  static_assert(Traits<KIND>::kragged, "weight-gradient kinds only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairSmem* sm = reinterpret_cast<PairSmem*>(smem + P_NS * P_STAGE + NUM_EPI_WARPS * W_STG);
  const int* __restrict__ offs = p.offsets;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank(), peer = rank ^ 1u;
  const int cid = static_cast<int>(ptx::cluster_id_x()), ncl = static_cast<int>(ptx::n_clusters_x());
  auto in_cta = [&](const void* x, uint32_t r) { return ptx::mapa(ptx::smem_u32(x), r); };
  const uint32_t peer_abort = in_cta(&sm->abort_flag, peer);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_NS; ++s) {
      ptx::mbar_init(&sm->full[s], rank == 0 ? 2 : 1);
      ptx::mbar_init(&sm->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm->tfull[b], 1);
      ptx::mbar_init(&sm->tempty[b], 2 * NUM_EPI_WARPS);
    }
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

  const int per = p.m_tiles * p.n_tiles;
  const int total = p.E * per;
  // the pair's r-th tile: experts largest first, a snake over the pairs
  auto tile_of = [&](int r) { return r * ncl + ((r & 1) ? ncl - 1 - cid : cid); };
  struct WT {
    int e, m0, n0, r0, r1, nkb;
  };
  auto decode_w = [&](int t) {
    WT w;
    w.e = p.order ? __ldg(p.order + t / per) : t / per;
    const int local = t % per;
    w.m0 = (local / p.n_tiles) * WBM;
    w.n0 = (local % p.n_tiles) * BN;
    w.r0 = __ldg(offs + w.e);
    w.r1 = __ldg(offs + w.e + 1);
    w.nkb = (w.r1 - w.r0 + PBK - 1) / PBK;
    return w;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    const bool ok = wait_pair(bar, parity, &sm->abort_flag, peer_abort, p.err);
    return __all_sync(0xffffffffu, ok) != 0;
  };
  // rows past the expert's end belong to the next expert: zero them in this
  // CTA's two A boxes of the stage (whole K steps of them are skipped)
  auto zero_tail = [&](uint8_t* a, int valid) {
    const int nks = (valid + 15) / 16;
    const int nrow = nks * 16 - valid, per_box = nrow * 8;
    for (int i = lane; i < 2 * per_box; i += 32) {
      const int box = i / per_box, rem = i % per_box;
      *reinterpret_cast<uint4*>(a + box * P_BOX + (valid + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    if (nrow > 0) ptx::fence_proxy_async_smem();
    return nks;
  };

  if (warp == 0) {
    // ===================================================== TMA producer
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
          const int s = it % P_NS;
          if (!warp_wait(&sm->empty[s], ((it / P_NS) & 1u) ^ 1u)) { ok = false; break; }
          if (lane == 0) {
            uint8_t* a = smem + s * P_STAGE;
            uint8_t* b = a + P_A_BYTES;
            uint64_t* fb = &sm->full[s];
            ptx::mbar_expect_tx(fb, P_STAGE);
            const int row = w.r0 + kb * PBK;
#pragma unroll
            for (int j = 0; j < 2; ++j) ptx::tma_load_2d(a + j * P_BOX, &tmA, fb, w.m0 + 128 * rank + 64 * j, row);
#pragma unroll
            for (int j = 0; j < 2; ++j) ptx::tma_load_2d(b + j * P_BOX, &tmB, fb, w.n0 + 128 * rank + 64 * j, row);
          }
          __syncwarp();
        }
      }
      // the even CTA's commits release these stages: wait for the last ones
      // to land before the CTA may finish
      for (int k = 0; k < P_NS && ok; ++k, ++it) ok = warp_wait(&sm->empty[it % P_NS], ((it / P_NS) & 1u) ^ 1u);
      if (!ok && lane == 0) {
        // let loads in flight finish (bounded) before the CTA leaves
        for (int s = 0; s < P_NS; ++s) {
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
        const int s = it % P_NS;
        if (!warp_wait(&sm->full[s], (it / P_NS) & 1u)) { ok = false; break; }
        const int valid = w.r1 - (w.r0 + kb * PBK);
        if (valid < PBK) zero_tail(smem + s * P_STAGE, valid);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(leader_full0 + 8u * s);
      }
    }
  } else if (warp == 1) {
    // ============================================ MMA issuer (even CTA)
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, BN, 1, 1);
    const uint32_t peer_empty0 = in_cta(&sm->empty[0], 1), peer_tfull0 = in_cta(&sm->tfull[0], 1);
    uint32_t it = 0, acc_it = 0;
    bool ok = run;
    for (int r = 0, t = tile_of(0); t < total && ok; t = tile_of(++r)) {
      const WT w = decode_w(t);
      if (w.nkb == 0) continue;
      const uint32_t buf = acc_it & 1u;
      if (!warp_wait(&sm->tempty[buf], ((acc_it >> 1) & 1u) ^ 1u)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + buf * BN;
      for (int kb = 0; kb < w.nkb; ++kb, ++it) {
        const int s = it % P_NS;
        if (!warp_wait(&sm->full[s], (it / P_NS) & 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        uint8_t* a = smem + s * P_STAGE;
        const int valid = w.r1 - (w.r0 + kb * PBK);
        const int nks = valid < PBK ? zero_tail(a, valid) : PBK / 16;
        __syncwarp();
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_u32(a), b_addr = a_addr + P_A_BYTES;
          for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + ks * 2048, P_BOX, 1024);
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 2048, P_BOX, 1024);
            ptx::mma_f16_pair(d_tmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit_pair(ptx::smem_u32(&sm->empty[s]));
          ptx::mma_commit_pair(peer_empty0 + 8u * s);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        ptx::mma_commit_pair(ptx::smem_u32(&sm->tfull[buf]));
        ptx::mma_commit_pair(peer_tfull0 + 8u * buf);
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
    // warp (q, ch): TMEM lanes 32q..32q+31 (this CTA's rows), columns
    // 128ch..128ch+127 of the accumulator, read and stored 64 at a time.
    const int ew = warp - 2, q = warp & 3, ch = ew >> 2;
    const uint32_t leader_tempty0 = in_cta(&sm->tempty[0], 0);
    uint8_t* stg = smem + P_NS * P_STAGE + ew * W_STG;
    uint32_t acc_it = 0;
    for (int r = 0, t = tile_of(0); t < total && run; t = tile_of(++r)) {
      const WT w = decode_w(t);
      const uint32_t buf = acc_it & 1u;
      if (w.nkb > 0) {
        if (!warp_wait(&sm->tfull[buf], (acc_it >> 1) & 1u)) break;
        ptx::tc_fence_after();
      }
      const uint32_t tbase = tmem + buf * BN + static_cast<uint32_t>(ch * 128) + (static_cast<uint32_t>(q * 32) << 16);
      const int mb = w.m0 + 128 * static_cast<int>(rank) + 32 * q;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        if (w.nkb > 0) {
          uint32_t v0[32], v1[32];
          ptx::tmem_ld32(tbase + c * 64, v0);
          ptx::tmem_ld32(tbase + c * 64 + 32, v1);
          ptx::tmem_wait_ld();
          if (c == 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(leader_tempty0 + 8u * buf);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
            __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            v[i] = *reinterpret_cast<uint32_t*>(&h0);
            v[16 + i] = *reinterpret_cast<uint32_t*>(&h1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;  // expert with no rows: dW_e = 0
        }
        const int n = w.n0 + ch * 128 + c * 64;
        if (n >= p.N) continue;
        // each lane writes its row's 128 bytes; each instruction then stores
        // four rows' 128-byte segments (8 lanes per row)
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((g ^ (lane & 7)) << 4)) =
              make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        __syncwarp();
        const int g = lane & 7;
        __nv_bfloat16* base;
        size_t ld;
        if (KIND == WGRAD2) {
          base = static_cast<__nv_bfloat16*>(p.out0) + ((size_t)w.e * p.M + mb) * p.N + n;
          ld = p.N;
        } else {
          base = n < p.f ? static_cast<__nv_bfloat16*>(p.out0) + ((size_t)w.e * p.d + mb) * p.f + n
                         : static_cast<__nv_bfloat16*>(p.out1) + ((size_t)w.e * p.d + mb) * p.f + (n - p.f);
          ld = p.f;
        }
        base += 8 * g;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + (lane >> 3);
          const uint4 u = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((g ^ (rr & 7)) << 4));
          if (mb + rr < p.M) *reinterpret_cast<uint4*>(base + rr * ld) = u;
        }
        __syncwarp();
      }
      if (w.nkb > 0) ++acc_it;
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
  const size_t smem = 1024 + P_NS * P_STAGE + NUM_EPI_WARPS * W_STG + sizeof(PairSmem) + 64;
  cudaError_t e = cudaFuncSetAttribute(tc_wgrad_pair_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    e = cudaOccupancyMaxActiveClusters(&max_pairs, tc_wgrad_pair_kernel<KIND>, &cfg);
    if (e != cudaSuccess) return e;
    if (max_pairs <= 0) return cudaErrorLaunchOutOfResources;
    cached_pairs.store(max_pairs, std::memory_order_relaxed);
  }
  const long pairs = tiles < max_pairs ? tiles : max_pairs;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  return MOE_COUNTED_AS(::moe::gemm_kind_name(KIND, false), st)
      cudaLaunchKernelEx(&cfg, tc_wgrad_pair_kernel<KIND>, a, b, p);
}

constexpr CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

// Experts ordered by row count, largest first, ties by index (order[i] = the
// expert of rank i): the walk order of the weight-gradient tiles, whose cost
// is their expert's row count. One block; E <= 1024.
__global__ void __launch_bounds__(1024) expert_order_kernel(const int32_t* __restrict__ offsets, int E,
                                                            int32_t* __restrict__ order) {
  __shared__ int cnt[1024];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = offsets[e + 1] - offsets[e];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = cnt[e];
    int rank = 0;
    for (int j = 0; j < E; ++j) {
      const int cj = cnt[j];
      rank += (cj > c) | ((cj == c) & (j < e));
    }
    order[rank] = e;
  }
}

}  // namespace

// ------------------------------------------------------------ shared host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
            uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, rows > 0 ? rows : 1};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
            uint64_t rows, uint64_t E, uint32_t box_inner, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, E};
  const cuuint64_t strides[2] = {inner * esize, inner * rows * esize};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::atomic<int> cached{0};  // host threads may race to fill it with the same value
  int n = cached.load(std::memory_order_relaxed);
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached.store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace tc

using namespace tc;

// Weight-gradient kernel choice (moe_use_cta_pairs): single-CTA 256x256 tiles
// by default, CTA pairs on request.
static std::atomic<int> g_cta_pairs{0};

template <int KIND>
cudaError_t launch_wgrad_any(const CUtensorMap& a, const CUtensorMap& b, const Params& p, cudaStream_t st) {
  return g_cta_pairs.load(std::memory_order_relaxed) ? launch_wgrad_pair<KIND>(a, b, p, st)
                                                     : launch_wgrad<KIND>(a, b, p, st);
}

void set_cta_pairs(int on) { g_cta_pairs.store(on ? 1 : 0, std::memory_order_relaxed); }

cudaError_t launch_expert_order(const int32_t* offsets, int E, int32_t* order, cudaStream_t st) {
  if (E <= 0 || E > 1024) return cudaErrorInvalidValue;
  MOE_COUNTED_AS("expert_order", st) expert_order_kernel<<<1, 1024, 0, st>>>(offsets, E, order);
  return cudaGetLastError();
}

cudaError_t tc_mlp_fwd(const void* x_perm, const void* wg, const void* wu, const void* wd,
                       const int32_t* offsets, int R, int E, int d, int f, void* h, void* a, void* y,
                       cudaStream_t st, const int32_t* src_row, int gk, int T) {
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  // GEMM1 + SwiGLU: tiles of 128 f-columns (gate 128 | up 128 in one N=256 MMA). With src_row,
  // x_perm is x [T][d] and the A rows are gathered one box row at a time.
  const bool ok_a = src_row ? map_2d(&mA, x_perm, BF, 2, d, T, 64, 1) : map_2d(&mA, x_perm, BF, 2, d, R, 64, BM);
  if (!ok_a || !map_3d(&mB0, wg, BF, 2, f, d, E, 64, 64) || !map_3d(&mB1, wu, BF, 2, f, d, E, 64, 64))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + 127) / 128; p.out0 = h; p.out1 = a;
  p.src_row = src_row; p.gk = gk; p.T = T;
  const long fp1_tiles = ((long)(R + BM - 1) / BM + E) * p.n_tiles;
  cudaError_t e = src_row ? launch<FPROP1, true>(mA, mB0, mB1, p, fp1_tiles, st)
                          : launch<FPROP1>(mA, mB0, mB1, p, fp1_tiles, st);
  if (e != cudaSuccess) return e;
  p.src_row = nullptr;
  // GEMM2
  if (!map_2d(&mA, a, BF, 2, f, R, 64, BM) || !map_3d(&mB0, wd, BF, 2, d, f, E, 64, 64))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = y; p.out1 = nullptr;
  return launch_row256<FPROP2>(mA, mB0, mB0, p, R, st);
}

cudaError_t tc_mlp_bwd(const void* dy_perm, const void* x_perm, const void* h, const void* a, const void* wg,
                       const void* wu, const void* wd, const int32_t* offsets, int R, int E, int d, int f,
                       void* dx_perm, void* dwg, void* dwu, void* dwd, void* dh, cudaStream_t st,
                       const int32_t* src_row, int gk, int T) {
  CUtensorMap mA, mB0, mB1;
  Params p{};
  p.offsets = offsets; p.E = E; p.R = R; p.d = d; p.f = f; p.err = device_error_word();
  cudaError_t e;
  // the weight gradients walk their experts largest first (order table after dh)
  int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(dh) + (((size_t)R * 2 * f * 2 + 255) & ~size_t(255)));
  if ((e = launch_expert_order(offsets, E, order, st)) != cudaSuccess) return e;
  // dA = dy . Wd^T with the SwiGLU backward fused: writes dh
  if (!map_2d(&mA, dy_perm, BF, 2, d, R, 64, BM) || !map_3d(&mB0, wd, BF, 2, d, f, E, 64, BN))
    return cudaErrorInvalidValue;
  p.N = f; p.n_tiles = (f + BN - 1) / BN; p.out0 = dh; p.aux = h;
  e = launch<DGRAD2>(mA, mB0, mB0, p, ((long)(R + BM - 1) / BM + E) * p.n_tiles, st);
  if (e != cudaSuccess) return e;
  // dWd[e] = A_e^T dy_e
  // K rows per stage (TMA box height) of the weight-gradient kernel in use
  const int wbk = g_cta_pairs.load(std::memory_order_relaxed) ? PBK : BK;
  if (!map_2d(&mA, a, BF, 2, f, R, 64, wbk) || !map_2d(&mB0, dy_perm, BF, 2, d, R, 64, wbk))
    return cudaErrorInvalidValue;
  p.M = f; p.N = d; p.m_tiles = (f + WBM - 1) / WBM; p.n_tiles = (d + BN - 1) / BN; p.out0 = dwd;
  p.order = order;
  e = launch_wgrad_any<WGRAD2>(mA, mB0, p, st);
  p.order = nullptr;
  if (e != cudaSuccess) return e;
  // dx_perm = dh_g . Wg^T + dh_u . Wu^T
  if (!map_2d(&mA, dh, BF, 2, 2L * f, R, 64, BM) || !map_3d(&mB0, wg, BF, 2, f, d, E, 64, BN) ||
      !map_3d(&mB1, wu, BF, 2, f, d, E, 64, BN))
    return cudaErrorInvalidValue;
  p.N = d; p.n_tiles = (d + BN - 1) / BN; p.out0 = dx_perm; p.aux = nullptr;
  e = launch_row256<DGRAD1>(mA, mB0, mB1, p, R, st);
  if (e != cudaSuccess) return e;
  // [dWg | dWu][e] = x_perm_e^T dh_e (with src_row: K rows gathered from x [T][d])
  const int gbk = src_row ? 64 : wbk;
  const bool ok_a = src_row ? map_2d(&mA, x_perm, BF, 2, d, T, 64, 1) : map_2d(&mA, x_perm, BF, 2, d, R, 64, gbk);
  if (!ok_a || !map_2d(&mB0, dh, BF, 2, 2L * f, R, 64, gbk)) return cudaErrorInvalidValue;
  p.M = d; p.N = 2 * f; p.m_tiles = (d + WBM - 1) / WBM; p.n_tiles = (2 * f + BN - 1) / BN;
  p.out0 = dwg; p.out1 = dwu;
  p.src_row = src_row; p.gk = gk; p.T = T;
  p.order = order;
  if (src_row) return launch_wgrad<WGRAD1, true>(mA, mB0, p, st);
  return launch_wgrad_any<WGRAD1>(mA, mB0, p, st);
}

cudaError_t tc_router_logits(const void* x, const void* w_r, const float* bias, int T, int d, int E,
                             float* logits, cudaStream_t st) {
  CUtensorMap mA, mB;
  Params p{};
  p.offsets = nullptr; p.bias = bias; p.E = 1; p.R = T; p.d = d; p.f = 0; p.err = device_error_word();
  constexpr int RBN = 128;  // logits tile width: E is a multiple of 32, most often 128 or less
  if (!map_2d(&mA, x, BF, 2, d, T, 64, BM) || !map_2d(&mB, w_r, BF, 2, d, E, 64, RBN)) return cudaErrorInvalidValue;
  p.N = E; p.n_tiles = (E + RBN - 1) / RBN; p.out0 = logits;
  return launch<ROUTER, false, RBN>(mA, mB, mB, p, (long)((T + BM - 1) / BM) * p.n_tiles, st);
}

}  // namespace moe
