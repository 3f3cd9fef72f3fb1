// route.cu -- top-k gate selection, per-expert counts, offsets and row
// placement, all on the device ("Introducing Olmo-core 3", section "Scaling
// and optimizing MoE training": routing metadata stays on the GPU so the host
// never waits for a copy back; routed rows go straight into each expert's
// contiguous input buffer).
//
// Pipeline (all deterministic, no dependence on atomic ordering):
//   1. topk_hist: one CTA per chunk of kTokensPerChunk tokens, one warp per
//      token: warp-wide k-round argmax over 64-bit keys (ordered logit,
//      inverted index), gates as a softmax over the selected logits, and the
//      chunk's expert histogram written to hist[chunk][e].
//   2. chunk_scan: one CTA per expert; exclusive scan of hist[.][e] over the
//      chunks (in place) and the expert's total count.
//   3. offsets: exclusive scan of the counts.
//   4. rank: one warp per chunk again; pairs p = t*k + j in order, groups of
//      32 lanes, __match_any_sync finds lanes routed to the same expert and
//      each pair's row is offsets[e] + chunk prefix + rank among earlier pairs.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kWarps = 8;  // warps per CTA in the per-chunk kernels

// Map a float to a uint32 whose unsigned order is the float order; -0 and +0
// map to the same key and NaN maps below every number.
__device__ __forceinline__ uint32_t ordered_key(float v) {
  if (v != v) return 0u;
  uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  uint32_t b = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(b);
}

// One CTA per chunk, one warp per token (kWarps == kTokensPerChunk). NV:
// logits per lane (E <= 32 NV). The chunk's expert histogram is summed with
// shared-memory integer atomics (exact in any order), then written out.
template <int NV>
__global__ void __launch_bounds__(kWarps * 32)
topk_hist_kernel(const float* __restrict__ logits, int T, int E, int k, int nchunks,
                 int32_t* __restrict__ topk_idx, float* __restrict__ gates,
                 int32_t* __restrict__ hist) {
  static_assert(kWarps == kTokensPerChunk, "one warp per token of the chunk");
  extern __shared__ int32_t cnt[];  // [E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  const int t = c * kTokensPerChunk + warp;
  float row[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    row[i] = (t < T && e < E) ? __ldg(logits + (size_t)t * E + e) : 0.0f;
  }
  __syncthreads();  // counters cleared
  if (t < T) {
    uint32_t key[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? ordered_key(row[i]) : 0u;
    }
    uint32_t taken = 0u;
    int my_idx = 0;
    float my_val = 0.0f, top_val = 0.0f;
    for (int j = 0; j < k; ++j) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u)) {
          unsigned long long cand = ((unsigned long long)key[i] << 32) | (0xFFFFFFFFu - (uint32_t)e);
          best = cand > best ? cand : best;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      const int idx = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
      const float val = key_value((uint32_t)(best >> 32));
      if ((idx & 31) == lane) taken |= 1u << (idx >> 5);
      if (lane == j) { my_idx = idx; my_val = val; }
      if (j == 0) top_val = val;
      if (lane == 0) atomicAdd(&cnt[idx], 1);
    }
    const float ex = lane < k ? expf(my_val - top_val) : 0.0f;
    const float z = warp_sum(ex);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_idx;
      gates[(size_t)t * k + lane] = ex / z;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)c * E + e] = cnt[e];
}

// In-place exclusive scan of hist[.][e] over chunks for expert e = blockIdx.x.
__global__ void __launch_bounds__(1024)
chunk_scan_kernel(int32_t* __restrict__ hist, int nchunks, int E, int32_t* __restrict__ counts) {
  __shared__ int32_t warp_tot[32];
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t running = 0;
  for (int base = 0; base < nchunks; base += 1024) {
    const int c = base + tid;
    const int32_t v = c < nchunks ? hist[(size_t)c * E + e] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t w = warp_tot[lane], wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t n = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += n;
      }
      warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int32_t excl = running + warp_tot[warp] + incl - v;
    if (c < nchunks) hist[(size_t)c * E + e] = excl;
    // total of this block of chunks = last thread's inclusive value
    __shared__ int32_t block_total;
    if (tid == 1023) block_total = warp_tot[31] + incl;
    __syncthreads();
    running += block_total;
    __syncthreads();
  }
  if (tid == 0) counts[e] = running;
}

__global__ void __launch_bounds__(1024)
offsets_kernel(const int32_t* __restrict__ counts, int E, int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t v = tid < E ? counts[tid] : 0;
  int32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_tot[lane], wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_tot[lane] = wi - w;
  }
  __syncthreads();
  const int32_t excl = warp_tot[warp] + incl - v;
  if (tid < E) offsets[tid] = excl;
  if (tid == E - 1) offsets[E] = excl + v;
}

__global__ void __launch_bounds__(kWarps * 32)
rank_kernel(const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ chunk_prefix,
            const int32_t* __restrict__ offsets, int T, int E, int k, int nchunks,
            int32_t* __restrict__ dest_row, int32_t* __restrict__ src_row, int* err) {
  extern __shared__ int32_t cur_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  if (c >= nchunks) return;
  int32_t* cursor = cur_all + warp * E;
  for (int e = lane; e < E; e += 32) cursor[e] = offsets[e] + chunk_prefix[(size_t)c * E + e];
  __syncwarp();
  const long p_beg = (long)c * kTokensPerChunk * k;
  const long p_end = (long)min(T, (c + 1) * kTokensPerChunk) * k;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long p0 = p_beg; p0 < p_end; p0 += 32) {
    const long p = p0 + lane;
    const bool active = p < p_end;
    int e = active ? topk_idx[p] : -1;
    if (active && (e < 0 || e >= E)) {
      set_error(err, MOE_ERR_DEVICE_INDEX);
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int32_t dest = cursor[e] + __popc(peers & lt_mask);
      dest_row[p] = dest;
      src_row[dest] = (int32_t)p;
    }
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(peers)) cursor[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

int route_num_chunks(int T) { return (T + kTokensPerChunk - 1) / kTokensPerChunk; }

size_t route_workspace_bytes(int T, int E) {
  return (size_t)route_num_chunks(T) * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_route_meta(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* gates, int32_t* counts, int32_t* offsets, int32_t* dest_row,
                              int32_t* src_row, int32_t* hist, cudaStream_t st) {
  const int nchunks = route_num_chunks(T);
  if (nchunks > 0) {
    const size_t smem = (size_t)E * sizeof(int32_t);
    const int nv = (E + 31) / 32;
#define MOE_TOPK_CASE(NVV)                                                                           \
  MOE_COUNTED_AS("topk_hist", st) topk_hist_kernel<NVV><<<nchunks, kWarps * 32, smem, st>>>(          \
      logits, T, E, k, nchunks, topk_idx, gates, hist)
    if (nv <= 1) MOE_TOPK_CASE(1);
    else if (nv <= 2) MOE_TOPK_CASE(2);
    else if (nv <= 4) MOE_TOPK_CASE(4);
    else if (nv <= 8) MOE_TOPK_CASE(8);
    else if (nv <= 16) MOE_TOPK_CASE(16);
    else MOE_TOPK_CASE(32);
#undef MOE_TOPK_CASE
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  MOE_COUNTED_AS("chunk_scan", st) chunk_scan_kernel<<<E, 1024, 0, st>>>(hist, nchunks, E, counts);
  MOE_COUNTED_AS("offsets", st) offsets_kernel<<<1, 1024, 0, st>>>(counts, E, offsets);
  if (nchunks > 0) {
    const int grid = (nchunks + kWarps - 1) / kWarps;
    const size_t smem = (size_t)kWarps * E * sizeof(int32_t);
    MOE_COUNTED_AS("rank", st) rank_kernel<<<grid, kWarps * 32, smem, st>>>(topk_idx, hist, offsets, T, E, k, nchunks,
                                                 dest_row, src_row, device_error_word());
  }
  return cudaGetLastError();
}

}  // namespace moe
