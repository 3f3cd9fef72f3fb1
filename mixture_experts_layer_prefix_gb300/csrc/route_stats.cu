// route_stats.cu -- routing load statistics kept alongside the routing
// metadata ("Introducing Olmo-core 3", section "Scaling and optimizing MoE
// training": routing decides which experts see which tokens, and an unbalanced
// token distribution starves or overloads experts). The pages give no formula;
// the statistics are the plainest ones:
//   probs_mean[e] = (1/T) sum_t softmax(logits[t])_e     (softmax over all E)
//   stats[0] = E * sum_e (counts[e] / (T k)) * probs_mean[e]  (1 when balanced)
//   stats[1] = max_e counts[e] * E / (T k)
//   stats[2] = experts with no rows
//   stats[3] = population std of counts / mean count
// Deterministic: every sum runs in a fixed order (tokens of a warp in order,
// warps of a CTA in order, CTAs in order).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kStatWarps = 8;
constexpr int kStatTokensPerWarp = 32;
constexpr int kStatTokensPerCta = kStatWarps * kStatTokensPerWarp;
constexpr int kMaxE = 1024;

// partial[b][e] = sum over the CTA's tokens of softmax(logits[t])_e.
__global__ void __launch_bounds__(kStatWarps * 32)
route_stats_partial_kernel(const float* __restrict__ logits, int T, int E, float* __restrict__ partial) {
  extern __shared__ float wsum[];  // [kStatWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_lane = (E + 31) / 32;  // <= 32
  float acc[kMaxE / 32];
#pragma unroll
  for (int j = 0; j < kMaxE / 32; ++j) acc[j] = 0.0f;
  const int t0 = blockIdx.x * kStatTokensPerCta + warp * kStatTokensPerWarp;
  for (int i = 0; i < kStatTokensPerWarp; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    const float* l = logits + (size_t)t * E;
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j)
      if (j < per_lane && lane + 32 * j < E) m = fmaxf(m, l[lane + 32 * j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j)
      if (j < per_lane && lane + 32 * j < E) z += expf(l[lane + 32 * j] - m);
    z = warp_sum(z);
    const float inv = 1.0f / z;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j)
      if (j < per_lane && lane + 32 * j < E) acc[j] += expf(l[lane + 32 * j] - m) * inv;
  }
#pragma unroll
  for (int j = 0; j < kMaxE / 32; ++j)
    if (j < per_lane && lane + 32 * j < E) wsum[warp * E + lane + 32 * j] = acc[j];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.0f;
    for (int w = 0; w < kStatWarps; ++w) s += wsum[w * E + e];
    partial[(size_t)blockIdx.x * E + e] = s;
  }
}

// One CTA of 1024 threads: probs_mean from the partials, then the statistics.
__global__ void __launch_bounds__(1024)
route_stats_final_kernel(const float* __restrict__ partial, int nblk, const int32_t* __restrict__ counts, int T,
                         int E, int k, float* __restrict__ probs_mean, float* __restrict__ stats) {
  __shared__ float s_aux[1024], s_var[1024];
  __shared__ int s_max[1024], s_empty[1024];
  const int e = threadIdx.x;
  const double R = (double)T * k, mean = R / E;
  float aux = 0.0f, var = 0.0f;
  int mx = 0, empty = 0;
  if (e < E) {
    float s = 0.0f;
    for (int b = 0; b < nblk; ++b) s += partial[(size_t)b * E + e];
    const float pm = T > 0 ? s / (float)T : 0.0f;
    probs_mean[e] = pm;
    const int c = counts[e];
    aux = R > 0 ? (float)(c / R) * pm : 0.0f;
    const float dev = (float)(c - mean);
    var = dev * dev;
    mx = c;
    empty = c == 0;
  }
  s_aux[e] = aux;
  s_var[e] = var;
  s_max[e] = mx;
  s_empty[e] = empty;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {  // fixed-shape tree
    if (e < o) {
      s_aux[e] += s_aux[e + o];
      s_var[e] += s_var[e + o];
      s_max[e] = max(s_max[e], s_max[e + o]);
      s_empty[e] += s_empty[e + o];
    }
    __syncthreads();
  }
  if (e == 0) {
    stats[0] = (float)E * s_aux[0];
    stats[1] = mean > 0 ? (float)(s_max[0] / mean) : 0.0f;
    stats[2] = (float)s_empty[0];
    stats[3] = mean > 0 ? sqrtf(s_var[0] / (float)E) / (float)mean : 0.0f;
  }
}

}  // namespace

size_t route_stats_workspace_bytes(int T, int E) {
  return (size_t)((T + kStatTokensPerCta - 1) / kStatTokensPerCta) * E * sizeof(float);
}

cudaError_t launch_route_stats(const float* logits, const int32_t* counts, int T, int E, int k, float* probs_mean,
                               float* stats, float* partial, cudaStream_t st) {
  const int nblk = (T + kStatTokensPerCta - 1) / kStatTokensPerCta;
  if (nblk > 0)
    MOE_COUNTED_AS("route_stats_partial", st) route_stats_partial_kernel<<<nblk, kStatWarps * 32, kStatWarps * E * sizeof(float), st>>>(
        logits, T, E, partial);
  MOE_COUNTED_AS("route_stats_final", st) route_stats_final_kernel<<<1, 1024, 0, st>>>(partial, nblk, counts, T, E, k, probs_mean, stats);
  return cudaGetLastError();
}

}  // namespace moe
