/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, fp64 CPU definition of the single-GPU Mixture-of-Experts
 * layer (forward and backward) and of the MXFP8 block quantiser. It is the
 * oracle that the CUDA path is checked against. Only tests/, the smoke entry
 * point and the CPU-baseline leg of bench.py load it. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources of what is computed:
 *  - "Introducing Olmo-core 3" (page 1), section "Scaling and optimizing MoE
 *    training": routing picks experts per token, routed rows are placed
 *    directly into each expert's input buffer, routing metadata stays on the
 *    device, and a grouped GEMM runs all expert computations together; MXFP8
 *    (a lower-precision format) is supported for the expert feed-forward.
 *  - The layer's math is fixed by the workload definition of the 8/128-expert
 *    top-4 benchmark: softmax over E router logits, top-k, gates renormalised
 *    to sum to 1, a SwiGLU expert FFN, and MXFP8 = E4M3 elements with one
 *    E8M0 power-of-two scale per 32 contiguous elements along K.
 *  - E4M3/E8M0 encodings: OCP Microscaling Formats (MX) v1.0 and OCP 8-bit
 *    Floating Point (OFP8) specifications (bias 7, max normal 448,
 *    S.1111.111 is NaN; E8M0 bias 127).
 *
 * Readings taken where the pages are silent:
 *  - top-k compares logits (not probabilities); equal logits keep the
 *    smaller expert index; the k slots are ordered by (logit desc, index asc).
 *  - g_j = exp(l_j - m) / sum_{i in S} exp(l_i - m): softmax over E followed
 *    by renormalisation over the selected set is the same value.
 *  - dropless: every token gets exactly k rows; offsets are an unpadded
 *    exclusive prefix sum; inside an expert, rows follow token order.
 *  - the optional per-expert logit bias is a constant input (no gradient).
 *  - E8M0 exponent s = ceil(log2(amax / 448)) (smallest s that needs no
 *    saturation), clamped to [-127, 127]; amax == 0 gives s = -127.
 *  - E4M3 rounding is round-to-nearest-even with saturation to +-448.
 *
 * Inputs are float32 arrays (bf16 values widen exactly); every sum, product
 * and exp is done in double. Threads only split independent work (tokens,
 * experts, hidden columns); every sum runs in a fixed order, so results do
 * not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* a tiny static work splitter                                          */
/* ------------------------------------------------------------------ */
typedef void (*oc_range_fn)(void* ctx, long lo, long hi);
typedef struct { oc_range_fn fn; void* ctx; long lo, hi; } oc_job;

static void* oc_run_job(void* p) {
  oc_job* j = (oc_job*)p;
  if (j->lo < j->hi) j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void oc_parallel(oc_range_fn fn, void* ctx, long n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((long)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  if (nthreads == 1) { if (n > 0) fn(ctx, 0, n); return; }
  pthread_t th[256];
  oc_job jobs[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].fn = fn; jobs[i].ctx = ctx;
    jobs[i].lo = n * i / nthreads; jobs[i].hi = n * (i + 1) / nthreads;
    pthread_create(&th[i], NULL, oc_run_job, &jobs[i]);
  }
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

static double oc_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double oc_silu(double z) { return z * oc_sigmoid(z); }
static double oc_dsilu(double z) { double s = oc_sigmoid(z); return s * (1.0 + z * (1.0 - s)); }

/* ------------------------------------------------------------------ */
/* routing                                                             */
/* ------------------------------------------------------------------ */

/* logits[t][e] = bias[e] + sum_c x[t][c] * w_r[c][e];  w_r is [d][E]. */
typedef struct { const float *x, *wr, *bias; int d, E; double* out; } oc_logits_ctx;
static void oc_logits_rows(void* p, long lo, long hi) {
  oc_logits_ctx* c = (oc_logits_ctx*)p;
  for (long t = lo; t < hi; ++t)
    for (int e = 0; e < c->E; ++e) {
      double s = c->bias ? (double)c->bias[e] : 0.0;
      for (int i = 0; i < c->d; ++i) s += (double)c->x[t * c->d + i] * (double)c->wr[(long)i * c->E + e];
      c->out[t * c->E + e] = s;
    }
}
void oc_router_logits(const float* x, const float* w_r, const float* bias, int T, int d, int E,
                      double* logits, int nthreads) {
  oc_logits_ctx c = {x, w_r, bias, d, E, logits};
  oc_parallel(oc_logits_rows, &c, T, nthreads);
}

/* Top-k: repeatedly take the largest not-yet-taken logit; scanning experts in
   ascending order with a strict '>' keeps the smaller index on ties. */
void oc_topk(const double* logits, int T, int E, int k, int32_t* topk_idx) {
  char* taken = (char*)malloc((size_t)E);
  for (long t = 0; t < T; ++t) {
    memset(taken, 0, (size_t)E);
    const double* l = logits + t * E;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      topk_idx[t * k + j] = best;
    }
  }
  free(taken);
}

/* gates[t][j] = exp(l_{S_j} - m) / sum_{i in S} exp(l_i - m), m = max over S. */
/* Routing load statistics (the next step after routing: a load-balance
 * metric kept alongside the routing metadata). The pages name the concern
 * (experts gaming or starving the token distribution) but give no formula,
 * so this is the plainest set of statistics; parity is unpinned by the pages.
 *   probs_mean[e] = (1/T) sum_t softmax(logits[t])_e   (softmax over all E)
 *   f_e           = counts[e] / (T k)
 *   stats[0]      = E * sum_e f_e probs_mean[e]   (1 under perfect balance)
 *   stats[1]      = max_e counts[e] * E / (T k)   (largest load / mean load)
 *   stats[2]      = number of experts with counts[e] == 0
 *   stats[3]      = population std of counts / their mean               */
void oc_route_stats(const double* logits, const int32_t* counts, int T, int E, int k, double* probs_mean,
                    double* stats) {
  for (int e = 0; e < E; ++e) probs_mean[e] = 0.0;
  for (long t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double m = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp(l[e] - m);
    for (int e = 0; e < E; ++e) probs_mean[e] += exp(l[e] - m) / z;
  }
  for (int e = 0; e < E; ++e) probs_mean[e] = T > 0 ? probs_mean[e] / T : 0.0;
  const double R = (double)T * k, mean = R / E;
  double aux = 0.0, mx = 0.0, var = 0.0;
  int empty = 0;
  for (int e = 0; e < E; ++e) {
    const double f = R > 0 ? counts[e] / R : 0.0;
    aux += f * probs_mean[e];
    if (counts[e] > mx) mx = counts[e];
    if (counts[e] == 0) ++empty;
    var += (counts[e] - mean) * (counts[e] - mean);
  }
  stats[0] = E * aux;
  stats[1] = mean > 0 ? mx / mean : 0.0;
  stats[2] = empty;
  stats[3] = mean > 0 ? sqrt(var / E) / mean : 0.0;
}

void oc_gates(const double* logits, const int32_t* topk_idx, int T, int E, int k, double* gates) {
  for (long t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double m = l[topk_idx[t * k]];
    for (int j = 1; j < k; ++j) if (l[topk_idx[t * k + j]] > m) m = l[topk_idx[t * k + j]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += exp(l[topk_idx[t * k + j]] - m);
    for (int j = 0; j < k; ++j) gates[t * k + j] = exp(l[topk_idx[t * k + j]] - m) / z;
  }
}

/* Per-expert counts, exclusive offsets, and the placement of routed pair
   p = t*k + j at row dest_row[p] of its expert's contiguous block. Visiting
   tokens in ascending order and bumping a per-expert cursor gives rows
   ordered by (expert, token). src_row is the inverse map. */
void oc_dispatch(const int32_t* topk_idx, int T, int E, int k, int32_t* counts, int32_t* offsets,
                 int32_t* dest_row, int32_t* src_row) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long p = 0; p < (long)T * k; ++p) counts[topk_idx[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (long t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      long p = t * k + j;
      int32_t r = cursor[topk_idx[p]]++;
      dest_row[p] = r;
      src_row[r] = (int32_t)p;
    }
  free(cursor);
}

/* ------------------------------------------------------------------ */
/* expert SwiGLU MLP, token by token                                   */
/* ------------------------------------------------------------------ */
/* Layouts: w_gate, w_up [E][d][f]; w_down [E][f][d]; x [T][d].
   For pair p = t*k + j with expert e and gate g:
     hg = x[t] . w_gate[e], hu = x[t] . w_up[e], a = silu(hg) * hu,
     ye = a . w_down[e],   y[t] += g * ye (j ascending).               */
typedef struct {
  const float *x, *wg, *wu, *wd; const int32_t* idx; const double* gates;
  int d, E, k, f; double *hg, *hu, *a, *ye, *y;
} oc_fwd_ctx;

static void oc_fwd_tokens(void* p, long lo, long hi) {
  oc_fwd_ctx* c = (oc_fwd_ctx*)p;
  const int d = c->d, f = c->f, k = c->k;
  for (long t = lo; t < hi; ++t) {
    double* yt = c->y + t * d;
    for (int i = 0; i < d; ++i) yt[i] = 0.0;
    const float* xt = c->x + t * d;
    for (int j = 0; j < k; ++j) {
      long pr = t * k + j;
      int e = c->idx[pr];
      const float* wg = c->wg + (long)e * d * f;
      const float* wu = c->wu + (long)e * d * f;
      const float* wd = c->wd + (long)e * f * d;
      double *hg = c->hg + pr * f, *hu = c->hu + pr * f, *a = c->a + pr * f, *ye = c->ye + pr * d;
      for (int n = 0; n < f; ++n) {
        double sg = 0.0, su = 0.0;
        for (int i = 0; i < d; ++i) {
          sg += (double)xt[i] * (double)wg[(long)i * f + n];
          su += (double)xt[i] * (double)wu[(long)i * f + n];
        }
        hg[n] = sg; hu[n] = su; a[n] = oc_silu(sg) * su;
      }
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int n = 0; n < f; ++n) s += a[n] * (double)wd[(long)n * d + i];
        ye[i] = s;
      }
      double g = c->gates[pr];
      for (int i = 0; i < d; ++i) yt[i] += g * ye[i];
    }
  }
}

/* hg, hu, a: [T*k][f]; ye: [T*k][d]; y: [T][d], all indexed by pair p = t*k+j. */
void oc_forward(const float* x, const float* w_gate, const float* w_up, const float* w_down,
                const int32_t* topk_idx, const double* gates, int T, int d, int E, int k, int f,
                double* hg, double* hu, double* a, double* ye, double* y, int nthreads) {
  oc_fwd_ctx c = {x, w_gate, w_up, w_down, topk_idx, gates, d, E, k, f, hg, hu, a, ye, y};
  oc_parallel(oc_fwd_tokens, &c, T, nthreads);
}

/* ------------------------------------------------------------------ */
/* backward                                                            */
/* ------------------------------------------------------------------ */
/* Chain rule through y[t] = sum_j g_j ye_j with g = softmax over the
   selected logits, given dy = dL/dy:
     dg_j   = <dy[t], ye_j>
     dye_j  = g_j dy[t]
     da     = w_down[e] . dye           (da[n] = sum_i w_down[e][n][i] dye[i])
     dhg    = da * hu * silu'(hg),  dhu = da * silu(hg)
     dx[t] += w_gate[e] . dhg + w_up[e] . dhu
     dl_i   = sum_j dg_j * d g_j / d l_i,  d g_j / d l_i = g_j (delta_ij - g_i)
              for i in S, 0 for experts not selected
     dx[t] += w_r . dl
   Weight gradients (summed over tokens in ascending order):
     dw_down[e] += a^T dye,  dw_gate[e] += x[t]^T dhg,  dw_up[e] += x[t]^T dhu,
     dw_r += x[t]^T dl.                                                 */
typedef struct {
  const float *x, *wr, *wg, *wu, *wd, *dy; const int32_t* idx; const double *gates, *hg, *hu, *a, *ye;
  int T, d, E, k, f;
  double *dgates, *dlogits, *dx, *dye, *dhg, *dhu;       /* per-token / per-pair outputs */
  double *dwg, *dwu, *dwd, *dwr;                          /* weight gradients */
} oc_bwd_ctx;

static void oc_bwd_tokens(void* p, long lo, long hi) {
  oc_bwd_ctx* c = (oc_bwd_ctx*)p;
  const int d = c->d, f = c->f, k = c->k, E = c->E;
  double* da = (double*)malloc(sizeof(double) * (size_t)f);
  for (long t = lo; t < hi; ++t) {
    const float* dyt = c->dy + t * d;
    const float* xt = c->x + t * d;
    double* dxt = c->dx + t * d;
    for (int i = 0; i < d; ++i) dxt[i] = 0.0;
    for (int j = 0; j < k; ++j) {
      long pr = t * k + j;
      int e = c->idx[pr];
      const double g = c->gates[pr];
      const double *ye = c->ye + pr * d, *hg = c->hg + pr * f, *hu = c->hu + pr * f;
      double *dye = c->dye + pr * d, *dhg = c->dhg + pr * f, *dhu = c->dhu + pr * f;
      double dg = 0.0;
      for (int i = 0; i < d; ++i) dg += (double)dyt[i] * ye[i];
      c->dgates[pr] = dg;
      for (int i = 0; i < d; ++i) dye[i] = g * (double)dyt[i];
      const float* wd = c->wd + (long)e * f * d;
      for (int n = 0; n < f; ++n) {
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += (double)wd[(long)n * d + i] * dye[i];
        da[n] = s;
      }
      for (int n = 0; n < f; ++n) {
        dhg[n] = da[n] * hu[n] * oc_dsilu(hg[n]);
        dhu[n] = da[n] * oc_silu(hg[n]);
      }
      const float* wg = c->wg + (long)e * d * f;
      const float* wu = c->wu + (long)e * d * f;
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int n = 0; n < f; ++n)
          s += (double)wg[(long)i * f + n] * dhg[n] + (double)wu[(long)i * f + n] * dhu[n];
        dxt[i] += s;
      }
    }
    /* router: softmax Jacobian over the selected set */
    double* dl = c->dlogits + t * E;
    for (int e = 0; e < E; ++e) dl[e] = 0.0;
    for (int i = 0; i < k; ++i) {
      double gi = c->gates[t * k + i], s = 0.0;
      for (int j = 0; j < k; ++j) {
        double gj = c->gates[t * k + j];
        s += c->dgates[t * k + j] * gj * ((i == j ? 1.0 : 0.0) - gi);
      }
      dl[c->idx[t * k + i]] = s;
    }
    for (int i = 0; i < d; ++i) {
      double s = 0.0;
      for (int e = 0; e < E; ++e) s += (double)c->wr[(long)i * E + e] * dl[e];
      dxt[i] += s;
    }
    (void)xt;
  }
  free(da);
}

static void oc_bwd_experts(void* p, long lo, long hi) {
  oc_bwd_ctx* c = (oc_bwd_ctx*)p;
  const int d = c->d, f = c->f, k = c->k;
  for (long e = lo; e < hi; ++e) {
    double* dwg = c->dwg + e * d * f;
    double* dwu = c->dwu + e * d * f;
    double* dwd = c->dwd + e * f * d;
    memset(dwg, 0, sizeof(double) * (size_t)d * f);
    memset(dwu, 0, sizeof(double) * (size_t)d * f);
    memset(dwd, 0, sizeof(double) * (size_t)f * d);
    for (long t = 0; t < c->T; ++t)
      for (int j = 0; j < k; ++j) {
        long pr = t * k + j;
        if (c->idx[pr] != e) continue;
        const float* xt = c->x + t * d;
        const double *a = c->a + pr * f, *dye = c->dye + pr * d;
        const double *dhg = c->dhg + pr * f, *dhu = c->dhu + pr * f;
        for (int n = 0; n < f; ++n)
          for (int i = 0; i < d; ++i) dwd[(long)n * d + i] += a[n] * dye[i];
        for (int i = 0; i < d; ++i)
          for (int n = 0; n < f; ++n) {
            dwg[(long)i * f + n] += (double)xt[i] * dhg[n];
            dwu[(long)i * f + n] += (double)xt[i] * dhu[n];
          }
      }
  }
}

static void oc_bwd_router_w(void* p, long lo, long hi) {
  oc_bwd_ctx* c = (oc_bwd_ctx*)p;
  const int d = c->d, E = c->E;
  for (long i = lo; i < hi; ++i)
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (long t = 0; t < c->T; ++t) s += (double)c->x[t * d + i] * c->dlogits[t * E + e];
      c->dwr[i * E + e] = s;
    }
}

/* Outputs: dgates [T*k], dlogits [T][E], dx [T][d], dw_gate/dw_up [E][d][f],
   dw_down [E][f][d], dw_r [d][E]. Scratch: dye [T*k][d], dhg/dhu [T*k][f]
   (returned too: they are the per-row values of the backward GEMMs). */
void oc_backward(const float* x, const float* w_r, const float* w_gate, const float* w_up,
                 const float* w_down, const float* dy, const int32_t* topk_idx, const double* gates,
                 const double* hg, const double* hu, const double* a, const double* ye, int T, int d,
                 int E, int k, int f, double* dgates, double* dlogits, double* dx, double* dye,
                 double* dhg, double* dhu, double* dw_gate, double* dw_up, double* dw_down,
                 double* dw_r, int nthreads) {
  oc_bwd_ctx c = {x, w_r, w_gate, w_up, w_down, dy, topk_idx, gates, hg, hu, a, ye, T, d, E, k, f,
                  dgates, dlogits, dx, dye, dhg, dhu, dw_gate, dw_up, dw_down, dw_r};
  oc_parallel(oc_bwd_tokens, &c, T, nthreads);
  oc_parallel(oc_bwd_experts, &c, E, nthreads);
  oc_parallel(oc_bwd_router_w, &c, d, nthreads);
}

/* ------------------------------------------------------------------ */
/* MXFP8: E4M3 elements with one E8M0 scale per 32 elements            */
/* ------------------------------------------------------------------ */

/* OCP OFP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
   field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities. */
double oc_e4m3_decode(uint8_t code) {
  int s = code >> 7, ex = (code >> 3) & 15, m = code & 7;
  double v;
  if (ex == 15 && m == 7) return NAN;
  if (ex == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, ex - 7);
  return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating at +-448. The grid
   spacing is 2^(e-3) for |v| in [2^e, 2^(e+1)), e >= -6, and 2^-9 below. */
uint8_t oc_e4m3_encode(double v) {
  int neg = signbit(v) ? 1 : 0;
  double av = fabs(v);
  if (av >= 448.0) return (uint8_t)((neg << 7) | 0x7E);
  int e;
  if (av < ldexp(1.0, -6)) e = -6;          /* subnormal range shares the 2^-9 step */
  else { frexp(av, &e); e -= 1; }           /* av in [2^e, 2^(e+1)) */
  double step = ldexp(1.0, e - 3);
  double q = av / step;                     /* exact: step is a power of two */
  double fl = floor(q), rem = q - fl;
  double n = fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;
  double r = n * step;                      /* may round up to 2^(e+1): still on the grid */
  if (r >= 448.0) return (uint8_t)((neg << 7) | 0x7E);
  /* encode r exactly */
  uint8_t code;
  if (r < ldexp(1.0, -6)) {
    code = (uint8_t)(r / ldexp(1.0, -9));   /* 0..7 */
  } else {
    int er; double fr = frexp(r, &er);      /* r = fr * 2^er, fr in [0.5,1) */
    int ex = er - 1 + 7;
    int m = (int)((fr * 2.0 - 1.0) * 8.0);
    code = (uint8_t)((ex << 3) | m);
  }
  return (uint8_t)((neg << 7) | code);
}

/* Shared exponent of one block: the smallest s with amax / 2^s <= 448,
   i.e. ceil(log2(amax / 448)), clamped to [-127, 127]. amax == 0 -> -127. */
int oc_e8m0_exponent(double amax) {
  if (!(amax > 0.0)) return -127;
  int e; frexp(amax, &e); e -= 1;            /* amax in [2^e, 2^(e+1)) */
  int s = e - 8;
  if (amax > ldexp(448.0, s)) s += 1;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return s;
}

/* Quantise a [rows][K] matrix with one scale per 32 consecutive elements of
   a row (K % 32 == 0). q: [rows][K] codes, sc: [rows][K/32] E8M0 bytes. */
void oc_mxfp8_quantize_rows(const float* v, long rows, long K, uint8_t* q, uint8_t* sc) {
  for (long r = 0; r < rows; ++r)
    for (long b = 0; b < K / 32; ++b) {
      const float* blk = v + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) if (fabs((double)blk[i]) > amax) amax = fabs((double)blk[i]);
      int s = oc_e8m0_exponent(amax);
      sc[r * (K / 32) + b] = (uint8_t)(s + 127);
      for (int i = 0; i < 32; ++i) q[r * K + b * 32 + i] = oc_e4m3_encode(ldexp((double)blk[i], -s));
    }
}

/* Quantise along rows inside segments: column c of rows [seg[g], seg[g+1])
   is cut into blocks of 32 consecutive rows starting at seg[g]; the last
   block of a segment is zero-padded to 32. q: [rows][C] codes in place of the
   values; sc: [nblk_total][C] where segment g owns block rows starting at
   sum_{h<g} ceil(len_h / 32). */
void oc_mxfp8_quantize_cols_segmented(const float* v, long rows, long C, const int32_t* seg, int nseg,
                                      uint8_t* q, uint8_t* sc) {
  long brow = 0;
  for (int g = 0; g < nseg; ++g) {
    long r0 = seg[g], r1 = seg[g + 1];
    for (long b0 = r0; b0 < r1; b0 += 32, ++brow) {
      long b1 = b0 + 32 < r1 ? b0 + 32 : r1;
      for (long c = 0; c < C; ++c) {
        double amax = 0.0;
        for (long r = b0; r < b1; ++r) if (fabs((double)v[r * C + c]) > amax) amax = fabs((double)v[r * C + c]);
        int s = oc_e8m0_exponent(amax);
        sc[brow * C + c] = (uint8_t)(s + 127);
        for (long r = b0; r < b1; ++r) q[r * C + c] = oc_e4m3_encode(ldexp((double)v[r * C + c], -s));
      }
    }
  }
}

/* The two quantisers above on double input (intermediates of the MXFP8
   layer that the oracle keeps in double). Same block rule and rounding. */
void oc_mxfp8_quantize_rows_f64(const double* v, long rows, long K, uint8_t* q, uint8_t* sc) {
  for (long r = 0; r < rows; ++r)
    for (long b = 0; b < K / 32; ++b) {
      const double* blk = v + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) if (fabs(blk[i]) > amax) amax = fabs(blk[i]);
      int s = oc_e8m0_exponent(amax);
      sc[r * (K / 32) + b] = (uint8_t)(s + 127);
      for (int i = 0; i < 32; ++i) q[r * K + b * 32 + i] = oc_e4m3_encode(ldexp(blk[i], -s));
    }
}

void oc_mxfp8_quantize_cols_segmented_f64(const double* v, long rows, long C, const int32_t* seg, int nseg,
                                          uint8_t* q, uint8_t* sc) {
  long brow = 0;
  for (int g = 0; g < nseg; ++g) {
    long r0 = seg[g], r1 = seg[g + 1];
    for (long b0 = r0; b0 < r1; b0 += 32, ++brow) {
      long b1 = b0 + 32 < r1 ? b0 + 32 : r1;
      for (long c = 0; c < C; ++c) {
        double amax = 0.0;
        for (long r = b0; r < b1; ++r) if (fabs(v[r * C + c]) > amax) amax = fabs(v[r * C + c]);
        int s = oc_e8m0_exponent(amax);
        sc[brow * C + c] = (uint8_t)(s + 127);
        for (long r = b0; r < b1; ++r) q[r * C + c] = oc_e4m3_encode(ldexp(v[r * C + c], -s));
      }
    }
  }
}
