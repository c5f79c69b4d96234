/*
 * sv_oracle.c -- plain, slow, fp64 CPU oracle for the speculative-decoding
 * verification step.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests,
 * by the smoke check and by the CPU-baseline leg of the benchmark, never by
 * the product path.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (sources, cited by page title and section):
 *
 *   [SD-overview]  "猜想解码 (Speculative Decoding) 全景" page:
 *       考点2 -- acceptance probability min(1, P_target(x)/P_draft(x)), the
 *               residual distribution max(0, P_t - P_d) / sum_y max(0, P_t - P_d),
 *               and the losslessness identity P_final == P_target;
 *       考点4 -- expected tokens per step sum_{i=0..gamma} alpha^i, and the
 *               floor of one emitted token when alpha -> 0;
 *       第二章 -- the acceptance formula;
 *       第三章 -- the NumPy operator: accept iff u <= P_accept, otherwise
 *               sample from the normalised residual.
 *   [Deferred-SD]  deferred speculative decoding page (lqnn.cn), section
 *       "动态推迟投机验证调度器设计": temperature-scaled softmax of a logit
 *       row, per-position accept test in draft order, stop at the first
 *       rejection ("后续推迟序列作废"), inverse-CDF scan in vocabulary order.
 *
 * Readings taken where the pages are silent or disagree:
 *   R1  accept iff u <= r (the NumPy operator), not u < r.
 *   R2  P_draft(x) == 0 gives r = 1 (the limit of the formula), no epsilon.
 *   R3  the residual is formed from PROBABILITIES (考点2), not from raw
 *       logits as the C++ scheduler snippet does.
 *   R4  the bonus token: when all gamma drafts are accepted, one more token is
 *       sampled from target row gamma (gamma+1 verified positions, 考点1/考点4).
 *   R5  inverse CDF: tau = u * Z, token = smallest v with C_v > tau, C the
 *       index-order running sum (strict '>' so zero-mass tokens are never
 *       chosen).
 *   R6  Z == 0 after a rejection (impossible in exact arithmetic): fall back
 *       to the inverse CDF of the target row with the same u; flagged.
 *   R7  temperature T scales both rows (l / T) before the softmax; T must be
 *       finite and >= 2^-126 (a normal fp32), else the request is invalid.
 *   R8  NaN or +inf anywhere in a request's rows, an all -inf row, or a draft
 *       token outside [0, V) make the request invalid: n = 0, tokens all -1.
 *   R9  greedy (T = 0): argmax of the stored target logits, lowest index on
 *       ties; accept while draft == argmax; the first mismatch emits the
 *       argmax; all accepted emits the argmax of row gamma.
 *
 * Every loop below is the definition written out: no blocking, no fusion.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SVO_F32 0
#define SVO_BF16 1

/* per-request flag bits written to out_flags */
#define SVO_INVALID_NONFINITE 1
#define SVO_INVALID_TOKEN 2
#define SVO_INVALID_TEMP 4
#define SVO_NEAR_ACCEPT 16    /* |u_acc - r_i| < near_eps at a decided position */
#define SVO_NEAR_SAMPLE 32    /* |C_{v-1}/Z - u| or |C_v/Z - u| < near_eps */
#define SVO_DEGENERATE 64     /* reading R6 was used */

#define SVO_TREE_MAX_N 256    /* nodes per token tree */

#ifndef SVO_MUTANT
#define SVO_MUTANT 0 /* the mutation tests rebuild this file with planted mistakes */
#endif

/* exact widening of one stored logit to fp64 */
static double load_logit(const void* base, int dtype, size_t idx) {
  if (dtype == SVO_F32) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Temperature-scaled softmax of one row into p[0..V).  Returns 0 when the row
 * holds NaN or +inf or is entirely -inf (reading R8), 1 otherwise.
 * [Deferred-SD] scheduler section: exp((l - max) / T) / sum, here in fp64 and
 * without the snippet's epsilon on the sum. */
static int softmax_row(const void* base, int dtype, size_t row_off, int V, double T,
                       double* p) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double l = load_logit(base, dtype, row_off + (size_t)v);
    if (isnan(l) || (isinf(l) && l > 0)) return 0;
#if SVO_MUTANT == 8
    (void)m;
#else
    if (l / T > m) m = l / T;
#endif
  }
#if SVO_MUTANT == 8
  m = 0.0; /* planted: no max subtraction */
#else
  if (isinf(m)) return 0; /* all -inf */
#endif
  double S = 0.0;
#if SVO_MUTANT == 9
  for (int v = 0; v + 1 < V; ++v) { /* planted: last term dropped */
#else
  for (int v = 0; v < V; ++v) {
#endif
    double l = load_logit(base, dtype, row_off + (size_t)v);
    p[v] = exp(l / T - m);
    S += p[v];
  }
  if (!(S > 0.0) || isinf(S)) return 0;
  for (int v = 0; v < V; ++v) p[v] /= S;
  return 1;
}

/* Inverse CDF over nonnegative weights w[0..V) with total Z (reading R5):
 * smallest v whose index-order running sum exceeds tau = u * Z.  Sets *near
 * when the chosen token's CDF edges sit within near_eps of u. */
static int inverse_cdf(const double* w, int V, double Z, double u, double near_eps,
                       int* near, double* dist) {
  double tau = u * Z;
  double C = 0.0;
  int chosen = -1;
  double c_lo = 0.0, c_hi = 0.0;
  for (int v = 0; v < V; ++v) {
    double c_prev = C;
    C += w[v];
#if SVO_MUTANT == 5
    if (C >= tau) { /* planted: '>=' picks a zero-mass token at tau == C */
#else
    if (C > tau) {
#endif
      chosen = v;
      c_lo = c_prev;
      c_hi = C;
      break;
    }
  }
  if (chosen < 0) { /* tau >= total after rounding: last token with mass */
    for (int v = V - 1; v >= 0; --v)
      if (w[v] > 0.0) { chosen = v; break; }
    if (chosen < 0) chosen = 0;
    c_lo = C - w[chosen];
    c_hi = C;
    *near = 1;
  }
  *dist = fmin(fabs(c_lo / Z - u), fabs(c_hi / Z - u));
  if (*dist < near_eps) *near = 1;
  return chosen;
}

typedef struct {
  int dtype;
  const void *Lt, *Ld;
  const int32_t* x;
  const float *u_acc, *u_res, *temp;
  int B, gamma, V;
  int32_t *out_tokens, *out_n;
  double *out_pt, *out_pd, *out_Z, *out_dist;
  int32_t* out_flags;
  double near_eps;
  int b0, b1;
} verify_job;

/* One request of the sampling path: the definition, step by step. */
static void verify_request(const verify_job* J, int b, double* Pt, double* Pd, double* w) {
  const int g = J->gamma, V = J->V, R = g + 1;
  int32_t* tok = J->out_tokens + (size_t)b * R;
  int32_t flags = 0;
  for (int i = 0; i < R; ++i) tok[i] = -1;
  J->out_n[b] = 0;
  if (J->out_Z) J->out_Z[b] = NAN;
  double dist_acc = INFINITY, dist_smp = INFINITY;
  if (J->out_dist) J->out_dist[(size_t)b * 2] = J->out_dist[(size_t)b * 2 + 1] = INFINITY;
  for (int i = 0; i < g; ++i) {
    if (J->out_pt) J->out_pt[(size_t)b * g + i] = NAN;
    if (J->out_pd) J->out_pd[(size_t)b * g + i] = NAN;
  }

  double T = (double)J->temp[b];
  if (!(isfinite(T) && T >= 0x1p-126)) flags |= SVO_INVALID_TEMP; /* reading R7 */
  for (int i = 0; i < g; ++i) {
    int32_t xi = J->x[(size_t)b * g + i];
    if (xi < 0 || xi >= V) flags |= SVO_INVALID_TOKEN;
  }
  if (flags) { J->out_flags[b] = flags; return; }

  /* step 1: softmax of every target row 0..gamma and draft row 0..gamma-1 */
  for (int i = 0; i < R; ++i) {
    if (!softmax_row(J->Lt, J->dtype, ((size_t)b * R + i) * V, V, T, Pt + (size_t)i * V))
      flags |= SVO_INVALID_NONFINITE;
  }
  for (int i = 0; i < g; ++i) {
#if SVO_MUTANT == 4
    double Td = 1.0; /* planted: temperature not applied to the draft row */
#else
    double Td = T;
#endif
    if (!softmax_row(J->Ld, J->dtype, ((size_t)b * g + i) * V, V, Td, Pd + (size_t)i * V))
      flags |= SVO_INVALID_NONFINITE;
  }
  if (flags) { J->out_flags[b] = flags; return; }

  /* step 2: accept draft tokens in order, stop at the first rejection */
  int k = g;
  for (int i = 0; i < g; ++i) {
    int32_t xi = J->x[(size_t)b * g + i];
    double pt = Pt[(size_t)i * V + xi];
    double pd = Pd[(size_t)i * V + xi];
    if (J->out_pt) J->out_pt[(size_t)b * g + i] = pt;
    if (J->out_pd) J->out_pd[(size_t)b * g + i] = pd;
  }
  for (int i = 0; i < g; ++i) {
    int32_t xi = J->x[(size_t)b * g + i];
    double pt = Pt[(size_t)i * V + xi];
    double pd = Pd[(size_t)i * V + xi];
    double r = (pd > 0.0) ? fmin(1.0, pt / pd) : 1.0; /* reading R2 */
    double u = (double)J->u_acc[(size_t)b * g + i];
    if (fabs(u - r) < dist_acc) dist_acc = fabs(u - r);
    if (fabs(u - r) < J->near_eps) flags |= SVO_NEAR_ACCEPT;
#if SVO_MUTANT == 2
    int accept = (u < r); /* planted: strict test */
#else
    int accept = (u <= r); /* reading R1 */
#endif
    if (accept) {
      tok[i] = xi;
    } else {
      k = i;
      break;
    }
  }
#if SVO_MUTANT == 6
  if (k < g) k = (k + 1 < g) ? k + 1 : k; /* planted: resample from the wrong row */
#endif

  /* step 3/4: residual resample at k, or the bonus from target row gamma */
  double Z = 0.0;
  int near = 0, chosen;
  double u = (double)J->u_res[(size_t)b * R + k];
  if (k < g) {
    const double* pt = Pt + (size_t)k * V;
    const double* pd = Pd + (size_t)k * V;
    for (int v = 0; v < V; ++v) {
#if SVO_MUTANT == 1
      /* planted: residual over raw logits, as the C++ snippet has it */
      double lt = load_logit(J->Lt, J->dtype, ((size_t)b * R + k) * V + v);
      double ld = load_logit(J->Ld, J->dtype, ((size_t)b * g + k) * V + v);
      w[v] = fmax(0.0, lt - ld);
#elif SVO_MUTANT == 7
      w[v] = fmax(0.0, pd[v] - pt[v]); /* planted: operands swapped */
#else
      w[v] = fmax(0.0, pt[v] - pd[v]);
#endif
      Z += w[v];
    }
    if (!(Z > 0.0)) { /* reading R6 */
      flags |= SVO_DEGENERATE;
      Z = 0.0;
      for (int v = 0; v < V; ++v) { w[v] = pt[v]; Z += w[v]; }
    }
    chosen = inverse_cdf(w, V, Z, u, J->near_eps, &near, &dist_smp);
  } else {
#if SVO_MUTANT == 3
    J->out_n[b] = k; /* planted: no bonus token */
    J->out_flags[b] = flags;
    if (J->out_Z) J->out_Z[b] = 1.0;
    return;
#endif
    const double* pt = Pt + (size_t)g * V;
    for (int v = 0; v < V; ++v) { w[v] = pt[v]; Z += w[v]; }
    chosen = inverse_cdf(w, V, Z, u, J->near_eps, &near, &dist_smp);
  }
  if (near) flags |= SVO_NEAR_SAMPLE;
  tok[k] = chosen;
  J->out_n[b] = k;
  if (J->out_Z) J->out_Z[b] = Z;
  if (J->out_dist) {
    J->out_dist[(size_t)b * 2] = dist_acc;
    J->out_dist[(size_t)b * 2 + 1] = dist_smp;
  }
  J->out_flags[b] = flags;
}

static void* verify_worker(void* arg) {
  const verify_job* J = (const verify_job*)arg;
  size_t V = (size_t)J->V, R = (size_t)J->gamma + 1;
  double* Pt = (double*)malloc(R * V * sizeof(double));
  double* Pd = (double*)malloc((R > 1 ? R - 1 : 1) * V * sizeof(double));
  double* w = (double*)malloc(V * sizeof(double));
  if (!Pt || !Pd || !w) {
    for (int b = J->b0; b < J->b1; ++b) J->out_flags[b] = -1;
  } else {
    for (int b = J->b0; b < J->b1; ++b) verify_request(J, b, Pt, Pd, w);
  }
  free(Pt);
  free(Pd);
  free(w);
  return NULL;
}

/* Sampling-path oracle over B requests.  Layouts match the library's:
 * Lt [B][gamma+1][V], Ld [B][gamma][V] (fp32 or bf16 bits), x [B][gamma],
 * u_acc [B][gamma], u_res [B][gamma+1], temp [B].  Outputs: out_tokens
 * [B][gamma+1] (-1 padded), out_n [B]; optional out_pt/out_pd [B][gamma]
 * (the softmax probabilities of x_i), out_Z [B] (residual or bonus mass);
 * out_dist [B][2] optional: the smallest |u_acc - r_i| over the decided
 * positions, and the distance of u_resample to the nearer CDF edge of the
 * emitted token (INFINITY where there is none); out_flags [B] (SVO_* bits).
 * Returns 0, or -1 on a bad argument. */
int svo_verify(int dtype, const void* Lt, const void* Ld, const int32_t* x,
               const float* u_acc, const float* u_res, const float* temp, int B,
               int gamma, int V, int32_t* out_tokens, int32_t* out_n, double* out_pt,
               double* out_pd, double* out_Z, double* out_dist, int32_t* out_flags,
               double near_eps, int nthreads) {
  if (B < 0 || gamma < 0 || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16)) return -1;
  if (B == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > B) nthreads = B;
  verify_job* jobs = (verify_job*)calloc((size_t)nthreads, sizeof(verify_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    verify_job* J = &jobs[t];
    J->dtype = dtype; J->Lt = Lt; J->Ld = Ld; J->x = x;
    J->u_acc = u_acc; J->u_res = u_res; J->temp = temp;
    J->B = B; J->gamma = gamma; J->V = V;
    J->out_tokens = out_tokens; J->out_n = out_n;
    J->out_pt = out_pt; J->out_pd = out_pd; J->out_Z = out_Z; J->out_dist = out_dist;
    J->out_flags = out_flags;
    J->near_eps = near_eps;
    J->b0 = (int)((long long)B * t / nthreads);
    J->b1 = (int)((long long)B * (t + 1) / nthreads);
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, verify_worker, &jobs[t]);
  verify_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  for (int b = 0; b < B; ++b)
    if (out_flags[b] < 0) return -2;
  return 0;
}

typedef struct {
  int dtype;
  const void* Lt;
  const int32_t* x;
  int B, gamma, V;
  int32_t *out_tokens, *out_n, *out_argmax, *out_flags;
  int b0, b1;
} greedy_job;

/* Greedy oracle, reading R9: sequential scan with strict '>' so the lowest
 * index wins a tie; the stored values are compared, no temperature. */
static void* greedy_worker(void* arg) {
  const greedy_job* J = (const greedy_job*)arg;
  const int g = J->gamma, V = J->V, R = g + 1;
  for (int b = J->b0; b < J->b1; ++b) {
    int32_t* tok = J->out_tokens + (size_t)b * R;
    int32_t flags = 0;
    for (int i = 0; i < R; ++i) tok[i] = -1;
    J->out_n[b] = 0;
    for (int i = 0; i < g; ++i) {
      int32_t xi = J->x[(size_t)b * g + i];
      if (xi < 0 || xi >= V) flags |= SVO_INVALID_TOKEN;
    }
    int amax[64 + 1];
    for (int i = 0; i < R && !flags; ++i) {
      size_t off = ((size_t)b * R + i) * V;
      double best = -INFINITY;
      int arg = -1;
      for (int v = 0; v < V; ++v) {
        double l = load_logit(J->Lt, J->dtype, off + (size_t)v);
        if (isnan(l) || (isinf(l) && l > 0)) { flags |= SVO_INVALID_NONFINITE; break; }
#if SVO_MUTANT == 10
        if (l >= best) { best = l; arg = v; } /* planted: last index wins a tie */
#else
        if (l > best) { best = l; arg = v; }
#endif
      }
      if (arg < 0) flags |= SVO_INVALID_NONFINITE; /* all -inf */
      amax[i] = arg;
      if (J->out_argmax) J->out_argmax[(size_t)b * R + i] = arg;
    }
    if (!flags) {
      int k = g;
      for (int i = 0; i < g; ++i) {
        if (J->x[(size_t)b * g + i] == amax[i]) tok[i] = amax[i];
        else { k = i; break; }
      }
      tok[k] = amax[k];
      J->out_n[b] = k;
    }
    J->out_flags[b] = flags;
  }
  return NULL;
}

/* Greedy-path oracle.  Lt [B][gamma+1][V], x [B][gamma]; gamma <= 64.
 * out_argmax [B][gamma+1] optional.  Returns 0, or -1 on a bad argument. */
int svo_greedy(int dtype, const void* Lt, const int32_t* x, int B, int gamma, int V,
               int32_t* out_tokens, int32_t* out_n, int32_t* out_argmax,
               int32_t* out_flags, int nthreads) {
  if (B < 0 || gamma < 0 || gamma > 64 || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16))
    return -1;
  if (B == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > B) nthreads = B;
  greedy_job* jobs = (greedy_job*)calloc((size_t)nthreads, sizeof(greedy_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    greedy_job* J = &jobs[t];
    J->dtype = dtype; J->Lt = Lt; J->x = x; J->B = B; J->gamma = gamma; J->V = V;
    J->out_tokens = out_tokens; J->out_n = out_n; J->out_argmax = out_argmax;
    J->out_flags = out_flags;
    J->b0 = (int)((long long)B * t / nthreads);
    J->b1 = (int)((long long)B * (t + 1) / nthreads);
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, greedy_worker, &jobs[t]);
  greedy_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  return 0;
}

/* ---------------------------------------------------------------- draft side
 * Draft-token sampling, the step before verification.  [SD-overview] 考点2
 * and 第三章: the token x that verification tests is one the draft model
 * SAMPLED from its own distribution P_draft.  Here each draft row is sampled
 * from its tempered softmax (reading R7 for the temperature) by the same
 * index-order inverse CDF as the bonus token (reading R5), and the row's
 * normaliser is reported with it, so that verification can reuse it:
 *   m = the largest stored logit of the row,
 *   S = sum_v exp((l_v - m) / T),  P_draft[v] = exp((l_v - m) / T) / S.
 * Rows with NaN / +inf / only -inf, or a bad temperature, are invalid
 * (reading R8): token -1, m = S = NaN. */
typedef struct {
  int dtype;
  const void* L;
  const float *u, *temp;
  int B, n, V;
  int32_t* out_tokens;
  double *out_m, *out_S, *out_dist;
  int32_t* out_flags;
  double near_eps;
  int r0, r1; /* rows b * n + i in [r0, r1) */
} draft_job;

static void* draft_worker(void* arg) {
  const draft_job* J = (const draft_job*)arg;
  const int V = J->V;
  double* P = (double*)malloc((size_t)V * sizeof(double));
  for (int r = J->r0; r < J->r1; ++r) {
    const int b = r / J->n;
    const size_t off = (size_t)r * V;
    J->out_tokens[r] = -1;
    J->out_m[r] = J->out_S[r] = NAN;
    if (J->out_dist) J->out_dist[r] = INFINITY;
    if (!P) { J->out_flags[r] = -1; continue; }
    const double T = (double)J->temp[b];
    if (!(isfinite(T) && T >= 0x1p-126)) { /* reading R7 */
      J->out_flags[r] = SVO_INVALID_TEMP;
      continue;
    }
#if SVO_MUTANT == 11
    const double Ts = 1.0; /* planted: the draft sample ignores the temperature */
#else
    const double Ts = T;
#endif
    if (!softmax_row(J->L, J->dtype, off, V, Ts, P)) {
      J->out_flags[r] = SVO_INVALID_NONFINITE;
      continue;
    }
    /* the normaliser, from its definition */
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
      const double l = load_logit(J->L, J->dtype, off + (size_t)v);
      if (l > m) m = l;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += exp((load_logit(J->L, J->dtype, off + (size_t)v) - m) / T);
    double Z = 0.0;
    for (int v = 0; v < V; ++v) Z += P[v];
    int near = 0;
    double dist = INFINITY;
    J->out_tokens[r] = inverse_cdf(P, V, Z, (double)J->u[r], J->near_eps, &near, &dist);
    J->out_m[r] = m;
    J->out_S[r] = S;
    if (J->out_dist) J->out_dist[r] = dist;
    J->out_flags[r] = near ? SVO_NEAR_SAMPLE : 0;
  }
  free(P);
  return NULL;
}

/* Draft-sampling oracle.  L [B][n][V] (fp32 or bf16 bits), u [B][n] in
 * [0, 1), temp [B].  Outputs [B][n]: out_tokens, out_m, out_S, out_flags
 * (SVO_* bits), out_dist optional (distance of u to the nearer CDF edge of
 * the chosen token).  Returns 0, or -1 on a bad argument. */
int svo_draft_sample(int dtype, const void* L, const float* u, const float* temp, int B, int n,
                     int V, int32_t* out_tokens, double* out_m, double* out_S,
                     double* out_dist, int32_t* out_flags, double near_eps, int nthreads) {
  if (B < 0 || n < 0 || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16)) return -1;
  const int rows = B * n;
  if (rows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > rows) nthreads = rows;
  draft_job* jobs = (draft_job*)calloc((size_t)nthreads, sizeof(draft_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    draft_job* J = &jobs[t];
    J->dtype = dtype; J->L = L; J->u = u; J->temp = temp;
    J->B = B; J->n = n; J->V = V;
    J->out_tokens = out_tokens; J->out_m = out_m; J->out_S = out_S; J->out_dist = out_dist;
    J->out_flags = out_flags;
    J->near_eps = near_eps;
    J->r0 = (int)((long long)rows * t / nthreads);
    J->r1 = (int)((long long)rows * (t + 1) / nthreads);
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, draft_worker, &jobs[t]);
  draft_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  for (int r = 0; r < rows; ++r)
    if (out_flags[r] < 0) return -2;
  return 0;
}

/* Build-identity hook for the mutation tests. */
int svo_mutant_id(void) { return SVO_MUTANT; }

/* ---------------------------------------------------------------- token tree
 * Token-tree (multi-branch) verification.  The pages name candidate token
 * trees ([Deferred-SD], opening section: the draft "emits a candidate token
 * tree" into the proposal queue; [SD-overview] 考点3: tree attention checks
 * several branches in one forward pass) but give no acceptance rule for
 * sibling drafts.  Readings:
 *   T1  the rejection rule of 考点2 applied to the siblings of a node in
 *       index order, the target distribution replaced after every rejected
 *       sibling by the residual of 考点2 -- the multi-draft form of the same
 *       rejection sampling, lossless when the siblings were drawn
 *       independently from the node's draft distribution.  At node n:
 *       r = P_t[n]; for each child c of n, with token x = tokens[c] and
 *       Q = P_d[n]: accept iff u_acc[c] <= min(1, r(x) / Q(x)) (Q(x) = 0
 *       accepts, reading R2); an accepted child is emitted and the walk
 *       moves to it; a rejected one replaces r by
 *       max(0, r - Q) / sum_v max(0, r - Q).  When no child is accepted (or
 *       n is a leaf) one token is drawn from r by the inverse CDF of reading
 *       R5 with u_res[n] and the walk ends.  A residual that vanishes is
 *       replaced by P_t[n] (reading R6, flagged).
 *   T2  only the rows the walk reads decide validity: the target row of
 *       every node it visits and the draft row of every visited node that
 *       has children.  NaN / +inf in one of them, or one that is all -inf,
 *       makes the request invalid (reading R8); rows off the walk are never
 *       read.
 *   T3  layout: nodes 0..N-1 per request, node 0 the root (parent -1),
 *       0 <= parent[n] < n otherwise, so a node's children follow it; the
 *       children of n are the nodes naming n as parent, in index order.
 *       target row n = the target distribution after the path to n; draft
 *       row n = the distribution n's children were drawn from.  A malformed
 *       parent array or a token outside [0, V) makes the request invalid.
 * Arrays: Lt, Ld [B][N][V]; parent, tokens, u_acc, u_res [B][N] (entry 0 of
 * tokens and u_acc unused); temp [B].  Outputs: out_tokens [B][N] (tokens of
 * the accepted nodes, then the drawn token, then -1), out_n [B] (accepted
 * nodes), out_nodes [B][N] (the accepted nodes, then -1; may be NULL),
 * out_flags [B] (SVO_* bits).
 * The loop applies the definition one residual at a time; no closed form of
 * the repeated residual is used. */
typedef struct {
  int dtype;
  const void *Lt, *Ld;
  const int32_t *parent, *tokens;
  const float *u_acc, *u_res, *temp;
  int B, N, V;
  int32_t *out_tokens, *out_n, *out_nodes, *out_flags;
  double near_eps;
  int b0, b1;
} tree_job;

static void tree_request(const tree_job* J, int b, double* P, double* Q, double* r, double* w) {
  const int N = J->N, V = J->V;
  int32_t* tok = J->out_tokens + (size_t)b * N;
  int32_t* nodes = J->out_nodes ? J->out_nodes + (size_t)b * N : NULL;
  const int32_t* par = J->parent + (size_t)b * N;
  const int32_t* xt = J->tokens + (size_t)b * N;
  int32_t flags = 0;
  for (int i = 0; i < N; ++i) {
    tok[i] = -1;
    if (nodes) nodes[i] = -1;
  }
  J->out_n[b] = 0;
  const double T = (double)J->temp[b];
  if (!(isfinite(T) && T >= 0x1p-126)) flags |= SVO_INVALID_TEMP;
  if (par[0] != -1) flags |= SVO_INVALID_TOKEN;
  for (int n = 1; n < N; ++n)
    if (par[n] < 0 || par[n] >= n || xt[n] < 0 || xt[n] >= V) flags |= SVO_INVALID_TOKEN;
  if (flags) {
    J->out_flags[b] = flags;
    return;
  }
  int n = 0, k = 0;
  int32_t emitted[SVO_TREE_MAX_N], path[SVO_TREE_MAX_N];
  for (;;) {
    int has_child = 0;
    for (int c = n + 1; c < N; ++c) has_child |= (par[c] == n);
    if (!softmax_row(J->Lt, J->dtype, ((size_t)b * N + n) * V, V, T, P) ||
        (has_child && !softmax_row(J->Ld, J->dtype, ((size_t)b * N + n) * V, V, T, Q))) {
      J->out_flags[b] = flags | SVO_INVALID_NONFINITE; /* reading T2 */
      return;
    }
    for (int v = 0; v < V; ++v) r[v] = P[v];
    int next = -1;
    for (int c = n + 1; c < N && next < 0; ++c) {
      if (par[c] != n) continue;
      const int x = xt[c];
      const double ratio = (Q[x] > 0.0) ? fmin(1.0, r[x] / Q[x]) : 1.0; /* reading R2 */
      const double u = (double)J->u_acc[(size_t)b * N + c];
      if (fabs(u - ratio) < J->near_eps) flags |= SVO_NEAR_ACCEPT;
#if SVO_MUTANT == 16
      const int accept = u <= ((Q[x] > 0.0) ? fmin(1.0, P[x] / Q[x]) : 1.0); /* planted: r unused */
#else
      const int accept = u <= ratio;
#endif
      if (accept) {
        next = c;
        break;
      }
      double Z = 0.0;
      for (int v = 0; v < V; ++v) {
#if SVO_MUTANT == 17
        r[v] = fmax(0.0, P[v] - Q[v]); /* planted: the residual restarts from P_t */
#else
        r[v] = fmax(0.0, r[v] - Q[v]);
#endif
        Z += r[v];
      }
      if (!(Z > 0.0)) { /* reading R6 */
        flags |= SVO_DEGENERATE;
        for (int v = 0; v < V; ++v) r[v] = P[v];
      } else {
        for (int v = 0; v < V; ++v) r[v] /= Z;
      }
    }
    if (next < 0) {
      double Z = 0.0;
      for (int v = 0; v < V; ++v) {
        w[v] = r[v];
        Z += w[v];
      }
      int near = 0;
      double dist = INFINITY;
      emitted[k] = inverse_cdf(w, V, Z, (double)J->u_res[(size_t)b * N + n], J->near_eps, &near,
                               &dist);
      if (near) flags |= SVO_NEAR_SAMPLE;
      break;
    }
    emitted[k] = xt[next];
    path[k] = next;
    ++k;
    n = next;
  }
  for (int i = 0; i <= k; ++i) tok[i] = emitted[i];
  if (nodes)
    for (int i = 0; i < k; ++i) nodes[i] = path[i];
  J->out_n[b] = k;
  J->out_flags[b] = flags;
}

static void* tree_worker(void* arg) {
  const tree_job* J = (const tree_job*)arg;
  const size_t V = (size_t)J->V;
  double* P = (double*)malloc(V * sizeof(double));
  double* Q = (double*)malloc(V * sizeof(double));
  double* r = (double*)malloc(V * sizeof(double));
  double* w = (double*)malloc(V * sizeof(double));
  for (int b = J->b0; b < J->b1; ++b) {
    if (!P || !Q || !r || !w)
      J->out_flags[b] = -1;
    else
      tree_request(J, b, P, Q, r, w);
  }
  free(P);
  free(Q);
  free(r);
  free(w);
  return NULL;
}

/* Token-tree verification (readings T1-T3 above).  Returns 0, -1 on a bad
 * argument (N outside [1, SVO_TREE_MAX_N]), -2 when out of memory. */
int svo_tree_verify(int dtype, const void* Lt, const void* Ld, const int32_t* parent,
                    const int32_t* tokens, const float* u_acc, const float* u_res,
                    const float* temp, int B, int N, int V, int32_t* out_tokens, int32_t* out_n,
                    int32_t* out_nodes, int32_t* out_flags, double near_eps, int nthreads) {
  if (B < 0 || N < 1 || N > SVO_TREE_MAX_N || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16))
    return -1;
  if (B == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > B) nthreads = B;
  tree_job* jobs = (tree_job*)calloc((size_t)nthreads, sizeof(tree_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -2;
  }
  for (int t = 0; t < nthreads; ++t) {
    tree_job* J = &jobs[t];
    J->dtype = dtype;
    J->Lt = Lt;
    J->Ld = Ld;
    J->parent = parent;
    J->tokens = tokens;
    J->u_acc = u_acc;
    J->u_res = u_res;
    J->temp = temp;
    J->B = B;
    J->N = N;
    J->V = V;
    J->out_tokens = out_tokens;
    J->out_n = out_n;
    J->out_nodes = out_nodes;
    J->out_flags = out_flags;
    J->near_eps = near_eps;
    J->b0 = (int)((long long)B * t / nthreads);
    J->b1 = (int)((long long)B * (t + 1) / nthreads);
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, tree_worker, &jobs[t]);
  tree_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  for (int b = 0; b < B; ++b)
    if (out_flags[b] < 0) return -2;
  return 0;
}
