/*
 * oracle.c — plain, slow, fp64 CPU oracle for the speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file;
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares no
 * code, header, table or constant with the CUDA library: it restates the method from the
 * pages, in their order, one request at a time, in double precision.
 *
 * Sources (cited as host + section of the page):
 *   cf-1.com/news/5155685  §2.1  the draft guesses, the target checks, roll back to the first wrong position
 *   cf-1.com/news/5155685  §2.2  accept x with probability min(1, p(x)/q(x)); on rejection resample
 *                                from norm(max(0, p(x) - q(x))); the result is distributed as p
 *   2kiu.com/news/5895634  §2.2  the same rule, written with (p(x) - q(x))_+
 *   gsyq.cn/news/428210    §3.1  one target forward gives the K positions' logits; judge position by
 *                                position; keep the accepted part and start drafting again
 *   gsyq.cn/news/428210    §3.2  E = 1 + a + ... + a^K: the target emits one token beyond the accepted
 *                                drafts, which is the bonus token when all K are accepted
 *   gsyq.cn/news/428210    §3.3  temperature, top-k and top-p are sampling parameters that draft and
 *                                target must share
 *   2kiu.com/news/5895634  §7    the draft may sample at its own, lower temperature
 *
 * Readings taken where the pages are silent (each is also listed in the design notes):
 *   - temperature divides the logits of both p and q (q may have its own draft temperature);
 *     top-k keeps every logit >= the k-th largest (ties kept, flagged), on the raw logits;
 *   - top-p (nucleus) comes after temperature and top-k: it keeps the smallest set of most likely
 *     tokens whose mass reaches top_p, every token tied with the last one included, and
 *     renormalises; top_p >= 1 is off;
 *   - accept iff u * q(x) < p(x)  (strict; q(x) = 0 accepts iff p(x) > 0);
 *   - the inverse CDF runs in ascending token id with the strict rule u * R < C_v;
 *   - n_acc counts accepted drafts; one more token (resampled or bonus) is always emitted;
 *   - T == 0 is the greedy limit: accept iff x == argmax p (lowest index on ties).
 *
 * Pins (tests, not in this file): exhaustive breakpoint enumeration of the decision at V = 4,
 * K <= 3 (exact output law == p); chi-square over 1e6 seeded trials; the mean emitted count
 * against (1 - a^(K+1)) / (1 - a) on inputs with exactly known a; softmax against a library
 * softmax; top-k against a library top-k; greedy against a library argmax.
 * Parity unpinned (conventions fixed by reading, not by the pages): the top-k tie rule, the CDF
 * order, the uniform grid.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_DTYPE_F32 0
#define OR_DTYPE_BF16 1

#define OR_FLAG_RESIDUAL_ZERO 1   /* R == 0 after rounding: resampled from p instead   */
#define OR_FLAG_CDF_CLAMP 2       /* u * R beyond the last cumulative value (rounding) */
#define OR_FLAG_BAD_TOKEN 4       /* a draft token outside [0, V)                      */
#define OR_FLAG_BAD_K 8           /* k_per_row outside [0, K_max]                      */
#define OR_FLAG_NONFINITE 16      /* NaN / +inf logit, or nothing left to sample from  */
#define OR_FLAG_TOPK_TIE 32       /* top-k kept more than k logits because of ties     */

/* One logit as an exact double.  bf16 is the upper half of an IEEE binary32. */
static double logit_at(const void* base, int dtype, size_t i) {
  if (dtype == OR_DTYPE_F32) return (double)((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int cmp_desc(const void* a, const void* b) {
  double x = *(const double*)a, y = *(const double*)b;
  return (x < y) - (x > y);
}

/* (logit, token) pairs ordered by logit, descending; equal logits by token id. */
typedef struct {
  double z;
  int v;
} zv_t;

static int cmp_zv_desc(const void* a, const void* b) {
  const zv_t* x = (const zv_t*)a;
  const zv_t* y = (const zv_t*)b;
  if (x->z != y->z) return (x->z < y->z) - (x->z > y->z);
  return (x->v > y->v) - (x->v < y->v);
}

/*
 * Distribution of one row (gsyq.cn §3.3: temperature, top-k and top-p; 2kiu.com §7: a draft row
 * takes the draft's own temperature, passed here as T).
 *   z: V logits; T > 0; top_k: 0 or >= V means no truncation; top_p in (0, 1], >= 1 means off.
 *   P_out: V doubles, the normalised probabilities.
 *   info_out (nullable, 6 doubles): [0] m = max kept logit, [1] log-normaliser m/T + ln sum_v w_v
 *       over the kept set, [2] top-k threshold t (-inf when off), [3] kept count, [4] top-p
 *       threshold t_p (-inf when off), [5] nucleus margin: the distance of top_p to the nearer of
 *       the two cumulative masses around the cut, the mass before the first group (exactly 0)
 *       left out (inf when off).
 *   cut: NaN = find the nucleus as above.  Otherwise the nucleus cut is given instead of found
 *       (the parity tests pass the cut the CUDA library chose, once they have checked that it is a
 *       valid one): the row keeps, inside its top-k set, every logit >= cut and is renormalised,
 *       which is the nucleus's last step with t_p = cut; info_out[4] = cut, info_out[5] = NaN.
 * Returns OR_FLAG_NONFINITE if the row holds NaN or +inf or keeps nothing finite,
 * OR_FLAG_TOPK_TIE if ties made the top-k set larger than k.
 */
int oracle_row_dist_at(const void* z, int dtype, int V, double T, int top_k, double top_p, double cut,
                       double* P_out, double* info_out) {
  int flags = 0;
  double t = -INFINITY;
  double info[6] = {NAN, NAN, NAN, NAN, -INFINITY, INFINITY};
  for (int v = 0; v < V; ++v) {
    double x = logit_at(z, dtype, (size_t)v);
    if (isnan(x) || (isinf(x) && x > 0)) flags |= OR_FLAG_NONFINITE;
  }
  if (flags) {
    for (int v = 0; v < V; ++v) P_out[v] = NAN;
    info[4] = info[5] = NAN;
    if (info_out) memcpy(info_out, info, sizeof info);
    return flags;
  }
  if (top_k > 0 && top_k < V) {
    /* t = the k-th largest logit, counted with multiplicity (a library sort as the step). */
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    for (int v = 0; v < V; ++v) s[v] = logit_at(z, dtype, (size_t)v);
    qsort(s, (size_t)V, sizeof(double), cmp_desc);
    t = s[top_k - 1];
    free(s);
  }
  double m = -INFINITY;
  int kept = 0;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(z, dtype, (size_t)v);
    if (x >= t) {
      ++kept;
      if (x > m) m = x;
    }
  }
  if (top_k > 0 && top_k < V && kept > top_k) flags |= OR_FLAG_TOPK_TIE;
  info[0] = m;
  info[2] = t;
  info[3] = kept;
  if (!(m > -INFINITY)) { /* every kept logit is -inf: nothing to sample from */
    for (int v = 0; v < V; ++v) P_out[v] = NAN;
    if (info_out) memcpy(info_out, info, sizeof info);
    return flags | OR_FLAG_NONFINITE;
  }
  double sum = 0.0;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(z, dtype, (size_t)v);
    double w = (x >= t) ? exp((x - m) / T) : 0.0;
    P_out[v] = w;
    sum += w;
  }
  for (int v = 0; v < V; ++v) P_out[v] /= sum;
  info[1] = m / T + log(sum);

  if (!isnan(cut)) {
    /* a given cut: keep the logits >= cut inside the top-k set and renormalise */
    double wsum = 0.0, mass = 0.0;
    int nk = 0;
    for (int v = 0; v < V; ++v) {
      if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) >= cut) {
        mass += P_out[v];
        wsum += exp((logit_at(z, dtype, (size_t)v) - m) / T);
        ++nk;
      } else {
        P_out[v] = 0.0;
      }
    }
    if (!(mass > 0.0)) { /* the cut lies above every kept logit: nothing to sample from */
      for (int v = 0; v < V; ++v) P_out[v] = NAN;
      info[4] = cut;
      info[5] = NAN;
      if (info_out) memcpy(info_out, info, sizeof info);
      return flags | OR_FLAG_NONFINITE;
    }
    for (int v = 0; v < V; ++v) P_out[v] = P_out[v] / mass;
    info[1] = m / T + log(wsum);
    info[3] = nk;
    info[4] = cut;
    info[5] = NAN;
  } else if (top_p < 1.0) {
    /* Nucleus: walk the kept tokens from the most likely down (a library sort as the step),
       one group of equal logits at a time, until the mass taken reaches top_p; the group that
       reaches it is kept whole. */
    zv_t* o = (zv_t*)malloc(sizeof(zv_t) * (size_t)V);
    int n = 0;
    for (int v = 0; v < V; ++v)
      if (P_out[v] > 0.0) {
        o[n].z = logit_at(z, dtype, (size_t)v);
        o[n].v = v;
        ++n;
      }
    qsort(o, (size_t)n, sizeof(zv_t), cmp_zv_desc);
    double taken = 0.0, tp = o[n - 1].z, margin = 0.0;
    for (int i = 0; i < n;) {
      double g = 0.0;
      int j = i;
      while (j < n && o[j].z == o[i].z) g += P_out[o[j++].v];
      if (taken + g >= top_p) {
        tp = o[i].z;
        /* before the first group the mass taken is exactly 0: only the far side can move */
        margin = taken > 0.0 ? fmin(top_p - taken, taken + g - top_p) : taken + g - top_p;
        break;
      }
      taken += g;
      i = j;
    }
    free(o);
    /* keep z >= t_p and renormalise; the normaliser of the kept weights follows */
    double wsum = 0.0, mass = 0.0;
    int nk = 0;
    for (int v = 0; v < V; ++v) {
      if (P_out[v] > 0.0 && logit_at(z, dtype, (size_t)v) >= tp) {
        mass += P_out[v];
        wsum += exp((logit_at(z, dtype, (size_t)v) - m) / T);
        ++nk;
      } else {
        P_out[v] = 0.0;
      }
    }
    for (int v = 0; v < V; ++v) P_out[v] /= mass;
    info[1] = m / T + log(wsum);
    info[3] = nk;
    info[4] = tp;
    info[5] = margin;
  }
  if (info_out) memcpy(info_out, info, sizeof info);
  return flags;
}

/* The row's distribution with its nucleus found (oracle_row_dist_at with a NaN cut). */
int oracle_row_dist_ex(const void* z, int dtype, int V, double T, int top_k, double top_p,
                       double* P_out, double* info_out) {
  return oracle_row_dist_at(z, dtype, V, T, top_k, top_p, NAN, P_out, info_out);
}

/* The same without top-p; info_out (nullable) gets the first four entries. */
int oracle_row_dist(const void* z, int dtype, int V, double T, int top_k, double* P_out,
                    double* info_out) {
  double info[6];
  int f = oracle_row_dist_ex(z, dtype, V, T, top_k, 1.0, P_out, info);
  if (info_out) memcpy(info_out, info, 4 * sizeof(double));
  return f;
}

/*
 * Inverse-CDF draw from the non-negative weights r[0..V) with total R, in ascending token id:
 * y = the smallest v with u * R < C_v, C_v = r_0 + ... + r_v.  If rounding leaves no such v,
 * y = the last v with r_v > 0 and OR_FLAG_CDF_CLAMP is returned.  *margin = the distance of u
 * to the nearer edge of y's interval, min(u - C_{y-1}/R, C_y/R - u).
 */
static int inverse_cdf(const double* r, int V, double R, double u, int32_t* y, double* margin) {
  double target = u * R, C = 0.0;
  for (int v = 0; v < V; ++v) {
    double prev = C;
    C += r[v];
    if (target < C) {
      double lo = u - prev / R, hi = C / R - u;
      *y = v;
      *margin = lo < hi ? lo : hi;
      return 0;
    }
  }
  *y = -1;
  for (int v = V - 1; v >= 0; --v)
    if (r[v] > 0.0) {
      *y = v;
      break;
    }
  *margin = 0.0;
  return OR_FLAG_CDF_CLAMP;
}

/*
 * The decision for one request, on its normalised distributions (cf-1.com §2.2, 2kiu.com §2.2,
 * cf-1.com §2.1, gsyq.cn §3.1-§3.2).
 *   P: (K+1) rows of V doubles, p at positions 0..K (row K is the bonus position);
 *   Q: K rows of V doubles;  x: K draft tokens;  ua: K accept uniforms;  ur: resample uniform
 *   (uniforms in [0, 1), taken as doubles so a test can place them anywhere on the real line).
 *   out_tokens: K+1 entries (x_0..x_{n-1}, y, then -1);  *n_acc: accepted drafts.
 *   p_draft, q_draft, accept_margin: K entries each (NaN past the first rejection);
 *   sample_margin, residual_mass: scalars.  work: V doubles of scratch.
 * Returns the request's flags.
 */
int oracle_decide(const double* P, const double* Q, int V, int K, const int32_t* x,
                  const double* ua, double ur, int32_t* out_tokens, int32_t* n_acc, double* p_draft,
                  double* q_draft, double* accept_margin, double* sample_margin,
                  double* residual_mass, double* work) {
  int flags = 0;
  for (int j = 0; j <= K; ++j) out_tokens[j] = -1;
  for (int j = 0; j < K; ++j) p_draft[j] = q_draft[j] = accept_margin[j] = NAN;

  /* Acceptance, position by position, stopping at the first rejection. */
  int jstar = K;
  for (int j = 0; j < K; ++j) {
    double a = 0.0, c = 0.0;
    if (x[j] < 0 || x[j] >= V)
      flags |= OR_FLAG_BAD_TOKEN; /* p(x) = q(x) = 0: never accepted */
    else {
      a = P[(size_t)j * V + x[j]];
      c = Q[(size_t)j * V + x[j]];
    }
    double u = ua[j];
    p_draft[j] = a;
    q_draft[j] = c;
    accept_margin[j] = (c > 0.0) ? fabs(u - a / c) : INFINITY;
    if (u * c < a) { /* u < p/q, with q = 0 accepting iff p > 0 */
      out_tokens[j] = x[j];
      continue;
    }
    jstar = j;
    break;
  }
  *n_acc = jstar;

  const double* Pj = P + (size_t)jstar * V;
  double R = 0.0;
  if (jstar < K) {
    /* Residual max(0, p - q) at the first rejected position. */
    const double* Qj = Q + (size_t)jstar * V;
    for (int v = 0; v < V; ++v) {
      double d = Pj[v] - Qj[v];
      work[v] = d > 0.0 ? d : 0.0;
      R += work[v];
    }
    *residual_mass = R;
    if (!(R > 0.0)) { /* only reachable through rounding: fall back to p */
      flags |= OR_FLAG_RESIDUAL_ZERO;
      R = 0.0;
      for (int v = 0; v < V; ++v) {
        work[v] = Pj[v];
        R += work[v];
      }
    }
  } else {
    /* Every draft accepted: the bonus token from p at position K. */
    for (int v = 0; v < V; ++v) {
      work[v] = Pj[v];
      R += work[v];
    }
    *residual_mass = 0.0;
  }
  flags |= inverse_cdf(work, V, R, ur, &out_tokens[jstar], sample_margin);
  return flags;
}

/* Greedy limit (T == 0): g = argmax with the lowest index on ties.  -1 if the row has NaN. */
static int32_t argmax_row(const void* z, int dtype, int V, int* flags) {
  int32_t g = -1;
  double best = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double x = logit_at(z, dtype, (size_t)v);
    if (isnan(x)) {
      *flags |= OR_FLAG_NONFINITE;
      return -1;
    }
    if (g < 0 || x > best) {
      best = x;
      g = v;
    }
  }
  return g;
}

/*
 * The whole verify step over a batch, with the same argument meaning as the CUDA library's
 * spec_verify, on host arrays.  Layout: p [B, K_max+1, V], q [B, K_max, V] (dtype), draft [B, K_max],
 * k_per_row [B] (NULL = K_max for all), ua [B, K_max], ur [B].
 * Outputs (all host, all required): out_tokens [B, K_max+1], out_n_acc [B], p_draft / q_draft /
 * accept_margin [B, K_max], sample_margin / residual_mass [B], row_lognorm [B, 2*K_max+1]
 * (p rows 0..K_max, then q rows 0..K_max-1; NaN where unused), flags [B].
 * Sampling parameters: temperature (T_p of the target; 0 = greedy), draft_temperature (T_q of the
 * draft rows, > 0 unless greedy, where it is not used), top_k, top_p (in (0, 1]; 1 = off).
 * row_nucleus_margin (nullable) [B, 2*K_max+1]: each row's nucleus margin (inf when top-p is off,
 * NaN where unused).
 * row_cut_out (nullable) [B, 2*K_max+1]: each row's smallest kept logit bound, the larger of the
 * top-k threshold and the nucleus cut (-inf when neither is on; NaN where unused and in greedy mode).
 * row_cut_in (nullable) [B, 2*K_max+1]: per row, NaN = find the nucleus; a value = take it as the
 * nucleus cut (oracle_row_dist_at).  oracle_verify_ex is this call with both NULL.
 * A request whose rows are non-finite gets n_acc = 0 and tokens -1 (its result is unspecified).
 * nthreads > 1 runs requests in parallel (OpenMP); the result does not depend on it.
 */
int oracle_verify_cuts(const void* p, const void* q, const int32_t* draft, const int32_t* k_per_row,
                     const float* ua, const float* ur, float temperature, float draft_temperature,
                     int top_k, float top_p, int32_t* out_tokens, int32_t* out_n_acc, double* p_draft,
                     double* q_draft, double* accept_margin, double* sample_margin,
                     double* residual_mass, double* row_lognorm, double* row_nucleus_margin,
                       const double* row_cut_in, double* row_cut_out,
                     int32_t* out_flags, int B, int K_max, int V, int dtype, int nthreads) {
  if (B < 0 || K_max < 0 || K_max > 64 || V <= 0 || !(temperature >= 0.0f) || top_k < 0) return 1;
  if (temperature > 0.0f && !(draft_temperature > 0.0f)) return 1;
  if (!(top_p > 0.0f)) return 1;
  if (nthreads < 1) nthreads = 1;
  const int rows_lognorm = 2 * K_max + 1;
  const size_t es = dtype == OR_DTYPE_F32 ? 4 : 2;
  const double T = (double)temperature, Tq = (double)draft_temperature, tp = (double)top_p;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int b = 0; b < B; ++b) {
    int flags = 0;
    int K = k_per_row ? k_per_row[b] : K_max;
    if (K < 0 || K > K_max) {
      flags |= OR_FLAG_BAD_K;
      K = K < 0 ? 0 : K_max;
    }
    const char* pb = (const char*)p + (size_t)b * (K_max + 1) * V * es;
    const char* qb = q ? (const char*)q + (size_t)b * K_max * V * es : NULL;
    const int32_t* xb = draft + (size_t)b * K_max;
    const float* uab = ua ? ua + (size_t)b * K_max : NULL;
    int32_t* tok = out_tokens + (size_t)b * (K_max + 1);
    double* pd = p_draft + (size_t)b * K_max;
    double* qd = q_draft + (size_t)b * K_max;
    double* am = accept_margin + (size_t)b * K_max;
    double* ln = row_lognorm + (size_t)b * rows_lognorm;
    for (int j = 0; j <= K_max; ++j) tok[j] = -1;
    for (int j = 0; j < K_max; ++j) pd[j] = qd[j] = am[j] = NAN;
    double* nm = row_nucleus_margin ? row_nucleus_margin + (size_t)b * rows_lognorm : NULL;
    double* co = row_cut_out ? row_cut_out + (size_t)b * rows_lognorm : NULL;
    const double* ci = row_cut_in ? row_cut_in + (size_t)b * rows_lognorm : NULL;
    for (int r = 0; r < rows_lognorm; ++r) ln[r] = NAN;
    if (nm)
      for (int r = 0; r < rows_lognorm; ++r) nm[r] = NAN;
    if (co)
      for (int r = 0; r < rows_lognorm; ++r) co[r] = NAN;
    sample_margin[b] = NAN;
    residual_mass[b] = NAN;

    if (temperature == 0.0f) {
      /* Greedy: accept while the draft equals the target's argmax.  Every row 0..K is examined
         (so a NaN anywhere in the request is flagged), then the decision is taken. */
      int32_t g[64 + 1];
      for (int j = 0; j <= K; ++j) g[j] = argmax_row(pb + (size_t)j * V * es, dtype, V, &flags);
      int n = K;
      for (int j = 0; j <= K; ++j) {
        if (j == K) {
          tok[j] = g[j];
          break;
        }
        if (xb[j] < 0 || xb[j] >= V) flags |= OR_FLAG_BAD_TOKEN;
        if (xb[j] == g[j]) {
          tok[j] = xb[j];
          continue;
        }
        tok[j] = g[j];
        n = j;
        break;
      }
      sample_margin[b] = INFINITY;
      residual_mass[b] = 0.0;
      if (flags & OR_FLAG_NONFINITE) {
        for (int j = 0; j <= K_max; ++j) tok[j] = -1;
        n = 0;
      }
      out_n_acc[b] = n;
      out_flags[b] = flags;
      continue;
    }

    double uad[64];
    for (int j = 0; j < K; ++j) uad[j] = uab ? (double)uab[j] : 0.0;
    double* Pr = (double*)malloc(sizeof(double) * (size_t)(K + 1) * V);
    double* Qr = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * V);
    double* work = (double*)malloc(sizeof(double) * (size_t)V);
    double info[6];
    for (int j = 0; j <= K; ++j) {
      const double cp = ci ? ci[j] : NAN;
      flags |= oracle_row_dist_at(pb + (size_t)j * V * es, dtype, V, T, top_k, tp, cp, Pr + (size_t)j * V, info);
      ln[j] = info[1];
      if (nm) nm[j] = info[5];
      if (co) co[j] = info[4] > info[2] ? info[4] : info[2];
    }
    for (int j = 0; j < K; ++j) {
      const double cq = ci ? ci[K_max + 1 + j] : NAN;
      flags |= oracle_row_dist_at(qb + (size_t)j * V * es, dtype, V, Tq, top_k, tp, cq, Qr + (size_t)j * V, info);
      ln[K_max + 1 + j] = info[1];
      if (nm) nm[K_max + 1 + j] = info[5];
      if (co) co[K_max + 1 + j] = info[4] > info[2] ? info[4] : info[2];
    }
    int32_t n = 0;
    if (flags & OR_FLAG_NONFINITE) {
      for (int j = 0; j <= K_max; ++j) tok[j] = -1;
    } else {
      flags |= oracle_decide(Pr, Qr, V, K, xb, uad, (double)ur[b], tok, &n, pd, qd, am, &sample_margin[b],
                             &residual_mass[b], work);
    }
    out_n_acc[b] = n;
    out_flags[b] = flags;
    free(Pr);
    free(Qr);
    free(work);
  }
  return 0;
}

/* The whole verify step with every nucleus found by the oracle itself. */
int oracle_verify_ex(const void* p, const void* q, const int32_t* draft, const int32_t* k_per_row,
                     const float* ua, const float* ur, float temperature, float draft_temperature,
                     int top_k, float top_p, int32_t* out_tokens, int32_t* out_n_acc, double* p_draft,
                     double* q_draft, double* accept_margin, double* sample_margin,
                     double* residual_mass, double* row_lognorm, double* row_nucleus_margin,
                     int32_t* out_flags, int B, int K_max, int V, int dtype, int nthreads) {
  return oracle_verify_cuts(p, q, draft, k_per_row, ua, ur, temperature, draft_temperature, top_k, top_p,
                            out_tokens, out_n_acc, p_draft, q_draft, accept_margin, sample_margin,
                            residual_mass, row_lognorm, row_nucleus_margin, NULL, NULL, out_flags, B, K_max,
                            V, dtype, nthreads);
}

/* The verify step with one temperature for both sides and no top-p. */
int oracle_verify(const void* p, const void* q, const int32_t* draft, const int32_t* k_per_row,
                  const float* ua, const float* ur, float temperature, int top_k, int32_t* out_tokens,
                  int32_t* out_n_acc, double* p_draft, double* q_draft, double* accept_margin,
                  double* sample_margin, double* residual_mass, double* row_lognorm,
                  int32_t* out_flags, int B, int K_max, int V, int dtype, int nthreads) {
  return oracle_verify_ex(p, q, draft, k_per_row, ua, ur, temperature, temperature, top_k, 1.0f,
                          out_tokens, out_n_acc, p_draft, q_draft, accept_margin, sample_margin,
                          residual_mass, row_lognorm, NULL, out_flags, B, K_max, V, dtype, nthreads);
}

/*
 * Multi-draft verify: several drafts propose at once (2kiu.com §7 and cf-1.com §2.3 name ensembles
 * of draft models, the target keeping the draft it accepts).  The pages fix the property the step
 * must keep -- the emitted tokens are distributed as p (cf-1.com §2.2, 2kiu.com §2.2) -- but no rule
 * for several candidates, so the rule here applies the single-draft rule to the candidates in turn,
 * each against what the earlier rejections leave of p:
 *   r_0 = P_0, the target's distribution at the first position (the drafts share the prefix);
 *   candidate n, the first token x_n of chain n drawn from its draft distribution Q_n, is
 *     accepted iff u_n * Q_n(x_n) < r_n(x_n); a rejection leaves r_{n+1} = norm(max(0, r_n - Q_n));
 *   the first accepted candidate's chain is verified on from its second position with the
 *     single-draft rule (oracle_decide) on its own target and draft distributions;
 *   if every candidate is rejected, one token is drawn from r_N by the inverse CDF with ur.
 * Each candidate's step leaves the law of what follows equal to r_n (the single-draft argument), so
 * the first emitted token is distributed as P_0, and with N = 1 this is oracle_decide.
 *   P: [N, K+1, V] (row 0 of chain 0 is P_0; rows 1..K of chain n are its target distributions
 *      along its own prefix); Q: [N, K, V]; x, ua: [N, K]; ur: the resample uniform.
 *   out_tokens [K+1], *n_acc, *chain (the accepted chain, -1 when every candidate is rejected),
 *   accept_margin [N, K]: |u - r/q| of every test taken (inf when q = 0), NaN elsewhere;
 *   *sample_margin as in oracle_decide.  work: 2 V doubles.  Returns the request's flags.
 */
int oracle_decide_multi(const double* P, const double* Q, int V, int N, int K, const int32_t* x,
                        const double* ua, double ur, int32_t* out_tokens, int32_t* n_acc, int32_t* chain,
                        double* accept_margin, double* sample_margin, double* work) {
  int flags = 0;
  for (int j = 0; j <= K; ++j) out_tokens[j] = -1;
  for (int i = 0; i < N * K; ++i) accept_margin[i] = NAN;
  *chain = -1;
  *n_acc = 0;
  double* r = work;
  double* rest = work + V;
  for (int v = 0; v < V; ++v) r[v] = P[v];  /* r_0 = P_0 */
  if (K == 0) { /* no drafts: the one token is drawn from P_0 */
    double R = 0.0;
    for (int v = 0; v < V; ++v) R += r[v];
    return inverse_cdf(r, V, R, ur, &out_tokens[0], sample_margin);
  }
  int acc = -1;
  for (int n = 0; n < N && acc < 0; ++n) {
    const double* Qn = Q + (size_t)n * K * V;
    const int32_t xn = x[(size_t)n * K];
    double a = 0.0, c = 0.0;
    if (xn < 0 || xn >= V)
      flags |= OR_FLAG_BAD_TOKEN;
    else {
      a = r[xn];
      c = Qn[xn];
    }
    const double u = ua[(size_t)n * K];
    accept_margin[(size_t)n * K] = (c > 0.0) ? fabs(u - a / c) : INFINITY;
    if (u * c < a) {
      acc = n;
      break;
    }
    /* rejected: what is left of r after candidate n */
    double R = 0.0;
    for (int v = 0; v < V; ++v) {
      const double d = r[v] - Qn[v];
      rest[v] = d > 0.0 ? d : 0.0;
      R += rest[v];
    }
    if (R > 0.0)
      for (int v = 0; v < V; ++v) r[v] = rest[v] / R;
    else /* only reachable through rounding: r is kept */
      flags |= OR_FLAG_RESIDUAL_ZERO;
  }
  if (acc < 0) { /* every candidate rejected: one token from r_N */
    double R = 0.0;
    for (int v = 0; v < V; ++v) R += r[v];
    return flags | inverse_cdf(r, V, R, ur, &out_tokens[0], sample_margin);
  }
  *chain = acc;
  out_tokens[0] = x[(size_t)acc * K];
  /* the accepted chain from its second position: the single-draft rule on its own rows */
  const int K1 = K - 1;
  double pd[64], qd[64], rm;
  int32_t n1 = 0;
  flags |= oracle_decide(P + ((size_t)acc * (K + 1) + 1) * V, Q + ((size_t)acc * K + 1) * V, V, K1,
                         x + (size_t)acc * K + 1, ua + (size_t)acc * K + 1, ur, out_tokens + 1, &n1, pd, qd,
                         accept_margin + (size_t)acc * K + 1, sample_margin, &rm, rest);
  *n_acc = 1 + n1;
  return flags;
}

/*
 * The multi-draft step over a batch, with the argument meaning of the CUDA library's
 * spec_verify_multi, on host arrays: p [B, N, K+1, V], q [B, N, K, V] (dtype), draft, ua [B, N, K],
 * ur [B]; temperature T of the target rows (0 = greedy), draft_temperature of the q rows.  Row 0 of
 * chain 0 of every request is the shared first position (row 0 of the other chains is not read).
 * Outputs: out_tokens [B, K+1], out_n_acc [B], out_chain [B], accept_margin [B, N, K],
 * sample_margin [B], out_flags [B].  Greedy: the first chain whose first draft is the argmax of
 * P_0 (lowest index on ties) is followed with the greedy rule; none -> the argmax is emitted.
 */
int oracle_verify_multi(const void* p, const void* q, const int32_t* draft, const float* ua, const float* ur,
                        float temperature, float draft_temperature, int32_t* out_tokens, int32_t* out_n_acc,
                        int32_t* out_chain, double* accept_margin, double* sample_margin, int32_t* out_flags,
                        int B, int N, int K, int V, int dtype, int nthreads) {
  if (B < 0 || N < 1 || N > 16 || K < 0 || K > 64 || V <= 0 || !(temperature >= 0.0f)) return 1;
  if (temperature > 0.0f && !(draft_temperature > 0.0f)) return 1;
  if (nthreads < 1) nthreads = 1;
  const size_t es = dtype == OR_DTYPE_F32 ? 4 : 2;
  const double T = (double)temperature, Tq = (double)draft_temperature;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int b = 0; b < B; ++b) {
    int flags = 0;
    const char* pb = (const char*)p + (size_t)b * N * (K + 1) * V * es;
    const char* qb = q ? (const char*)q + (size_t)b * N * K * V * es : NULL;
    const int32_t* xb = draft + (size_t)b * N * K;
    int32_t* tok = out_tokens + (size_t)b * (K + 1);
    double* am = accept_margin + (size_t)b * N * K;
    for (int j = 0; j <= K; ++j) tok[j] = -1;
    for (int i = 0; i < N * K; ++i) am[i] = NAN;
    sample_margin[b] = NAN;
    out_chain[b] = -1;
    out_n_acc[b] = 0;
    if (temperature == 0.0f) {
      /* every row the step reads is examined, so a NaN anywhere in the request is flagged */
      int32_t gr[16 * 65];
      for (int n = 0; n < N; ++n)
        for (int j = (n == 0 ? 0 : 1); j <= K; ++j)
          gr[n * (K + 1) + j] = argmax_row(pb + ((size_t)n * (K + 1) + j) * V * es, dtype, V, &flags);
      const int32_t g = gr[0];
      int acc = -1;
      for (int n = 0; n < N && K > 0 && acc < 0; ++n) {
        if (xb[(size_t)n * K] < 0 || xb[(size_t)n * K] >= V) flags |= OR_FLAG_BAD_TOKEN;
        if (xb[(size_t)n * K] == g) acc = n;
      }
      int nacc = 0;
      if (acc < 0) {
        tok[0] = g;
      } else {
        tok[0] = g;
        nacc = 1;
        for (int j = 1; j <= K; ++j) {
          const int32_t gj = gr[acc * (K + 1) + j];
          if (j == K) {
            tok[j] = gj;
            break;
          }
          const int32_t xj = xb[(size_t)acc * K + j];
          if (xj < 0 || xj >= V) flags |= OR_FLAG_BAD_TOKEN;
          tok[j] = gj;
          if (xj != gj) break;
          ++nacc;
        }
      }
      if (flags & OR_FLAG_NONFINITE) {
        for (int j = 0; j <= K; ++j) tok[j] = -1;
        nacc = 0;
        acc = -1;
      }
      sample_margin[b] = INFINITY;
      out_chain[b] = acc;
      out_n_acc[b] = nacc;
      out_flags[b] = flags;
      continue;
    }
    double* Pr = (double*)malloc(sizeof(double) * (size_t)N * (K + 1) * V);
    double* Qr = (double*)malloc(sizeof(double) * (size_t)N * (K > 0 ? K : 1) * V);
    double* work = (double*)malloc(sizeof(double) * 2 * (size_t)V);
    double* uad = (double*)malloc(sizeof(double) * (size_t)N * (K > 0 ? K : 1));
    for (int n = 0; n < N; ++n) {
      for (int j = 0; j <= K; ++j) {
        double* dst = Pr + ((size_t)n * (K + 1) + j) * V;
        if (j == 0 && n > 0) { /* the shared first position: chain 0's row */
          memcpy(dst, Pr, sizeof(double) * (size_t)V);
          continue;
        }
        flags |= oracle_row_dist(pb + ((size_t)n * (K + 1) + j) * V * es, dtype, V, T, 0, dst, NULL);
      }
      for (int j = 0; j < K; ++j)
        flags |= oracle_row_dist(qb + ((size_t)n * K + j) * V * es, dtype, V, Tq, 0, Qr + ((size_t)n * K + j) * V, NULL);
      for (int j = 0; j < K; ++j) uad[(size_t)n * K + j] = ua ? (double)ua[((size_t)b * N + n) * K + j] : 0.0;
    }
    if (!(flags & OR_FLAG_NONFINITE)) {
      int32_t nacc = 0, ch = -1;
      flags |= oracle_decide_multi(Pr, Qr, V, N, K, xb, uad, (double)ur[b], tok, &nacc, &ch, am,
                                   &sample_margin[b], work);
      out_n_acc[b] = nacc;
      out_chain[b] = ch;
    }
    out_flags[b] = flags;
    free(Pr);
    free(Qr);
    free(work);
    free(uad);
  }
  return 0;
}

/*
 * Many independent trials of oracle_decide on one shared pair of distributions (the pins'
 * chi-square and Monte-Carlo checks): P [(K+1), V], Q [K, V]; x, ua [N, K]; ur [N].
 * Outputs out_tokens [N, K+1], out_n_acc [N], out_flags [N].
 */
int oracle_decide_trials(const double* P, const double* Q, int V, int K, int N, const int32_t* x,
                         const float* ua, const float* ur, int32_t* out_tokens, int32_t* out_n_acc,
                         int32_t* out_flags, int nthreads) {
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* work = (double*)malloc(sizeof(double) * (size_t)V);
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(4 * (K > 0 ? K : 1)));
    double sm, rm;
#pragma omp for schedule(static)
    for (int i = 0; i < N; ++i) {
      double* uad = scratch + 3 * K;
      for (int j = 0; j < K; ++j) uad[j] = (double)ua[(size_t)i * K + j];
      out_flags[i] = oracle_decide(P, Q, V, K, x + (size_t)i * K, uad, (double)ur[i],
                                   out_tokens + (size_t)i * (K + 1), &out_n_acc[i], scratch,
                                   scratch + K, scratch + 2 * K, &sm, &rm, work);
    }
    free(work);
    free(scratch);
  }
  return 0;
}
