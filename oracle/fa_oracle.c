/*
 * CPU oracle for the flash-attention backward over a raw K/V cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA
 * path.
 *
 * What it computes (plain definition, double precision), following the
 * FLASH_ATTN_BACK operator described in "CUDA: FLASH_ATTN_BACK kernels"
 * (CambrianTech/llama.cpp pull request 63, review of the first revision:
 * the math of the q and kv kernels), with the GQA map, additive mask,
 * fully-masked-row rule and causal tail given there and in its perf cases:
 *
 *   hk      = h / (H / Hkv)                                   (GQA map)
 *   allowed = (mask absent or mask[h % Hm][i][j] != -inf)
 *             and (not causal or j <= M - N + i)              (causal tail)
 *   s_ij    = scale * sum_c Q[i,h,c] * K^[j,hk,c] + mask[h % Hm][i][j]
 *   lse_ih  = log sum_{allowed j} exp(s_ij)   (-inf if no j is allowed)
 *   p_ij    = exp(s_ij - lse_ih)   (0 if not allowed or lse = -inf)
 *   dP_ij   = sum_c dO[i,h,c] * V^[j,hk,c]
 *   delta_ih= sum_j p_ij * dP_ij   (equals rowsum(dO o O) without forming O)
 *   dS_ij   = p_ij * (dP_ij - delta_ih)
 *   dQ[i,h] = scale * sum_j dS_ij * K^[j,hk]
 *   dK[j,hk]= scale * sum_{h in group(hk)} sum_i dS_ij * Q[i,h]
 *   dV[j,hk]= sum_{h in group(hk)} sum_i p_ij * dO[i,h]
 *
 * The forward output, for oracle_fa_forward (the attention the backward
 * differentiates; 0 for a row without an allowed key):
 *
 *   O[i,h]  = sum_j p_ij * V^[j,hk]
 *
 * Extensions (oracle_fa_back_ext).  The pages exclude these and define none,
 * so the definitions are the common ones, each optional:
 *   soft-capping, c > 0:  s_ij = c * tanh(scale * q_i . k^_j / c) + mask
 *                          (the cap applies to the scaled product only), and
 *                          dS_ij = p_ij (dP_ij - delta_ih) (1 - tanh^2(.))
 *                          since ds/d(scale q.k) = 1 - tanh^2
 *   ALiBi slope m_h:       s_ij += m_h * (j - (M - N + i))   (query i sits
 *                          at position M - N + i, as in the causal tail)
 *   sink logit sigma_h:    e^sigma_h joins the softmax denominator:
 *                          lse_ih = log(e^sigma_h + sum_allowed e^s_ij)
 *                          (finite even without an allowed key); the sink
 *                          has no value, so delta and dS keep their form;
 *                          dsigma_h = -sum_i e^(sigma_h - lse_ih) delta_ih
 *
 * K^ and V^ are the cache rows decoded exactly as the block formats define
 * them (a q8_0 block: binary16 scale d, then 32 int8 codes, value code*d;
 * a q4_0 block: binary16 scale d, then 16 bytes whose low nibble is element
 * b and high nibble element b+16, value (nibble-8)*d; the q4_0 layout is the
 * one the raw-cache forward kernel in torad-labs/llama.cpp pull request 71
 * reads).  Binary16 is decoded from its IEEE 754 bit fields here.
 *
 * Layouts: Q, dO, dQ [N][H][D]; K, V, dK, dV [M][Hkv][D]; lse, delta [N][H];
 * mask element (j, i, hm) at (hm*N + i)*M + j.
 *
 * Evaluation order: rows of one KV head are taken 32 at a time so each key
 * row is read once per group, and the per-row dot products are run side by
 * side.  Every dot product and every sum is still formed term by term in
 * the order of the definition above (c = 0..D-1, j = 0..M-1, rows in
 * (i, h) order), so the result equals the one-row-at-a-time loop.  The
 * softmax takes two passes over j: max and sum first, then the rest.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OT_F32 = 0, OT_F16 = 1, OT_Q8_0 = 2, OT_Q4_0 = 3 };
#define RB 32 /* rows (or keys) evaluated side by side */

double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

long oracle_row_bytes(int type, int D) {
  switch (type) {
    case OT_F32: return 4L * D;
    case OT_F16: return 2L * D;
    case OT_Q8_0: return (D % 32) ? -1 : (D / 32) * 34L;
    case OT_Q4_0: return (D % 32) ? -1 : (D / 32) * 18L;
  }
  return -1;
}

static void decode_row(const uint8_t* row, int type, int D, double* out) {
  if (type == OT_F32) {
    for (int c = 0; c < D; ++c) {
      float f;
      memcpy(&f, row + 4 * c, 4);
      out[c] = (double)f;
    }
  } else if (type == OT_F16) {
    for (int c = 0; c < D; ++c) out[c] = oracle_half_to_double((uint16_t)(row[2 * c] | (row[2 * c + 1] << 8)));
  } else if (type == OT_Q8_0) {
    for (int b = 0; b < D / 32; ++b) {
      const uint8_t* blk = row + 34 * b;
      double d = oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
      for (int t = 0; t < 32; ++t) out[32 * b + t] = (double)(int8_t)blk[2 + t] * d;
    }
  } else { /* OT_Q4_0 */
    for (int b = 0; b < D / 32; ++b) {
      const uint8_t* blk = row + 18 * b;
      double d = oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
      for (int t = 0; t < 16; ++t) {
        int lo = blk[2 + t] & 15, hi = blk[2 + t] >> 4;
        out[32 * b + t] = (double)(lo - 8) * d;
        out[32 * b + t + 16] = (double)(hi - 8) * d;
      }
    }
  }
}

int oracle_dequant(const uint8_t* raw, int type, int64_t nrows, int D, double* out) {
  long rb = oracle_row_bytes(type, D);
  if (rb <= 0) return 1;
  for (int64_t r = 0; r < nrows; ++r) decode_row(raw + r * rb, type, D, out + r * (int64_t)D);
  return 0;
}

typedef struct {
  /* problem */
  const double *Qd, *dOd, *Kh, *Vh; /* Q [N][H][D], dO [N][H][Dv], K^ [M][Hkv][D], V^ [M][Hkv][Dv] */
  const uint16_t* mask;
  int Hm, N, M, H, Hkv, D, Dv, G, causal;
  double scale;
  /* selection */
  const int64_t* dq_index; /* [N]: position in the dQ output or -1 */
  const int64_t* keys;
  int nkeys;
  /* extensions (all optional) */
  const double* alibi; /* [H] slopes, or NULL */
  double softcap;      /* c > 0, or 0 */
  const double* sinks; /* [H] sink logits, or NULL */
  /* outputs */
  double *lse, *delta, *dQ, *dK, *dV;
  double* O; /* [N][H][Dv] forward output, or NULL */
  /* scheduling */
  int phase, nitems;
  int next;
  pthread_mutex_t mu;
  int err;
} Job;

/* mask value for (row i, key j, head h); 0 without a mask */
static double mask_at(const Job* J, int i, int j, int h) {
  if (!J->mask) return 0.0;
  int hm = h % J->Hm;
  return oracle_half_to_double(J->mask[((int64_t)hm * J->N + i) * J->M + j]);
}

static int is_allowed(const Job* J, int i, int j, double mval) {
  if (J->causal && (int64_t)j > (int64_t)J->M - J->N + i) return 0;
  if (J->mask && isinf(mval) && mval < 0) return 0;
  return 1;
}

/* Phase 1: for a group of RB rows r = i*G + g of KV head hk, form s and dP for
 * every key, then lse, delta and (for selected i) dQ row by row. */
/* The logit from the scaled product: soft-capping, then the mask and the ALiBi bias.  *fac is
 * d(logit)/d(scaled product): 1 - tanh^2 under the cap, else 1. */
static double logit_of(const Job* J, double raw, double mv, int i, int j, int h, double* fac) {
  double s = raw;
  *fac = 1.0;
  if (J->softcap > 0.0) {
    const double t = tanh(raw / J->softcap);
    s = J->softcap * t;
    *fac = 1.0 - t * t;
  }
  s += mv;
  if (J->alibi) s += J->alibi[h] * ((double)j - ((double)J->M - J->N + i));
  return s;
}

static void phase1_item(Job* J, int item, double* S, double* DP, double* qt, double* dot, double* F) {
  const int G = J->G, D = J->D, Dv = J->Dv, M = J->M, N = J->N, H = J->H, Hkv = J->Hkv;
  const int rows_per_hk = N * G;
  const int nblk = (rows_per_hk + RB - 1) / RB;
  const int hk = item / nblk, r0 = (item % nblk) * RB;
  int nr = rows_per_hk - r0;
  if (nr > RB) nr = RB;
  /* gather Q and dO of the group's rows, transposed so the RB dot products run side by side */
  for (int c = 0; c < D; ++c)
    for (int r = 0; r < RB; ++r) {
      double x = 0.0;
      if (r < nr) {
        int rr = r0 + r, i = rr / G, h = hk * G + rr % G;
        x = J->Qd[((int64_t)i * H + h) * D + c];
      }
      qt[(int64_t)c * RB + r] = x;
    }
  for (int c = 0; c < Dv; ++c)
    for (int r = 0; r < RB; ++r) {
      double x = 0.0;
      if (r < nr) {
        int rr = r0 + r, i = rr / G, h = hk * G + rr % G;
        x = J->dOd[((int64_t)i * H + h) * Dv + c];
      }
      dot[(int64_t)c * RB + r] = x; /* dO^T */
    }
  const double* dOt = dot;
  for (int j = 0; j < M; ++j) {
    const double* k = J->Kh + ((int64_t)j * Hkv + hk) * D;
    const double* v = J->Vh + ((int64_t)j * Hkv + hk) * Dv;
    double acc[RB], acc2[RB];
    for (int r = 0; r < RB; ++r) acc[r] = 0.0, acc2[r] = 0.0;
    for (int c = 0; c < D; ++c) {
      const double kc = k[c];
      const double* qc = qt + (int64_t)c * RB;
      for (int r = 0; r < RB; ++r) acc[r] += qc[r] * kc;
    }
    for (int c = 0; c < Dv; ++c) {
      const double vc = v[c];
      const double* oc = dOt + (int64_t)c * RB;
      for (int r = 0; r < RB; ++r) acc2[r] += oc[r] * vc;
    }
    for (int r = 0; r < nr; ++r) {
      S[(int64_t)r * M + j] = J->scale * acc[r];
      DP[(int64_t)r * M + j] = acc2[r];
    }
  }
  for (int r = 0; r < nr; ++r) {
    const int rr = r0 + r, i = rr / G, h = hk * G + rr % G;
    double* s = S + (int64_t)r * M;
    const double* dp = DP + (int64_t)r * M;
    double* fac = F + (int64_t)r * M;
    /* the logits (cap, mask, bias); keys that are not allowed are marked with -inf */
    double mx = -INFINITY;
    int any = 0;
    for (int j = 0; j < M; ++j) {
      double mv = mask_at(J, i, j, h);
      if (!is_allowed(J, i, j, mv)) {
        s[j] = -INFINITY;
        continue;
      }
      s[j] = logit_of(J, s[j], mv, i, j, h, &fac[j]);
      if (!any || s[j] > mx) mx = s[j];
      any = 1;
    }
    const int64_t o = (int64_t)i * H + h;
    int64_t qi = J->dq_index ? J->dq_index[i] : -1;
    const double sink = J->sinks ? J->sinks[h] : -INFINITY;
    if (!any && !J->sinks) {
      J->lse[o] = -INFINITY;
      J->delta[o] = 0.0;
      if (qi >= 0) memset(J->dQ + (qi * H + h) * (int64_t)D, 0, sizeof(double) * D);
      if (J->O) memset(J->O + o * Dv, 0, sizeof(double) * Dv);
      continue;
    }
    if (J->sinks && (!any || sink > mx)) mx = sink;
    double sum = 0.0;
    for (int j = 0; j < M; ++j)
      if (s[j] != -INFINITY) sum += exp(s[j] - mx);
    if (J->sinks) sum += exp(sink - mx);
    const double lse = mx + log(sum);
    double delta = 0.0;
    for (int j = 0; j < M; ++j)
      if (s[j] != -INFINITY) delta += exp(s[j] - lse) * dp[j];
    J->lse[o] = lse;
    J->delta[o] = delta;
    if (J->O) {
      double* out = J->O + o * Dv;
      for (int c = 0; c < Dv; ++c) out[c] = 0.0;
      for (int j = 0; j < M; ++j) {
        if (s[j] == -INFINITY) continue;
        const double p = exp(s[j] - lse);
        const double* v = J->Vh + ((int64_t)j * Hkv + (h / G)) * Dv;
        for (int c = 0; c < Dv; ++c) out[c] += p * v[c];
      }
    }
    if (qi >= 0) {
      double* out = J->dQ + (qi * H + h) * (int64_t)D;
      for (int c = 0; c < D; ++c) out[c] = 0.0;
      for (int j = 0; j < M; ++j) {
        if (s[j] == -INFINITY) continue;
        const double p = exp(s[j] - lse);
        const double ds = p * (dp[j] - delta) * fac[j];
        const double* k = J->Kh + ((int64_t)j * Hkv + (h / G)) * D;
        for (int c = 0; c < D; ++c) out[c] += ds * k[c];
      }
      for (int c = 0; c < D; ++c) out[c] *= J->scale;
    }
  }
}

/* Phase 2: for a group of RB selected keys of KV head hk, sum dS*Q and p*dO over
 * every (i, h in group) row. */
static void phase2_item(Job* J, int item, double* kt, double* vt) {
  const int G = J->G, D = J->D, Dv = J->Dv, N = J->N, H = J->H, Hkv = J->Hkv;
  const int nblk = (J->nkeys + RB - 1) / RB;
  const int hk = item / nblk, k0 = (item % nblk) * RB;
  int nk = J->nkeys - k0;
  if (nk > RB) nk = RB;
  for (int c = 0; c < D; ++c)
    for (int t = 0; t < RB; ++t)
      kt[(int64_t)c * RB + t] = t < nk ? J->Kh[((int64_t)J->keys[k0 + t] * Hkv + hk) * D + c] : 0.0;
  for (int c = 0; c < Dv; ++c)
    for (int t = 0; t < RB; ++t)
      vt[(int64_t)c * RB + t] = t < nk ? J->Vh[((int64_t)J->keys[k0 + t] * Hkv + hk) * Dv + c] : 0.0;
  for (int t = 0; t < nk; ++t) {
    int64_t ko = ((int64_t)(k0 + t) * Hkv + hk);
    memset(J->dK + ko * D, 0, sizeof(double) * D);
    memset(J->dV + ko * Dv, 0, sizeof(double) * Dv);
  }
  for (int i = 0; i < N; ++i)
    for (int g = 0; g < G; ++g) {
      const int h = hk * G + g;
      const int64_t o = (int64_t)i * H + h;
      const double lse = J->lse[o];
      if (lse == -INFINITY) continue;
      const double* q = J->Qd + o * D;
      const double* d = J->dOd + o * Dv;
      double acc[RB], acc2[RB];
      for (int t = 0; t < RB; ++t) acc[t] = 0.0, acc2[t] = 0.0;
      for (int c = 0; c < D; ++c) {
        const double qc = q[c];
        const double* kc = kt + (int64_t)c * RB;
        for (int t = 0; t < RB; ++t) acc[t] += qc * kc[t];
      }
      for (int c = 0; c < Dv; ++c) {
        const double oc = d[c];
        const double* vc = vt + (int64_t)c * RB;
        for (int t = 0; t < RB; ++t) acc2[t] += oc * vc[t];
      }
      for (int t = 0; t < nk; ++t) {
        const int j = (int)J->keys[k0 + t];
        const double mv = mask_at(J, i, j, h);
        if (!is_allowed(J, i, j, mv)) continue;
        double fac;
        const double s = logit_of(J, J->scale * acc[t], mv, i, j, h, &fac);
        const double p = exp(s - lse);
        const double ds = p * (acc2[t] - J->delta[o]) * fac;
        const int64_t ko = ((int64_t)(k0 + t) * Hkv + hk);
        double* dk = J->dK + ko * D;
        double* dv = J->dV + ko * Dv;
        for (int c = 0; c < D; ++c) dk[c] += J->scale * ds * q[c];
        for (int c = 0; c < Dv; ++c) dv[c] += p * d[c];
      }
    }
}

static void* worker(void* arg) {
  Job* J = (Job*)arg;
  const int RBmax = RB;
  double *S = NULL, *DP = NULL, *F = NULL, *bufA = NULL, *bufB = NULL;
  int64_t dmax = J->D > J->Dv ? J->D : J->Dv;
  bufA = (double*)malloc(sizeof(double) * dmax * RBmax);
  bufB = (double*)malloc(sizeof(double) * dmax * RBmax);
  if (J->phase == 1) {
    S = (double*)malloc(sizeof(double) * ((int64_t)RBmax * J->M + 1));
    DP = (double*)malloc(sizeof(double) * ((int64_t)RBmax * J->M + 1));
    F = (double*)malloc(sizeof(double) * ((int64_t)RBmax * J->M + 1));
  }
  if (!bufA || !bufB || (J->phase == 1 && (!S || !DP || !F))) {
    pthread_mutex_lock(&J->mu);
    J->err = 2;
    pthread_mutex_unlock(&J->mu);
  } else {
    for (;;) {
      pthread_mutex_lock(&J->mu);
      int it = J->next++;
      pthread_mutex_unlock(&J->mu);
      if (it >= J->nitems) break;
      if (J->phase == 1)
        phase1_item(J, it, S, DP, bufA, bufB, F);
      else
        phase2_item(J, it, bufA, bufB);
    }
  }
  free(S);
  free(DP);
  free(F);
  free(bufA);
  free(bufB);
  return NULL;
}

static int run_phase(Job* J, int nthreads) {
  J->next = 0;
  if (nthreads > J->nitems) nthreads = J->nitems;
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
  if (!th) return 2;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, worker, J) != 0) break;
    ++started;
  }
  if (started == 0) worker(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  return J->err;
}

int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Full or sampled backward.
 *   dq_rows  : query positions i whose dQ rows (all H heads) are produced, or NULL for all N
 *   dkv_keys : key positions j whose dK/dV rows (all Hkv heads) are produced, or NULL for all M
 * lse and delta are always produced for every (i, h).
 * Outputs: lse, delta [N][H]; dQ [n_dq][H][D]; dK [n_keys][Hkv][D]; dV [n_keys][Hkv][Dv].
 * Returns 0 on success, 1 on a bad argument, 2 when memory runs out.
 */
static int run_oracle(const float* q, const uint8_t* k, int k_type, const uint8_t* v, int v_type,
                      const uint16_t* mask, int mask_heads, const float* dO, double scale, int N, int M, int H,
                      int Hkv, int D, int Dv, int causal, const int64_t* dq_rows, int n_dq_rows,
                      const int64_t* dkv_keys, int n_dkv_keys, double* lse, double* delta, double* dQ, double* dK,
                      double* dV, double* O, const double* alibi, double softcap, const double* sinks,
                      double* dsinks, int nthreads) {
  if (!q || !k || !v || !dO || !lse || !delta) return 1;
  if (!(softcap >= 0.0) || isinf(softcap)) return 1;
  if (N < 0 || M < 0 || H <= 0 || Hkv <= 0 || D <= 0 || Dv <= 0 || H % Hkv) return 1;
  if (mask && mask_heads != 1 && mask_heads != H) return 1;
  if (oracle_row_bytes(k_type, D) <= 0 || oracle_row_bytes(v_type, Dv) <= 0) return 1;
  if (nthreads <= 0) nthreads = oracle_default_threads();
  Job J;
  memset(&J, 0, sizeof(J));
  pthread_mutex_init(&J.mu, NULL);
  J.N = N, J.M = M, J.H = H, J.Hkv = Hkv, J.D = D, J.Dv = Dv, J.G = H / Hkv, J.causal = causal;
  J.scale = scale, J.mask = mask, J.Hm = mask ? mask_heads : 1;
  J.lse = lse, J.delta = delta, J.dQ = dQ, J.dK = dK, J.dV = dV, J.O = O;
  J.alibi = alibi, J.softcap = softcap, J.sinks = sinks;
  int rc = 0;
  double* Qd = (double*)malloc(sizeof(double) * ((int64_t)N * H * D + 1));
  double* dOd = (double*)malloc(sizeof(double) * ((int64_t)N * H * Dv + 1));
  double* Kh = (double*)malloc(sizeof(double) * ((int64_t)M * Hkv * D + 1));
  double* Vh = (double*)malloc(sizeof(double) * ((int64_t)M * Hkv * Dv + 1));
  int64_t* dq_index = (int64_t*)malloc(sizeof(int64_t) * (N + 1));
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * ((dkv_keys ? n_dkv_keys : M) + 1));
  if (!Qd || !dOd || !Kh || !Vh || !dq_index || !keys) {
    rc = 2;
    goto done;
  }
  for (int64_t x = 0; x < (int64_t)N * H * D; ++x) Qd[x] = (double)q[x];
  for (int64_t x = 0; x < (int64_t)N * H * Dv; ++x) dOd[x] = (double)dO[x];
  oracle_dequant(k, k_type, (int64_t)M * Hkv, D, Kh);
  oracle_dequant(v, v_type, (int64_t)M * Hkv, Dv, Vh);
  for (int i = 0; i < N; ++i) dq_index[i] = dq_rows ? -1 : i;
  if (dq_rows) {
    for (int t = 0; t < n_dq_rows; ++t) {
      if (dq_rows[t] < 0 || dq_rows[t] >= N) {
        rc = 1;
        goto done;
      }
      dq_index[dq_rows[t]] = t;
    }
  }
  if (!dQ) {
    for (int i = 0; i < N; ++i) dq_index[i] = -1;
  }
  J.nkeys = dkv_keys ? n_dkv_keys : M;
  for (int t = 0; t < J.nkeys; ++t) {
    keys[t] = dkv_keys ? dkv_keys[t] : t;
    if (keys[t] < 0 || keys[t] >= M) {
      rc = 1;
      goto done;
    }
  }
  J.Qd = Qd, J.dOd = dOd, J.Kh = Kh, J.Vh = Vh, J.dq_index = dq_index, J.keys = keys;
  if (N > 0) {
    J.phase = 1;
    J.nitems = Hkv * ((N * J.G + RB - 1) / RB);
    rc = run_phase(&J, nthreads);
    if (rc) goto done;
  }
  /* the sink logits' gradient, rows in order: dsigma_h = -sum_i e^(sigma_h - lse_ih) delta_ih */
  if (sinks && dsinks) {
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int i = 0; i < N; ++i) {
        const int64_t o = (int64_t)i * H + h;
        acc -= exp(sinks[h] - lse[o]) * delta[o];
      }
      dsinks[h] = acc;
    }
  }
  if (dK && dV && J.nkeys > 0) {
    J.phase = 2;
    J.nitems = Hkv * ((J.nkeys + RB - 1) / RB);
    rc = run_phase(&J, nthreads);
  }
done:
  free(Qd);
  free(dOd);
  free(Kh);
  free(Vh);
  free(dq_index);
  free(keys);
  pthread_mutex_destroy(&J.mu);
  return rc;
}

int oracle_fa_back(const float* q, const uint8_t* k, int k_type, const uint8_t* v, int v_type,
                   const uint16_t* mask, int mask_heads, const float* dO, double scale, int N, int M, int H,
                   int Hkv, int D, int Dv, int causal, const int64_t* dq_rows, int n_dq_rows,
                   const int64_t* dkv_keys, int n_dkv_keys, double* lse, double* delta, double* dQ, double* dK,
                   double* dV, int nthreads) {
  return run_oracle(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dq_rows,
                    n_dq_rows, dkv_keys, n_dkv_keys, lse, delta, dQ, dK, dV, NULL, NULL, 0.0, NULL, NULL, nthreads);
}

/*
 * oracle_fa_back with the extensions of the header comment: alibi [H] slopes or NULL, softcap
 * c > 0 or 0, sinks [H] logits or NULL, and dsinks [H] (written when sinks and dsinks are given).
 */
int oracle_fa_back_ext(const float* q, const uint8_t* k, int k_type, const uint8_t* v, int v_type,
                       const uint16_t* mask, int mask_heads, const float* dO, double scale, int N, int M, int H,
                       int Hkv, int D, int Dv, int causal, const int64_t* dq_rows, int n_dq_rows,
                       const int64_t* dkv_keys, int n_dkv_keys, double* lse, double* delta, double* dQ, double* dK,
                       double* dV, const double* alibi, double softcap, const double* sinks, double* dsinks,
                       int nthreads) {
  return run_oracle(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal, dq_rows,
                    n_dq_rows, dkv_keys, n_dkv_keys, lse, delta, dQ, dK, dV, NULL, alibi, softcap, sinks, dsinks,
                    nthreads);
}

/*
 * Forward: lse [N][H] and O [N][H][Dv] of the same attention (no gradients).  The backward's
 * first phase is run with a zero dO, whose delta is discarded.  Same return codes.
 */
int oracle_fa_forward(const float* q, const uint8_t* k, int k_type, const uint8_t* v, int v_type,
                      const uint16_t* mask, int mask_heads, double scale, int N, int M, int H, int Hkv, int D,
                      int Dv, int causal, double* lse, double* O, int nthreads) {
  if (!lse || !O || N < 0 || H <= 0 || Dv <= 0) return 1;
  float* dO = (float*)calloc((size_t)N * H * Dv + 1, sizeof(float));
  double* delta = (double*)malloc(sizeof(double) * ((size_t)N * H + 1));
  int rc = (!dO || !delta) ? 2
                           : run_oracle(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv,
                                        causal, NULL, 0, NULL, 0, lse, delta, NULL, NULL, NULL, O, NULL, 0.0, NULL,
                                        NULL, nthreads);
  free(dO);
  free(delta);
  return rc;
}
