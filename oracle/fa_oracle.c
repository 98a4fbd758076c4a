/*
 * Test infrastructure, not product code: a plain, slow fp64 CPU oracle for
 * exact scaled-dot-product attention. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load or call it; the CUDA library never
 * does, and this file shares no code with it.
 *
 * It computes the definition of attention written out, not a tiled
 * algorithm. The pages state that the IO-aware method returns exactly
 * softmax(Q K^T) V, without approximating it ("FlashAttention does more
 * arithmetic to move less data", section "FlashAttention never writes the
 * full score table to HBM"; "FlashAttention and GPU Memory", chapter 01 and
 * chapter 12), so the definition is the oracle.
 *
 * Layout: q, k, v, dO, o, dq, dk, dv are [BH][N][d] row-major doubles; lse
 * and D are [BH][N]. Row i attends to A(i) = {0..N-1}, or {0..i} when causal
 * (the pages name a fused "mask" without defining it; the causal reading
 * j <= i is the plainest one and makes row 0 attend to key 0 only).
 *
 * oracle_fwd_kv is the same forward with Nq query rows against Nk keys
 * (q, o: [BH][Nq][d]; k, v: [BH][Nk][d]; lse: [BH][Nq]). Causal then aligns
 * the queries with the last Nq keys: row i attends to {0..i + Nk - Nq}, so
 * that the last row sees every key, as a decoding step does (the pages list
 * unequal lengths and decode-style attention without defining their mask;
 * this is the reading under which Nq = Nk gives the mask above). Causal needs
 * Nq <= Nk, so that every row sees at least one key.
 *
 * Both _kv functions optionally take per-head sequence lengths sq[h] <= Nq and
 * sk[h] <= Nk (padding masks): head h then has only its first sq[h] query
 * rows and sk[h] keys, with the causal rule above written for those lengths
 * (row i sees keys 0..i + sk - sq). Padding rows get o = 0 and lse = -inf in
 * the forward and dq = 0, D = 0 in the backward; padding keys get dk = dv = 0
 * and are seen by no row.
 *
 * Forward, per head and row i (chapter 08 defines the row max m and the sum
 * of exponentials l that the tiled method carries; here they are taken over
 * the whole row at once):
 *   s_ij = scale * q_i . k_j          (j in A(i))
 *   M_i  = max_j s_ij
 *   l_i  = sum_j exp(s_ij - M_i)
 *   P_ij = exp(s_ij - M_i) / l_i
 *   o_i  = sum_j P_ij v_j
 *   lse_i = M_i + ln l_i              (the natural-log logsumexp of the row)
 *
 * Backward, by the chain rule on the same definition (the pages only say that
 * the backward recomputes the score and probability tiles from Q, K, V and
 * the per-row values the forward kept, chapter 09):
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_{j in A(i)} P_ij dP_ij   (summed explicitly, not as dO_i . o_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dq_i  = scale * sum_j dS_ij k_j
 *   dk_j  = scale * sum_i dS_ij q_i
 *   dv_j  = sum_i P_ij dO_i
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
  for (int t = 0; t < d; ++t) acc += a[t] * b[t];
  return acc;
}

/* Keys visible to query row i of Nq against Nk keys. */
static int row_len_kv(int i, int Nq, int Nk, int causal) { return causal ? i + 1 + (Nk - Nq) : Nk; }

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Scores, max and sum of exponentials for row i of one head. s has room for N. */
static void score_row(const double* qi, const double* k, int n, int d, double scale, double* s, double* M_out,
                      double* l_out) {
  double M = -INFINITY;
  for (int j = 0; j < n; ++j) {
    s[j] = scale * dot(qi, k + (size_t)j * d, d);
    if (s[j] > M) M = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < n; ++j) l += exp(s[j] - M);
  *M_out = M;
  *l_out = l;
}

/*
 * Forward pass, Nq query rows against Nk keys. rows == NULL computes every
 * row; otherwise only the nrows listed rows of every head are written (o rows
 * and lse entries elsewhere are left untouched). Returns 0, or -1 on a bad
 * argument (including causal with Nq > Nk) or allocation failure.
 */
static int bad_lengths(int BH, int Nq, int Nk, int causal, const int* sq, const int* sk) {
  for (int h = 0; h < BH; ++h) {
    const int a = sq ? sq[h] : Nq, b = sk ? sk[h] : Nk;
    if (a < 1 || a > Nq || b < 1 || b > Nk || (causal && a > b)) return 1;
  }
  return 0;
}

int oracle_fwd_kv(const double* q, const double* k, const double* v, double* o, double* lse, int BH, int Nq, int Nk,
                  int d, double scale, int causal, const int* sq, const int* sk, const int* rows, int nrows,
                  int nthreads) {
  if (BH < 1 || Nq < 1 || Nk < 1 || d < 1 || !q || !k || !v || !o || !lse) return -1;
  if (bad_lengths(BH, Nq, Nk, causal, sq, sk)) return -1;
  if (!rows) nrows = Nq;
  for (int r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= Nq) return -1;
  set_threads(nthreads);
  int failed = 0;
  const long long total = (long long)BH * nrows;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long long w = 0; w < total; ++w) {
      if (!s) continue;
      const int h = (int)(w / nrows);
      const int i = rows ? rows[w % nrows] : (int)(w % nrows);
      const double* qi = q + ((size_t)h * Nq + i) * d;
      const double* kh = k + (size_t)h * Nk * d;
      const double* vh = v + (size_t)h * Nk * d;
      const int a = sq ? sq[h] : Nq, b = sk ? sk[h] : Nk;
      double* oi = o + ((size_t)h * Nq + i) * d;
      for (int t = 0; t < d; ++t) oi[t] = 0.0;
      if (i >= a) { /* a padding row */
        lse[(size_t)h * Nq + i] = -INFINITY;
        continue;
      }
      const int n = row_len_kv(i, a, b, causal);
      double M, l;
      score_row(qi, kh, n, d, scale, s, &M, &l);
      for (int j = 0; j < n; ++j) {
        const double p = exp(s[j] - M) / l;
        const double* vj = vh + (size_t)j * d;
        for (int t = 0; t < d; ++t) oi[t] += p * vj[t];
      }
      lse[(size_t)h * Nq + i] = M + log(l);
    }
    free(s);
  }
  return failed ? -1 : 0;
}

/* Forward pass of self-attention (Nq = Nk = N): the listed rows, or all. */
int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse, int BH, int N, int d,
               double scale, int causal, const int* rows, int nrows, int nthreads) {
  return oracle_fwd_kv(q, k, v, o, lse, BH, N, N, d, scale, causal, NULL, NULL, rows, nrows, nthreads);
}

/*
 * Backward pass, Nq query rows against Nk keys (causal: row i sees keys
 * 0..i + Nk - Nq; needs Nq <= Nk). Every row's lse and D are computed (both
 * are needed by every key's gradient). dq is written for the listed query rows
 * (qrows == NULL: all rows), dk and dv for the listed keys (keys == NULL: all
 * keys). D, if non-NULL, receives D_i for every row. Returns 0, or -1 on error.
 */
int oracle_bwd_kv(const double* q, const double* k, const double* v, const double* dO, double* dq, double* dk,
                  double* dv, double* D, int BH, int Nq, int Nk, int d, double scale, int causal, const int* sq,
                  const int* sk, const int* qrows, int nqr, const int* keys, int nkr, int nthreads) {
  if (BH < 1 || Nq < 1 || Nk < 1 || d < 1 || !q || !k || !v || !dO || !dq || !dk || !dv) return -1;
  if (bad_lengths(BH, Nq, Nk, causal, sq, sk)) return -1;
  if (!qrows) nqr = Nq;
  if (!keys) nkr = Nk;
  for (int r = 0; qrows && r < nqr; ++r)
    if (qrows[r] < 0 || qrows[r] >= Nq) return -1;
  for (int r = 0; keys && r < nkr; ++r)
    if (keys[r] < 0 || keys[r] >= Nk) return -1;
  set_threads(nthreads);
  double* lse_all = (double*)malloc(sizeof(double) * (size_t)BH * Nq);
  double* D_all = (double*)malloc(sizeof(double) * (size_t)BH * Nq);
  char* want_q = (char*)calloc((size_t)Nq, 1);
  if (!lse_all || !D_all || !want_q) {
    free(lse_all);
    free(D_all);
    free(want_q);
    return -1;
  }
  for (int r = 0; r < nqr; ++r) want_q[qrows ? qrows[r] : r] = 1;
  int failed = 0;

  /* Pass 1, one query row at a time: P, dP, D and dS of the row; dq. */
  const long long total_rows = (long long)BH * Nq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
    double* dp = (double*)malloc(sizeof(double) * (size_t)Nk);
    if (!s || !dp) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long long w = 0; w < total_rows; ++w) {
      if (!s || !dp) continue;
      const int h = (int)(w / Nq), i = (int)(w % Nq);
      const size_t qb = (size_t)h * Nq * d, kb = (size_t)h * Nk * d;
      const double* qi = q + qb + (size_t)i * d;
      const double* dOi = dO + qb + (size_t)i * d;
      const int a = sq ? sq[h] : Nq, b = sk ? sk[h] : Nk;
      if (i >= a) { /* a padding row: no gradient, and it sees no key */
        lse_all[w] = INFINITY;
        D_all[w] = 0.0;
        if (want_q[i])
          for (int t = 0; t < d; ++t) dq[qb + (size_t)i * d + t] = 0.0;
        continue;
      }
      const int n = row_len_kv(i, a, b, causal);
      double M, l;
      score_row(qi, k + kb, n, d, scale, s, &M, &l);
      double Di = 0.0;
      for (int j = 0; j < n; ++j) {
        s[j] = exp(s[j] - M) / l; /* s now holds P_ij */
        dp[j] = dot(dOi, v + kb + (size_t)j * d, d);
        Di += s[j] * dp[j];
      }
      lse_all[w] = M + log(l);
      D_all[w] = Di;
      if (want_q[i]) {
        double* dqi = dq + qb + (size_t)i * d;
        for (int t = 0; t < d; ++t) dqi[t] = 0.0;
        for (int j = 0; j < n; ++j) {
          const double ds = s[j] * (dp[j] - Di);
          const double* kj = k + kb + (size_t)j * d;
          for (int t = 0; t < d; ++t) dqi[t] += scale * ds * kj[t];
        }
      }
    }
    free(s);
    free(dp);
  }

  /* Pass 2, one key at a time: dk and dv sum over the rows that see key j. */
  const long long total_keys = (long long)BH * nkr;
  if (!failed) {
#pragma omp parallel for schedule(dynamic, 4)
    for (long long w = 0; w < total_keys; ++w) {
      const int h = (int)(w / nkr);
      const int j = keys ? keys[w % nkr] : (int)(w % nkr);
      const size_t qb = (size_t)h * Nq * d, kb = (size_t)h * Nk * d;
      const double* kj = k + kb + (size_t)j * d;
      const double* vj = v + kb + (size_t)j * d;
      double* dkj = dk + kb + (size_t)j * d;
      double* dvj = dv + kb + (size_t)j * d;
      for (int t = 0; t < d; ++t) {
        dkj[t] = 0.0;
        dvj[t] = 0.0;
      }
      const int a = sq ? sq[h] : Nq, b = sk ? sk[h] : Nk, off = b - a;
      if (j >= b) continue; /* a padding key */
      for (int i = causal && j > off ? j - off : 0; i < a; ++i) {
        const double* qi = q + qb + (size_t)i * d;
        const double* dOi = dO + qb + (size_t)i * d;
        const double p = exp(scale * dot(qi, kj, d) - lse_all[(size_t)h * Nq + i]);
        const double ds = p * (dot(dOi, vj, d) - D_all[(size_t)h * Nq + i]);
        for (int t = 0; t < d; ++t) {
          dkj[t] += scale * ds * qi[t];
          dvj[t] += p * dOi[t];
        }
      }
    }
  }
  if (D && !failed) memcpy(D, D_all, sizeof(double) * (size_t)BH * Nq);
  free(lse_all);
  free(D_all);
  free(want_q);
  return failed ? -1 : 0;
}

/* Backward pass of self-attention (Nq = Nk = N). */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dO, double* dq, double* dk,
               double* dv, double* D, int BH, int N, int d, double scale, int causal, const int* qrows, int nq,
               const int* keys, int nk, int nthreads) {
  return oracle_bwd_kv(q, k, v, dO, dq, dk, dv, D, BH, N, N, d, scale, causal, NULL, NULL, qrows, nq, keys, nk,
                       nthreads);
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_max_threads(int nthreads) {
  set_threads(nthreads);
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * 8-bit forward (the FP8 mode of the third version: "FlashAttention does more
 * arithmetic to move less data", the section on the later versions, and
 * "FlashAttention and GPU Memory", chapter 11). The pages say only that the
 * inputs are 8-bit floats and that rounding to them loses precision; the
 * readings taken here:
 *
 *   - q, k, v arrive as E4M3 codes (the OCP 8-bit float: 1 sign bit, 4
 *     exponent bits with bias 7, 3 mantissa bits, subnormals, no infinities,
 *     S.1111.111 = NaN, largest finite 448) with one dequantisation factor per
 *     tensor: q = desc_q * e4m3(q8), and so on;
 *   - the scores, the row maximum and the row sum of exponentials are exact
 *     functions of those values (lse is the exact logsumexp);
 *   - the probabilities feed the second product as E4M3 too (both operands of
 *     an 8-bit product are 8-bit). They are rounded at a per-row power-of-two
 *     scale: with x_ij = s_ij log2(e) and X_i = ceil(max_j x_ij),
 *       w_ij = 2^(x_ij - X_i + 6)          (in (0, 64], so never saturated)
 *       p_ij = rn_e4m3(w_ij)               (round to nearest, ties to even)
 *       o_i  = sum_j p_ij v_j / sum_j w_ij
 *     Because the scale is a power of two, rounding at any other integer
 *     reference gives the same p_ij up to that power of two (away from the
 *     subnormal range), so the result does not depend on the order in which
 *     the keys are visited. With round_p = 0, p_ij = w_ij and o_i is exact.
 */
#define E4M3_MAX 448.0

/* Value of an E4M3 code. */
double oracle_e4m3_decode(int code) {
  const int b = code & 0xFF;
  const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: m/8 * 2^(1 - 7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* x rounded to the nearest E4M3 value (ties to even), saturated at +-448. */
double oracle_e4m3_round(double x) {
  if (isnan(x)) return NAN;
  const double a = fabs(x);
  double r;
  if (a >= E4M3_MAX) {
    r = E4M3_MAX;
  } else if (a < ldexp(1.0, -6)) {
    r = ldexp(nearbyint(ldexp(a, 9)), -9); /* subnormal spacing 2^-9 */
  } else {
    int ex;
    frexp(a, &ex); /* a = f 2^ex, f in [0.5, 1): leading bit 2^(ex - 1) */
    const int q = ex - 1 - 3; /* three mantissa bits: spacing 2^(ex - 4) */
    r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > E4M3_MAX) r = E4M3_MAX;
  }
  return x < 0 ? -r : r;
}

int oracle_fwd_fp8(const unsigned char* q8, const unsigned char* k8, const unsigned char* v8, double desc_q,
                   double desc_k, double desc_v, double* o, double* lse, int BH, int N, int d, double scale,
                   int causal, int round_p, const int* rows, int nrows, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q8 || !k8 || !v8 || !o || !lse) return -1;
  if (!rows) nrows = N;
  for (int r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return -1;
  set_threads(nthreads);
  const double log2e = 1.4426950408889634074;
  int failed = 0;
  const long long total = (long long)BH * nrows;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* qi = (double*)malloc(sizeof(double) * (size_t)d);
    double* kj = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !qi || !kj) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long long w = 0; w < total; ++w) {
      if (!s || !qi || !kj) continue;
      const int h = (int)(w / nrows);
      const int i = rows ? rows[w % nrows] : (int)(w % nrows);
      const unsigned char* qrow = q8 + ((size_t)h * N + i) * d;
      for (int t = 0; t < d; ++t) qi[t] = desc_q * oracle_e4m3_decode(qrow[t]);
      const int n = causal ? i + 1 : N;
      double M = -INFINITY;
      for (int j = 0; j < n; ++j) {
        const unsigned char* krow = k8 + ((size_t)h * N + j) * d;
        for (int t = 0; t < d; ++t) kj[t] = desc_k * oracle_e4m3_decode(krow[t]);
        s[j] = scale * dot(qi, kj, d);
        if (s[j] > M) M = s[j];
      }
      double l = 0.0; /* exact logsumexp */
      for (int j = 0; j < n; ++j) l += exp(s[j] - M);
      lse[(size_t)h * N + i] = M + log(l);
      const double X = ceil(M * log2e);
      double wsum = 0.0;
      double* oi = o + ((size_t)h * N + i) * d;
      for (int t = 0; t < d; ++t) oi[t] = 0.0;
      for (int j = 0; j < n; ++j) {
        const double wj = exp2(s[j] * log2e - X + 6.0);
        const double pj = round_p ? oracle_e4m3_round(wj) : wj;
        wsum += wj;
        const unsigned char* vrow = v8 + ((size_t)h * N + j) * d;
        for (int t = 0; t < d; ++t) oi[t] += pj * desc_v * oracle_e4m3_decode(vrow[t]);
      }
      for (int t = 0; t < d; ++t) oi[t] /= wsum;
    }
    free(s);
    free(qi);
    free(kj);
  }
  return failed ? -1 : 0;
}

/*
 * Dropout ("FlashAttention and GPU Memory", chapter 07: dropout is one of
 * the steps fused into the single kernel; chapter 09: the backward stores no
 * mask, only what is needed to regenerate it). The pages
 * fix neither the generator nor the mask's layout; the readings taken here:
 *
 *   - the generator is Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 *     "Parallel random numbers: as easy as 1, 2, 3", SC 2011), a counter-based
 *     generator: ten rounds of
 *       (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 *     with M0 = 0xD2511F53, M1 = 0xCD9E8D57 and the key (k0, k1) advanced by
 *     (0x9E3779B9, 0xBB67AE85) after every round;
 *   - one call covers a block of 4 queries by 4 keys of one head: counter
 *     (j / 4, i / 4, bh, offset), key (seed mod 2^32, seed / 2^32); output
 *     word i mod 4, byte j mod 4 (bits 8 (j mod 4) .. + 7) is the element's
 *     random byte u;
 *   - the element is kept iff u >= p256, so the dropout probability is
 *     p256 / 256 (p256 in 0 .. 255), and kept elements are scaled by
 *     256 / (256 - p256);
 *   - dropout applies to P after the softmax: lse, m and l are those of the
 *     undropped scores, and o_i = sum_j P_ij Z_ij v_j with Z_ij = keep / (1 - p).
 * The backward, by the chain rule with the mask fixed:
 *   dv_j  = sum_i P_ij Z_ij dO_i
 *   dP_ij = Z_ij (dO_i . v_j)
 *   D_i   = sum_j P_ij dP_ij            (= dO_i . o_i)
 *   dS_ij = P_ij (dP_ij - D_i), dq and dk as without dropout.
 */
void oracle_philox4x32_10(const unsigned int ctr[4], const unsigned int key[2], unsigned int out[4]) {
  unsigned int c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    const unsigned long long p0 = 0xD2511F53ull * c0, p1 = 0xCD9E8D57ull * c2;
    const unsigned int n0 = (unsigned int)(p1 >> 32) ^ c1 ^ k0, n1 = (unsigned int)p1;
    const unsigned int n2 = (unsigned int)(p0 >> 32) ^ c3 ^ k1, n3 = (unsigned int)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The random byte of element (query i, key j) of head bh. */
int oracle_dropout_byte(unsigned long long seed, unsigned int offset, int bh, int i, int j) {
  const unsigned int ctr[4] = {(unsigned int)j >> 2, (unsigned int)i >> 2, (unsigned int)bh, offset};
  const unsigned int key[2] = {(unsigned int)(seed & 0xFFFFFFFFull), (unsigned int)(seed >> 32)};
  unsigned int out[4];
  oracle_philox4x32_10(ctr, key, out);
  return (int)((out[i & 3] >> (8 * (j & 3))) & 0xFFu);
}

/* The keep decisions of every element of heads 0 .. BH - 1 with N queries and
 * N keys: keep[(bh * N + i) * N + j] = 1 iff byte(bh, i, j) >= p256. */
int oracle_dropout_keep(unsigned long long seed, unsigned int offset, int BH, int N, int p256, unsigned char* keep,
                        int nthreads) {
  if (BH < 1 || N < 1 || p256 < 0 || p256 > 255 || !keep) return 1;
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (long long r = 0; r < (long long)BH * N; ++r) {
    const int bh = (int)(r / N), i = (int)(r % N);
    for (int j = 0; j < N; ++j) keep[r * N + j] = oracle_dropout_byte(seed, offset, bh, i, j) >= p256;
  }
  return 0;
}

/* Z_ij: 0 if the element is dropped, else 256 / (256 - p256). */
static double drop_factor(unsigned long long seed, unsigned int offset, int bh, int i, int j, int p256) {
  return oracle_dropout_byte(seed, offset, bh, i, j) >= p256 ? 256.0 / (256.0 - p256) : 0.0;
}

/* Forward with dropout, self-attention (N query rows and keys); rows as in oracle_fwd. */
int oracle_fwd_drop(const double* q, const double* k, const double* v, double* o, double* lse, int BH, int N, int d,
                    double scale, int causal, int p256, unsigned long long seed, unsigned int offset, const int* rows,
                    int nrows, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !lse || p256 < 0 || p256 > 255) return -1;
  if (!rows) nrows = N;
  for (int r = 0; rows && r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return -1;
  set_threads(nthreads);
  int failed = 0;
  const long long total = (long long)BH * nrows;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long long w = 0; w < total; ++w) {
      if (!s) continue;
      const int h = (int)(w / nrows);
      const int i = rows ? rows[w % nrows] : (int)(w % nrows);
      const double* qi = q + ((size_t)h * N + i) * d;
      const double* kh = k + (size_t)h * N * d;
      const double* vh = v + (size_t)h * N * d;
      double* oi = o + ((size_t)h * N + i) * d;
      const int n_vis = causal ? i + 1 : N;
      double M, l;
      score_row(qi, kh, n_vis, d, scale, s, &M, &l);
      for (int t = 0; t < d; ++t) oi[t] = 0.0;
      for (int j = 0; j < n_vis; ++j) {
        const double pz = exp(s[j] - M) / l * drop_factor(seed, offset, h, i, j, p256);
        const double* vj = vh + (size_t)j * d;
        for (int t = 0; t < d; ++t) oi[t] += pz * vj[t];
      }
      lse[(size_t)h * N + i] = M + log(l);
    }
    free(s);
  }
  return failed ? -1 : 0;
}

/* Backward with dropout, self-attention: dq, dk, dv for every row and key; D if non-NULL. */
int oracle_bwd_drop(const double* q, const double* k, const double* v, const double* dO, double* dq, double* dk,
                    double* dv, double* D, int BH, int N, int d, double scale, int causal, int p256,
                    unsigned long long seed, unsigned int offset, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !dO || !dq || !dk || !dv || p256 < 0 || p256 > 255) return -1;
  set_threads(nthreads);
  double* lse_all = (double*)malloc(sizeof(double) * (size_t)BH * N);
  double* D_all = (double*)malloc(sizeof(double) * (size_t)BH * N);
  if (!lse_all || !D_all) {
    free(lse_all);
    free(D_all);
    return -1;
  }
  int failed = 0;
  /* Pass 1, per query row: P, the dropped dP, D, dS; dq. */
  const long long total_rows = (long long)BH * N;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* dp = (double*)malloc(sizeof(double) * (size_t)N);
    if (!s || !dp) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long long w = 0; w < total_rows; ++w) {
      if (!s || !dp) continue;
      const int h = (int)(w / N), i = (int)(w % N);
      const size_t hb = (size_t)h * N * d;
      const double* qi = q + hb + (size_t)i * d;
      const double* dOi = dO + hb + (size_t)i * d;
      const int n_vis = causal ? i + 1 : N;
      double M, l;
      score_row(qi, k + hb, n_vis, d, scale, s, &M, &l);
      double Dsum = 0.0;
      for (int j = 0; j < n_vis; ++j) {
        s[j] = exp(s[j] - M) / l; /* P_ij */
        dp[j] = drop_factor(seed, offset, h, i, j, p256) * dot(dOi, v + hb + (size_t)j * d, d);
        Dsum += s[j] * dp[j];
      }
      lse_all[w] = M + log(l);
      D_all[w] = Dsum;
      double* dq_row = dq + hb + (size_t)i * d;
      for (int t = 0; t < d; ++t) dq_row[t] = 0.0;
      for (int j = 0; j < n_vis; ++j) {
        const double ds = s[j] * (dp[j] - Dsum);
        const double* kj = k + hb + (size_t)j * d;
        for (int t = 0; t < d; ++t) dq_row[t] += scale * ds * kj[t];
      }
    }
    free(s);
    free(dp);
  }
  /* Pass 2, per key: dk and dv over the rows that see it. */
  if (!failed) {
#pragma omp parallel for schedule(dynamic, 4)
    for (long long w = 0; w < total_rows; ++w) {
      const int h = (int)(w / N), j = (int)(w % N);
      const size_t hb = (size_t)h * N * d;
      const double* kj = k + hb + (size_t)j * d;
      const double* vj = v + hb + (size_t)j * d;
      double* dkj = dk + hb + (size_t)j * d;
      double* dvj = dv + hb + (size_t)j * d;
      for (int t = 0; t < d; ++t) {
        dkj[t] = 0.0;
        dvj[t] = 0.0;
      }
      for (int i = causal ? j : 0; i < N; ++i) {
        const double* qi = q + hb + (size_t)i * d;
        const double* dOi = dO + hb + (size_t)i * d;
        const double p = exp(scale * dot(qi, kj, d) - lse_all[(size_t)h * N + i]);
        const double z = drop_factor(seed, offset, h, i, j, p256);
        const double ds = p * (z * dot(dOi, vj, d) - D_all[(size_t)h * N + i]);
        for (int t = 0; t < d; ++t) {
          dkj[t] += scale * qi[t] * ds;
          dvj[t] += p * z * dOi[t];
        }
      }
    }
  }
  if (D && !failed) memcpy(D, D_all, sizeof(double) * (size_t)BH * N);
  free(lse_all);
  free(D_all);
  return failed ? -1 : 0;
}
