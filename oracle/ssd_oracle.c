/*
 * ssd_oracle.c -- plain fp64 CPU oracle for the SSD selective-scan forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: it exists so that tests/, the smoke check and the benchmark's
 * CPU-baseline leg can compare the CUDA library against an obviously correct,
 * independent statement of what the method computes.  It shares no code, no
 * header and no constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [M3-02]  "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of SSM)"
 *            §2.1.1 (continuous LTV system with skip term D),
 *            §2.1.2 (Euler/ZOH discretisation h_t = e^{Δ_t A_t} h_{t-1} + Δ_t B_t x_t,
 *                    forget gate α_t = e^{Δ_t A_t}, input gate γ_t = Δ_t,
 *                    boxed recurrence h_t = α_t h_{t-1} + γ_t B_t x_t, y_t = C_tᵀ h_t),
 *            §2.2.1 (matrix form Y = (L ⊙ C Bᵀ) X and the mask
 *                    L_ij = ∏_{k=j+1}^{i} α_k for i>j, 1 for i=j, 0 for i<j),
 *            §2.2.2 / mask figure (block decomposition of the mask; the text is
 *                    cut off there, so the chunked form below is the plain
 *                    reading: split time into chunks, exact within a chunk by
 *                    the matrix form, carry the state between chunks by the
 *                    recurrence).
 *   [T2M]    "从Transformer到Mamba：状态空间模型（SSM）如何改变序列建模的未来"
 *            §2.1 (y = M x with M_ji = C_jᵀ A_{j:i} B_i).
 *   [TaS]    "Transformers are SSMs" §1, §1.1 (semiseparable matrix; both paths
 *            compute the same matrix product).
 *
 * Readings where the pages are silent (the plainest reading each time):
 *   - the input term is Δ_t·B_t·x_t (Euler, as printed in [M3-02] §2.1.2);
 *   - y_t reads h_t after the update (so y_t sees x_t; the mask has L_ii = 1);
 *   - y_t += D_h·x_t, the skip term of the continuous system in [M3-02] §2.1.1;
 *   - A is one real scalar per head ([M3-02] §2.3.1), so α_t is a scalar per
 *     (token, head) and the state of a head is a P×N matrix h[p][n];
 *   - heads are split into G contiguous groups; head h reads B/C of group
 *     h / (H/G)  (the pages give no mapping -- parity unpinned for the order);
 *   - an optional initial state h_{-1} enters as the state before token 0.
 *
 * Layouts (all row-major, contiguous):
 *   x [Bsz][L][H][P], dt [Bsz][L][H], A [H], Bm/Cm [Bsz][L][G][N], D [H],
 *   h0/hT [Bsz][H][P][N], y [Bsz][L][H][P].
 *   Chunked intermediates: dA_cs [Bsz][H][nc][Q], chunk states and the states
 *   entering each chunk [Bsz][nc][H][P][N].
 *
 * Every function returns 0 on success, nonzero on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted-mistake switch used only by the pin tests: they compile extra copies
 * of this file with -DORACLE_MUTANT=k and check that the pins reject each
 * copy.  The default build (0) is the oracle.
 *   1: y_t reads the state before the update (y_t = C_tᵀ h_{t-1})
 *   2: the input gate Δ_t is dropped from the input term
 *   3: the skip term D x_t is dropped
 *   4: the sign of the exponent in α_t is flipped
 *   5: the roles of B and C are swapped                                      */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static int g_threads = 0; /* 0: OpenMP default */

void oracle_set_threads(int n) { g_threads = n; }

int oracle_max_threads(void) {
#ifdef _OPENMP
  return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
  return 1;
#endif
}

static int bad_dims(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N) {
  return Bsz <= 0 || L < 0 || H <= 0 || P <= 0 || G <= 0 || N <= 0 || (H % G) != 0;
}

/* ------------------------------------------------------------------------- */
/* 1. The sequential recurrence -- the plain definition, the primary oracle.  */
/*    [M3-02] §2.1.2: α_t = exp(Δ_t A), h_t = α_t h_{t-1} + Δ_t B_t x_t,      */
/*    y_t = C_tᵀ h_t; [M3-02] §2.1.1: + D x_t.                                */
/*    For one head the state is h[p][n] (P input channels, N state entries).   */
/* ------------------------------------------------------------------------- */
int oracle_ssd_recurrent(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                         const double* x, const double* dt, const double* A,
                         const double* Bm, const double* Cm, const double* D,
                         const double* h0, double* y, double* hT) {
  if (bad_dims(Bsz, L, H, P, G, N)) return 1;
  const int64_t heads_per_group = H / G;
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / heads_per_group;
      double* st = (double*)malloc((size_t)(P * N) * sizeof(double));
      if (!st) {
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t i = 0; i < P * N; ++i)
        st[i] = h0 ? h0[((b * H + h) * P) * N + i] : 0.0;
      for (int64_t t = 0; t < L; ++t) {
        const double delta = dt[(b * L + t) * H + h];
        const double alpha = exp((ORACLE_MUTANT == 4 ? -1.0 : 1.0) * delta * A[h]); /* forget gate */
        const double gain = (ORACLE_MUTANT == 2) ? 1.0 : delta;                      /* input gate */
        const double* xt = x + ((b * L + t) * H + h) * P;
        const double* Bt = ((ORACLE_MUTANT == 5) ? Cm : Bm) + ((b * L + t) * G + g) * N;
        const double* Ct = ((ORACLE_MUTANT == 5) ? Bm : Cm) + ((b * L + t) * G + g) * N;
        const double dskip = (D && ORACLE_MUTANT != 3) ? D[h] : 0.0;
        double* yt = y + ((b * L + t) * H + h) * P;
        for (int pass = 0; pass < 2; ++pass) {
          /* pass 0 updates the state, pass 1 reads it out (the mutant 1 copy
             reads first) */
          const int do_update = (ORACLE_MUTANT == 1) ? (pass == 1) : (pass == 0);
          if (do_update) {
            for (int64_t p = 0; p < P; ++p)
              for (int64_t n = 0; n < N; ++n)
                st[p * N + n] = alpha * st[p * N + n] + gain * Bt[n] * xt[p];
          } else {
            for (int64_t p = 0; p < P; ++p) {
              double acc = 0.0;
              for (int64_t n = 0; n < N; ++n) acc += Ct[n] * st[p * N + n];
              yt[p] = acc + dskip * xt[p];
            }
          }
        }
      }
      if (hT)
        memcpy(hT + ((b * H + h) * P) * N, st, (size_t)(P * N) * sizeof(double));
      free(st);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* 2. The quadratic ("attention") form -- diagnostic.                        */
/*    [M3-02] §2.2.1: Y = (L ⊙ C Bᵀ) X with L_ij = ∏_{k=j+1}^{i} α_k (i>j),   */
/*    1 (i=j), 0 (i<j); [T2M] §2.1: M_ji = C_jᵀ A_{j:i} B_i.  The input gate   */
/*    Δ_j scales column j (the recurrence writes Δ_j B_j x_j).  The initial    */
/*    state reaches token i decayed by ∏_{k=0}^{i} α_k.  The mask entries are */
/*    running products of α, never differences of logarithms.                 */
/*    O(L²) per head: tiny inputs only.                                       */
/* ------------------------------------------------------------------------- */
int oracle_ssd_quadratic(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                         const double* x, const double* dt, const double* A,
                         const double* Bm, const double* Cm, const double* D,
                         const double* h0, double* y, double* hT) {
  if (bad_dims(Bsz, L, H, P, G, N)) return 1;
  const int64_t heads_per_group = H / G;
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / heads_per_group;
      double* alpha = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
      if (!alpha) {
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t t = 0; t < L; ++t) alpha[t] = exp(dt[(b * L + t) * H + h] * A[h]);
      for (int64_t i = 0; i < L; ++i) {
        const double* Ci = Cm + ((b * L + i) * G + g) * N;
        double* yi = y + ((b * L + i) * H + h) * P;
        for (int64_t p = 0; p < P; ++p) yi[p] = 0.0;
        /* L_ij for j = i, i-1, ..., 0, built as a running product. */
        double Lij = 1.0;
        for (int64_t j = i; j >= 0; --j) {
          if (j < i) Lij *= alpha[j + 1];
          const double* Bj = Bm + ((b * L + j) * G + g) * N;
          double cb = 0.0;
          for (int64_t n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
          const double Mij = Lij * cb * dt[(b * L + j) * H + h];
          const double* xj = x + ((b * L + j) * H + h) * P;
          for (int64_t p = 0; p < P; ++p) yi[p] += Mij * xj[p];
        }
        if (h0) {
          double decay = 1.0; /* ∏_{k=0}^{i} α_k */
          for (int64_t k = 0; k <= i; ++k) decay *= alpha[k];
          const double* s0 = h0 + ((b * H + h) * P) * N;
          for (int64_t p = 0; p < P; ++p) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += Ci[n] * s0[p * N + n];
            yi[p] += decay * acc;
          }
        }
        if (D) {
          const double* xi = x + ((b * L + i) * H + h) * P;
          for (int64_t p = 0; p < P; ++p) yi[p] += D[h] * xi[p];
        }
      }
      if (hT) {
        /* h_{L-1} = Σ_j (∏_{k=j+1}^{L-1} α_k) Δ_j x_j B_jᵀ + (∏_k α_k) h0 */
        double* s = hT + ((b * H + h) * P) * N;
        for (int64_t e = 0; e < P * N; ++e) s[e] = 0.0;
        double tail = 1.0;
        for (int64_t j = L - 1; j >= 0; --j) {
          if (j < L - 1) tail *= alpha[j + 1];
          const double dj = dt[(b * L + j) * H + h];
          const double* xj = x + ((b * L + j) * H + h) * P;
          const double* Bj = Bm + ((b * L + j) * G + g) * N;
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) s[p * N + n] += tail * dj * xj[p] * Bj[n];
        }
        if (h0) {
          double decay = 1.0;
          for (int64_t k = 0; k < L; ++k) decay *= alpha[k];
          const double* s0 = h0 + ((b * H + h) * P) * N;
          for (int64_t e = 0; e < P * N; ++e) s[e] += decay * s0[e];
        }
      }
      free(alpha);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* 3. The chunked form -- diagnostic, and the source of the per-step          */
/*    intermediates.  Time is cut into chunks of Q tokens (nc = ceil(L/Q)).    */
/*    Inside chunk c, with log-decays a_k = Δ_k A (log α_k) and the in-chunk   */
/*    inclusive sums cs_i = Σ_{k≤i} a_k, the mask of [M3-02] §2.2.1 restricted */
/*    to the chunk is L_ij = exp(cs_i − cs_j) for j ≤ i.  Positions past L     */
/*    (tail of the last chunk) carry Δ = 0, i.e. α = 1 and no input.           */
/*      dA_cs[c][i] = cs_i                                                     */
/*      S_c         = Σ_i exp(cs_{Q−1} − cs_i) Δ_i x_i B_iᵀ   (chunk state)     */
/*      hin[0] = h0, hin[c+1] = exp(cs_{Q−1}) hin[c] + S_c, hT = hin[nc]         */
/*                 (the recurrence of §2.1.2 lifted to chunk granularity)      */
/*      y_i = Σ_{j≤i} (C_i·B_j) exp(cs_i − cs_j) Δ_j x_j                       */
/*            + exp(cs_i) C_iᵀ hin[c] + D x_i                                  */
/*    Any of dA_cs, states, hin, y, hT may be NULL.                            */
/* ------------------------------------------------------------------------- */
int oracle_ssd_chunked(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                       int64_t Q, const double* x, const double* dt, const double* A,
                       const double* Bm, const double* Cm, const double* D,
                       const double* h0, double* dA_cs, double* states, double* hin,
                       double* y, double* hT) {
  if (bad_dims(Bsz, L, H, P, G, N) || Q <= 0) return 1;
  const int64_t heads_per_group = H / G;
  const int64_t nc = (L + Q - 1) / Q;
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / heads_per_group;
      double* cs = (double*)malloc((size_t)Q * sizeof(double));
      double* dl = (double*)malloc((size_t)Q * sizeof(double));
      double* run = (double*)malloc((size_t)(P * N) * sizeof(double));
      double* sc = (double*)malloc((size_t)(P * N) * sizeof(double));
      if (!cs || !dl || !run || !sc) {
        free(cs); free(dl); free(run); free(sc);
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t e = 0; e < P * N; ++e) run[e] = h0 ? h0[((b * H + h) * P) * N + e] : 0.0;
      for (int64_t c = 0; c < nc; ++c) {
        /* in-chunk inclusive sum of log α */
        double acc = 0.0;
        for (int64_t i = 0; i < Q; ++i) {
          const int64_t t = c * Q + i;
          dl[i] = (t < L) ? dt[(b * L + t) * H + h] : 0.0;
          acc += dl[i] * A[h];
          cs[i] = acc;
          if (dA_cs) dA_cs[((b * H + h) * nc + c) * Q + i] = acc;
        }
        /* state entering this chunk */
        if (hin) {
          double* dst = hin + (((b * nc + c) * H + h) * P) * N;
          for (int64_t e = 0; e < P * N; ++e) dst[e] = run[e];
        }
        /* outputs of the chunk */
        if (y) {
          for (int64_t i = 0; i < Q; ++i) {
            const int64_t ti = c * Q + i;
            if (ti >= L) break;
            const double* Ci = Cm + ((b * L + ti) * G + g) * N;
            double* yi = y + ((b * L + ti) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) yi[p] = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
              const int64_t tj = c * Q + j;
              const double* Bj = Bm + ((b * L + tj) * G + g) * N;
              double cb = 0.0;
              for (int64_t n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
              const double m = cb * exp(cs[i] - cs[j]) * dl[j];
              const double* xj = x + ((b * L + tj) * H + h) * P;
              for (int64_t p = 0; p < P; ++p) yi[p] += m * xj[p];
            }
            const double ein = exp(cs[i]);
            const double* xi = x + ((b * L + ti) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) {
              double r = 0.0;
              for (int64_t n = 0; n < N; ++n) r += Ci[n] * run[p * N + n];
              yi[p] += ein * r + (D ? D[h] * xi[p] : 0.0);
            }
          }
        }
        /* chunk state S_c and the carried state */
        for (int64_t e = 0; e < P * N; ++e) sc[e] = 0.0;
        for (int64_t i = 0; i < Q; ++i) {
          const int64_t t = c * Q + i;
          if (t >= L) break;
          const double w = exp(cs[Q - 1] - cs[i]) * dl[i];
          const double* xi = x + ((b * L + t) * H + h) * P;
          const double* Bi = Bm + ((b * L + t) * G + g) * N;
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) sc[p * N + n] += w * xi[p] * Bi[n];
        }
        if (states) {
          double* dst = states + (((b * nc + c) * H + h) * P) * N;
          for (int64_t e = 0; e < P * N; ++e) dst[e] = sc[e];
        }
        const double dec = exp(cs[Q - 1]);
        for (int64_t e = 0; e < P * N; ++e) run[e] = dec * run[e] + sc[e];
      }
      if (hT) memcpy(hT + ((b * H + h) * P) * N, run, (size_t)(P * N) * sizeof(double));
      free(cs); free(dl); free(run); free(sc);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* 4. The gradient of the recurrence (reverse mode) -- the backward oracle.   */
/*    The function differentiated is the recurrence of section 1 ([M3-02]     */
/*    §2.1.2 plus the skip term of §2.1.1); the scalar being differentiated   */
/*    is  Lsum = Σ dy ⊙ y + Σ dhT ⊙ hT  for given cotangents dy (and dhT).    */
/*    The page "从 SSM 的长期记忆问题，到 Mamba 的选择性机制与硬件感知扫描"   */
/*    (paragraph on the hardware-aware scan) has the backward pass recompute  */
/*    the states instead of storing them; here every sqrt(L)-th state is kept */
/*    on the forward sweep and each span is recomputed from it on the way     */
/*    back.  Writing G_t = ∂Lsum/∂h_t (the whole dependence of Lsum on h_t):  */
/*      G_{L-1} = dhT + dy_{L-1} C_{L-1}ᵀ,  G_t = dy_t C_tᵀ + α_{t+1} G_{t+1}  */
/*      u_t     = G_t B_t                      (P-vector)                     */
/*      dx_t    = D dy_t + Δ_t u_t                                            */
/*      dB_t   += Δ_t G_tᵀ x_t,   dC_t += h_tᵀ dy_t    (summed over the heads  */
/*                                                      of the group)         */
/*      da_t    = <G_t, α_t h_{t-1}>          (a_t = Δ_t A, log α_t)          */
/*      dΔ_t    = x_t·u_t + A da_t,   dA += Δ_t da_t,   dD += dy_t·x_t        */
/*      dh0     = α_0 G_0                                                      */
/*    Parallel over (batch, group) with the heads of a group in order, so the */
/*    group sums are deterministic.  dhT, h0, D may be NULL; dh0 may be NULL. */
/*    Planted mistakes for the pin tests (ORACLE_BWD_MUTANT):                 */
/*      1: dΔ drops the decay term A da_t                                     */
/*      2: G is decayed before dy_t C_tᵀ is added (an index shift)            */
/*      3: dB uses the state h_{t-1} in place of x_t                           */
/* ------------------------------------------------------------------------- */
#ifndef ORACLE_BWD_MUTANT
#define ORACLE_BWD_MUTANT 0
#endif

int oracle_ssd_recurrent_bwd(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                             const double* x, const double* dt, const double* A,
                             const double* Bm, const double* Cm, const double* D,
                             const double* h0, const double* dy, const double* dhT,
                             double* dx, double* ddt, double* dA, double* dBm, double* dCm,
                             double* dD, double* dh0) {
  if (bad_dims(Bsz, L, H, P, G, N)) return 1;
  const int64_t hpg = H / G;
  const int64_t PN = P * N;
  int64_t K = 1; /* span between kept states */
  while (K * K < L) ++K;
  const int64_t nck = L > 0 ? (L + K - 1) / K : 0;
  double* dA_part = (double*)calloc((size_t)(Bsz * H), sizeof(double));
  double* dD_part = (double*)calloc((size_t)(Bsz * H), sizeof(double));
  if (!dA_part || !dD_part) {
    free(dA_part); free(dD_part);
    return 2;
  }
  memset(dBm, 0, (size_t)(Bsz * L * G * N) * sizeof(double));
  memset(dCm, 0, (size_t)(Bsz * L * G * N) * sizeof(double));
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t g = 0; g < G; ++g) {
      /* kept[k] = h_{kK-1} (the state before token kK); span[j] = h_{t0+j} */
      double* kept = (double*)malloc((size_t)((nck + 1) * PN) * sizeof(double));
      double* span = (double*)malloc((size_t)((K + 1) * PN) * sizeof(double));
      double* Gt = (double*)malloc((size_t)PN * sizeof(double));
      double* u = (double*)malloc((size_t)P * sizeof(double));
      if (!kept || !span || !Gt || !u) {
        free(kept); free(span); free(Gt); free(u);
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
        const double* x_bh = x + (b * L * H + h) * P;     /* token t at + t*H*P */
        const double dskip = D ? D[h] : 0.0;
        /* forward sweep: keep every K-th state */
        double* run = span;
        for (int64_t e = 0; e < PN; ++e) run[e] = h0 ? h0[(b * H + h) * PN + e] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
          if (t % K == 0) memcpy(kept + (t / K) * PN, run, (size_t)PN * sizeof(double));
          const double delta = dt[(b * L + t) * H + h];
          const double alpha = exp(delta * A[h]);
          const double* xt = x_bh + t * H * P;
          const double* Bt = Bm + ((b * L + t) * G + g) * N;
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n)
              run[p * N + n] = alpha * run[p * N + n] + delta * xt[p] * Bt[n];
        }
        /* backward sweep */
        for (int64_t e = 0; e < PN; ++e) Gt[e] = dhT ? dhT[(b * H + h) * PN + e] : 0.0;
        double dA_acc = 0.0, dD_acc = 0.0;
        for (int64_t k = nck - 1; k >= 0; --k) {
          const int64_t t0 = k * K;
          const int64_t t1 = (t0 + K < L) ? t0 + K : L;
          /* recompute span[j] = h_{t0-1+j}, j = 0 .. t1-t0 */
          memcpy(span, kept + k * PN, (size_t)PN * sizeof(double));
          for (int64_t t = t0; t < t1; ++t) {
            const double delta = dt[(b * L + t) * H + h];
            const double alpha = exp(delta * A[h]);
            const double* xt = x_bh + t * H * P;
            const double* Bt = Bm + ((b * L + t) * G + g) * N;
            const double* prev = span + (t - t0) * PN;
            double* cur = span + (t - t0 + 1) * PN;
            for (int64_t p = 0; p < P; ++p)
              for (int64_t n = 0; n < N; ++n)
                cur[p * N + n] = alpha * prev[p * N + n] + delta * xt[p] * Bt[n];
          }
          for (int64_t t = t1 - 1; t >= t0; --t) {
            const double delta = dt[(b * L + t) * H + h];
            const double alpha = exp(delta * A[h]);
            const double* xt = x_bh + t * H * P;
            const double* Bt = Bm + ((b * L + t) * G + g) * N;
            const double* Ct = Cm + ((b * L + t) * G + g) * N;
            const double* dyt = dy + ((b * L + t) * H + h) * P;
            const double* hprev = span + (t - t0) * PN;   /* h_{t-1} */
            const double* hcur = span + (t - t0 + 1) * PN; /* h_t */
            if (ORACLE_BWD_MUTANT == 2) {
              for (int64_t e = 0; e < PN; ++e) Gt[e] *= alpha;
            }
            for (int64_t p = 0; p < P; ++p)
              for (int64_t n = 0; n < N; ++n) Gt[p * N + n] += dyt[p] * Ct[n];
            /* G_t is complete */
            double xu = 0.0, da = 0.0;
            for (int64_t p = 0; p < P; ++p) {
              double s = 0.0;
              for (int64_t n = 0; n < N; ++n) s += Gt[p * N + n] * Bt[n];
              u[p] = s;
              xu += xt[p] * s;
              dD_acc += dyt[p] * xt[p];
              dx[((b * L + t) * H + h) * P + p] = dskip * dyt[p] + delta * s;
            }
            double* dBt = dBm + ((b * L + t) * G + g) * N;
            double* dCt = dCm + ((b * L + t) * G + g) * N;
            for (int64_t n = 0; n < N; ++n) {
              double sb = 0.0, sc = 0.0;
              for (int64_t p = 0; p < P; ++p) {
                sb += Gt[p * N + n] * (ORACLE_BWD_MUTANT == 3 ? hprev[p * N + n] : xt[p]);
                sc += hcur[p * N + n] * dyt[p];
              }
              dBt[n] += delta * sb;
              dCt[n] += sc;
            }
            for (int64_t e = 0; e < PN; ++e) da += Gt[e] * alpha * hprev[e];
            ddt[(b * L + t) * H + h] = xu + (ORACLE_BWD_MUTANT == 1 ? 0.0 : A[h] * da);
            dA_acc += delta * da;
            if (ORACLE_BWD_MUTANT != 2) {
              for (int64_t e = 0; e < PN; ++e) Gt[e] *= alpha; /* toward G_{t-1} */
            }
          }
        }
        if (ORACLE_BWD_MUTANT == 2 && L > 0) {
          const double alpha0 = exp(dt[(b * L + 0) * H + h] * A[h]);
          for (int64_t e = 0; e < PN; ++e) Gt[e] *= alpha0;
        }
        if (dh0) memcpy(dh0 + (b * H + h) * PN, Gt, (size_t)PN * sizeof(double));
        dA_part[b * H + h] = dA_acc;
        dD_part[b * H + h] = dD_acc;
      }
      free(kept); free(span); free(Gt); free(u);
    }
  }
  for (int64_t h = 0; h < H; ++h) {
    double sa = 0.0, sd = 0.0;
    for (int64_t b = 0; b < Bsz; ++b) {
      sa += dA_part[b * H + h];
      sd += dD_part[b * H + h];
    }
    dA[h] = sa;
    if (dD) dD[h] = sd;
  }
  free(dA_part); free(dD_part);
  return err;
}

/* ------------------------------------------------------------------------- */
/* 5. The complex (rotational) decay -- the Mamba-3 variant.                  */
/*    [M3-02] §2.3 (the limit of real decays: a real eigenvalue cannot rotate */
/*    or oscillate, e^{iθ} = cos θ + i sin θ can; the parity task as the      */
/*    motivating example) and the page's summary (complex dynamics).  The    */
/*    plainest reading: the scalar decay of a head gains                    */
/*    a rotation angle θ_t per token and head (input-dependent like Δ_t),     */
/*      α_t = exp(Δ_t A) · (cos θ_t + i sin θ_t),                             */
/*      h_t = α_t h_{t-1} + Δ_t x_t B_tᵀ      (complex state, real input)     */
/*      y_t = Re(h_t) C_t + D x_t,                                            */
/*    θ = 0 is the real recurrence of section 1.  The state is kept as its    */
/*    real and imaginary parts; h0_re/h0_im and hT_re/hT_im may be NULL.      */
/* ------------------------------------------------------------------------- */
int oracle_ssd_recurrent_rot(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                             const double* x, const double* dt, const double* theta, const double* A,
                             const double* Bm, const double* Cm, const double* D,
                             const double* h0_re, const double* h0_im,
                             double* y, double* hT_re, double* hT_im) {
  if (bad_dims(Bsz, L, H, P, G, N)) return 1;
  const int64_t hpg = H / G;
  const int64_t PN = P * N;
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / hpg;
      double* re = (double*)malloc((size_t)PN * sizeof(double));
      double* im = (double*)malloc((size_t)PN * sizeof(double));
      if (!re || !im) {
        free(re); free(im);
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t e = 0; e < PN; ++e) {
        re[e] = h0_re ? h0_re[(b * H + h) * PN + e] : 0.0;
        im[e] = h0_im ? h0_im[(b * H + h) * PN + e] : 0.0;
      }
      for (int64_t t = 0; t < L; ++t) {
        const double delta = dt[(b * L + t) * H + h];
        const double th = theta[(b * L + t) * H + h];
        const double mag = exp(delta * A[h]);
        const double ar = mag * cos(th), ai = mag * sin(th);
        const double* xt = x + ((b * L + t) * H + h) * P;
        const double* Bt = Bm + ((b * L + t) * G + g) * N;
        const double* Ct = Cm + ((b * L + t) * G + g) * N;
        double* yt = y + ((b * L + t) * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; ++n) {
            const int64_t e = p * N + n;
            const double r = ar * re[e] - ai * im[e] + delta * xt[p] * Bt[n];
            const double i = ar * im[e] + ai * re[e];
            re[e] = r;
            im[e] = i;
            acc += r * Ct[n];
          }
          yt[p] = acc + (D ? D[h] * xt[p] : 0.0);
        }
      }
      if (hT_re) memcpy(hT_re + (b * H + h) * PN, re, (size_t)PN * sizeof(double));
      if (hT_im) memcpy(hT_im + (b * H + h) * PN, im, (size_t)PN * sizeof(double));
      free(re); free(im);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* 6. Retrieval rank R > 1 (MIMO) -- page "状态空间模型的对角等价：检索秩与选择性 */
/*    扩展新解", section "从 MIMO 到 HybridMamba": the retrieval rank is the     */
/*    number of independent value channels written and read in parallel at  */
/*    a local interface (the width of the state update); SSD-MIMO routes an   */
/*    independent value per rank; SISO (R = 1) is recovered exactly.  The     */
/*    page gives no formula.  Reading taken: per token and head, R channels   */
/*    r with their own x_t^(r) (P), B_t^(r), C_t^(r) (N, per group) share the */
/*    token's decay; the update writes all R values at once and each rank     */
/*    reads its own output from the updated state:                            */
/*      h_t = α_t h_{t-1} + Δ_t Σ_r x_t^(r) B_t^(r)ᵀ                           */
/*      y_t^(r) = h_t C_t^(r) + D x_t^(r)                                      */
/*    Layouts: x, y [Bsz][L][R][H][P]; dt [Bsz][L][H]; Bm, Cm                  */
/*    [Bsz][L][R][G][N]; h0, hT [Bsz][H][P][N].                                */
/* ------------------------------------------------------------------------- */
int oracle_ssd_recurrent_mimo(int64_t Bsz, int64_t L, int64_t R, int64_t H, int64_t P, int64_t G, int64_t N,
                              const double* x, const double* dt, const double* A,
                              const double* Bm, const double* Cm, const double* D,
                              const double* h0, double* y, double* hT) {
  if (bad_dims(Bsz, L, H, P, G, N) || R < 1) return 1;
  const int64_t heads_per_group = H / G;
  const int nthr = oracle_max_threads();
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthr)
  for (int64_t b = 0; b < Bsz; ++b) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / heads_per_group;
      double* st = (double*)malloc((size_t)(P * N) * sizeof(double));
      if (!st) {
#pragma omp atomic write
        err = 2;
        continue;
      }
      for (int64_t i = 0; i < P * N; ++i)
        st[i] = h0 ? h0[((b * H + h) * P) * N + i] : 0.0;
      for (int64_t t = 0; t < L; ++t) {
        const double delta = dt[(b * L + t) * H + h];
        const double alpha = exp(delta * A[h]);
        /* decay once per token, then the R writes */
        for (int64_t i = 0; i < P * N; ++i) st[i] *= alpha;
        for (int64_t r = 0; r < R; ++r) {
          const double* xr = x + (((b * L + t) * R + r) * H + h) * P;
          const double* Br = Bm + (((b * L + t) * R + r) * G + g) * N;
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) st[p * N + n] += delta * Br[n] * xr[p];
        }
        /* each rank reads its own output from the updated state */
        for (int64_t r = 0; r < R; ++r) {
          const double* xr = x + (((b * L + t) * R + r) * H + h) * P;
          const double* Cr = Cm + (((b * L + t) * R + r) * G + g) * N;
          double* yr = y + (((b * L + t) * R + r) * H + h) * P;
          for (int64_t p = 0; p < P; ++p) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) acc += Cr[n] * st[p * N + n];
            yr[p] = acc + (D ? D[h] * xr[p] : 0.0);
          }
        }
      }
      if (hT) memcpy(hT + ((b * H + h) * P) * N, st, (size_t)(P * N) * sizeof(double));
      free(st);
    }
  }
  return err;
}
