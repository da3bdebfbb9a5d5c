/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle for the Gated DeltaNet
 * forward pass.  TEST INFRASTRUCTURE ONLY: nothing on the product path may
 * link, load or call this file; only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py use it.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Two independent forms are given:
 *
 *  1. oracle_recurrent -- the token-by-token gated delta rule, i.e. the plain
 *     definition of the operator ("Gated DeltaNet" chunk-recurrence pages:
 *     MegaGDN-PTO walkthrough, section 1.1, and the TileLang x xLLM page,
 *     Step 1, where the state h is [K, V] fp32 and carries h0 -> ht):
 *
 *        S_t = exp(g_t) * (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *        o_t = scale * S_t^T q_t
 *
 *     with S in [K][V] orientation (the transpose of the [V][K] statement
 *     S_t = e^{g_t} S_{t-1}(I - beta k k^T) + beta v k^T, o_t = scale S_t q_t;
 *     I - beta k k^T is symmetric, so the two are the same map).
 *
 *  2. oracle_chunked -- the chunked form, written out step by step in the
 *     order of the MegaGDN-PTO walkthrough's seven-stage list (section 1.1:
 *     cumsum, scaled_dot_kkt, solve_tril, wy_fast, chunk_h, chunk_o), with a
 *     generic Gauss-Jordan inverse standing in for solve_tril:
 *
 *        gamma_i = sum_{r<=i} g_r                      (in-chunk cumsum)
 *        A_ij    = beta_i exp(gamma_i - gamma_j) k_i.k_j   for i > j, else 0
 *        T       = (I + A)^{-1}
 *        W       = T diag(beta exp(gamma)) K,   U = T diag(beta) V
 *        V'      = U - W S0
 *        O       = scale (diag(exp(gamma)) Q S0 + (Q K^T o [j<=i] o exp(gamma_i-gamma_j)) V')
 *        S1      = exp(gamma_last) S0 + K^T diag(exp(gamma_last - gamma)) V'
 *
 *     A tail chunk is simply shorter (equivalent to zero padding).
 *
 * Layouts (row-major, float64):  q,k [Ttot][Hqk][K];  v [Ttot][Hv][V];
 * g,beta [Ttot][Hv];  h0,ht [N][Hv][K][V];  o [Ttot][Hv][V];
 * cu [N+1] int64 token offsets of the N packed sequences.
 * GQA: value head h reads q/k head h / (Hv/Hqk).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2
#define ORACLE_ESINGULAR 3

static int check_args(int64_t Ttot, int N, const int64_t* cu, int Hqk, int Hv, int K, int V) {
  if (Ttot < 0 || N <= 0 || !cu || Hqk <= 0 || Hv <= 0 || K <= 0 || V <= 0) return ORACLE_EINVAL;
  if (Hv % Hqk != 0) return ORACLE_EINVAL;
  if (cu[0] != 0 || cu[N] != Ttot) return ORACLE_EINVAL;
  for (int n = 0; n < N; ++n)
    if (cu[n + 1] < cu[n]) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- form 1 */

/* One (sequence, value head) chain of the token recurrence. */
static void recurrent_chain(int64_t t0, int64_t L, int Hqk, int Hv, int K, int V, int h,
                            const double* q, const double* k, const double* v,
                            const double* g, const double* beta, double scale,
                            double* S /* [K][V], in: h0, out: ht */, double* o,
                            double* ktS /* [V] */) {
  const int hq = h / (Hv / Hqk);
  for (int64_t t = t0; t < t0 + L; ++t) {
    const double* kt = k + (t * Hqk + hq) * (int64_t)K;
    const double* qt = q + (t * Hqk + hq) * (int64_t)K;
    const double* vt = v + (t * Hv + h) * (int64_t)V;
    const double a = exp(g[t * Hv + h]);
    const double b = beta[t * Hv + h];
    /* (I - b k k^T) S  =  S - b k (k^T S) */
    for (int e = 0; e < V; ++e) ktS[e] = 0.0;
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e) ktS[e] += kt[d] * S[(int64_t)d * V + e];
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e) {
        const double proj = S[(int64_t)d * V + e] - b * kt[d] * ktS[e];
        /* S_t = a (I - b k k^T) S_{t-1} + b k v^T */
        S[(int64_t)d * V + e] = a * proj + b * kt[d] * vt[e];
      }
    /* o_t = scale S_t^T q_t */
    double* ot = o + (t * Hv + h) * (int64_t)V;
    for (int e = 0; e < V; ++e) {
      double acc = 0.0;
      for (int d = 0; d < K; ++d) acc += S[(int64_t)d * V + e] * qt[d];
      ot[e] = scale * acc;
    }
  }
}

/* chain_ids: optional list of chains (n * Hv + h) to compute; NULL = all.
 * Outputs of chains not listed are left untouched. */
int oracle_recurrent(int64_t Ttot, int N, const int64_t* cu, int Hqk, int Hv, int K, int V,
                     const double* q, const double* k, const double* v, const double* g,
                     const double* beta, double scale, const double* h0, double* o, double* ht,
                     const int32_t* chain_ids, int n_chain_ids, int nthreads) {
  int rc = check_args(Ttot, N, cu, Hqk, Hv, K, V);
  if (rc) return rc;
  const int nchains = chain_ids ? n_chain_ids : N * Hv;
  int err = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int c = 0; c < nchains; ++c) {
    const int id = chain_ids ? chain_ids[c] : c;
    const int n = id / Hv, h = id % Hv;
    double* S = (double*)malloc(sizeof(double) * ((size_t)K * V + V));
    if (!S) { err = 1; continue; }
    double* ktS = S + (size_t)K * V;
    if (h0) memcpy(S, h0 + ((int64_t)n * Hv + h) * K * (int64_t)V, sizeof(double) * (size_t)K * V);
    else memset(S, 0, sizeof(double) * (size_t)K * V);
    recurrent_chain(cu[n], cu[n + 1] - cu[n], Hqk, Hv, K, V, h, q, k, v, g, beta, scale, S, o, ktS);
    if (ht) memcpy(ht + ((int64_t)n * Hv + h) * K * (int64_t)V, S, sizeof(double) * (size_t)K * V);
    free(S);
  }
  (void)nthreads;
  return err ? ORACLE_ENOMEM : ORACLE_OK;
}

/* ------------------------------------------------------- form 1, backward */

/*
 * Gradients of the token recurrence (reverse mode, written out by hand from
 * the forward above; the FlashQLA notes list a backward of the chunk form
 * among the variants, section 4.3).  For upstream gradients dout = dL/do and
 * dht = dL/dht, with a_t = exp(g_t), b_t = beta_t, P_t = I - b_t k_t k_t^T
 * (symmetric) and S_t the state after token t (S_0 = h0):
 *
 *   G     <- G + scale q_t dout_t^T            (G = dL/dS_t, starts at dht)
 *   dq_t   = scale S_t dout_t
 *   u      = S_{t-1}^T k_t,   w = G^T k_t      (V-vectors)
 *   dv_t   = b_t w
 *   dg_t   = a_t (<G, S_{t-1}> - b_t w.u)      (<,> = sum of elementwise products)
 *   dbeta_t= -a_t w.u + w.v_t
 *   dk_t   = -a_t b_t (G u + S_{t-1} w) + b_t G v_t
 *   G     <- a_t (G - b_t k_t w^T)             (= a_t P_t G, the gradient w.r.t. S_{t-1})
 *
 * and dh0 = the final G.  With GQA, dq and dk of a q/k head sum over the
 * value heads that read it.  Chains keep every state of the sequence (tests
 * use small sizes).
 */
static void recurrent_chain_bwd(int64_t t0, int64_t L, int Hqk, int Hv, int K, int V, int h,
                                const double* q, const double* k, const double* v, const double* g,
                                const double* beta, double scale, const double* h0c, const double* dout,
                                const double* dhtc, double* dq, double* dk, double* dv, double* dg,
                                double* dbeta, double* dh0c, double* St /* [(L+1)][K][V] */,
                                double* G /* [K][V] */, double* u /* [V] */, double* w /* [V] */) {
  const int hq = h / (Hv / Hqk);
  const int64_t KV = (int64_t)K * V;
  /* forward, keeping every state */
  if (h0c) memcpy(St, h0c, sizeof(double) * (size_t)KV);
  else memset(St, 0, sizeof(double) * (size_t)KV);
  for (int64_t i = 0; i < L; ++i) {
    const int64_t t = t0 + i;
    const double* kt = k + (t * Hqk + hq) * (int64_t)K;
    const double* vt = v + (t * Hv + h) * (int64_t)V;
    const double a = exp(g[t * Hv + h]), b = beta[t * Hv + h];
    const double* Sp = St + i * KV;
    double* Sn = St + (i + 1) * KV;
    for (int e = 0; e < V; ++e) {
      u[e] = 0.0;
      for (int d = 0; d < K; ++d) u[e] += kt[d] * Sp[(int64_t)d * V + e];
    }
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e)
        Sn[(int64_t)d * V + e] = a * (Sp[(int64_t)d * V + e] - b * kt[d] * u[e]) + b * kt[d] * vt[e];
  }
  /* backward */
  if (dhtc) memcpy(G, dhtc, sizeof(double) * (size_t)KV);
  else memset(G, 0, sizeof(double) * (size_t)KV);
  for (int64_t i = L - 1; i >= 0; --i) {
    const int64_t t = t0 + i;
    const double* kt = k + (t * Hqk + hq) * (int64_t)K;
    const double* qt = q + (t * Hqk + hq) * (int64_t)K;
    const double* vt = v + (t * Hv + h) * (int64_t)V;
    const double* dot = dout + (t * Hv + h) * (int64_t)V;
    const double a = exp(g[t * Hv + h]), b = beta[t * Hv + h];
    const double* Sp = St + i * KV;        /* S_{t-1} */
    const double* Sc = St + (i + 1) * KV;  /* S_t */
    double* dqt = dq + (t * Hqk + hq) * (int64_t)K;
    double* dkt = dk + (t * Hqk + hq) * (int64_t)K;
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e) G[(int64_t)d * V + e] += scale * qt[d] * dot[e];
    for (int d = 0; d < K; ++d) {
      double acc = 0.0;
      for (int e = 0; e < V; ++e) acc += Sc[(int64_t)d * V + e] * dot[e];
      dqt[d] += scale * acc;
    }
    for (int e = 0; e < V; ++e) {
      u[e] = 0.0;
      w[e] = 0.0;
      for (int d = 0; d < K; ++d) {
        u[e] += Sp[(int64_t)d * V + e] * kt[d];
        w[e] += G[(int64_t)d * V + e] * kt[d];
      }
    }
    double wu = 0.0, wv = 0.0, gs = 0.0;
    for (int e = 0; e < V; ++e) {
      wu += w[e] * u[e];
      wv += w[e] * vt[e];
    }
    for (int64_t x = 0; x < KV; ++x) gs += G[x] * Sp[x];
    double* dvt = dv + (t * Hv + h) * (int64_t)V;
    for (int e = 0; e < V; ++e) dvt[e] = b * w[e];
    dg[t * Hv + h] = a * (gs - b * wu);
    dbeta[t * Hv + h] = -a * wu + wv;
    for (int d = 0; d < K; ++d) {
      double gu = 0.0, sw = 0.0, gv = 0.0;
      for (int e = 0; e < V; ++e) {
        gu += G[(int64_t)d * V + e] * u[e];
        sw += Sp[(int64_t)d * V + e] * w[e];
        gv += G[(int64_t)d * V + e] * vt[e];
      }
      dkt[d] += -a * b * (gu + sw) + b * gv;
    }
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e) G[(int64_t)d * V + e] = a * (G[(int64_t)d * V + e] - b * kt[d] * w[e]);
  }
  memcpy(dh0c, G, sizeof(double) * (size_t)KV);
}

/* dq, dk [Ttot][Hqk][K] are overwritten (accumulated over the value heads of
 * each q/k head); dv [Ttot][Hv][V], dg, dbeta [Ttot][Hv], dh0 [N][Hv][K][V].
 * dht may be NULL (zero). */
int oracle_recurrent_bwd(int64_t Ttot, int N, const int64_t* cu, int Hqk, int Hv, int K, int V,
                         const double* q, const double* k, const double* v, const double* g,
                         const double* beta, double scale, const double* h0, const double* dout,
                         const double* dht, double* dq, double* dk, double* dv, double* dg, double* dbeta,
                         double* dh0, int nthreads) {
  int rc = check_args(Ttot, N, cu, Hqk, Hv, K, V);
  if (rc) return rc;
  memset(dq, 0, sizeof(double) * (size_t)Ttot * Hqk * K);
  memset(dk, 0, sizeof(double) * (size_t)Ttot * Hqk * K);
  const int G_ = Hv / Hqk;
  int err = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int c = 0; c < N * Hqk; ++c) {   /* one q/k head group per task: dq / dk have one writer */
    const int n = c / Hqk, hq = c % Hqk;
    const int64_t L = cu[n + 1] - cu[n];
    const int64_t KV = (int64_t)K * V;
    double* buf = (double*)malloc(sizeof(double) * ((size_t)(L + 2) * KV + 2 * (size_t)V));
    if (!buf) { err = 1; continue; }
    double* St = buf;
    double* G = buf + (L + 1) * KV;
    double* u = G + KV;
    double* w = u + V;
    for (int j = 0; j < G_; ++j) {
      const int h = hq * G_ + j;
      const int64_t off = ((int64_t)n * Hv + h) * KV;
      recurrent_chain_bwd(cu[n], L, Hqk, Hv, K, V, h, q, k, v, g, beta, scale, h0 ? h0 + off : NULL, dout,
                          dht ? dht + off : NULL, dq, dk, dv, dg, dbeta, dh0 + off, St, G, u, w);
    }
    free(buf);
  }
  (void)nthreads;
  return err ? ORACLE_ENOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------- form 2 */

/* Generic Gauss-Jordan inverse with partial pivoting: Minv = M^{-1}, n x n.
 * Deliberately not a triangular solve, so it cannot share a mistake with one. */
static int gauss_jordan_inverse(int n, const double* M, double* Minv, double* work /* [n][2n] */) {
  const int w = 2 * n;
  for (int i = 0; i < n; ++i) {
    for (int j = 0; j < n; ++j) work[i * w + j] = M[i * n + j];
    for (int j = 0; j < n; ++j) work[i * w + n + j] = (i == j) ? 1.0 : 0.0;
  }
  for (int col = 0; col < n; ++col) {
    int piv = col;
    for (int r = col + 1; r < n; ++r)
      if (fabs(work[r * w + col]) > fabs(work[piv * w + col])) piv = r;
    if (work[piv * w + col] == 0.0) return ORACLE_ESINGULAR;
    if (piv != col)
      for (int j = 0; j < w; ++j) {
        double t = work[col * w + j];
        work[col * w + j] = work[piv * w + j];
        work[piv * w + j] = t;
      }
    const double p = work[col * w + col];
    for (int j = 0; j < w; ++j) work[col * w + j] /= p;
    for (int r = 0; r < n; ++r) {
      if (r == col) continue;
      const double f = work[r * w + col];
      if (f == 0.0) continue;
      for (int j = 0; j < w; ++j) work[r * w + j] -= f * work[col * w + j];
    }
  }
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) Minv[i * n + j] = work[i * w + n + j];
  return ORACLE_OK;
}

typedef struct {
  double *gamma, *A, *M, *T, *work, *W, *U, *Vn, *QK, *S0;
} chunk_scratch;

/* Optional per-chunk intermediates of one chain (rows past the chunk length
 * are left zero):  gamma [NT][C], A [NT][C][C], T [NT][C][C], W [NT][C][K],
 * U [NT][C][V], S0 [NT][K][V] (state at chunk start), Vn [NT][C][V]. */
typedef struct {
  double *gamma, *A, *T, *W, *U, *S0, *Vn;
} chunk_dump;

static int chunked_chain(int64_t t0, int64_t L, int C, int Hqk, int Hv, int K, int V, int h,
                         const double* q, const double* k, const double* v, const double* g,
                         const double* beta, double scale, double* S /* [K][V] in h0 / out ht */,
                         double* o, chunk_scratch* sc, const chunk_dump* dump) {
  const int hq = h / (Hv / Hqk);
  int64_t ci = 0;
  for (int64_t s = t0; s < t0 + L; s += C, ++ci) {
    const int n = (int)((t0 + L - s) < C ? (t0 + L - s) : C); /* rows in this chunk */
#define KR(i) (k + ((s + (i)) * Hqk + hq) * (int64_t)K)
#define QR(i) (q + ((s + (i)) * Hqk + hq) * (int64_t)K)
#define VR(i) (v + ((s + (i)) * Hv + h) * (int64_t)V)
#define GV(i) (g[(s + (i)) * Hv + h])
#define BV(i) (beta[(s + (i)) * Hv + h])
    /* stage: cumsum */
    double acc = 0.0;
    for (int i = 0; i < n; ++i) { acc += GV(i); sc->gamma[i] = acc; }
    const double glast = sc->gamma[n - 1];
    /* stage: scaled_dot_kkt, A strictly lower triangular */
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        double a = 0.0;
        if (i > j) {
          double dot = 0.0;
          for (int d = 0; d < K; ++d) dot += KR(i)[d] * KR(j)[d];
          a = BV(i) * exp(sc->gamma[i] - sc->gamma[j]) * dot;
        }
        sc->A[i * n + j] = a;
      }
    /* stage: solve_tril, T = (I + A)^{-1} */
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) sc->M[i * n + j] = sc->A[i * n + j] + (i == j ? 1.0 : 0.0);
    int rc = gauss_jordan_inverse(n, sc->M, sc->T, sc->work);
    if (rc) return rc;
    /* stage: wy_fast, W = T diag(beta e^gamma) K, U = T diag(beta) V */
    for (int i = 0; i < n; ++i) {
      for (int d = 0; d < K; ++d) {
        double a = 0.0;
        for (int c = 0; c < n; ++c) a += sc->T[i * n + c] * BV(c) * exp(sc->gamma[c]) * KR(c)[d];
        sc->W[(int64_t)i * K + d] = a;
      }
      for (int e = 0; e < V; ++e) {
        double a = 0.0;
        for (int c = 0; c < n; ++c) a += sc->T[i * n + c] * BV(c) * VR(c)[e];
        sc->U[(int64_t)i * V + e] = a;
      }
    }
    /* stage: chunk_h, first half: V' = U - W S0 */
    for (int i = 0; i < n; ++i)
      for (int e = 0; e < V; ++e) {
        double a = 0.0;
        for (int d = 0; d < K; ++d) a += sc->W[(int64_t)i * K + d] * S[(int64_t)d * V + e];
        sc->Vn[(int64_t)i * V + e] = sc->U[(int64_t)i * V + e] - a;
      }
    if (dump) {
      const int64_t C2 = (int64_t)C * C;
      for (int i = 0; i < n; ++i) dump->gamma[ci * C + i] = sc->gamma[i];
      for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
          dump->A[ci * C2 + (int64_t)i * C + j] = sc->A[i * n + j];
          dump->T[ci * C2 + (int64_t)i * C + j] = sc->T[i * n + j];
        }
      memcpy(dump->W + ci * C * (int64_t)K, sc->W, sizeof(double) * (size_t)n * K);
      memcpy(dump->U + ci * C * (int64_t)V, sc->U, sizeof(double) * (size_t)n * V);
      memcpy(dump->Vn + ci * C * (int64_t)V, sc->Vn, sizeof(double) * (size_t)n * V);
      memcpy(dump->S0 + ci * (int64_t)K * V, S, sizeof(double) * (size_t)K * V);
    }
    /* stage: chunk_o,
     * O = scale (diag(e^gamma) Q S0 + (Q K^T o [j<=i] o e^{gamma_i-gamma_j}) V') */
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        double a = 0.0;
        if (j <= i) {
          double dot = 0.0;
          for (int d = 0; d < K; ++d) dot += QR(i)[d] * KR(j)[d];
          a = dot * exp(sc->gamma[i] - sc->gamma[j]);
        }
        sc->QK[i * n + j] = a;
      }
    for (int i = 0; i < n; ++i) {
      double* oi = o + ((s + i) * Hv + h) * (int64_t)V;
      for (int e = 0; e < V; ++e) {
        double inter = 0.0, intra = 0.0;
        for (int d = 0; d < K; ++d) inter += QR(i)[d] * S[(int64_t)d * V + e];
        for (int j = 0; j <= i; ++j) intra += sc->QK[i * n + j] * sc->Vn[(int64_t)j * V + e];
        oi[e] = scale * (exp(sc->gamma[i]) * inter + intra);
      }
    }
    /* stage: chunk_h, second half: S1 = e^{gamma_last} S0 + K^T diag(e^{gamma_last-gamma}) V' */
    for (int d = 0; d < K; ++d)
      for (int e = 0; e < V; ++e) {
        double a = 0.0;
        for (int c = 0; c < n; ++c) a += KR(c)[d] * exp(glast - sc->gamma[c]) * sc->Vn[(int64_t)c * V + e];
        S[(int64_t)d * V + e] = exp(glast) * S[(int64_t)d * V + e] + a;
      }
#undef KR
#undef QR
#undef VR
#undef GV
#undef BV
  }
  return ORACLE_OK;
}

static int alloc_scratch(chunk_scratch* sc, int C, int K, int V) {
  const size_t C2 = (size_t)C * C;
  size_t total = C + 4 * C2 + 2 * C2 /* work [C][2C] */ + (size_t)C * K + 2 * (size_t)C * V + (size_t)K * V;
  double* p = (double*)calloc(total, sizeof(double));
  if (!p) return ORACLE_ENOMEM;
  sc->gamma = p; p += C;
  sc->A = p; p += C2;
  sc->M = p; p += C2;
  sc->T = p; p += C2;
  sc->QK = p; p += C2;
  sc->work = p; p += 2 * C2;
  sc->W = p; p += (size_t)C * K;
  sc->U = p; p += (size_t)C * V;
  sc->Vn = p; p += (size_t)C * V;
  sc->S0 = p;
  return ORACLE_OK;
}

int oracle_chunked(int64_t Ttot, int N, const int64_t* cu, int Hqk, int Hv, int K, int V, int C,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, double scale, const double* h0, double* o, double* ht,
                   const int32_t* chain_ids, int n_chain_ids, int nthreads) {
  int rc = check_args(Ttot, N, cu, Hqk, Hv, K, V);
  if (rc) return rc;
  if (C <= 0) return ORACLE_EINVAL;
  const int nchains = chain_ids ? n_chain_ids : N * Hv;
  int err = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int c = 0; c < nchains; ++c) {
    const int id = chain_ids ? chain_ids[c] : c;
    const int n = id / Hv, h = id % Hv;
    chunk_scratch sc;
    if (alloc_scratch(&sc, C, K, V)) { err = ORACLE_ENOMEM; continue; }
    double* S = sc.S0;
    if (h0) memcpy(S, h0 + ((int64_t)n * Hv + h) * K * (int64_t)V, sizeof(double) * (size_t)K * V);
    int r = chunked_chain(cu[n], cu[n + 1] - cu[n], C, Hqk, Hv, K, V, h, q, k, v, g, beta, scale, S, o, &sc, NULL);
    if (r) err = r;
    if (ht) memcpy(ht + ((int64_t)n * Hv + h) * K * (int64_t)V, S, sizeof(double) * (size_t)K * V);
    free(sc.gamma);
  }
  (void)nthreads;
  return err;
}

/* Chunked form of one chain (n, h) with its per-chunk intermediates written
 * to the dump arrays (sized for NT = ceil(len / C) chunks, zero-filled by the
 * caller).  o / ht receive the chain's outputs as in oracle_chunked. */
int oracle_chunked_stages(int64_t Ttot, int N, const int64_t* cu, int Hqk, int Hv, int K, int V, int C,
                          const double* q, const double* k, const double* v, const double* g,
                          const double* beta, double scale, const double* h0, int n, int h,
                          double* o, double* ht, double* gamma, double* A, double* T, double* W,
                          double* U, double* S0, double* Vn) {
  int rc = check_args(Ttot, N, cu, Hqk, Hv, K, V);
  if (rc) return rc;
  if (C <= 0 || n < 0 || n >= N || h < 0 || h >= Hv) return ORACLE_EINVAL;
  chunk_scratch sc;
  if (alloc_scratch(&sc, C, K, V)) return ORACLE_ENOMEM;
  double* S = sc.S0;
  if (h0) memcpy(S, h0 + ((int64_t)n * Hv + h) * K * (int64_t)V, sizeof(double) * (size_t)K * V);
  chunk_dump dump = {gamma, A, T, W, U, S0, Vn};
  rc = chunked_chain(cu[n], cu[n + 1] - cu[n], C, Hqk, Hv, K, V, h, q, k, v, g, beta, scale, S, o, &sc, &dump);
  if (!rc && ht) memcpy(ht + ((int64_t)n * Hv + h) * K * (int64_t)V, S, sizeof(double) * (size_t)K * V);
  free(sc.gamma);
  return rc;
}
