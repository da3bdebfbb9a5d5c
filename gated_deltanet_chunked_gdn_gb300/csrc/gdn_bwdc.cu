// gdn_bwdc.cu -- chunked backward pass of the Gated DeltaNet forward for
// equal-length sequences (fp32 arithmetic on the stored inputs).
//
// Per 64-token chunk (rows i, j; padding rows have g = beta = 0 and zero
// k, q, v, dout) the forward is, with gamma the in-chunk cumsum of g,
// e = e^gamma, e_l = e at the last row, E_ij = e_i / e_j, D = e_l / e:
//   A = strict-lower(beta_i E_ij k_i.k_j),  T = (I + A)^-1
//   W = T diag(beta e) K,  U = T diag(beta) V,  V' = U - W S0
//   O = scale (diag(e) Q S0 + P V'),  P = lower(E_ij q_i.k_j)
//   S1 = e_l S0 + K^T diag(D) V'
// and its reverse mode, for G = dL/dS1:
//   dV' = D (K G) + scale P^T dO
//   dS0 = e_l G + scale Q^T diag(e) dO - W^T dV'            (the serial part)
//   dQ  = scale diag(e) dO S0^T + (dP o E) K,   dP = lower(scale dO V'^T)
//   dK  = diag(D) V' G^T + (dP o E)^T Q + diag(beta e) T^T dW + dKK K + dKK^T K
//   dW  = -dV' S0^T,  dT = dW (diag(beta e) K)^T + dV' (diag(beta) V)^T
//   dA  = strict-lower(-T^T dT T^T),  dKK = dA o beta_i E
//   dV  = diag(beta) T^T dV',  dbeta = e (K o T^T dW) 1 + (V o T^T dV') 1 + (dA o E o KK) 1
//   dgamma: <S1, G> at the last row, - D_i (K G)_i . V'_i,
//           scale e_i (Q S0)_i . dO_i, rowsum - colsum of dP o P and dA o A,
//           beta_i e_i k_i . (T^T dW)_i;   dg = reverse cumsum of dgamma.
// The chunk-start states S0 come from a serial forward over the chunks and G
// from a serial reverse (one CTA per chain and 32-column slice of V); every
// other product is a batched fp32 GEMM over all (chunk, head) pairs at once.
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kC = 64;      // chunk length
constexpr int kDh = 128;    // K = V
constexpr int kSl = 32;     // V columns per CTA of the serial kernels

// ---------------------------------------------------------------- batched GEMM
// C[b] = alpha diag(rs[b]) op(A[b]) op(B[b]) + beta C[b] for M, N multiples of
// 64 and Kd a multiple of 16; op(A)(i, k) = tA ? A[k lda + i] : A[i lda + k],
// op(B)(k, j) = tB ? B[j ldb + k] : B[k ldb + j]; rs may be null (all ones).
struct GemmArgs {
  const float* A;
  const float* B;
  float* C;
  const float* rs;
  int64_t sA, sB, sC, sR;
  int lda, ldb, ldc, M, N, Kd;
  bool tA, tB;
  float alpha, beta;
};

__global__ void __launch_bounds__(256) bgemm_kernel(const GemmArgs g) {
  __shared__ __align__(16) float As[16][64 + 4];
  __shared__ __align__(16) float Bs[16][64 + 4];
  const int64_t b = blockIdx.z;
  const int i0 = 64 * blockIdx.y, j0 = 64 * blockIdx.x;
  const float* A = g.A + b * g.sA;
  const float* B = g.B + b * g.sB;
  const int tid = threadIdx.x, ti = 4 * (tid >> 4), tj = 4 * (tid & 15);
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.Kd; k0 += 16) {
    for (int u = tid; u < 16 * 64; u += 256) {
      // A tile: (row i, k) -> As[k][i];  B tile: (k, col j) -> Bs[k][j]
      int kk, i;
      if (g.tA) { kk = u >> 6; i = u & 63; } else { i = u >> 4; kk = u & 15; }
      As[kk][i] = g.tA ? A[(int64_t)(k0 + kk) * g.lda + i0 + i] : A[(int64_t)(i0 + i) * g.lda + k0 + kk];
      int kb, j;
      if (g.tB) { j = u >> 4; kb = u & 15; } else { kb = u >> 6; j = u & 63; }
      Bs[kb][j] = g.tB ? B[(int64_t)(j0 + j) * g.ldb + k0 + kb] : B[(int64_t)(k0 + kb) * g.ldb + j0 + j];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ti]);
      const float4 c = *reinterpret_cast<const float4*>(&Bs[kk][tj]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(av[r], bv[s], acc[r][s]);
    }
    __syncthreads();
  }
  float* C = g.C + b * g.sC;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = i0 + ti + r;
    const float f = g.alpha * (g.rs ? g.rs[b * g.sR + i] : 1.f);
    float* c = C + (int64_t)i * g.ldc + j0 + tj;
#pragma unroll
    for (int s = 0; s < 4; ++s) c[s] = f * acc[r][s] + (g.beta != 0.f ? g.beta * c[s] : 0.f);
  }
}

// ------------------------------------------------------------ per-chunk data
// Workspace per (chunk, head) pair b, fp32 (padded to 64 rows):
struct Lay {
  int64_t nb;                 // pairs: N * Hv * NC
  float *K, *Q, *V, *dO;      // [nb][64][128]
  float *W, *U, *Vp, *dVp;    // [nb][64][128]
  float *X1, *X2, *X3, *X4;   // [nb][64][128] scratch
  float *dQ, *dK;             // [nb][64][128]
  float *KK, *P, *A, *T;      // [nb][64][64]
  float *M1, *M2, *M3;        // [nb][64][64] scratch
  float *S0, *G;              // [nb][128][128]
  float *vec;                 // [nb][8][64]: gamma, e, beta, D, beta e, dgamma, dbeta, spare
  size_t bytes;
};

Lay layout(const gdn_problem& p, uint8_t* base) {
  Lay L;
  const int64_t NC = ((int64_t)p.T + kC - 1) / kC;
  L.nb = (int64_t)p.N * p.Hv * NC;
  size_t off = 0;
  auto take = [&](size_t floats) {
    float* r = reinterpret_cast<float*>(base ? base + off : nullptr);
    off += ((floats * sizeof(float) + kAlign - 1) / kAlign) * kAlign;
    return r;
  };
  const size_t big = (size_t)L.nb * kC * kDh, sq = (size_t)L.nb * kC * kC, st = (size_t)L.nb * kDh * kDh;
  L.K = take(big); L.Q = take(big); L.V = take(big); L.dO = take(big);
  L.W = take(big); L.U = take(big); L.Vp = take(big); L.dVp = take(big);
  L.X1 = take(big); L.X2 = take(big); L.X3 = take(big); L.X4 = take(big);
  L.dQ = take(big); L.dK = take(big);
  L.KK = take(sq); L.P = take(sq); L.A = take(sq); L.T = take(sq);
  L.M1 = take(sq); L.M2 = take(sq); L.M3 = take(sq);
  L.S0 = take(st); L.G = take(st);
  L.vec = take((size_t)L.nb * 8 * kC);
  L.bytes = off;
  return L;
}

enum { kGam = 0, kE = 1, kBeta = 2, kD = 3, kBe = 4, kDgam = 5, kDbeta = 6 };
__device__ __forceinline__ float* vecp(const Lay& L, int64_t b, int which) { return L.vec + (b * 8 + which) * kC; }

template <typename Tin>
__device__ __forceinline__ float ldf(const Tin* p, int64_t i) { return to_f(p[i]); }

// Gather one pair's rows (fp32, zero-padded) and its per-row scalars.
// Grid nb, 256 threads.  Pair b = ((n Hv + h) NC + c).
template <typename Tin>
__global__ void __launch_bounds__(256) bwdc_gather(const Lay L, const Tin* q, const Tin* k, const Tin* v,
                                                   const Tin* dout, const float* g, const float* beta, int T, int NC,
                                                   int Hqk, int Hv) {
  const int64_t b = blockIdx.x;
  const int c = (int)(b % NC), h = (int)((b / NC) % Hv), n = (int)(b / ((int64_t)NC * Hv));
  const int hq = h / (Hv / Hqk);
  const int64_t t0 = (int64_t)n * T + (int64_t)c * kC;
  const int Lc = T - c * kC < kC ? T - c * kC : kC;
  const int tid = threadIdx.x;
  for (int u = tid; u < kC * kDh; u += 256) {
    const int i = u / kDh, d = u % kDh;
    const bool in = i < Lc;
    const int64_t qk = ((t0 + i) * Hqk + hq) * (int64_t)kDh + d, vo = ((t0 + i) * Hv + h) * (int64_t)kDh + d;
    L.K[b * kC * kDh + u] = in ? ldf(k, qk) : 0.f;
    L.Q[b * kC * kDh + u] = in ? ldf(q, qk) : 0.f;
    L.V[b * kC * kDh + u] = in ? ldf(v, vo) : 0.f;
    L.dO[b * kC * kDh + u] = in ? ldf(dout, vo) : 0.f;
  }
  if (tid < 32) {
    // gamma by a warp scan over two rows per lane
    float ga = 0.f, gb = 0.f, ba = 0.f, bb = 0.f;
    const int r0 = 2 * tid, r1 = 2 * tid + 1;
    if (r0 < Lc) { ga = g[(t0 + r0) * Hv + h]; ba = beta[(t0 + r0) * Hv + h]; }
    if (r1 < Lc) { gb = g[(t0 + r1) * Hv + h]; bb = beta[(t0 + r1) * Hv + h]; }
    float s = ga + gb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, off);
      if (tid >= off) s += y;
    }
    const float g0 = s - gb, g1 = s;
    const float gl = __shfl_sync(0xffffffffu, s, 31);
    float* gam = vecp(L, b, kGam);
    gam[r0] = g0; gam[r1] = g1;
    const float e0 = expf(g0), e1 = expf(g1);
    vecp(L, b, kE)[r0] = e0; vecp(L, b, kE)[r1] = e1;
    vecp(L, b, kBeta)[r0] = ba; vecp(L, b, kBeta)[r1] = bb;
    vecp(L, b, kD)[r0] = expf(gl - g0); vecp(L, b, kD)[r1] = expf(gl - g1);
    vecp(L, b, kBe)[r0] = ba * e0; vecp(L, b, kBe)[r1] = bb * e1;
    vecp(L, b, kDgam)[r0] = 0.f; vecp(L, b, kDgam)[r1] = 0.f;
    vecp(L, b, kDbeta)[r0] = 0.f; vecp(L, b, kDbeta)[r1] = 0.f;
  }
}

// A = strict-lower(beta_i E_ij KK_ij) and P = lower(E_ij QK_ij) (in place of
// the QK^T product in P).  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_masks(const Lay L) {
  const int64_t b = blockIdx.x;
  const float* gam = vecp(L, b, kGam);
  const float* bet = vecp(L, b, kBeta);
  for (int u = threadIdx.x; u < kC * kC; u += 256) {
    const int i = u / kC, j = u % kC;
    const float E = expf(gam[i] - gam[j]);
    const int64_t x = b * kC * kC + u;
    L.A[x] = i > j ? bet[i] * E * L.KK[x] : 0.f;
    L.P[x] = i >= j ? E * L.P[x] : 0.f;
  }
}

// T = (I + A)^-1 by forward substitution: thread l owns column l.  Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_solve(const Lay L) {
  const int64_t b = blockIdx.x;
  __shared__ float As[kC][kC + 1];
  const int l = threadIdx.x;
  for (int u = l; u < kC * kC; u += 64) As[u / kC][u % kC] = L.A[b * kC * kC + u];
  __syncthreads();
  float* T = L.T + b * kC * kC;
  float t[kC];
#pragma unroll
  for (int i = 0; i < kC; ++i) {
    float x = i == l ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < i; ++j) x = fmaf(-As[i][j], t[j], x);
    t[i] = x;
    T[i * kC + l] = x;
  }
}

// X1 = diag(beta e) K, X2 = diag(beta) V.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_scale_kv(const Lay L) {
  const int64_t b = blockIdx.x;
  const float* be = vecp(L, b, kBe);
  const float* bet = vecp(L, b, kBeta);
  for (int u = threadIdx.x; u < kC * kDh; u += 256) {
    const int i = u / kDh;
    const int64_t x = b * kC * kDh + u;
    L.X1[x] = be[i] * L.K[x];
    L.X2[x] = bet[i] * L.V[x];
  }
}

// Serial forward over a chain's chunks for 32 state columns: S0 of every
// chunk and V' = U - W S0.  Grid (N Hv, 4), 256 threads.
__global__ void __launch_bounds__(256) bwdc_fwd_states(const Lay L, const float* h0, int NC) {
  __shared__ __align__(16) float S[kDh][kSl];
  __shared__ __align__(16) float Vp[kC][kSl];
  const int64_t chain = blockIdx.x;
  const int e0 = kSl * blockIdx.y, tid = threadIdx.x;
  for (int u = tid; u < kDh * kSl; u += 256) {
    const int d = u / kSl, e = u % kSl;
    S[d][e] = h0 ? h0[(chain * kDh + d) * kDh + e0 + e] : 0.f;
  }
  __syncthreads();
  for (int c = 0; c < NC; ++c) {
    const int64_t b = chain * NC + c;
    // S0 out
    for (int u = tid; u < kDh * kSl; u += 256) {
      const int d = u / kSl, e = u % kSl;
      L.S0[(b * kDh + d) * kDh + e0 + e] = S[d][e];
    }
    // V' = U - W S0 (64 x 32): thread -> rows 4 (tid / 8) .. + 3... (64 rows x 32 cols / 256 = 8 per thread)
    {
      const int i = tid >> 2, c0 = 8 * (tid & 3);
      const float* Wr = L.W + (b * kC + i) * kDh;
      float acc[8];
#pragma unroll
      for (int s = 0; s < 8; ++s) acc[s] = L.U[(b * kC + i) * kDh + e0 + c0 + s];
      for (int d = 0; d < kDh; ++d) {
        const float w = Wr[d];
#pragma unroll
        for (int s = 0; s < 8; ++s) acc[s] = fmaf(-w, S[d][c0 + s], acc[s]);
      }
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        Vp[i][c0 + s] = acc[s];
        L.Vp[(b * kC + i) * kDh + e0 + c0 + s] = acc[s];
      }
    }
    __syncthreads();
    // S <- e_l S + K^T diag(D) V'  (128 x 32: 16 per thread)
    {
      const float* Dv = vecp(L, b, kD);
      const float el = vecp(L, b, kE)[kC - 1];
      const int d = tid >> 1, c0 = 16 * (tid & 1);
      float acc[16];
#pragma unroll
      for (int s = 0; s < 16; ++s) acc[s] = el * S[d][c0 + s];
      for (int i = 0; i < kC; ++i) {
        const float kd = L.K[(b * kC + i) * kDh + d] * Dv[i];
#pragma unroll
        for (int s = 0; s < 16; ++s) acc[s] = fmaf(kd, Vp[i][c0 + s], acc[s]);
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < 16; ++s) S[d][c0 + s] = acc[s];
    }
    __syncthreads();
  }
}

// Serial reverse over a chain's chunks for 32 columns of G = dL/dS1:
// G of every chunk (before its update), dV' = D (K G) + scale P^T dO, then
// G <- e_l G + scale Q^T diag(e) dO - W^T dV'.  dh0 = the last G.
// Grid (N Hv, 4), 256 threads.
__global__ void __launch_bounds__(256) bwdc_rev(const Lay L, const float* dht, float* dh0, int NC, float scale) {
  __shared__ __align__(16) float Gs[kDh][kSl];
  __shared__ __align__(16) float dV[kC][kSl];
  __shared__ __align__(16) float eD[kC][kSl];   // scale e_i dO_i
  const int64_t chain = blockIdx.x;
  const int e0 = kSl * blockIdx.y, tid = threadIdx.x;
  for (int u = tid; u < kDh * kSl; u += 256) {
    const int d = u / kSl, e = u % kSl;
    Gs[d][e] = dht ? dht[(chain * kDh + d) * kDh + e0 + e] : 0.f;
  }
  __syncthreads();
  for (int c = NC - 1; c >= 0; --c) {
    const int64_t b = chain * NC + c;
    const float* ev = vecp(L, b, kE);
    const float* Dv = vecp(L, b, kD);
    for (int u = tid; u < kDh * kSl; u += 256) {
      const int d = u / kSl, e = u % kSl;
      L.G[(b * kDh + d) * kDh + e0 + e] = Gs[d][e];
    }
    for (int u = tid; u < kC * kSl; u += 256) {
      const int i = u / kSl, e = u % kSl;
      eD[i][e] = scale * ev[i] * L.dO[(b * kC + i) * kDh + e0 + e];
    }
    __syncthreads();
    // dV' (64 x 32): D_i sum_d K_id G_de + scale sum_j P_ji dO_je
    {
      const int i = tid >> 2, c0 = 8 * (tid & 3);
      float acc[8] = {}, acc2[8] = {};
      const float* Kr = L.K + (b * kC + i) * kDh;
      for (int d = 0; d < kDh; ++d) {
        const float kd = Kr[d];
#pragma unroll
        for (int s = 0; s < 8; ++s) acc[s] = fmaf(kd, Gs[d][c0 + s], acc[s]);
      }
      for (int j = 0; j < kC; ++j) {
        const float pj = L.P[(b * kC + j) * kC + i];   // P^T(i, j) = P(j, i)
        const float* dOr = L.dO + (b * kC + j) * kDh + e0 + c0;
#pragma unroll
        for (int s = 0; s < 8; ++s) acc2[s] = fmaf(pj, dOr[s], acc2[s]);
      }
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float x = Dv[i] * acc[s] + scale * acc2[s];
        dV[i][c0 + s] = x;
        L.dVp[(b * kC + i) * kDh + e0 + c0 + s] = x;
      }
    }
    __syncthreads();
    // G <- e_l G + Q^T (scale e dO) - W^T dV'   (128 x 32)
    {
      const float el = ev[kC - 1];
      const int d = tid >> 1, c0 = 16 * (tid & 1);
      float acc[16];
#pragma unroll
      for (int s = 0; s < 16; ++s) acc[s] = el * Gs[d][c0 + s];
      for (int i = 0; i < kC; ++i) {
        const float qd = L.Q[(b * kC + i) * kDh + d], wd = L.W[(b * kC + i) * kDh + d];
#pragma unroll
        for (int s = 0; s < 16; ++s) acc[s] = fmaf(qd, eD[i][c0 + s], fmaf(-wd, dV[i][c0 + s], acc[s]));
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < 16; ++s) Gs[d][c0 + s] = acc[s];
    }
    __syncthreads();
  }
  if (dh0)
    for (int u = tid; u < kDh * kSl; u += 256) {
      const int d = u / kSl, e = u % kSl;
      dh0[(chain * kDh + d) * kDh + e0 + e] = Gs[d][e];
    }
}

// Row sums over the 128 columns of products of two [64][128] matrices: out[i]
// += f(i) sum_d X[i][d] Y[i][d].  mode 0: dgamma -= D_i (KG)_i . V'_i and
// dgamma[last] += e_l <S0, G> + sum_i D_i (KG)_i . V'_i (the <S1, G> term);
// mode 1: dgamma += scale e_i (Q S0)_i . dO_i.  Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_rowdots(const Lay L, int mode, float scale) {
  const int64_t b = blockIdx.x;
  const int i = threadIdx.x;
  const float* X = (mode == 0 ? L.X1 : L.X2) + (b * kC + i) * kDh;
  const float* Y = (mode == 0 ? L.Vp : L.dO) + (b * kC + i) * kDh;
  float s = 0.f;
  for (int d = 0; d < kDh; ++d) s = fmaf(X[d], Y[d], s);
  float* dg = vecp(L, b, kDgam);
  if (mode == 0) {
    const float t = vecp(L, b, kD)[i] * s;
    dg[i] -= t;
    // <S1, G> = e_l <S0, G> + sum_i t_i
    __shared__ float red[64], red2[64];
    const float* S0 = L.S0 + b * kDh * kDh;
    const float* G = L.G + b * kDh * kDh;
    float sg = 0.f;
    for (int x = i; x < kDh * kDh; x += 64) sg = fmaf(S0[x], G[x], sg);
    red[i] = t;
    red2[i] = sg;
    __syncthreads();
    if (i == 0) {
      float tot = 0.f, sgt = 0.f;
      for (int r = 0; r < 64; ++r) {
        tot += red[r];
        sgt += red2[r];
      }
      dg[kC - 1] += vecp(L, b, kE)[kC - 1] * sgt + tot;
    }
  } else {
    dg[i] += scale * vecp(L, b, kE)[i] * s;
  }
}

// dP = lower(M1) (M1 = scale dO V'^T): dgamma += rowsum(dP o P) - colsum(dP o P);
// M1 <- dP o E (for dQ += M1 K, dK += M1^T Q).  Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_dp(const Lay L) {
  const int64_t b = blockIdx.x;
  const int r = threadIdx.x;
  __shared__ float col[64][65];
  const float* gam = vecp(L, b, kGam);
  float rs = 0.f;
  for (int j = 0; j < kC; ++j) {
    const int64_t x = b * kC * kC + r * kC + j;
    const float dp = r >= j ? L.M1[x] : 0.f;
    const float pp = dp * L.P[x];
    rs += pp;
    col[r][j] = pp;
    L.M1[x] = r >= j ? dp * expf(gam[r] - gam[j]) : 0.f;
  }
  __syncthreads();
  float cs = 0.f;
  for (int i = 0; i < kC; ++i) cs += col[i][r];
  vecp(L, b, kDgam)[r] += rs - cs;
}

// From TdW = T^T dW and TdV = T^T dV': dK += diag(beta e) TdW, dbeta += e rowsum(K o TdW)
// + rowsum(V o TdV), dgamma += beta e rowsum(K o TdW), TdV <- diag(beta) TdV (= dV).
// Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_wy(const Lay L, const float* TdW, float* TdV) {
  const int64_t b = blockIdx.x;
  const int i = threadIdx.x;
  const float be = vecp(L, b, kBe)[i], bt = vecp(L, b, kBeta)[i], e = vecp(L, b, kE)[i];
  const int64_t r = (b * kC + i) * kDh;
  float kx = 0.f, vx = 0.f;
  for (int d = 0; d < kDh; ++d) {
    const float x3 = TdW[r + d], x4 = TdV[r + d];
    kx = fmaf(L.K[r + d], x3, kx);
    vx = fmaf(L.V[r + d], x4, vx);
    L.dK[r + d] = fmaf(be, x3, L.dK[r + d]);
    TdV[r + d] = bt * x4;
  }
  vecp(L, b, kDbeta)[i] += e * kx + vx;
  vecp(L, b, kDgam)[i] += be * kx;
}

// dA = strict-lower(M3) (M3 = -T^T dT T^T): dbeta += rowsum(dA o E o KK),
// dgamma += rowsum(dA o A) - colsum(dA o A), M3 <- dKK = dA o beta_i E.
// Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_da(const Lay L) {
  const int64_t b = blockIdx.x;
  const int r = threadIdx.x;
  __shared__ float col[64][65];
  const float* gam = vecp(L, b, kGam);
  const float bt = vecp(L, b, kBeta)[r];
  float db = 0.f, rs = 0.f;
  for (int j = 0; j < kC; ++j) {
    const int64_t x = b * kC * kC + r * kC + j;
    const float da = r > j ? L.M3[x] : 0.f;
    const float E = r > j ? expf(gam[r] - gam[j]) : 0.f;
    db = fmaf(da, E * L.KK[x], db);
    const float aa = da * L.A[x];
    rs += aa;
    col[r][j] = aa;
    L.M3[x] = da * bt * E;
  }
  __syncthreads();
  float cs = 0.f;
  for (int i = 0; i < kC; ++i) cs += col[i][r];
  vecp(L, b, kDgam)[r] += rs - cs;
  vecp(L, b, kDbeta)[r] += db;
}

// Scatter a pair's gradients: dq, dk (atomics across the value heads of a
// qk group), dv, dg (reverse cumsum of dgamma), dbeta.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_scatter(const Lay L, float* dq, float* dk, float* dv, float* dg,
                                                    float* dbeta, int T, int NC, int Hqk, int Hv) {
  const int64_t b = blockIdx.x;
  const int c = (int)(b % NC), h = (int)((b / NC) % Hv), n = (int)(b / ((int64_t)NC * Hv));
  const int hq = h / (Hv / Hqk);
  const int64_t t0 = (int64_t)n * T + (int64_t)c * kC;
  const int Lc = T - c * kC < kC ? T - c * kC : kC;
  const bool share = Hv != Hqk;
  for (int u = threadIdx.x; u < Lc * kDh; u += 256) {
    const int i = u / kDh, d = u % kDh;
    const int64_t qk = ((t0 + i) * Hqk + hq) * (int64_t)kDh + d, vo = ((t0 + i) * Hv + h) * (int64_t)kDh + d;
    const int64_t x = b * kC * kDh + u;
    if (share) {
      atomicAdd(dq + qk, L.dQ[x]);
      atomicAdd(dk + qk, L.dK[x]);
    } else {
      dq[qk] = L.dQ[x];
      dk[qk] = L.dK[x];
    }
    dv[vo] = L.X4[x];
  }
  if (threadIdx.x < 32) {
    // dg_s = sum_{i >= s} dgamma_i over all 64 rows (padding rows included:
    // the last row's <S1, G> term sits at row 63 of a tail chunk)
    const float* dgam = vecp(L, b, kDgam);
    const int lane = threadIdx.x;
    float a = dgam[2 * lane], bb = dgam[2 * lane + 1];
    float s = a + bb;   // suffix scan over lanes in reverse
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, s, off);
      if (lane + off < 32) s += y;
    }
    const float s0 = s, s1 = s - a;   // dg at rows 2 lane and 2 lane + 1
    const float* db = vecp(L, b, kDbeta);
    if (2 * lane < Lc) {
      dg[(t0 + 2 * lane) * Hv + h] = s0;
      dbeta[(t0 + 2 * lane) * Hv + h] = db[2 * lane];
    }
    if (2 * lane + 1 < Lc) {
      dg[(t0 + 2 * lane + 1) * Hv + h] = s1;
      dbeta[(t0 + 2 * lane + 1) * Hv + h] = db[2 * lane + 1];
    }
  }
}

// ------------------------------------------------------------------- host side
bool gemm(cudaStream_t s, int64_t nb, int M, int N, int Kd, float alpha, const float* A, int64_t sA, int lda,
          bool tA, const float* B, int64_t sB, int ldb, bool tB, float beta, float* C, int64_t sC, int ldc,
          const float* rs = nullptr, int64_t sR = 0) {
  GemmArgs g{A, B, C, rs, sA, sB, sC, sR, lda, ldb, ldc, M, N, Kd, tA, tB, alpha, beta};
  bgemm_kernel<<<dim3(N / 64, M / 64, (unsigned)nb), 256, 0, s>>>(g);
  return cudaGetLastError() == cudaSuccess;
}

template <typename Tin>
gdn_status run(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g, const float* beta,
               float scale, const float* h0, const void* dout, const float* dht, float* dq, float* dk, float* dv,
               float* dg, float* dbeta, float* dh0, void* ws, cudaStream_t s) {
  const int NC = (p.T + kC - 1) / kC;
  const Lay L = layout(p, static_cast<uint8_t*>(ws));
  const int64_t nb = L.nb, B2 = (int64_t)kC * kDh, Q2 = (int64_t)kC * kC, S2 = (int64_t)kDh * kDh, V8 = 8 * kC;
  const unsigned nbu = (unsigned)nb;
  const int64_t chains = (int64_t)p.N * p.Hv;
  bool ok = true;
  bwdc_gather<Tin><<<nbu, 256, 0, s>>>(L, static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                        static_cast<const Tin*>(v), static_cast<const Tin*>(dout), g, beta, p.T, NC,
                                        p.Hqk, p.Hv);
  // KK = K K^T, P <- Q K^T, then the masks, T, W and U
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.K, B2, kDh, false, L.K, B2, kDh, true, 0.f, L.KK, Q2, kC);
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.Q, B2, kDh, false, L.K, B2, kDh, true, 0.f, L.P, Q2, kC);
  bwdc_masks<<<nbu, 256, 0, s>>>(L);
  bwdc_solve<<<nbu, 64, 0, s>>>(L);
  bwdc_scale_kv<<<nbu, 256, 0, s>>>(L);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, false, L.X1, B2, kDh, false, 0.f, L.W, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, false, L.X2, B2, kDh, false, 0.f, L.U, B2, kDh);
  // the serial passes
  bwdc_fwd_states<<<dim3((unsigned)chains, kDh / kSl), 256, 0, s>>>(L, h0, NC);
  bwdc_rev<<<dim3((unsigned)chains, kDh / kSl), 256, 0, s>>>(L, dht, dh0, NC, scale);
  // dQ = scale diag(e) dO S0^T ;  dK = diag(D) V' G^T
  ok = ok && gemm(s, nb, kC, kDh, kDh, scale, L.dO, B2, kDh, false, L.S0, S2, kDh, true, 0.f, L.dQ, B2, kDh,
                  L.vec + kE * kC, V8);
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.Vp, B2, kDh, false, L.G, S2, kDh, true, 0.f, L.dK, B2, kDh,
                  L.vec + kD * kC, V8);
  // X1 = K G (the D (K G) . V' terms), X2 = Q S0 (the e (Q S0) . dO terms)
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.K, B2, kDh, false, L.G, S2, kDh, false, 0.f, L.X1, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.Q, B2, kDh, false, L.S0, S2, kDh, false, 0.f, L.X2, B2, kDh);
  bwdc_rowdots<<<nbu, 64, 0, s>>>(L, 0, scale);
  bwdc_rowdots<<<nbu, 64, 0, s>>>(L, 1, scale);
  // dP = lower(scale dO V'^T) -> (dP o E): dQ += . K, dK += .^T Q
  ok = ok && gemm(s, nb, kC, kC, kDh, scale, L.dO, B2, kDh, false, L.Vp, B2, kDh, true, 0.f, L.M1, Q2, kC);
  bwdc_dp<<<nbu, 64, 0, s>>>(L);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M1, Q2, kC, false, L.K, B2, kDh, false, 1.f, L.dQ, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M1, Q2, kC, true, L.Q, B2, kDh, false, 1.f, L.dK, B2, kDh);
  // dW = -dV' S0^T (X1); dT = dW (beta e K)^T + dV' (beta V)^T (M2)
  bwdc_scale_kv<<<nbu, 256, 0, s>>>(L);   // X1 = beta e K, X2 = beta V again (X1, X2 were reused)
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.dVp, B2, kDh, false, L.X2, B2, kDh, true, 0.f, L.M2, Q2, kC);
  ok = ok && gemm(s, nb, kC, kDh, kDh, -1.f, L.dVp, B2, kDh, false, L.S0, S2, kDh, true, 0.f, L.X3, B2, kDh);
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.X3, B2, kDh, false, L.X1, B2, kDh, true, 1.f, L.M2, Q2, kC);
  // X1 <- T^T dW, X4 = T^T dV'
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, true, L.X3, B2, kDh, false, 0.f, L.X1, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, true, L.dVp, B2, kDh, false, 0.f, L.X4, B2, kDh);
  bwdc_wy<<<nbu, 64, 0, s>>>(L, L.X1, L.X4);
  // dA = strict-lower(-T^T dT T^T): M1 = T^T dT, M3 = -M1 T^T
  ok = ok && gemm(s, nb, kC, kC, kC, 1.f, L.T, Q2, kC, true, L.M2, Q2, kC, false, 0.f, L.M1, Q2, kC);
  ok = ok && gemm(s, nb, kC, kC, kC, -1.f, L.M1, Q2, kC, false, L.T, Q2, kC, true, 0.f, L.M3, Q2, kC);
  bwdc_da<<<nbu, 64, 0, s>>>(L);
  // dK += dKK K + dKK^T K
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M3, Q2, kC, false, L.K, B2, kDh, false, 1.f, L.dK, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M3, Q2, kC, true, L.K, B2, kDh, false, 1.f, L.dK, B2, kDh);
  if (p.Hv != p.Hqk) {
    const size_t tq = sizeof(float) * (size_t)p.B * p.T * p.Hqk * p.K;
    if (cudaMemsetAsync(dq, 0, tq, s) != cudaSuccess || cudaMemsetAsync(dk, 0, tq, s) != cudaSuccess) return GDN_ERR_CUDA;
  }
  bwdc_scatter<<<nbu, 256, 0, s>>>(L, dq, dk, dv, dg, dbeta, p.T, NC, p.Hqk, p.Hv);
  ok = ok && cudaGetLastError() == cudaSuccess;
  return ok ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool bwdc_supported(const gdn_problem& p) { return !p.varlen && p.K == kDh && p.V == kDh && p.T > 0; }

size_t bwdc_workspace_bytes(const gdn_problem& p) { return kAlign + layout(p, nullptr).bytes; }

gdn_status run_bwdc(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                    const float* beta, float scale, const float* h0, const void* dout, const float* dht, float* dq,
                    float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws, cudaStream_t s) {
  int32_t* status = static_cast<int32_t*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  void* w = static_cast<uint8_t*>(ws) + kAlign;
  if (p.dt == GDN_F32) return run<float>(p, q, k, v, g, beta, scale, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, w, s);
  return run<__nv_bfloat16>(p, q, k, v, g, beta, scale, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, w, s);
}

}  // namespace gdn
