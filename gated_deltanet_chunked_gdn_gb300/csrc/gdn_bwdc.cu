// gdn_bwdc.cu -- chunked backward pass of the Gated DeltaNet forward for
// K = V = 128, equal-length or packed sequences (fp32 accuracy on the stored
// inputs: every product on the tensor cores as tf32 in three terms).
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
// from a serial reverse (one CTA per chain and 16-column slice of V); every
// other product is a batched GEMM over all (chunk, head) pairs at once.
#include <type_traits>

#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kC = 64;      // chunk length
constexpr int kDh = 128;    // K = V
constexpr int kSl = 16;     // V columns per CTA of the serial kernels

// ---------------------------------------------------------------- batched GEMM
// C[b] = alpha diag(rs[b]) op(A[b]) op(B[b]) diag(cs[b]) + beta C[b] for M, N
// multiples of 64 and Kd a multiple of 32; op(A)(i, k) = tA ? A[k lda + i] :
// A[i lda + k], op(B)(k, j) = tB ? B[j ldb + k] : B[k ldb + j]; rs and cs may
// be null (all ones).
struct GemmArgs {
  const float* A;
  const float* B;
  float* C;
  const float* rs;
  int64_t sA, sB, sC, sR;
  int lda, ldb, ldc, M, N, Kd;
  bool tA, tB;
  float alpha, beta;
  int exact;   // bit 0: op(A) is exact in tf32 (its lo part is zero), bit 1: op(B) is
  const float* cs;
  int64_t sCs;
};

// x = hi + lo, hi = x cut to its top 10 mantissa bits (exact tf32), lo = x - hi
// (exact in fp32); the three-term products hi hi + hi lo + lo hi leave about
// 2^-19 of each product (the lo lo term and the unit's truncation of lo, whose
// low 13 bits it ignores).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  // no side effects: not volatile, so that the compiler may schedule the
  // operand loads of later k-steps ahead of it
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64 x 64 tile of C per CTA on the tensor cores (mma.sync m16n8k8, tf32
// in three terms): warp w computes rows 16 (w % 4) .. + 15 and columns
// 32 (w / 4) .. + 31 as four 16 x 8 accumulators.  k-tiles of 32 go from global
// to shared memory by cp.async through a ring of three stages (two k-tiles in
// flight while the tensor cores work on the third), in the operands' own
// orientation (A as [m][k] with row stride 36 or [k][m] with 72, B as [k][n]
// with 72 or [n][k] with 36: the fragment loads of a warp then hit 32
// different banks).  Dynamic shared memory kGemmSmem.
constexpr int kGemmStages = 3, kGemmBuf = 64 * 36;
constexpr int kGemmSmem = 2 * kGemmStages * kGemmBuf * 4;
template <bool TA, bool TB>
__global__ void __launch_bounds__(256, 4) bgemm_kernel(const GemmArgs g) {
  constexpr int kT = 32, kBuf = kGemmBuf;
  constexpr int sAm = TA ? 1 : 36, sAk = TA ? 72 : 1;   // A(m, k) at As[m sAm + k sAk]
  constexpr int sBk = TB ? 1 : 36 * 2, sBn = TB ? 36 : 1;
  extern __shared__ __align__(16) float gsm[];
  float* const As = gsm;
  float* const Bs = gsm + kGemmStages * kBuf;
  const int64_t b = blockIdx.z;
  const int i0 = 64 * blockIdx.y, j0 = 64 * blockIdx.x;
  const float* A = g.A + b * g.sA;
  const float* B = g.B + b * g.sB;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, gq = lane >> 2, tq = lane & 3;
  const int mt = w & 3, nh = w >> 2;
  // this thread's float4 pieces: row (TA: k, else m) ar + {0, half}, column aq
  const int ar = TA ? tid >> 4 : tid >> 3, aq = TA ? 4 * (tid & 15) : 4 * (tid & 7), ah_ = TA ? 16 : 32;
  const int br = TB ? tid >> 3 : tid >> 4, bq = TB ? 4 * (tid & 7) : 4 * (tid & 15), bh_ = TB ? 32 : 16;
  const int sa = TA ? 72 : 36, sb = TB ? 36 : 72;   // shared row strides
  // this thread's 16-byte pieces of a k-tile, straight to shared memory
  auto issue = [&](int stage, int k0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      cp_async16(As + stage * kBuf + (ar + r * ah_) * sa + aq,
                 TA ? A + (int64_t)(k0 + ar + r * ah_) * g.lda + i0 + aq : A + (int64_t)(i0 + ar + r * ah_) * g.lda + k0 + aq);
      cp_async16(Bs + stage * kBuf + (br + r * bh_) * sb + bq,
                 TB ? B + (int64_t)(j0 + br + r * bh_) * g.ldb + k0 + bq : B + (int64_t)(k0 + br + r * bh_) * g.ldb + j0 + bq);
    }
    cp_async_commit();
  };
  float acc[4][4] = {};
  const int nk = g.Kd / kT;
  issue(0, 0);
  if (nk > 1) issue(1, kT);
  for (int kt = 0; kt < nk; ++kt) {
    // k-tile kt has landed once at most one later group is still pending
    if (kt + 1 < nk) cp_async_wait_prev(); else cp_async_wait_all();
    __syncthreads();   // every thread's pieces are in; stage (kt + 2) % 3 is free
    if (kt + 2 < nk) issue((kt + 2) % kGemmStages, (kt + 2) * kT);
    const int buf = kt % kGemmStages;
    const float* as = As + buf * kBuf + (16 * mt + gq) * sAm + tq * sAk;
    const float* bs = Bs + buf * kBuf + (32 * nh + gq) * sBn + tq * sBk;
#pragma unroll
    for (int ks = 0; ks < kT; ks += 8) {
      // A fragment: (row g, k t), (g + 8, t), (g, t + 4), (g + 8, t + 4) of m-tile mt
      uint32_t ah[4], al[4];
      split_tf32(as[ks * sAk], ah[0], al[0]);
      split_tf32(as[ks * sAk + 8 * sAm], ah[1], al[1]);
      split_tf32(as[(ks + 4) * sAk], ah[2], al[2]);
      split_tf32(as[(ks + 4) * sAk + 8 * sAm], ah[3], al[3]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        // B fragment: (k t, col g), (k t + 4, col g) of n-tile nt
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(bs[ks * sBk + 8 * nt * sBn], bh0, bl0);
        split_tf32(bs[(ks + 4) * sBk + 8 * nt * sBn], bh1, bl1);
        if (!(g.exact & 1)) mma_tf32(acc[nt], al[0], al[1], al[2], al[3], bh0, bh1);
        if (!(g.exact & 2)) mma_tf32(acc[nt], ah[0], ah[1], ah[2], ah[3], bl0, bl1);
        mma_tf32(acc[nt], ah[0], ah[1], ah[2], ah[3], bh0, bh1);
      }
    }
  }
  // accumulator nt: (row g, cols 2t, 2t + 1) and (row g + 8, same cols).  All
  // loads of the epilogue (row and column scales, C for beta) are issued before
  // its first store: the compiler cannot reorder them past stores to C.
  float* C = g.C + b * g.sC;
  const int jc = j0 + 32 * nh + 2 * tq;
  float2 cv[4], cx[2][4];
  float f[2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
    cv[nt] = g.cs ? *reinterpret_cast<const float2*>(g.cs + b * g.sCs + jc + 8 * nt) : make_float2(1.f, 1.f);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = i0 + 16 * mt + gq + 8 * h;
    f[h] = g.alpha * (g.rs ? g.rs[b * g.sR + i] : 1.f);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      cx[h][nt] = g.beta != 0.f ? *reinterpret_cast<const float2*>(C + (int64_t)i * g.ldc + jc + 8 * nt)
                                : make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = i0 + 16 * mt + gq + 8 * h;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float2 o = make_float2(fmaf(f[h] * acc[nt][2 * h], cv[nt].x, g.beta * cx[h][nt].x),
                                   fmaf(f[h] * acc[nt][2 * h + 1], cv[nt].y, g.beta * cx[h][nt].y));
      *reinterpret_cast<float2*>(C + (int64_t)i * g.ldc + jc + 8 * nt) = o;
    }
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
  float *S0, *G, *H;          // [nb][128][128]
  float *vec;                 // [nb][8][64]: gamma, e, beta, D, beta e, dgamma, dbeta, spare
  int4* pinfo;                // packed sequences: [nb] {first token, rows, value head, chain} of pair b
                              // (rows = 0: a padding pair); null for equal lengths
  int2* cinfo;                // packed sequences: [N Hv] {first pair, chunks} of chain n Hv + h
  size_t bytes;
};

// Pairs of a packed batch: at most ceil(T / 64) + N chunks a value head.
int64_t varlen_pairs(const gdn_problem& p) {
  const int64_t Ttot = (int64_t)p.B * p.T;
  return (int64_t)p.Hv * ((Ttot + kC - 1) / kC + p.N);
}

Lay layout(const gdn_problem& p, uint8_t* base) {
  Lay L;
  const int64_t NC = ((int64_t)p.T + kC - 1) / kC;
  L.nb = p.varlen ? varlen_pairs(p) : (int64_t)p.N * p.Hv * NC;
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
  L.S0 = take(st); L.G = take(st); L.H = take(st);
  L.pinfo = p.varlen ? reinterpret_cast<int4*>(take((size_t)L.nb * 4)) : nullptr;
  L.cinfo = p.varlen ? reinterpret_cast<int2*>(take((size_t)p.N * p.Hv * 2)) : nullptr;
  L.vec = take((size_t)L.nb * 8 * kC);
  L.bytes = off;
  return L;
}

enum { kGam = 0, kE = 1, kBeta = 2, kD = 3, kBe = 4, kDgam = 5, kDbeta = 6 };
__device__ __forceinline__ float* vecp(const Lay& L, int64_t b, int which) { return L.vec + (b * 8 + which) * kC; }

// Packed sequences: validates cu_seqlens (0 <= cu[n] <= cu[n + 1] <= Ttot,
// cu[0] = 0, cu[N] = Ttot) and writes the chain and pair tables.  Chain
// n Hv + h owns pairs Hv P_n + h C_n .. + C_n - 1 (C_n = ceil(L_n / 64) chunks,
// P_n their exclusive prefix over the sequences); its pair c holds tokens
// cu[n] + 64 c .. + min(64, L_n - 64 c) - 1.  The pairs past the last chain's
// are padding (no rows: they compute zeros and scatter nothing).  A malformed
// cu_seqlens sets the status word and leaves every chain and pair empty.  One
// CTA of 1024 threads.
__global__ void __launch_bounds__(1024) bwdc_prepare(const Lay L, const int32_t* cu, int N, int64_t Ttot, int Hv,
                                                     int32_t* status) {
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int ok = 1;
  for (int n = tid; n < N; n += 1024) {
    const int64_t a = cu[n], e = cu[n + 1];
    if (!(0 <= a && a <= e && e <= Ttot)) ok = 0;
  }
  if (tid == 0 && (cu[0] != 0 || cu[N] != Ttot)) ok = 0;
  ok = __syncthreads_and(ok);
  for (int64_t b = tid; b < L.nb; b += 1024) L.pinfo[b] = make_int4(0, 0, 0, 0);
  if (!ok) {
    if (tid == 0) atomicExch(status, GDN_DEV_BAD_CU_SEQLENS);
    for (int64_t c = tid; c < (int64_t)N * Hv; c += 1024) L.cinfo[c] = make_int2(0, 0);
    return;
  }
  __syncthreads();   // the padding entries are written before the real ones
  int carry = 0;     // chunks of the sequences before this tile
  for (int n0 = 0; n0 < N; n0 += 1024) {
    const int n = n0 + tid;
    const int64_t t0 = n < N ? cu[n] : 0, len = n < N ? cu[n + 1] - t0 : 0;
    const int nc = (int)((len + kC - 1) / kC);
    int x = nc;   // inclusive scan within the warp, then over the warp sums
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int v = wsum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      wsum[lane] = v;   // inclusive over warps
    }
    __syncthreads();
    const int pre = carry + (warp > 0 ? wsum[warp - 1] : 0) + x - nc;
    if (n < N) {
      for (int h = 0; h < Hv; ++h) {
        const int base = Hv * pre + h * nc;
        L.cinfo[(int64_t)n * Hv + h] = make_int2(base, nc);
        for (int c = 0; c < nc; ++c) {
          const int64_t rest = len - (int64_t)kC * c;
          L.pinfo[base + c] = make_int4((int)(t0 + (int64_t)kC * c), rest < kC ? (int)rest : kC, h, n * Hv + h);
        }
      }
    }
    carry += wsum[31];
    __syncthreads();   // wsum is rewritten by the next tile
  }
}

// First token, valid rows and value head of pair b: from the pair table for
// packed sequences, else b = (n Hv + h) NC + c over sequences of T tokens.
__device__ __forceinline__ void pair_rows(const Lay& L, int64_t b, int T, int NC, int Hv, int64_t& t0, int& Lc,
                                          int& h) {
  if (L.pinfo) {
    const int4 pi = L.pinfo[b];
    t0 = pi.x;
    Lc = pi.y;
    h = pi.z;
  } else {
    const int c = (int)(b % NC), n = (int)(b / ((int64_t)NC * Hv));
    h = (int)((b / NC) % Hv);
    t0 = (int64_t)n * T + (int64_t)c * kC;
    Lc = T - c * kC < kC ? T - c * kC : kC;
  }
}

// Four consecutive elements (16-byte aligned for fp32, 8-byte for bf16) as fp32.
__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4f(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// Gather one pair's rows (fp32, zero-padded) and its per-row scalars.
// Grid nb, 256 threads.  Pair b = ((n Hv + h) NC + c).
template <typename Tin>
__global__ void __launch_bounds__(256) bwdc_gather(const Lay L, const Tin* q, const Tin* k, const Tin* v,
                                                   const Tin* dout, const float* g, const float* beta, int T, int NC,
                                                   int Hqk, int Hv) {
  const int64_t b = blockIdx.x;
  int64_t t0;
  int Lc, h;
  pair_rows(L, b, T, NC, Hv, t0, Lc, h);
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int u = tid; u < kC * kDh / 4; u += 256) {
    const int i = (4 * u) / kDh, d = (4 * u) % kDh;
    const bool in = i < Lc;
    const int64_t qk = ((t0 + i) * Hqk + hq) * (int64_t)kDh + d, vo = ((t0 + i) * Hv + h) * (int64_t)kDh + d;
    reinterpret_cast<float4*>(L.K + b * kC * kDh)[u] = in ? ld4f(k + qk) : z;
    reinterpret_cast<float4*>(L.Q + b * kC * kDh)[u] = in ? ld4f(q + qk) : z;
    reinterpret_cast<float4*>(L.V + b * kC * kDh)[u] = in ? ld4f(v + vo) : z;
    reinterpret_cast<float4*>(L.dO + b * kC * kDh)[u] = in ? ld4f(dout + vo) : z;
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

// T = (I + A)^-1 by forward substitution: thread l owns column l; also
// T diag(beta e) (in M1) and T diag(beta) (in M2), the left factors of W and
// U.  Grid nb, 64 threads.
__global__ void __launch_bounds__(64) bwdc_solve(const Lay L) {
  const int64_t b = blockIdx.x;
  __shared__ float As[kC][kC + 1];
  const int l = threadIdx.x;
  for (int u = l; u < kC * kC; u += 64) As[u / kC][u % kC] = L.A[b * kC * kC + u];
  __syncthreads();
  float* T = L.T + b * kC * kC;
  float* Tbe = L.M1 + b * kC * kC;
  float* Tb = L.M2 + b * kC * kC;
  const float fbe = vecp(L, b, kBe)[l], fb = vecp(L, b, kBeta)[l];
  float t[kC];
#pragma unroll
  for (int i = 0; i < kC; ++i) {
    float x = i == l ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < i; ++j) x = fmaf(-As[i][j], t[j], x);
    t[i] = x;
    T[i * kC + l] = x;
    Tbe[i * kC + l] = x * fbe;
    Tb[i * kC + l] = x * fb;
  }
}

// L2 prefetch of rows x (cols floats) of a row-major matrix.
__device__ __forceinline__ void prefetch_rows(const float* src, int64_t ld, int rows, int cols, int tid, int nthreads) {
  const int lines = (cols * 4 + 127) / 128;
  for (int u = tid; u < rows * lines; u += nthreads) {
    const float* p = src + (u / lines) * ld + 32 * (u % lines);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  }
}

// The serial passes run their two products per chunk on the same three-term
// tf32 MMAs.  Operands that sit in shared memory are stored in fp32, in the
// order of the MMA fragments, so that a lane reads its four values of a
// k-step with one 16-byte load; every warp splits what it reads into hi and lo
// (a few integer and FMA operations, where shared-memory reads are the scarce
// resource: the V' product's warps all read the whole state slice).
// A [128][16] slice X (the state, or G) as the A operand of X^T R^T: k-step
// ks = 2 kk + p covers rows d = 16 kk + 4 t + 2 p (fragment column t) and
// d + 1 (column t + 4), fragment row g = column c % 8, c / 8 = the lower or
// upper 8 rows; lane 4 g + t holds {(d, g), (d, g + 8), (d + 1, g), (d + 1, g + 8)}
// in 16-byte chunk ks * 32 + lane.  Within each 128-byte row of chunks (row =
// chunk / 8) the chunk position is XORed with xf_swz(row): a lane's read stays
// one 16-byte load, a quarter warp still reads one row (conflict-free), and the
// scattered stores of the state meet at most two to a bank instead of eight.
__device__ __forceinline__ int xf_swz(int row) { return 2 * (row & 3) + ((row >> 2) & 1); }
__device__ __forceinline__ int xf_index(int d, int c) {
  const int ks = 2 * (d >> 4) + ((d >> 1) & 1), t = (d >> 2) & 3;
  const int ch = ks * 32 + 4 * (c & 7) + t;
  return (((ch & ~7) | ((ch & 7) ^ xf_swz(ch >> 3))) << 2) + 2 * (d & 1) + (c >> 3);
}
// Chunk of lane `lane` in k-step ks of the X array (rows ks * 4 + lane / 8).
__device__ __forceinline__ int xf_chunk(int ks, int lane) {
  return ks * 32 + (lane & ~7) + ((lane & 7) ^ (2 * (lane >> 3) + (ks & 1)));
}
// A [64][16] slice V as the B operand of Col^T V: k-step ks covers rows
// 8 ks + t (fragment row t) and 8 ks + t + 4 (row t + 4), fragment column g
// = c % 8 of n-tile c / 8; lane 4 g + t holds {b0, b1} of n-tile 0, then of 1,
// in chunk ks * 32 + lane, XORed within its row by (row / 2) % 2 (the stores
// of V' then meet at most two to a bank instead of four).
__device__ __forceinline__ int vf_index(int i, int c) {
  const int ch = (i >> 3) * 32 + 4 * (c & 7) + (i & 3);
  return (((ch & ~7) | ((ch & 7) ^ ((ch >> 4) & 1))) << 2) + 2 * (c >> 3) + ((i >> 2) & 1);
}
__device__ __forceinline__ int vf_chunk(int ks, int lane) {
  return ks * 32 + (lane & ~7) + ((lane & 7) ^ ((lane >> 4) & 1));
}
constexpr int kXF = kDh * kSl;   // floats of one XF array
constexpr int kVF = kC * kSl;    // floats of one VF array

// hi and lo parts of a 16-byte fragment load
__device__ __forceinline__ void split4(const float4& x, uint4& hi, uint4& lo) {
  split_tf32(x.x, hi.x, lo.x);
  split_tf32(x.y, hi.y, lo.y);
  split_tf32(x.z, hi.z, lo.z);
  split_tf32(x.w, hi.w, lo.w);
}

// out = (R X)[i][c] at i = 8 w + 2 t (+1), c = g (+8): out[0] = (i, c),
// out[1] = (i + 1, c), out[2] = (i, c + 8), out[3] = (i + 1, c + 8).  The warp
// computes n-tile w of X^T R^T over 16 k-steps; r[kk] holds R[8 w + g][16 kk + 4 t .. + 3].
template <bool REXACT>   // R exact in tf32: its lo term is dropped
__device__ __forceinline__ void row_product(const float4 (&r)[8], const float* xs, int lane, float (&out)[4]) {
  // four independent accumulators (even / odd k-steps x main / correction
  // terms) keep the MMA dependency chains short
  float acc[4][4] = {};
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const float rv[4] = {r[kk].x, r[kk].y, r[kk].z, r[kk].w};
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int ks = 2 * kk + p;
      uint32_t bh0, bl0, bh1, bl1;
      split_tf32(rv[2 * p], bh0, bl0);
      split_tf32(rv[2 * p + 1], bh1, bl1);
      uint4 ah, al;
      split4(*reinterpret_cast<const float4*>(xs + (xf_chunk(ks, lane) << 2)), ah, al);
      mma_tf32(acc[2 * p + 1], al.x, al.y, al.z, al.w, bh0, bh1);
      if (!REXACT) mma_tf32(acc[2 * p + 1], ah.x, ah.y, ah.z, ah.w, bl0, bl1);
      mma_tf32(acc[2 * p], ah.x, ah.y, ah.z, ah.w, bh0, bh1);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) out[q] = (acc[1][q] + acc[3][q]) + (acc[0][q] + acc[2][q]);
}

// st[nt] += sign Col^T V for the rows d = 16 w + g (+8) and columns 8 nt + 2 t
// (+1) (the C fragments of m-tile w); col[4 ks + r] holds Col[8 ks + t (+4 for
// r >= 2)][16 w + g (+8 for odd r)].
template <bool CEXACT>   // Col exact in tf32: its lo term is dropped
__device__ __forceinline__ void col_product(float (&st)[2][4], const float (&col)[32], const float* vs, int lane,
                                            float sign) {
  float cor[2][4] = {};   // the correction terms, in their own accumulators
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t ah[4], al[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) split_tf32(sign * col[4 * ks + r], ah[r], al[r]);
    uint4 bh, bl;
    split4(*reinterpret_cast<const float4*>(vs + (vf_chunk(ks, lane) << 2)), bh, bl);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t h0 = nt ? bh.z : bh.x, h1 = nt ? bh.w : bh.y;
      const uint32_t l0 = nt ? bl.z : bl.x, l1 = nt ? bl.w : bl.y;
      if (!CEXACT) mma_tf32(cor[nt], al[0], al[1], al[2], al[3], h0, h1);
      mma_tf32(cor[nt], ah[0], ah[1], ah[2], ah[3], l0, l1);
      mma_tf32(st[nt], ah[0], ah[1], ah[2], ah[3], h0, h1);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) st[nt][q] += cor[nt][q];
}

// Row d and column c of state element r of the C fragment st[nt][r].
__device__ __forceinline__ int st_row(int w, int g, int r) { return 16 * w + g + 8 * (r >> 1); }
__device__ __forceinline__ int st_col(int t, int nt, int r) { return 8 * nt + 2 * t + (r & 1); }

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Serial forward over a chain's chunks for the 16 state columns e0 .. e0 + 15:
// S0 of every chunk, V' = U - W S0 and S <- e_l S + K^T diag(D) V'.  The
// state slice lives in the MMA accumulators of the state update (warp w: rows
// 16 w .. 16 w + 15) and, split for the next V' product, in shared memory;
// each lane holds its fragments of the chunk's W rows and K columns in
// registers, loaded one chunk ahead so that their latency hides behind the
// arithmetic of the chunk before.  KEXACT: K holds bf16 values (exact in
// tf32).  Grid (N Hv, 8), 256 threads.
template <bool KEXACT>
__global__ void __launch_bounds__(256, 2) bwdc_fwd_states(const Lay L, const float* h0, int NC) {
  __shared__ __align__(16) float xs[kXF], vs[kVF];
  const int64_t chain = blockIdx.x;
  int64_t b0 = chain * NC;
  int nc = NC;
  if (L.cinfo) {
    const int2 ci = L.cinfo[chain];
    b0 = ci.x;
    nc = ci.y;
  }
  if (nc == 0) return;   // an empty sequence has no chunk states
  const int e0 = kSl * blockIdx.y, tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int i0 = 8 * w + 2 * t;   // rows i0, i0 + 1 of the V' product's output
  float st[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = st_row(w, g, r), c = st_col(t, nt, r);
      st[nt][r] = h0 ? h0[(chain * kDh + d) * kDh + e0 + c] : 0.f;   // h0 may be 4-byte aligned only
      xs[xf_index(d, c)] = st[nt][r];
    }
  auto put_s0 = [&](int64_t b) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        *reinterpret_cast<float2*>(L.S0 + (b * kDh + st_row(w, g, 2 * h)) * kDh + e0 + st_col(t, nt, 0)) =
            make_float2(st[nt][2 * h], st[nt][2 * h + 1]);
  };
  put_s0(b0);
  float4 wr[8];
  float ur[4], dr[2], kc[32], el;
  auto load_r = [&](int64_t b) {   // W rows 8 w + g; U and D at the V' product's output
    const float* wp = L.W + (b * kC + 8 * w + g) * kDh + 4 * t;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) wr[kk] = ldg4(wp + 16 * kk);
    const float* up = L.U + (b * kC + i0) * kDh + e0 + g;
    ur[0] = __ldg(up), ur[1] = __ldg(up + kDh), ur[2] = __ldg(up + 8), ur[3] = __ldg(up + kDh + 8);
    const float* dp = vecp(L, b, kD) + i0;
    dr[0] = __ldg(dp), dr[1] = __ldg(dp + 1);
  };
  auto load_c = [&](int64_t b) {   // K columns 16 w + g (+8) at rows 8 ks + t (+4)
    const float* kp = L.K + (b * kC + t) * kDh + 16 * w + g;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      kc[4 * ks] = __ldg(kp + 8 * ks * kDh);
      kc[4 * ks + 1] = __ldg(kp + 8 * ks * kDh + 8);
      kc[4 * ks + 2] = __ldg(kp + (8 * ks + 4) * kDh);
      kc[4 * ks + 3] = __ldg(kp + (8 * ks + 4) * kDh + 8);
    }
    el = __ldg(vecp(L, b, kE) + kC - 1);
  };
  load_r(b0);
  load_c(b0);
  __syncthreads();
#pragma unroll 1
  for (int c = 0; c < nc; ++c) {
    const int64_t b = b0 + c;
    if (c + 2 < nc) {
      prefetch_rows(L.W + (b + 2) * kC * kDh, kDh, kC, kDh, tid, 256);
      prefetch_rows(L.K + (b + 2) * kC * kDh, kDh, kC, kDh, tid, 256);
    }
    {
      // V' = U - W S0 at rows i0, i0 + 1 and columns g, g + 8
      float o[4];
      row_product<false>(wr, xs, lane, o);
      const float v[4] = {ur[0] - o[0], ur[1] - o[1], ur[2] - o[2], ur[3] - o[3]};
      const float d0 = dr[0], d1 = dr[1];
      if (c + 1 < nc) load_r(b + 1);
      float* vp = L.Vp + (b * kC + i0) * kDh + e0 + g;
      vp[0] = v[0], vp[kDh] = v[1], vp[8] = v[2], vp[kDh + 8] = v[3];
      vs[vf_index(i0, g)] = d0 * v[0];
      vs[vf_index(i0 + 1, g)] = d1 * v[1];
      vs[vf_index(i0, g + 8)] = d0 * v[2];
      vs[vf_index(i0 + 1, g + 8)] = d1 * v[3];
    }
    __syncthreads();
    {
      // S <- e_l S + K^T (D V')
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) st[nt][r] *= el;
      col_product<KEXACT>(st, kc, vs, lane, 1.f);
      if (c + 1 < nc) {
        load_c(b + 1);
        put_s0(b + 1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) xs[xf_index(st_row(w, g, r), st_col(t, nt, r))] = st[nt][r];
      }
    }
    __syncthreads();
  }
}

// Serial reverse over a chain's chunks for 16 columns of G = dL/dS1, with the
// G-independent terms computed beforehand by batched GEMMs (X = scale P^T dO
// in dVp, H = scale Q^T diag(e) dO): G of every chunk (before its update),
// dV' = D (K G) + X (over X in dVp), G <- e_l G + H - W^T dV'; dh0 = the last
// G.  Same arrangement as the forward pass, with K rows and W columns.  Grid
// (N Hv, 8), 256 threads.
template <bool KEXACT>
__global__ void __launch_bounds__(256, 2) bwdc_rev(const Lay L, const float* dht, float* dh0, int NC) {
  __shared__ __align__(16) float xs[kXF], vs[kVF];
  const int64_t chain = blockIdx.x;
  int64_t b0 = chain * NC;
  int nc = NC;
  if (L.cinfo) {
    const int2 ci = L.cinfo[chain];
    b0 = ci.x;
    nc = ci.y;
  }
  const int e0 = kSl * blockIdx.y, tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int i0 = 8 * w + 2 * t;
  if (nc == 0) {
    // an empty sequence passes dht through: dh0 = dht
    if (dh0)
      for (int u = tid; u < kDh * kSl; u += 256) {
        const int64_t at = (chain * kDh + u / kSl) * kDh + e0 + u % kSl;
        dh0[at] = dht ? dht[at] : 0.f;
      }
    return;
  }
  float st[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = st_row(w, g, r), cc = st_col(t, nt, r);
      st[nt][r] = dht ? dht[(chain * kDh + d) * kDh + e0 + cc] : 0.f;   // dht may be 4-byte aligned only
      xs[xf_index(d, cc)] = st[nt][r];
    }
  auto put_g = [&](int64_t b) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        *reinterpret_cast<float2*>(L.G + (b * kDh + st_row(w, g, 2 * h)) * kDh + e0 + st_col(t, nt, 0)) =
            make_float2(st[nt][2 * h], st[nt][2 * h + 1]);
  };
  put_g(b0 + nc - 1);
  float4 kr[8];
  float xr[4], dr[2], wc[32], hr[2][4], el;
  auto load_r = [&](int64_t b) {   // K rows 8 w + g; X and D at the dV' product's output
    const float* kp = L.K + (b * kC + 8 * w + g) * kDh + 4 * t;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) kr[kk] = ldg4(kp + 16 * kk);
    const float* xp = L.dVp + (b * kC + i0) * kDh + e0 + g;
    xr[0] = xp[0], xr[1] = xp[kDh], xr[2] = xp[8], xr[3] = xp[kDh + 8];   // plain loads: this kernel writes dVp
    const float* dp = vecp(L, b, kD) + i0;
    dr[0] = __ldg(dp), dr[1] = __ldg(dp + 1);
  };
  auto load_c = [&](int64_t b) {   // W columns 16 w + g (+8) at rows 8 ks + t (+4); H at the state's places
    const float* wp = L.W + (b * kC + t) * kDh + 16 * w + g;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      wc[4 * ks] = __ldg(wp + 8 * ks * kDh);
      wc[4 * ks + 1] = __ldg(wp + 8 * ks * kDh + 8);
      wc[4 * ks + 2] = __ldg(wp + (8 * ks + 4) * kDh);
      wc[4 * ks + 3] = __ldg(wp + (8 * ks + 4) * kDh + 8);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 x = __ldg(reinterpret_cast<const float2*>(L.H + (b * kDh + st_row(w, g, 2 * h)) * kDh + e0 +
                                                               st_col(t, nt, 0)));
        hr[nt][2 * h] = x.x, hr[nt][2 * h + 1] = x.y;
      }
    el = __ldg(vecp(L, b, kE) + kC - 1);
  };
  load_r(b0 + nc - 1);
  load_c(b0 + nc - 1);
  __syncthreads();
#pragma unroll 1
  for (int c = nc - 1; c >= 0; --c) {
    const int64_t b = b0 + c;
    if (c >= 2) {
      prefetch_rows(L.K + (b - 2) * kC * kDh, kDh, kC, kDh, tid, 256);
      prefetch_rows(L.W + (b - 2) * kC * kDh, kDh, kC, kDh, tid, 256);
    }
    {
      // dV' = D (K G) + X at rows i0, i0 + 1 and columns g, g + 8 (X was read
      // by this lane from the places dV' now overwrites)
      float o[4];
      row_product<KEXACT>(kr, xs, lane, o);
      const float v[4] = {fmaf(dr[0], o[0], xr[0]), fmaf(dr[1], o[1], xr[1]), fmaf(dr[0], o[2], xr[2]),
                          fmaf(dr[1], o[3], xr[3])};
      if (c > 0) load_r(b - 1);
      float* vp = L.dVp + (b * kC + i0) * kDh + e0 + g;
      vp[0] = v[0], vp[kDh] = v[1], vp[8] = v[2], vp[kDh + 8] = v[3];
      vs[vf_index(i0, g)] = v[0];
      vs[vf_index(i0 + 1, g)] = v[1];
      vs[vf_index(i0, g + 8)] = v[2];
      vs[vf_index(i0 + 1, g + 8)] = v[3];
    }
    __syncthreads();
    {
      // G <- e_l G + H - W^T dV'
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) st[nt][r] = fmaf(el, st[nt][r], hr[nt][r]);
      col_product<false>(st, wc, vs, lane, -1.f);
      if (c > 0) {
        load_c(b - 1);
        put_g(b - 1);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) xs[xf_index(st_row(w, g, r), st_col(t, nt, r))] = st[nt][r];
      } else if (dh0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            dh0[(chain * kDh + st_row(w, g, r)) * kDh + e0 + st_col(t, nt, r)] = st[nt][r];
      }
    }
    __syncthreads();
  }
}

// dst[i][:] = vec[i] src[i][:] for a pair's [64][128] rows.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_scale_rows(float* dst, const float* src, const Lay L, int which) {
  const int64_t b = blockIdx.x;
  const float* v = vecp(L, b, which);
  for (int u = threadIdx.x; u < kC * kDh / 4; u += 256) {
    const int i = (4 * u) / kDh;
    const float4 x = reinterpret_cast<const float4*>(src + b * kC * kDh)[u];
    const float f = v[i];
    reinterpret_cast<float4*>(dst + b * kC * kDh)[u] = make_float4(f * x.x, f * x.y, f * x.z, f * x.w);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Row sums over the 128 columns of products of two [64][128] matrices (warp
// w takes rows w, w + 8, ..; lane l the float4 column l).  mode 0: dgamma -=
// D_i (KG)_i . V'_i and dgamma[last] += e_l <S0, G> + sum_i D_i (KG)_i . V'_i
// (the <S1, G> term); mode 1: dgamma += scale e_i (Q S0)_i . dO_i.  Grid nb,
// 256 threads.
__global__ void __launch_bounds__(256) bwdc_rowdots(const Lay L, int mode, float scale) {
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const float4* X = reinterpret_cast<const float4*>((mode == 0 ? L.X1 : L.X2) + b * kC * kDh) + lane;
  const float4* Y = reinterpret_cast<const float4*>((mode == 0 ? L.Vp : L.dO) + b * kC * kDh) + lane;
  float* dg = vecp(L, b, kDgam);
  const float* f = vecp(L, b, mode == 0 ? kD : kE);
  float tt = 0.f;   // mode 0: sum over this warp's rows of D_i (KG)_i . V'_i
#pragma unroll 2
  for (int i = w; i < kC; i += 8) {
    const float4 x = X[i * (kDh / 4)], y = Y[i * (kDh / 4)];
    const float s = warp_sum(fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w))));
    const float t = (mode == 0 ? 1.f : scale) * f[i] * s;
    if (lane == 0) dg[i] += mode == 0 ? -t : t;
    tt += t;
  }
  if (mode == 1) return;
  // <S1, G> = e_l <S0, G> + sum_i t_i
  const float4* S0 = reinterpret_cast<const float4*>(L.S0 + b * kDh * kDh);
  const float4* G = reinterpret_cast<const float4*>(L.G + b * kDh * kDh);
  float sg = 0.f;
  for (int x = tid; x < kDh * kDh / 4; x += 256) {
    const float4 u = S0[x], v = G[x];
    sg = fmaf(u.x, v.x, fmaf(u.y, v.y, fmaf(u.z, v.z, fmaf(u.w, v.w, sg))));
  }
  sg = warp_sum(sg);
  __shared__ float red[8], red2[8];
  if (lane == 0) {
    red[w] = tt;
    red2[w] = sg;
  }
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f, sgt = 0.f;
    for (int v = 0; v < 8; ++v) {
      tot += red[v];
      sgt += red2[v];
    }
    dg[kC - 1] += vecp(L, b, kE)[kC - 1] * sgt + tot;
  }
}

// dP = lower(M1) (M1 = scale dO V'^T): dgamma += rowsum(dP o P) - colsum(dP o P);
// M1 <- dP o E (for dQ += M1 K, dK += M1^T Q).  Warp w takes rows w, w + 8, ..;
// lane l columns 2 l, 2 l + 1.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_dp(const Lay L) {
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, j = 2 * lane;
  __shared__ float csum[8][kC], rsum[kC];
  const float* gam = vecp(L, b, kGam);
  const float gj0 = gam[j], gj1 = gam[j + 1];
  float c0 = 0.f, c1 = 0.f;
#pragma unroll 2
  for (int r = w; r < kC; r += 8) {
    float2* mp = reinterpret_cast<float2*>(L.M1 + b * kC * kC + r * kC + j);
    const float2 m = *mp, pv = *reinterpret_cast<const float2*>(L.P + b * kC * kC + r * kC + j);
    const float gr = gam[r];
    const float d0 = r >= j ? m.x : 0.f, d1 = r >= j + 1 ? m.y : 0.f;
    const float p0 = d0 * pv.x, p1 = d1 * pv.y;
    c0 += p0;
    c1 += p1;
    const float rs = warp_sum(p0 + p1);
    if (lane == 0) rsum[r] = rs;
    *mp = make_float2(r >= j ? d0 * expf(gr - gj0) : 0.f, r >= j + 1 ? d1 * expf(gr - gj1) : 0.f);
  }
  csum[w][j] = c0;
  csum[w][j + 1] = c1;
  __syncthreads();
  if (tid < kC) {
    float cs = 0.f;
#pragma unroll
    for (int v = 0; v < 8; ++v) cs += csum[v][tid];
    vecp(L, b, kDgam)[tid] += rsum[tid] - cs;
  }
}

// From TdW = T^T dW and TdV = T^T dV': dK += diag(beta e) TdW, dbeta += e rowsum(K o TdW)
// + rowsum(V o TdV), dgamma += beta e rowsum(K o TdW), TdV <- diag(beta) TdV (= dV).
// Warp w takes rows w, w + 8, ..; lane l the float4 column l.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_wy(const Lay L, const float* TdW, float* TdV) {
  const int64_t b = blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* vbe = vecp(L, b, kBe);
  const float* vbt = vecp(L, b, kBeta);
  const float* ve = vecp(L, b, kE);
#pragma unroll 2
  for (int i = w; i < kC; i += 8) {
    const int64_t r = (b * kC + i) * kDh + 4 * lane;
    const float be = vbe[i], bt = vbt[i];
    const float4 x3 = *reinterpret_cast<const float4*>(TdW + r);
    const float4 x4 = *reinterpret_cast<const float4*>(TdV + r);
    const float4 k4 = *reinterpret_cast<const float4*>(L.K + r);
    const float4 v4 = *reinterpret_cast<const float4*>(L.V + r);
    float4 dk = *reinterpret_cast<const float4*>(L.dK + r);
    const float kx = warp_sum(fmaf(k4.x, x3.x, fmaf(k4.y, x3.y, fmaf(k4.z, x3.z, k4.w * x3.w))));
    const float vx = warp_sum(fmaf(v4.x, x4.x, fmaf(v4.y, x4.y, fmaf(v4.z, x4.z, v4.w * x4.w))));
    dk.x = fmaf(be, x3.x, dk.x); dk.y = fmaf(be, x3.y, dk.y); dk.z = fmaf(be, x3.z, dk.z); dk.w = fmaf(be, x3.w, dk.w);
    *reinterpret_cast<float4*>(L.dK + r) = dk;
    *reinterpret_cast<float4*>(TdV + r) = make_float4(bt * x4.x, bt * x4.y, bt * x4.z, bt * x4.w);
    if (lane == 0) {
      vecp(L, b, kDbeta)[i] += ve[i] * kx + vx;
      vecp(L, b, kDgam)[i] += be * kx;
    }
  }
}

// dA = strict-lower(M3) (M3 = -T^T dT T^T): dbeta += rowsum(dA o E o KK),
// dgamma += rowsum(dA o A) - colsum(dA o A), M3 <- dKK = dA o beta_i E.  Warp
// w takes rows w, w + 8, ..; lane l columns 2 l, 2 l + 1.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_da(const Lay L) {
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, j = 2 * lane;
  __shared__ float csum[8][kC], rsum[kC], dbs[kC];
  const float* gam = vecp(L, b, kGam);
  const float* bet = vecp(L, b, kBeta);
  const float gj0 = gam[j], gj1 = gam[j + 1];
  float c0 = 0.f, c1 = 0.f;
#pragma unroll 2
  for (int r = w; r < kC; r += 8) {
    const int64_t x = b * kC * kC + r * kC + j;
    float2* mp = reinterpret_cast<float2*>(L.M3 + x);
    const float2 m = *mp, kk = *reinterpret_cast<const float2*>(L.KK + x),
                 av = *reinterpret_cast<const float2*>(L.A + x);
    const float gr = gam[r], bt = bet[r];
    const float d0 = r > j ? m.x : 0.f, d1 = r > j + 1 ? m.y : 0.f;
    const float E0 = r > j ? expf(gr - gj0) : 0.f, E1 = r > j + 1 ? expf(gr - gj1) : 0.f;
    const float a0 = d0 * av.x, a1 = d1 * av.y;
    c0 += a0;
    c1 += a1;
    const float db = warp_sum(fmaf(d0, E0 * kk.x, d1 * (E1 * kk.y)));
    const float rs = warp_sum(a0 + a1);
    if (lane == 0) {
      rsum[r] = rs;
      dbs[r] = db;
    }
    *mp = make_float2(d0 * bt * E0, d1 * bt * E1);
  }
  csum[w][j] = c0;
  csum[w][j + 1] = c1;
  __syncthreads();
  if (tid < kC) {
    float cs = 0.f;
#pragma unroll
    for (int v = 0; v < 8; ++v) cs += csum[v][tid];
    vecp(L, b, kDgam)[tid] += rsum[tid] - cs;
    vecp(L, b, kDbeta)[tid] += dbs[tid];
  }
}

// Scatter a pair's gradients: dq, dk (atomics across the value heads of a
// qk group), dv, dg (reverse cumsum of dgamma), dbeta.  vec: dq, dk and dv are
// 16-byte aligned (float4 copies).  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) bwdc_scatter(const Lay L, float* dq, float* dk, float* dv, float* dg,
                                                    float* dbeta, int T, int NC, int Hqk, int Hv, bool vec) {
  const int64_t b = blockIdx.x;
  int64_t t0;
  int Lc, h;
  pair_rows(L, b, T, NC, Hv, t0, Lc, h);
  const int hq = h / (Hv / Hqk);
  const bool share = Hv != Hqk;
  if (vec) {
    for (int u = threadIdx.x; u < Lc * kDh / 4; u += 256) {
      const int i = (4 * u) / kDh, d = (4 * u) % kDh;
      const int64_t qk = ((t0 + i) * Hqk + hq) * (int64_t)kDh + d, vo = ((t0 + i) * Hv + h) * (int64_t)kDh + d;
      const int64_t x = b * kC * kDh + 4 * u;
      const float4 a = *reinterpret_cast<const float4*>(L.dQ + x), k4 = *reinterpret_cast<const float4*>(L.dK + x);
      if (share) {
        atomicAdd(dq + qk, a.x); atomicAdd(dq + qk + 1, a.y); atomicAdd(dq + qk + 2, a.z); atomicAdd(dq + qk + 3, a.w);
        atomicAdd(dk + qk, k4.x); atomicAdd(dk + qk + 1, k4.y); atomicAdd(dk + qk + 2, k4.z); atomicAdd(dk + qk + 3, k4.w);
      } else {
        *reinterpret_cast<float4*>(dq + qk) = a;
        *reinterpret_cast<float4*>(dk + qk) = k4;
      }
      *reinterpret_cast<float4*>(dv + vo) = *reinterpret_cast<const float4*>(L.X4 + x);
    }
  } else {
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
          int exact = 0, const float* rs = nullptr, int64_t sR = 0, const float* cs = nullptr, int64_t sCs = 0) {
  GemmArgs g{A, B, C, rs, sA, sB, sC, sR, lda, ldb, ldc, M, N, Kd, tA, tB, alpha, beta, exact, cs, sCs};
  // dynamic shared memory above 48 KB (set on every call: the attribute is
  // cheap and the caller's device may change between calls)
  const auto set = [](const void* f) {
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) == cudaSuccess;
  };
  const void* kf = tA ? (tB ? reinterpret_cast<const void*>(bgemm_kernel<true, true>)
                            : reinterpret_cast<const void*>(bgemm_kernel<true, false>))
                      : (tB ? reinterpret_cast<const void*>(bgemm_kernel<false, true>)
                            : reinterpret_cast<const void*>(bgemm_kernel<false, false>));
  if (!set(kf)) return false;
  const dim3 grid(N / 64, M / 64, (unsigned)nb);
  if (tA)
    tB ? bgemm_kernel<true, true><<<grid, 256, kGemmSmem, s>>>(g) : bgemm_kernel<true, false><<<grid, 256, kGemmSmem, s>>>(g);
  else
    tB ? bgemm_kernel<false, true><<<grid, 256, kGemmSmem, s>>>(g) : bgemm_kernel<false, false><<<grid, 256, kGemmSmem, s>>>(g);
  return cudaGetLastError() == cudaSuccess;
}

template <typename Tin>
gdn_status run(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g, const float* beta,
               float scale, const float* h0, const int32_t* cu, const void* dout, const float* dht, float* dq,
               float* dk, float* dv, float* dg, float* dbeta, float* dh0, int32_t* status, void* ws, cudaStream_t s) {
  const int NC = (p.T + kC - 1) / kC;   // equal lengths (packed sequences: the tables)
  const Lay L = layout(p, static_cast<uint8_t*>(ws));
  const int64_t nb = L.nb, B2 = (int64_t)kC * kDh, Q2 = (int64_t)kC * kC, S2 = (int64_t)kDh * kDh, V8 = 8 * kC;
  const unsigned nbu = (unsigned)nb;
  const int64_t chains = (int64_t)p.N * p.Hv;
  // with bf16 inputs K, Q, V and dO hold bf16 values, exact in tf32: products
  // with them drop the lo terms of those operands (xA, xB: op(A), op(B) exact)
  constexpr bool kBf = std::is_same<Tin, __nv_bfloat16>::value;
  const int xA = kBf ? 1 : 0, xB = kBf ? 2 : 0;
  bool ok = true;
  if (p.varlen) bwdc_prepare<<<1, 1024, 0, s>>>(L, cu, p.N, (int64_t)p.B * p.T, p.Hv, status);
  bwdc_gather<Tin><<<nbu, 256, 0, s>>>(L, static_cast<const Tin*>(q), static_cast<const Tin*>(k),
                                        static_cast<const Tin*>(v), static_cast<const Tin*>(dout), g, beta, p.T, NC,
                                        p.Hqk, p.Hv);
  // KK = K K^T, P <- Q K^T, then the masks, T, W and U
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.K, B2, kDh, false, L.K, B2, kDh, true, 0.f, L.KK, Q2, kC, xA | xB);
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.Q, B2, kDh, false, L.K, B2, kDh, true, 0.f, L.P, Q2, kC, xA | xB);
  bwdc_masks<<<nbu, 256, 0, s>>>(L);
  bwdc_solve<<<nbu, 64, 0, s>>>(L);
  // W = (T diag(beta e)) K, U = (T diag(beta)) V
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M1, Q2, kC, false, L.K, B2, kDh, false, 0.f, L.W, B2, kDh, xB);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M2, Q2, kC, false, L.V, B2, kDh, false, 0.f, L.U, B2, kDh, xB);
  // the serial passes
  bwdc_fwd_states<kBf><<<dim3((unsigned)chains, kDh / kSl), 256, 0, s>>>(L, h0, NC);
  // the reverse pass's G-independent terms: X = scale P^T dO (in dVp), H = scale Q^T diag(e) dO
  ok = ok && gemm(s, nb, kC, kDh, kC, scale, L.P, Q2, kC, true, L.dO, B2, kDh, false, 0.f, L.dVp, B2, kDh, xB);
  bwdc_scale_rows<<<nbu, 256, 0, s>>>(L.X3, L.dO, L, kE);
  ok = ok && gemm(s, nb, kDh, kDh, kC, scale, L.Q, B2, kDh, true, L.X3, B2, kDh, false, 0.f, L.H, S2, kDh, xA);
  bwdc_rev<kBf><<<dim3((unsigned)chains, kDh / kSl), 256, 0, s>>>(L, dht, dh0, NC);
  // dQ = scale diag(e) dO S0^T ;  dK = diag(D) V' G^T
  ok = ok && gemm(s, nb, kC, kDh, kDh, scale, L.dO, B2, kDh, false, L.S0, S2, kDh, true, 0.f, L.dQ, B2, kDh, xA,
                  L.vec + kE * kC, V8);
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.Vp, B2, kDh, false, L.G, S2, kDh, true, 0.f, L.dK, B2, kDh, 0,
                  L.vec + kD * kC, V8);
  // X1 = K G (the D (K G) . V' terms), X2 = Q S0 (the e (Q S0) . dO terms)
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.K, B2, kDh, false, L.G, S2, kDh, false, 0.f, L.X1, B2, kDh, xA);
  ok = ok && gemm(s, nb, kC, kDh, kDh, 1.f, L.Q, B2, kDh, false, L.S0, S2, kDh, false, 0.f, L.X2, B2, kDh, xA);
  bwdc_rowdots<<<nbu, 256, 0, s>>>(L, 0, scale);
  bwdc_rowdots<<<nbu, 256, 0, s>>>(L, 1, scale);
  // dP = lower(scale dO V'^T) -> (dP o E): dQ += . K, dK += .^T Q
  ok = ok && gemm(s, nb, kC, kC, kDh, scale, L.dO, B2, kDh, false, L.Vp, B2, kDh, true, 0.f, L.M1, Q2, kC, xA);
  bwdc_dp<<<nbu, 256, 0, s>>>(L);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M1, Q2, kC, false, L.K, B2, kDh, false, 1.f, L.dQ, B2, kDh, xB);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M1, Q2, kC, true, L.Q, B2, kDh, false, 1.f, L.dK, B2, kDh, xB);
  // dW = -dV' S0^T (X3); dT = (dW K^T) diag(beta e) + (dV' V^T) diag(beta) (M2)
  ok = ok && gemm(s, nb, kC, kDh, kDh, -1.f, L.dVp, B2, kDh, false, L.S0, S2, kDh, true, 0.f, L.X3, B2, kDh);
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.X3, B2, kDh, false, L.K, B2, kDh, true, 0.f, L.M2, Q2, kC, xB,
                  nullptr, 0, L.vec + kBe * kC, V8);
  ok = ok && gemm(s, nb, kC, kC, kDh, 1.f, L.dVp, B2, kDh, false, L.V, B2, kDh, true, 1.f, L.M2, Q2, kC, xB,
                  nullptr, 0, L.vec + kBeta * kC, V8);
  // X1 <- T^T dW, X4 = T^T dV'
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, true, L.X3, B2, kDh, false, 0.f, L.X1, B2, kDh);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.T, Q2, kC, true, L.dVp, B2, kDh, false, 0.f, L.X4, B2, kDh);
  bwdc_wy<<<nbu, 256, 0, s>>>(L, L.X1, L.X4);
  // dA = strict-lower(-T^T dT T^T): M1 = T^T dT, M3 = -M1 T^T
  ok = ok && gemm(s, nb, kC, kC, kC, 1.f, L.T, Q2, kC, true, L.M2, Q2, kC, false, 0.f, L.M1, Q2, kC);
  ok = ok && gemm(s, nb, kC, kC, kC, -1.f, L.M1, Q2, kC, false, L.T, Q2, kC, true, 0.f, L.M3, Q2, kC);
  bwdc_da<<<nbu, 256, 0, s>>>(L);
  // dK += dKK K + dKK^T K
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M3, Q2, kC, false, L.K, B2, kDh, false, 1.f, L.dK, B2, kDh, xB);
  ok = ok && gemm(s, nb, kC, kDh, kC, 1.f, L.M3, Q2, kC, true, L.K, B2, kDh, false, 1.f, L.dK, B2, kDh, xB);
  if (p.Hv != p.Hqk) {
    const size_t tq = sizeof(float) * (size_t)p.B * p.T * p.Hqk * p.K;
    if (cudaMemsetAsync(dq, 0, tq, s) != cudaSuccess || cudaMemsetAsync(dk, 0, tq, s) != cudaSuccess) return GDN_ERR_CUDA;
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
                     reinterpret_cast<uintptr_t>(dv)) & 15) == 0;
  bwdc_scatter<<<nbu, 256, 0, s>>>(L, dq, dk, dv, dg, dbeta, p.T, NC, p.Hqk, p.Hv, vec);
  ok = ok && cudaGetLastError() == cudaSuccess;
  return ok ? GDN_OK : GDN_ERR_CUDA;
}

// Sequences per group: the batch runs in groups of whole sequences whose
// per-(chunk, head) data fits kGroupBytes (at least one sequence a group).
constexpr size_t kGroupBytes = size_t(16) << 30;

int group_seqs(const gdn_problem& p) {
  gdn_problem one = p;
  one.N = one.B = 1;
  const size_t per = layout(one, nullptr).bytes;
  int64_t g = (int64_t)(kGroupBytes / (per > 0 ? per : 1));
  if (g < 1) g = 1;
  return (int)(g < p.N ? g : p.N);
}

gdn_problem group_problem(const gdn_problem& p, int n) {
  gdn_problem q = p;
  q.N = q.B = n;
  return q;
}

}  // namespace

// Packed sequences run as one group, sized for the bound of ceil(T / 64) + N
// chunks a value head; larger packed batches take the token recurrence.
constexpr size_t kVarlenBytes = size_t(32) << 30;

bool bwdc_supported(const gdn_problem& p) {
  if (p.K != kDh || p.V != kDh || p.T <= 0) return false;
  return !p.varlen || layout(p, nullptr).bytes <= kVarlenBytes;
}

size_t bwdc_workspace_bytes(const gdn_problem& p) {
  if (p.varlen) return kAlign + layout(p, nullptr).bytes;
  return kAlign + layout(group_problem(p, group_seqs(p)), nullptr).bytes;
}

gdn_status run_bwdc(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                    const float* beta, float scale, const float* h0, const int32_t* cu_seqlens, const void* dout,
                    const float* dht, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws,
                    cudaStream_t s) {
  int32_t* status = static_cast<int32_t*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  void* w = static_cast<uint8_t*>(ws) + kAlign;
  if (p.varlen) {
    if (p.dt == GDN_F32)
      return run<float>(p, q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, status, w,
                        s);
    return run<__nv_bfloat16>(p, q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0,
                              status, w, s);
  }
  const int G = group_seqs(p);
  const size_t e = p.dt == GDN_F32 ? 4 : 2;
  const int64_t kv = (int64_t)p.K * p.V;
  for (int n0 = 0; n0 < p.N; n0 += G) {
    const int n = p.N - n0 < G ? p.N - n0 : G;
    const gdn_problem gp = group_problem(p, n);
    const int64_t t0 = (int64_t)n0 * p.T;   // first token of the group
    auto off = [&](const void* x, int64_t elems) {
      return x ? static_cast<const void*>(static_cast<const uint8_t*>(x) + elems * e) : nullptr;
    };
    auto offf = [&](const float* x, int64_t elems) { return x ? x + elems : nullptr; };
    auto offw = [&](float* x, int64_t elems) { return x ? x + elems : nullptr; };
    const int64_t tq = t0 * p.Hqk * p.K, tv = t0 * p.Hv * p.V, tg = t0 * p.Hv, ts = (int64_t)n0 * p.Hv * kv;
    gdn_status st;
    if (p.dt == GDN_F32)
      st = run<float>(gp, off(q, tq), off(k, tq), off(v, tv), g + tg, beta + tg, scale, offf(h0, ts), nullptr,
                      off(dout, tv), offf(dht, ts), dq + tq, dk + tq, dv + tv, dg + tg, dbeta + tg, offw(dh0, ts),
                      status, w, s);
    else
      st = run<__nv_bfloat16>(gp, off(q, tq), off(k, tq), off(v, tv), g + tg, beta + tg, scale, offf(h0, ts),
                              nullptr, off(dout, tv), offf(dht, ts), dq + tq, dk + tq, dv + tv, dg + tg, dbeta + tg,
                              offw(dh0, ts), status, w, s);
    if (st != GDN_OK) return st;
  }
  return GDN_OK;
}

}  // namespace gdn
