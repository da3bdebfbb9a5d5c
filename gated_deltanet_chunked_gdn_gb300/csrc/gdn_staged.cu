// gdn_staged.cu -- the staged path: one sm_103a kernel per stage of the chunk
// pipeline, fp32 arithmetic, intermediates kept in the caller's workspace.
//
// This is the pages' staged execution mode (MegaGDN-PTO walkthrough, section
// 7.4: every stage runs alone and its intermediates can be inspected, the
// MEGA_STOP_AFTER_* hooks).  Stages, in the order of section 1.1:
//   0 prepare     chunk tables from cu_seqlens (section 5.3 varlen packing)
//   1 cumsum      gamma = in-chunk prefix sum of g          (section 4.1)
//   2 kkt         A = strict-lower(beta_i exp(gamma_i - gamma_j) k_i.k_j)
//                                                            (section 4.2)
//   3 solve_tril  T = (I + A)^{-1}: 16x16 diagonal blocks by forward
//                 substitution, then recursive merges T21 = -T22 A21 T11
//                                                            (section 4.4)
//   4 wy_fast     W = T diag(beta e^gamma) K, U = T diag(beta) V (section 4.3)
//   5 chunk_h     serial over chunks: V' = U - W S, S <- e^{g_last} S +
//                 K^T diag(e^{g_last - gamma}) V'  (TileLang x xLLM page, Step 1)
//   6 chunk_o     O = scale (diag(e^gamma) Q S + (Q K^T o causal o e^{gamma_i -
//                 gamma_j}) V')                              (section 1.1)
// Rows past a chunk's length are zero in every intermediate and never stored
// to o.  It is also the path for fp32 inputs and for head dims the fused
// kernel does not cover.
#include "gdn_internal.h"

namespace gdn {
namespace {

// ------------------------------------------------------------------ stage 0
// One CTA.  Thread 0 validates cu_seqlens and scans the per-sequence chunk
// counts (N is small next to the token count); all threads then fill the
// per-chunk tables.
__global__ void prepare_kernel(const int32_t* __restrict__ cu, int N, int T, int C, int nc_max, Tables t,
                               int32_t* status) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    int good = 1;
    int64_t acc = 0;
    if (cu) {
      if (cu[0] != 0 || cu[N] != T) good = 0;
      for (int n = 0; n < N && good; ++n) {
        const int64_t L = (int64_t)cu[n + 1] - cu[n];
        if (L < 0) { good = 0; break; }
        t.seq_chunk0[n] = (int32_t)acc;
        acc += ceil_div(L, C);
      }
    } else {
      for (int n = 0; n < N; ++n) {
        t.seq_chunk0[n] = (int32_t)acc;
        acc += ceil_div(T, C);
      }
    }
    if (acc > nc_max) good = 0;
    if (good) {
      t.seq_chunk0[N] = (int32_t)acc;
      *t.nc = (int32_t)acc;
    } else {
      *t.nc = -1;
      atomicExch(status, GDN_DEV_BAD_CU_SEQLENS);
    }
    ok = good;
  }
  __syncthreads();
  if (!ok) return;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const int64_t tok0 = cu ? (int64_t)cu[n] : (int64_t)n * T;
    const int64_t L = cu ? (int64_t)cu[n + 1] - cu[n] : T;
    const int c0 = t.seq_chunk0[n];
    const int nch = (int)ceil_div(L, C);
    for (int j = 0; j < nch; ++j) {
      t.chunk_seq[c0 + j] = n;
      t.chunk_tok0[c0 + j] = (int32_t)(tok0 + (int64_t)j * C);
      t.chunk_len[c0 + j] = (int32_t)((L - (int64_t)j * C) < C ? (L - (int64_t)j * C) : C);
    }
  }
}

// ------------------------------------------------------------------ stage 1
__global__ void cumsum_kernel(const float* __restrict__ g, Tables t, int Hv, int C, float* __restrict__ gamma) {
  const int c = blockIdx.x;
  if (c >= *t.nc) return;
  const int h = threadIdx.x;
  if (h >= Hv) return;
  const int64_t tok0 = t.chunk_tok0[c];
  const int len = t.chunk_len[c];
  float acc = 0.f;
  float* out = gamma + ((int64_t)c * Hv + h) * C;
  for (int i = 0; i < C; ++i) {
    if (i < len) acc += g[(tok0 + i) * Hv + h];
    out[i] = (i < len) ? acc : 0.f;
  }
}

// Gram tile: acc[r][s] = sum_d X[ty + 16 r][d] * Y[tx + 16 s][d] over the C
// rows of a chunk, X and Y read from [tok][H][D] tensors through 32-wide
// shared-memory slabs.  R = C / 16.
template <typename Tin, int R>
__device__ __forceinline__ void chunk_gram(const Tin* __restrict__ X, const Tin* __restrict__ Y, int64_t tok0, int len,
                                           int H, int hq, int D, float (*xs)[33], float (*ys)[33],
                                           float (&acc)[R][R]) {
  constexpr int C = R * 16;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int s = 0; s < R; ++s) acc[r][s] = 0.f;
  for (int d0 = 0; d0 < D; d0 += 32) {
    for (int idx = tid; idx < C * 32; idx += blockDim.x) {
      const int i = idx / 32, dd = idx % 32;
      const int64_t off = ((tok0 + i) * H + hq) * (int64_t)D + d0 + dd;
      xs[i][dd] = (i < len) ? to_f(X[off]) : 0.f;
      ys[i][dd] = (i < len) ? to_f(Y[off]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int dd = 0; dd < 32; ++dd) {
      float a[R], b[R];
#pragma unroll
      for (int r = 0; r < R; ++r) a[r] = xs[ty + 16 * r][dd];
#pragma unroll
      for (int s = 0; s < R; ++s) b[s] = ys[tx + 16 * s][dd];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int s = 0; s < R; ++s) acc[r][s] = fmaf(a[r], b[s], acc[r][s]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ stage 2
template <typename Tin, int C>
__global__ void __launch_bounds__(256) kkt_kernel(const Tin* __restrict__ k, const float* __restrict__ beta,
                                                  const float* __restrict__ gamma, Tables t, int Hqk, int Hv, int K,
                                                  float* __restrict__ A) {
  constexpr int R = C / 16;
  __shared__ float ks[C][33];
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= *t.nc) return;
  const int hq = h / (Hv / Hqk);
  const int64_t tok0 = t.chunk_tok0[c];
  const int len = t.chunk_len[c];
  float acc[R][R];
  chunk_gram<Tin, R>(k, k, tok0, len, Hqk, hq, K, ks, ks, acc);
  const float* gam = gamma + ((int64_t)c * Hv + h) * C;
  float* out = A + ((int64_t)c * Hv + h) * C * C;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = ty + 16 * r;
    const float bi = (i < len) ? beta[(tok0 + i) * Hv + h] : 0.f;
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const int j = tx + 16 * s;
      float val = 0.f;
      if (i > j && i < len) val = bi * expf(gam[i] - gam[j]) * acc[r][s];
      out[i * C + j] = val;
    }
  }
}

// ------------------------------------------------------------------ stage 3
template <int C>
__global__ void __launch_bounds__(128) solve_kernel(const float* __restrict__ A, Tables t, int Hv,
                                                    float* __restrict__ Tinv) {
  extern __shared__ float smem[];
  float* As = smem;                    // [C][C+1]
  float* Ts = As + C * (C + 1);        // [C][C+1]
  float* tmp = Ts + C * (C + 1);       // [C/2 * 64] scratch for A21 T11
  constexpr int LD = C + 1;
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= *t.nc) return;
  const float* a = A + ((int64_t)c * Hv + h) * C * C;
  for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
    As[(idx / C) * LD + idx % C] = a[idx];
    Ts[(idx / C) * LD + idx % C] = 0.f;
  }
  __syncthreads();
  // Diagonal 16x16 blocks of (I + A)^{-1} by forward substitution: lane l owns
  // column l of its block, so each lane's recurrence is independent.
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int b = warp; b < C / 16; b += blockDim.x / 32) {
    if (lane < 16) {
      const int base = 16 * b;
      for (int i = 0; i < 16; ++i) {
        float x = (i == lane) ? 1.f : 0.f;
        for (int j = lane; j < i; ++j) x -= As[(base + i) * LD + base + j] * Ts[(base + j) * LD + base + lane];
        Ts[(base + i) * LD + base + lane] = x;
      }
    }
  }
  __syncthreads();
  // Merge neighbouring blocks: [[T11, 0], [T21, T22]] with T21 = -T22 A21 T11.
  for (int s = 16; s < C; s *= 2) {
    const int npairs = C / (2 * s);
    for (int idx = threadIdx.x; idx < npairs * s * s; idx += blockDim.x) {
      const int p = idx / (s * s), i = (idx / s) % s, m = idx % s;
      const int o = 2 * s * p;
      float x = 0.f;
      for (int j = m; j < s; ++j) x += As[(o + s + i) * LD + o + j] * Ts[(o + j) * LD + o + m];
      tmp[idx] = x;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < npairs * s * s; idx += blockDim.x) {
      const int p = idx / (s * s), i = (idx / s) % s, m = idx % s;
      const int o = 2 * s * p;
      float x = 0.f;
      for (int j = 0; j <= i; ++j) x += Ts[(o + s + i) * LD + o + s + j] * tmp[p * s * s + j * s + m];
      Ts[(o + s + i) * LD + o + m] = -x;
    }
    __syncthreads();
  }
  float* out = Tinv + ((int64_t)c * Hv + h) * C * C;
  for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) out[idx] = Ts[(idx / C) * LD + idx % C];
}

// ------------------------------------------------------------------ stage 4
// blockIdx.z < K/64: a 64-column tile of W, else of U.
template <typename Tin, int C>
__global__ void __launch_bounds__(256) wy_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                                                 const float* __restrict__ beta, const float* __restrict__ gamma,
                                                 const float* __restrict__ Tinv, Tables t, int Hqk, int Hv, int K,
                                                 int V, float* __restrict__ W, float* __restrict__ U) {
  extern __shared__ float smem[];
  float* Ts = smem;                 // [C][C+1]
  float* Xs = Ts + C * (C + 1);     // [C][65]
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= *t.nc) return;
  const bool isW = blockIdx.z < K / 64;
  const int col0 = 64 * (isW ? blockIdx.z : blockIdx.z - K / 64);
  const int hq = h / (Hv / Hqk);
  const int64_t tok0 = t.chunk_tok0[c];
  const int len = t.chunk_len[c];
  const float* tin = Tinv + ((int64_t)c * Hv + h) * C * C;
  const float* gam = gamma + ((int64_t)c * Hv + h) * C;
  for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) Ts[(idx / C) * (C + 1) + idx % C] = tin[idx];
  for (int idx = threadIdx.x; idx < C * 64; idx += blockDim.x) {
    const int r = idx / 64, cc = idx % 64;
    float x = 0.f;
    if (r < len) {
      const float b = beta[(tok0 + r) * Hv + h];
      if (isW) x = b * expf(gam[r]) * to_f(k[((tok0 + r) * Hqk + hq) * (int64_t)K + col0 + cc]);
      else x = b * to_f(v[((tok0 + r) * Hv + h) * (int64_t)V + col0 + cc]);
    }
    Xs[r * 65 + cc] = x;
  }
  __syncthreads();
  constexpr int RR = C / 4;
  const int col = threadIdx.x % 64, rg = threadIdx.x / 64;
  float acc[RR];
#pragma unroll
  for (int r = 0; r < RR; ++r) acc[r] = 0.f;
  for (int cc = 0; cc < C; ++cc) {
    const float x = Xs[cc * 65 + col];
#pragma unroll
    for (int r = 0; r < RR; ++r) acc[r] = fmaf(Ts[(rg + 4 * r) * (C + 1) + cc], x, acc[r]);
  }
  const int D = isW ? K : V;
  float* out = (isW ? W : U) + ((int64_t)c * Hv + h) * C * (int64_t)D;
#pragma unroll
  for (int r = 0; r < RR; ++r) {
    const int i = rg + 4 * r;
    out[(int64_t)i * D + col0 + col] = (i < len) ? acc[r] : 0.f;
  }
}

// ------------------------------------------------------------------ stage 5
// One CTA per (sequence, value head, 32-column slice of V); the state slice
// S[K][32] lives in shared memory for the whole sequence.
template <typename Tin, int C>
__global__ void __launch_bounds__(256) chunk_h_kernel(const Tin* __restrict__ k, const float* __restrict__ gamma,
                                                      const float* __restrict__ W, const float* __restrict__ U,
                                                      const float* __restrict__ h0, Tables t, int Hqk, int Hv,
                                                      int K, int V, float* __restrict__ S0, float* __restrict__ Vn,
                                                      float* __restrict__ ht) {
  extern __shared__ float smem[];
  float* S = smem;               // [K][33]
  float* vn = S + K * 33;        // [C][33]
  if (*t.nc < 0) return;
  const int n = blockIdx.x, h = blockIdx.y, e0 = 32 * blockIdx.z;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, e = tid % 32, grp = tid / 32;
  const int64_t sbase = ((int64_t)n * Hv + h) * K * (int64_t)V;
  for (int idx = tid; idx < K * 32; idx += blockDim.x) {
    const int d = idx / 32, ee = idx % 32;
    S[d * 33 + ee] = h0 ? h0[sbase + (int64_t)d * V + e0 + ee] : 0.f;
  }
  __syncthreads();
  const int c0 = t.seq_chunk0[n], c1 = t.seq_chunk0[n + 1];
  for (int c = c0; c < c1; ++c) {
    const int64_t tok0 = t.chunk_tok0[c];
    const int len = t.chunk_len[c];
    const int64_t ch = (int64_t)c * Hv + h;
    for (int idx = tid; idx < K * 32; idx += blockDim.x) {
      const int d = idx / 32, ee = idx % 32;
      S0[ch * K * (int64_t)V + (int64_t)d * V + e0 + ee] = S[d * 33 + ee];
    }
    // V' = U - W S
    constexpr int RI = C / 8;
    float acc[RI];
#pragma unroll
    for (int r = 0; r < RI; ++r) acc[r] = 0.f;
    const float* w = W + ch * C * (int64_t)K;
    for (int d = 0; d < K; ++d) {
      const float s = S[d * 33 + e];
#pragma unroll
      for (int r = 0; r < RI; ++r) acc[r] = fmaf(w[(int64_t)(grp + 8 * r) * K + d], s, acc[r]);
    }
    const float* u = U + ch * C * (int64_t)V;
    float* vout = Vn + ch * C * (int64_t)V;
    const float* gam = gamma + ch * C;
    const float gl = gam[len - 1];
#pragma unroll
    for (int r = 0; r < RI; ++r) {
      const int i = grp + 8 * r;
      const float x = (i < len) ? u[(int64_t)i * V + e0 + e] - acc[r] : 0.f;
      vout[(int64_t)i * V + e0 + e] = x;
      vn[i * 33 + e] = (i < len) ? expf(gl - gam[i]) * x : 0.f;   // e^{g_last - gamma_i} V'_i
    }
    __syncthreads();
    // S <- e^{g_last} S + K^T diag(e^{g_last - gamma}) V'
    const float decay = expf(gl);
    for (int d = grp; d < K; d += 8) {
      float a = 0.f;
      for (int i = 0; i < len; ++i) a = fmaf(to_f(k[((tok0 + i) * Hqk + hq) * (int64_t)K + d]), vn[i * 33 + e], a);
      S[d * 33 + e] = decay * S[d * 33 + e] + a;
    }
    __syncthreads();
  }
  if (ht)
    for (int idx = tid; idx < K * 32; idx += blockDim.x) {
      const int d = idx / 32, ee = idx % 32;
      ht[sbase + (int64_t)d * V + e0 + ee] = S[d * 33 + ee];
    }
}

// ------------------------------------------------------------------ stage 6
template <typename Tin, int C>
__global__ void __launch_bounds__(256) chunk_o_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                      const float* __restrict__ gamma, const float* __restrict__ S0,
                                                      const float* __restrict__ Vn, Tables t, int Hqk, int Hv,
                                                      int K, int V, float scale, Tin* __restrict__ o) {
  constexpr int R = C / 16;
  extern __shared__ float smem[];
  float (*qs)[33] = reinterpret_cast<float (*)[33]>(smem);            // [C][33]
  float (*ks)[33] = reinterpret_cast<float (*)[33]>(smem + C * 33);   // [C][33]
  float* Ps = smem + 2 * C * 33;                                      // [C][C+1]
  const int c = blockIdx.x, h = blockIdx.y, e0 = 64 * blockIdx.z;
  if (c >= *t.nc) return;
  const int hq = h / (Hv / Hqk);
  const int64_t tok0 = t.chunk_tok0[c];
  const int len = t.chunk_len[c];
  const int64_t ch = (int64_t)c * Hv + h;
  const float* gam = gamma + ch * C;
  {
    float acc[R][R];
    chunk_gram<Tin, R>(q, k, tok0, len, Hqk, hq, K, qs, ks, acc);
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int i = ty + 16 * r, j = tx + 16 * s;
        Ps[i * (C + 1) + j] = (j <= i && i < len) ? expf(gam[i] - gam[j]) * acc[r][s] : 0.f;
      }
  }
  __syncthreads();
  constexpr int RR = C / 4;
  const int col = threadIdx.x % 64, rg = threadIdx.x / 64;
  float inter[RR], intra[RR];
#pragma unroll
  for (int r = 0; r < RR; ++r) inter[r] = intra[r] = 0.f;
  const float* s0 = S0 + ch * K * (int64_t)V;
  for (int d = 0; d < K; ++d) {
    const float s = s0[(int64_t)d * V + e0 + col];
#pragma unroll
    for (int r = 0; r < RR; ++r) {
      const int i = rg + 4 * r;
      const float qv = (i < len) ? to_f(q[((tok0 + i) * Hqk + hq) * (int64_t)K + d]) : 0.f;
      inter[r] = fmaf(qv, s, inter[r]);
    }
  }
  const float* vn = Vn + ch * C * (int64_t)V;
  for (int j = 0; j < len; ++j) {
    const float x = vn[(int64_t)j * V + e0 + col];
#pragma unroll
    for (int r = 0; r < RR; ++r) intra[r] = fmaf(Ps[(rg + 4 * r) * (C + 1) + j], x, intra[r]);
  }
#pragma unroll
  for (int r = 0; r < RR; ++r) {
    const int i = rg + 4 * r;
    if (i < len)
      o[((tok0 + i) * Hv + h) * (int64_t)V + e0 + col] = from_f<Tin>(scale * (expf(gam[i]) * inter[r] + intra[r]));
  }
}

template <typename KernelT>
cudaError_t set_smem(KernelT kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin, int C>
gdn_status run_staged_t(const gdn_problem& p, int stop_after, const Tin* q, const Tin* k, const Tin* v,
                        const float* g, const float* beta, float scale, const float* h0, const int32_t* cu, Tin* o,
                        float* ht, void* ws, cudaStream_t s) {
  gdn_staged_layout_t L;
  gdn_status st = staged_layout(p, &L);
  if (st != GDN_OK) return st;
  char* base = static_cast<char*>(ws);
  Tables t = tables_at(base + L.tables, p.N, L.nc_max);
  int32_t* status = reinterpret_cast<int32_t*>(base + L.status);
  float* gamma = reinterpret_cast<float*>(base + L.gamma);
  float* A = reinterpret_cast<float*>(base + L.A);
  float* Tinv = reinterpret_cast<float*>(base + L.Tinv);
  float* W = reinterpret_cast<float*>(base + L.W);
  float* U = reinterpret_cast<float*>(base + L.U);
  float* S0 = reinterpret_cast<float*>(base + L.S0);
  float* Vn = reinterpret_cast<float*>(base + L.Vn);
  const int nc = L.nc_max;
#define GDN_CK(x)                               \
  do {                                          \
    cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return GDN_ERR_CUDA; \
  } while (0)
  GDN_CK(cudaMemsetAsync(status, 0, sizeof(int32_t), s));
  GDN_CK(launch_prepare(p, C, cu, t, nc, status, s));
  if (stop_after < 1) return GDN_OK;
  if (nc == 0) return GDN_OK;   // fixed-length problems have T >= 1, varlen ones N >= 1
  const int hb = ((p.Hv + 31) / 32) * 32;
  cumsum_kernel<<<nc, hb, 0, s>>>(g, t, p.Hv, C, gamma);
  GDN_CK(cudaGetLastError());
  if (stop_after < 2) return GDN_OK;
  kkt_kernel<Tin, C><<<dim3(nc, p.Hv), 256, 0, s>>>(k, beta, gamma, t, p.Hqk, p.Hv, p.K, A);
  GDN_CK(cudaGetLastError());
  if (stop_after < 3) return GDN_OK;
  {
    const size_t sm = sizeof(float) * (2 * C * (C + 1) + (C / 2) * 64);
    GDN_CK(set_smem(solve_kernel<C>, sm));
    solve_kernel<C><<<dim3(nc, p.Hv), 128, sm, s>>>(A, t, p.Hv, Tinv);
    GDN_CK(cudaGetLastError());
  }
  if (stop_after < 4) return GDN_OK;
  {
    const size_t sm = sizeof(float) * (C * (C + 1) + C * 65);
    GDN_CK(set_smem(wy_kernel<Tin, C>, sm));
    wy_kernel<Tin, C><<<dim3(nc, p.Hv, (p.K + p.V) / 64), 256, sm, s>>>(k, v, beta, gamma, Tinv, t, p.Hqk, p.Hv,
                                                                        p.K, p.V, W, U);
    GDN_CK(cudaGetLastError());
  }
  if (stop_after < 5) return GDN_OK;
  {
    const size_t sm = sizeof(float) * (p.K * 33 + C * 33);
    GDN_CK(set_smem(chunk_h_kernel<Tin, C>, sm));
    chunk_h_kernel<Tin, C><<<dim3(p.N, p.Hv, p.V / 32), 256, sm, s>>>(k, gamma, W, U, h0, t, p.Hqk, p.Hv, p.K,
                                                                      p.V, S0, Vn, ht);
    GDN_CK(cudaGetLastError());
  }
  if (stop_after < 6) return GDN_OK;
  {
    const size_t sm = sizeof(float) * (2 * C * 33 + C * (C + 1));
    GDN_CK(set_smem(chunk_o_kernel<Tin, C>, sm));
    chunk_o_kernel<Tin, C><<<dim3(nc, p.Hv, p.V / 64), 256, sm, s>>>(q, k, gamma, S0, Vn, t, p.Hqk, p.Hv, p.K,
                                                                     p.V, scale, o);
    GDN_CK(cudaGetLastError());
  }
#undef GDN_CK
  return GDN_OK;
}

}  // namespace

cudaError_t launch_prepare(const gdn_problem& p, int C, const int32_t* cu_seqlens, Tables t, int nc_max,
                           int32_t* status, cudaStream_t s) {
  prepare_kernel<<<1, 256, 0, s>>>(p.varlen ? cu_seqlens : nullptr, p.N, p.T, C, nc_max, t, status);
  return cudaGetLastError();
}

gdn_status staged_layout(const gdn_problem& p, gdn_staged_layout_t* out) {
  const int nc = nc_max_of(p, p.C);
  const size_t f = sizeof(float);
  const size_t H = p.Hv, C = p.C, K = p.K, V = p.V;
  size_t off = 0;
  gdn_staged_layout_t L;
  L.nc_max = nc;
  L.tables = off; off = align_up(off + tables_bytes(p.N, nc));
  L.status = off; off = align_up(off + sizeof(int32_t));
  L.gamma = off;  off = align_up(off + f * nc * H * C);
  L.A = off;      off = align_up(off + f * nc * H * C * C);
  L.Tinv = off;   off = align_up(off + f * nc * H * C * C);
  L.W = off;      off = align_up(off + f * nc * H * C * K);
  L.U = off;      off = align_up(off + f * nc * H * C * V);
  L.S0 = off;     off = align_up(off + f * nc * H * K * V);
  L.Vn = off;     off = align_up(off + f * nc * H * C * V);
  L.total = off;
  *out = L;
  return GDN_OK;
}

gdn_status run_staged(const gdn_problem& p, int stop_after, const void* q, const void* k, const void* v,
                      const float* g, const float* beta, float scale, const float* h0, const int32_t* cu, void* o,
                      float* ht, void* ws, cudaStream_t s) {
  if (p.dt == GDN_F32) {
    using T = float;
    if (p.C == 64)
      return run_staged_t<T, 64>(p, stop_after, (const T*)q, (const T*)k, (const T*)v, g, beta, scale, h0, cu,
                                 (T*)o, ht, ws, s);
    return run_staged_t<T, 128>(p, stop_after, (const T*)q, (const T*)k, (const T*)v, g, beta, scale, h0, cu,
                                (T*)o, ht, ws, s);
  }
  using T = __nv_bfloat16;
  if (p.C == 64)
    return run_staged_t<T, 64>(p, stop_after, (const T*)q, (const T*)k, (const T*)v, g, beta, scale, h0, cu, (T*)o,
                               ht, ws, s);
  return run_staged_t<T, 128>(p, stop_after, (const T*)q, (const T*)k, (const T*)v, g, beta, scale, h0, cu, (T*)o,
                              ht, ws, s);
}

}  // namespace gdn
