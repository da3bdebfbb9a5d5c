// gdn_bwd.cu -- backward pass of the Gated DeltaNet forward (gradients of o
// and ht with respect to q, k, v, g, beta and h0; the FlashQLA notes list a
// backward among the variants of the chunk kernel, section 4.3).
//
// Reverse mode of the token recurrence S_t = a_t P_t S_{t-1} + b_t k_t v_t^T,
// P_t = I - b_t k_t k_t^T, o_t = scale S_t^T q_t (a_t = e^{g_t}, b_t = beta_t),
// with G = dL/dS_t walked from dht back to dh0:
//   G += scale q_t dout_t^T;   dq_t = scale S_t dout_t
//   u = S_{t-1}^T k_t, w = G^T k_t;   dv_t = b_t w
//   dg_t = a_t (<G, S_{t-1}> - b_t w.u);   dbeta_t = -a_t w.u + w.v_t
//   dk_t = -a_t b_t (G u + S_{t-1} w) + b_t G v_t;   G <- a_t (G - b_t k_t w^T)
//
// Columns of S (and of G) evolve independently, so a CTA owns one
// (sequence, value head, 16-column slice of V); thread d holds row d of the
// slice of S and of G in registers.  Sums over d (u, w, <G, S>) are block
// reductions; sums over the 16 columns are per thread, and the column slices
// and the value heads of a GQA group meet in fp32 atomics on dq, dk, dg and
// dbeta (order of addition not fixed).
//
// States S_{t-1} are needed in reverse order: a forward pass stores every
// chain's state at the start of each 64-token chunk; the backward recomputes
// a chunk from its checkpoint keeping the states at 16-token steps, then
// each 16-token block from its start keeping all 17 states in shared memory,
// and walks back through the block.  About three forward recurrences of work
// plus the reverse one, all in fp32.
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

constexpr int kCols = 16;   // V columns per CTA
constexpr int kChunkB = 64;  // checkpoint interval
constexpr int kSub = 16;     // tokens per recomputed block
constexpr int kRow = 20;     // padded row length of the state tiles in shared memory (floats)

template <int K>
struct BwdSmem {
  float st[kSub + 1][K][kRow];        // states before each token of a block, and after its last
  float lvl[kChunkB / kSub][K][kRow];  // block-start states of a chunk
  float u[kSub][kCols];                // S_{t-1}^T k_t of the block's tokens
  float red[K / 32][kCols + 1];
  float sum[kCols + 1];
};

// Sum of NV values over the K threads of the block; the total lands in out[].
template <int K, int NV>
__device__ __forceinline__ void block_sum(float (&x)[NV], float (*red)[kCols + 1], float* out, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x[j] += __shfl_xor_sync(0xffffffffu, x[j], off);
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < NV; ++j) red[warp][j] = x[j];
  __syncthreads();
  if (tid < NV) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < K / 32; ++w) s += red[w][tid];
    out[tid] = s;
  }
  __syncthreads();
}

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;
  const void* dout;
  const float* dht;
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dh0;
  float* ckpt;   // [slots][Hv][K][V]
  int32_t* status;
  int64_t Ttot;
  int N, Tseq, Hqk, Hv, V;
  float scale;
};

// Sequence bounds; false (status set) for malformed cu_seqlens.
__device__ __forceinline__ bool bwd_bounds(const BwdArgs& a, int n, int64_t& tok0, int64_t& L) {
  if (a.cu) {
    const int64_t s = a.cu[n], e = a.cu[n + 1];
    bool ok = 0 <= s && s <= e && e <= a.Ttot;
    if (n == 0 && (a.cu[0] != 0 || a.cu[a.N] != a.Ttot)) ok = false;
    if (!ok) {
      if (threadIdx.x == 0) atomicExch(a.status, GDN_DEV_BAD_CU_SEQLENS);
      return false;
    }
    tok0 = s;
    L = e - s;
  } else {
    tok0 = (int64_t)n * a.Tseq;
    L = a.Tseq;
  }
  return true;
}

// Checkpoint slot of the chunk that starts at token t0 of sequence n: distinct
// for all chunks of all sequences, below ceil(Ttot / 64) + N.
__device__ __forceinline__ int64_t ckpt_slot(int64_t t0, int n) { return t0 / kChunkB + n; }

// One forward token: S <- a (S - b k (k^T S)) + b k v^T for this thread's row.
template <typename T, int K>
__device__ __forceinline__ void fwd_token(const BwdArgs& a, BwdSmem<K>& s, int tid, int64_t t, int hq, int h, int e0,
                                          float (&S)[kCols], float* u_out) {
  const float kd = to_f(static_cast<const T*>(a.k)[(t * a.Hqk + hq) * (int64_t)K + tid]);
  float x[kCols];
#pragma unroll
  for (int e = 0; e < kCols; ++e) x[e] = S[e] * kd;
  block_sum<K, kCols>(x, s.red, s.sum, tid);
  const float ag = expf(a.g[t * a.Hv + h]), b = a.beta[t * a.Hv + h];
  const T* vt = static_cast<const T*>(a.v) + (t * a.Hv + h) * (int64_t)a.V + e0;
#pragma unroll
  for (int e = 0; e < kCols; ++e) {
    const float ue = s.sum[e];
    S[e] = ag * (S[e] - b * kd * ue) + b * kd * to_f(vt[e]);
  }
  if (u_out && tid < kCols) u_out[tid] = s.sum[tid];
  __syncthreads();   // s.sum is reused by the next reduction
}

// Checkpoints: the forward recurrence of every chain, the state slice saved at
// each chunk start.  Grid (N, Hv, V / 16), K threads.
template <typename T, int K>
__global__ void __launch_bounds__(K) gdn_bwd_ckpt_kernel(const BwdArgs a) {
  __shared__ float red[K / 32][kCols + 1];
  __shared__ float sum[kCols + 1];
  const int n = blockIdx.x, h = blockIdx.y, e0 = kCols * blockIdx.z, tid = threadIdx.x;
  const int hq = h / (a.Hv / a.Hqk);
  int64_t tok0, L;
  if (!bwd_bounds(a, n, tok0, L)) return;
  float S[kCols];
  const size_t KV = (size_t)K * a.V;
  const float* h0p = a.h0 ? a.h0 + ((size_t)n * a.Hv + h) * KV + (size_t)tid * a.V + e0 : nullptr;
#pragma unroll
  for (int e = 0; e < kCols; ++e) S[e] = h0p ? h0p[e] : 0.f;
  for (int64_t i = 0; i < L; ++i) {
    const int64_t t = tok0 + i;
    if (i % kChunkB == 0) {
      float* cp = a.ckpt + ((size_t)ckpt_slot(t, n) * a.Hv + h) * KV + (size_t)tid * a.V + e0;
#pragma unroll
      for (int e = 0; e < kCols; e += 4) *reinterpret_cast<float4*>(cp + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
    }
    const float kd = to_f(static_cast<const T*>(a.k)[(t * a.Hqk + hq) * (int64_t)K + tid]);
    float x[kCols];
#pragma unroll
    for (int e = 0; e < kCols; ++e) x[e] = S[e] * kd;
    block_sum<K, kCols>(x, red, sum, tid);
    const float ag = expf(a.g[t * a.Hv + h]), b = a.beta[t * a.Hv + h];
    const T* vt = static_cast<const T*>(a.v) + (t * a.Hv + h) * (int64_t)a.V + e0;
#pragma unroll
    for (int e = 0; e < kCols; ++e) S[e] = ag * (S[e] - b * kd * sum[e]) + b * kd * to_f(vt[e]);
    __syncthreads();
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(K) gdn_bwd_kernel(const BwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdSmem<K>& s = *reinterpret_cast<BwdSmem<K>*>(smem_raw);
  const int n = blockIdx.x, h = blockIdx.y, e0 = kCols * blockIdx.z, tid = threadIdx.x;
  const int hq = h / (a.Hv / a.Hqk);
  int64_t tok0, L;
  if (!bwd_bounds(a, n, tok0, L)) return;
  const size_t KV = (size_t)K * a.V;
  const size_t row = ((size_t)n * a.Hv + h) * KV + (size_t)tid * a.V + e0;   // this thread's row of the slice
  float G[kCols];
#pragma unroll
  for (int e = 0; e < kCols; ++e) G[e] = a.dht ? a.dht[row + e] : 0.f;
  const int nchunks = (int)((L + kChunkB - 1) / kChunkB);
  auto put = [&](float* p, const float (&x)[kCols]) {
#pragma unroll
    for (int e = 0; e < kCols; e += 4) *reinterpret_cast<float4*>(p + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
  };
  auto get = [&](const float* p, float (&x)[kCols]) {
#pragma unroll
    for (int e = 0; e < kCols; e += 4) {
      const float4 y = *reinterpret_cast<const float4*>(p + e);
      x[e] = y.x, x[e + 1] = y.y, x[e + 2] = y.z, x[e + 3] = y.w;
    }
  };
  for (int c = nchunks - 1; c >= 0; --c) {
    const int64_t t0 = tok0 + (int64_t)kChunkB * c;
    const int Lc = (int)(L - (int64_t)kChunkB * c < kChunkB ? L - (int64_t)kChunkB * c : kChunkB);
    float S[kCols];
    get(a.ckpt + ((size_t)ckpt_slot(t0, n) * a.Hv + h) * KV + (size_t)tid * a.V + e0, S);
    // block-start states of the chunk
    for (int i = 0; i < Lc; ++i) {
      if (i % kSub == 0) put(&s.lvl[i / kSub][tid][0], S);
      fwd_token<T, K>(a, s, tid, t0 + i, hq, h, e0, S, nullptr);
    }
    const int nsub = (Lc + kSub - 1) / kSub;
    for (int sb = nsub - 1; sb >= 0; --sb) {
      const int64_t tb = t0 + (int64_t)kSub * sb;
      const int nb = Lc - kSub * sb < kSub ? Lc - kSub * sb : kSub;
      get(&s.lvl[sb][tid][0], S);
      put(&s.st[0][tid][0], S);
      for (int i = 0; i < nb; ++i) {
        fwd_token<T, K>(a, s, tid, tb + i, hq, h, e0, S, &s.u[i][0]);
        put(&s.st[i + 1][tid][0], S);
      }
      __syncthreads();   // u of the block visible to every thread
      for (int i = nb - 1; i >= 0; --i) {
        const int64_t t = tb + i;
        const float qd = to_f(static_cast<const T*>(a.q)[(t * a.Hqk + hq) * (int64_t)K + tid]);
        const float kd = to_f(static_cast<const T*>(a.k)[(t * a.Hqk + hq) * (int64_t)K + tid]);
        const T* dot = static_cast<const T*>(a.dout) + (t * a.Hv + h) * (int64_t)a.V + e0;
        const T* vt = static_cast<const T*>(a.v) + (t * a.Hv + h) * (int64_t)a.V + e0;
        const float ag = expf(a.g[t * a.Hv + h]), b = a.beta[t * a.Hv + h];
        float dov[kCols], vv[kCols], Sn[kCols], Sp[kCols], uu[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          dov[e] = to_f(dot[e]);
          vv[e] = to_f(vt[e]);
          uu[e] = s.u[i][e];
        }
        get(&s.st[i + 1][tid][0], Sn);
        get(&s.st[i][tid][0], Sp);
        float dq = 0.f;
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          G[e] = fmaf(a.scale * qd, dov[e], G[e]);
          dq = fmaf(Sn[e], dov[e], dq);
        }
        float x[kCols + 1];
        float gs = 0.f;
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          x[e] = G[e] * kd;
          gs = fmaf(G[e], Sp[e], gs);
        }
        x[kCols] = gs;
        block_sum<K, kCols + 1>(x, s.red, s.sum, tid);
        float w[kCols];
        float wu = 0.f, wv = 0.f;
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          w[e] = s.sum[e];
          wu = fmaf(w[e], uu[e], wu);
          wv = fmaf(w[e], vv[e], wv);
        }
        const float gsum = s.sum[kCols];
        if (tid < kCols) a.dv[(t * a.Hv + h) * (int64_t)a.V + e0 + tid] = b * s.sum[tid];
        if (tid == 0) {
          atomicAdd(a.dg + t * a.Hv + h, ag * (gsum - b * wu));
          atomicAdd(a.dbeta + t * a.Hv + h, -ag * wu + wv);
        }
        float gu = 0.f, sw = 0.f, gv = 0.f;
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          gu = fmaf(G[e], uu[e], gu);
          sw = fmaf(Sp[e], w[e], sw);
          gv = fmaf(G[e], vv[e], gv);
        }
        atomicAdd(a.dq + (t * a.Hqk + hq) * (int64_t)K + tid, a.scale * dq);
        atomicAdd(a.dk + (t * a.Hqk + hq) * (int64_t)K + tid, -ag * b * (gu + sw) + b * gv);
#pragma unroll
        for (int e = 0; e < kCols; ++e) G[e] = ag * (G[e] - b * kd * w[e]);
        __syncthreads();   // s.sum is reused by the next reduction
      }
    }
  }
  if (a.dh0) {
    float* dh = a.dh0 + row;
#pragma unroll
    for (int e = 0; e < kCols; e += 4) *reinterpret_cast<float4*>(dh + e) = make_float4(G[e], G[e + 1], G[e + 2], G[e + 3]);
  }
}

template <typename T, int K>
gdn_status launch_bwd(const BwdArgs& a, cudaStream_t s) {
  const dim3 grid(a.N, a.Hv, a.V / kCols);
  gdn_bwd_ckpt_kernel<T, K><<<grid, K, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  const int smem = (int)sizeof(BwdSmem<K>);
  if (cudaFuncSetAttribute(gdn_bwd_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  gdn_bwd_kernel<T, K><<<grid, K, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

bool bwd_supported(const gdn_problem& p) { return (p.K == 64 || p.K == 128) && p.V % kCols == 0; }

size_t bwd_workspace_bytes(const gdn_problem& p) {
  const int64_t Ttot = (int64_t)p.B * p.T;
  const int64_t slots = (Ttot + kChunkB - 1) / kChunkB + p.N;
  return kAlign + align_up(sizeof(float) * (size_t)slots * p.Hv * p.K * p.V);
}

gdn_status run_bwd(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                   const float* beta, float scale, const float* h0, const int32_t* cu, const void* dout,
                   const float* dht, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws,
                   cudaStream_t s) {
  if (!bwd_supported(p)) return GDN_ERR_UNSUPPORTED;
  uint8_t* w = static_cast<uint8_t*>(ws);
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.h0 = h0;
  a.cu = p.varlen ? cu : nullptr;
  a.dout = dout;
  a.dht = dht;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dg = dg;
  a.dbeta = dbeta;
  a.dh0 = dh0;
  a.status = reinterpret_cast<int32_t*>(w);
  a.ckpt = reinterpret_cast<float*>(w + kAlign);
  a.Ttot = (int64_t)p.B * p.T;
  a.N = p.N;
  a.Tseq = p.T;
  a.Hqk = p.Hqk;
  a.Hv = p.Hv;
  a.V = p.V;
  a.scale = scale;
  if (cudaMemsetAsync(a.status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  const size_t tq = sizeof(float) * (size_t)a.Ttot * p.Hqk * p.K, tg = sizeof(float) * (size_t)a.Ttot * p.Hv;
  if (tq && (cudaMemsetAsync(dq, 0, tq, s) != cudaSuccess || cudaMemsetAsync(dk, 0, tq, s) != cudaSuccess))
    return GDN_ERR_CUDA;
  if (tg && (cudaMemsetAsync(dg, 0, tg, s) != cudaSuccess || cudaMemsetAsync(dbeta, 0, tg, s) != cudaSuccess))
    return GDN_ERR_CUDA;
  if ((int64_t)p.N * p.Hv == 0) return GDN_OK;
  if (p.dt == GDN_F32) return p.K == 64 ? launch_bwd<float, 64>(a, s) : launch_bwd<float, 128>(a, s);
  using B16 = __nv_bfloat16;
  return p.K == 64 ? launch_bwd<B16, 64>(a, s) : launch_bwd<B16, 128>(a, s);
}

}  // namespace gdn
