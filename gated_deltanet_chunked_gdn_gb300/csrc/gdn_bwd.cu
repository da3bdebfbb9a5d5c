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
// (sequence, value head, 8-column slice of V); thread d holds row d of the
// slice of S and of G in registers.  Sums over d (u, w, <G, S>) are block
// reductions; sums over the 8 columns are per thread, and the column slices
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

constexpr int kCols = 8;    // V columns per CTA
constexpr int kChunkB = 64;  // checkpoint interval
constexpr int kSub = 16;     // tokens per recomputed block
constexpr int kRow = kCols;  // row length of the state tiles in shared memory (floats)

// One 16-token block of the inputs, converted to fp32 (k, q: full rows; v,
// dout: this CTA's 16 columns; e^g and beta).
template <int K>
struct TokBlock {
  float k[kSub][K];
  float q[kSub][K];
  float v[kSub][kCols];
  float dout[kSub][kCols];
  float a[kSub];
  float b[kSub];
};

template <int K>
struct BwdSmem {
  float st[kSub + 1][K][kRow];        // states before each token of a block, and after its last
  float lvl[kChunkB / kSub][K][kRow];  // block-start states of a chunk
  float u[kSub][kCols];                // S_{t-1}^T k_t of the block's tokens
  TokBlock<K> tb;
  float red[K / 32][kCols + 1];
  float sum[kCols + 1];
};

// Warp sum of NC (8 or 16) values by reduce-scatter: at each of the first
// log2(NC) levels a lane keeps half of its values and adds its partner's copy
// of that half (NC / 2, NC / 4, ..., 1 exchanges), the remaining levels add
// the last partials; lanes (32 / NC) j .. (32 / NC) (j + 1) - 1 end with the
// total of value j.  2 NC - 1 + 5 - log2(NC) shuffles instead of 5 NC.
template <int NC>
__device__ __forceinline__ float warp_sum_rs(float (&x)[NC], int lane) {
  constexpr int kLevels = NC == 16 ? 4 : 3;
#pragma unroll
  for (int lvl = 0; lvl < kLevels; ++lvl) {
    const int half = (NC / 2) >> lvl;       // values kept after this level
    const int off = 16 >> lvl;              // partner lane distance
    const bool upper = (lane & off) != 0;   // keep the upper half of the live values
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? x[j] : x[j + half];
      const float keep = upper ? x[j + half] : x[j];
      x[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = x[0];
#pragma unroll
  for (int off = (16 >> kLevels); off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// Index (0..NC-1) of the value whose total lane `lane` holds after warp_sum_rs.
template <int NC>
__device__ __forceinline__ int warp_sum_rs_index(int lane) {
  // level l kept the upper half when bit (16 >> l) of the lane was set; the
  // kept half's offset adds (NC / 2) >> l
  int i = 0;
#pragma unroll
  for (int lvl = 0; lvl < (NC == 16 ? 4 : 3); ++lvl)
    if (lane & (16 >> lvl)) i += (NC / 2) >> lvl;
  return i;
}

// Sum of NV (kCols or kCols + 1) values over the K threads of the block; the
// totals land in out[].
template <int K, int NV>
__device__ __forceinline__ void block_sum(float (&x)[NV], float (*red)[kCols + 1], float* out, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  float y[kCols];
#pragma unroll
  for (int j = 0; j < kCols; ++j) y[j] = x[j];
  const float tot = warp_sum_rs<kCols>(y, lane);
  if ((lane & (32 / kCols - 1)) == 0) red[warp][warp_sum_rs_index<kCols>(lane)] = tot;
  if (NV > kCols) {
    float z = x[NV - 1];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane == 0) red[warp][kCols] = z;
  }
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

// Token block [t0, t0 + n) into shared memory (fp32), all threads.
template <typename T, int K>
__device__ __forceinline__ void stage_block(const BwdArgs& a, TokBlock<K>& tb, int64_t t0, int n, int hq, int h,
                                            int e0, bool with_q, int tid) {
  const T* kp = static_cast<const T*>(a.k);
  const T* qp = static_cast<const T*>(a.q);
  for (int i = tid; i < n * K; i += K) {
    const int r = i / K, d = i % K;
    const int64_t off = ((t0 + r) * a.Hqk + hq) * (int64_t)K + d;
    tb.k[r][d] = to_f(kp[off]);
    if (with_q) tb.q[r][d] = to_f(qp[off]);
  }
  for (int i = tid; i < n * kCols; i += K) {
    const int r = i / kCols, e = i % kCols;
    const int64_t off = ((t0 + r) * a.Hv + h) * (int64_t)a.V + e0 + e;
    tb.v[r][e] = to_f(static_cast<const T*>(a.v)[off]);
    if (with_q) tb.dout[r][e] = to_f(static_cast<const T*>(a.dout)[off]);
  }
  if (tid < n) {
    tb.a[tid] = expf(a.g[(t0 + tid) * a.Hv + h]);
    tb.b[tid] = a.beta[(t0 + tid) * a.Hv + h];
  }
  __syncthreads();
}

// One forward token (row i of the staged block): S <- a (S - b k (k^T S)) + b k v^T
// for this thread's row of the state.
template <int K>
__device__ __forceinline__ void fwd_token(const TokBlock<K>& tb, int i, float (*red)[kCols + 1], float* sum, int tid,
                                          float (&S)[kCols], float* u_out) {
  const float kd = tb.k[i][tid];
  float x[kCols];
#pragma unroll
  for (int e = 0; e < kCols; ++e) x[e] = S[e] * kd;
  block_sum<K, kCols>(x, red, sum, tid);
  const float ag = tb.a[i], b = tb.b[i];
#pragma unroll
  for (int e = 0; e < kCols; ++e) S[e] = ag * (S[e] - b * kd * sum[e]) + b * kd * tb.v[i][e];
  if (u_out && tid < kCols) u_out[tid] = sum[tid];
  __syncthreads();   // sum is reused by the next reduction
}

// Checkpoints: the forward recurrence of every chain, the state slice saved at
// each chunk start.  Grid (N, Hv, V / 16), K threads.
template <typename T, int K>
__global__ void __launch_bounds__(K) gdn_bwd_ckpt_kernel(const BwdArgs a) {
  __shared__ float red[K / 32][kCols + 1];
  __shared__ float sum[kCols + 1];
  __shared__ TokBlock<K> tb;
  const int n = blockIdx.x, h = blockIdx.y, e0 = kCols * blockIdx.z, tid = threadIdx.x;
  const int hq = h / (a.Hv / a.Hqk);
  int64_t tok0, L;
  if (!bwd_bounds(a, n, tok0, L)) return;
  float S[kCols];
  const size_t KV = (size_t)K * a.V;
  const float* h0p = a.h0 ? a.h0 + ((size_t)n * a.Hv + h) * KV + (size_t)tid * a.V + e0 : nullptr;
#pragma unroll
  for (int e = 0; e < kCols; ++e) S[e] = h0p ? h0p[e] : 0.f;
  for (int64_t i0 = 0; i0 < L; i0 += kSub) {
    const int64_t t0 = tok0 + i0;
    if (i0 % kChunkB == 0) {
      float* cp = a.ckpt + ((size_t)ckpt_slot(t0, n) * a.Hv + h) * KV + (size_t)tid * a.V + e0;
#pragma unroll
      for (int e = 0; e < kCols; e += 4) *reinterpret_cast<float4*>(cp + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
    }
    const int nb = L - i0 < kSub ? (int)(L - i0) : kSub;
    stage_block<T, K>(a, tb, t0, nb, hq, h, e0, false, tid);
    for (int i = 0; i < nb; ++i) fwd_token<K>(tb, i, red, sum, tid, S, nullptr);
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
    for (int i0 = 0; i0 < Lc; i0 += kSub) {
      put(&s.lvl[i0 / kSub][tid][0], S);
      const int nb = Lc - i0 < kSub ? Lc - i0 : kSub;
      stage_block<T, K>(a, s.tb, t0 + i0, nb, hq, h, e0, false, tid);
      for (int i = 0; i < nb; ++i) fwd_token<K>(s.tb, i, s.red, s.sum, tid, S, nullptr);
    }
    const int nsub = (Lc + kSub - 1) / kSub;
    for (int sb = nsub - 1; sb >= 0; --sb) {
      const int64_t tb = t0 + (int64_t)kSub * sb;
      const int nb = Lc - kSub * sb < kSub ? Lc - kSub * sb : kSub;
      get(&s.lvl[sb][tid][0], S);
      put(&s.st[0][tid][0], S);
      stage_block<T, K>(a, s.tb, tb, nb, hq, h, e0, true, tid);
      for (int i = 0; i < nb; ++i) {
        fwd_token<K>(s.tb, i, s.red, s.sum, tid, S, &s.u[i][0]);
        put(&s.st[i + 1][tid][0], S);
      }
      __syncthreads();   // u of the block visible to every thread
      for (int i = nb - 1; i >= 0; --i) {
        const int64_t t = tb + i;
        const float qd = s.tb.q[i][tid], kd = s.tb.k[i][tid];
        const float ag = s.tb.a[i], b = s.tb.b[i];
        float dov[kCols], vv[kCols], Sn[kCols], Sp[kCols], uu[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) {
          dov[e] = s.tb.dout[i][e];
          vv[e] = s.tb.v[i][e];
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
