// gdn_decode.cu -- the fused recurrent (decode) step: sigmoid / softplus
// gating and the gated delta-rule state update in one kernel, token by token
// (TileLang x xLLM page, "fused_sigmoid_gating_delta_rule": the decode-phase
// operator that fuses the sigmoid activation, the gate computation from the
// decay rate A_log, and the delta-rule update of the fp32 state; per-sequence
// state offsets for packed batches).
//
// Gating (the usual Gated DeltaNet parameterisation; the page names A_log,
// the sigmoid and exp but prints no formula):
//     g_t    = -exp(A_log[h]) * softplus(a_t + dt_bias[h])      (log-decay)
//     beta_t = sigmoid(b_t)
// then, with S the [K][V] fp32 state of (sequence, value head):
//     S <- e^{g_t} (I - beta_t k_t k_t^T) S + beta_t k_t v_t^T,   o_t = scale S^T q_t
//
// One CTA per (sequence, value head, 64-column slice of V); the slice S[K][64]
// lives in registers (256 threads: 16 float4 column groups x 16 row groups)
// for all of the sequence's tokens and is read and written once.  The step is
// bound by HBM traffic on the state (2 * K * V * 4 bytes per head): the state
// goes through L2 with the evict-first (streaming) hint, since a pool larger
// than L2 is touched once a step, and K <= 128 runs four CTAs an SM (64
// registers) so that more state loads are in flight.
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;
constexpr int kCols = 64;   // V slice per CTA

template <typename Tin, int K>
__global__ void __launch_bounds__(kDecThreads, K <= 128 ? 4 : 2) gdn_recurrent_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v, const float* __restrict__ a,
    const float* __restrict__ b, const float* __restrict__ A_log, const float* __restrict__ dt_bias, float scale,
    float* __restrict__ state, const int32_t* __restrict__ state_indices, int state_slots,
    const int32_t* __restrict__ cu, int Tseq, int64_t Ttot, int Hqk, int Hv, int V, Tin* __restrict__ o) {
  constexpr int RG = 16;         // row groups
  constexpr int RPG = K / RG;    // rows per group
  __shared__ float ks[K], qs[K];
  __shared__ float part[RG][kCols];
  __shared__ float vec[kCols];
  __shared__ float gb[2];
  const int n = blockIdx.x, h = blockIdx.y, e0 = kCols * blockIdx.z;
  const int tid = threadIdx.x, cg = tid & 15, rg = tid >> 4;
  const int hq = h / (Hv / Hqk);
  const int64_t tok0 = cu ? cu[n] : (int64_t)n * Tseq;
  const int64_t L = cu ? (int64_t)cu[n + 1] - cu[n] : Tseq;
  if (L < 0 || tok0 < 0 || tok0 + L > Ttot) return;   // malformed cu_seqlens: touch nothing
  const int slot = state_indices ? state_indices[n] : n;
  if (slot < 0 || slot >= state_slots) {
    // no state for this sequence: its outputs are zero, nothing else is touched
    for (int64_t t = 0; t < L; ++t)
      for (int e = tid; e < kCols; e += kDecThreads) o[((tok0 + t) * Hv + h) * (int64_t)V + e0 + e] = from_f<Tin>(0.f);
    return;
  }
  float* S = state + (((int64_t)slot * Hv + h) * K) * (int64_t)V;
  const int col = e0 + 4 * cg;
  float s[RPG][4];
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rg * RPG + r) * V + col));
    s[r][0] = x.x, s[r][1] = x.y, s[r][2] = x.z, s[r][3] = x.w;
  }
  const float decay_rate = expf(A_log[h]);
  const float bias = dt_bias ? dt_bias[h] : 0.f;
  for (int64_t t = 0; t < L; ++t) {
    const int64_t tok = tok0 + t;
    for (int d = tid; d < K; d += kDecThreads) {
      ks[d] = to_f(k[(tok * Hqk + hq) * (int64_t)K + d]);
      qs[d] = to_f(q[(tok * Hqk + hq) * (int64_t)K + d]);
    }
    if (tid < kCols) vec[tid] = to_f(v[(tok * Hv + h) * (int64_t)V + e0 + tid]);
    if (tid == 0) {
      const float x = a[tok * Hv + h] + bias;
      const float softplus = x > 20.f ? x : log1pf(expf(x));   // log(1 + e^x), exact above 20 in fp32
      gb[0] = expf(-decay_rate * softplus);                    // e^{g_t}
      gb[1] = 1.f / (1.f + expf(-b[tok * Hv + h]));            // beta_t
    }
    __syncthreads();
    const float eg = gb[0], beta = gb[1];
    // k^T S for this thread's 4 columns over its rows
    float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const float kd = ks[rg * RPG + r];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = fmaf(kd, s[r][j], p[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[rg][4 * cg + j] = p[j];
    __syncthreads();
    // delta_e = beta (v_e - e^g k^T S_e);  S <- e^g S + k delta^T
    float dlt[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float ktS = 0.f;
#pragma unroll
      for (int r = 0; r < RG; ++r) ktS += part[r][4 * cg + j];
      dlt[j] = beta * (vec[4 * cg + j] - eg * ktS);
    }
    __syncthreads();   // part is reused below
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = 0.f;
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const float kd = ks[rg * RPG + r], qd = qs[rg * RPG + r];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[r][j] = fmaf(eg, s[r][j], kd * dlt[j]);
        p[j] = fmaf(qd, s[r][j], p[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[rg][4 * cg + j] = p[j];
    __syncthreads();
    if (tid < kCols) {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < RG; ++r) acc += part[r][tid];
      o[(tok * Hv + h) * (int64_t)V + e0 + tid] = from_f<Tin>(scale * acc);
    }
    __syncthreads();   // ks, qs, vec, part, gb reused by the next token
  }
#pragma unroll
  for (int r = 0; r < RPG; ++r)
    __stcs(reinterpret_cast<float4*>(S + (int64_t)(rg * RPG + r) * V + col), make_float4(s[r][0], s[r][1], s[r][2], s[r][3]));
}

template <typename Tin>
gdn_status launch_recurrent(const gdn_problem& p, const Tin* q, const Tin* k, const Tin* v, const float* a,
                            const float* b, const float* A_log, const float* dt_bias, float scale, float* state,
                            const int32_t* idx, int slots, const int32_t* cu, Tin* o, cudaStream_t s) {
  const dim3 grid(p.N, p.Hv, p.V / kCols);
  const int32_t* cup = p.varlen ? cu : nullptr;
  switch (p.K) {
    case 64:
      gdn_recurrent_kernel<Tin, 64><<<grid, kDecThreads, 0, s>>>(q, k, v, a, b, A_log, dt_bias, scale, state, idx,
                                                                 slots, cup, p.T, (int64_t)p.B * p.T, p.Hqk, p.Hv, p.V, o);
      break;
    case 128:
      gdn_recurrent_kernel<Tin, 128><<<grid, kDecThreads, 0, s>>>(q, k, v, a, b, A_log, dt_bias, scale, state, idx,
                                                                  slots, cup, p.T, (int64_t)p.B * p.T, p.Hqk, p.Hv, p.V, o);
      break;
    default:
      gdn_recurrent_kernel<Tin, 256><<<grid, kDecThreads, 0, s>>>(q, k, v, a, b, A_log, dt_bias, scale, state, idx,
                                                                  slots, cup, p.T, (int64_t)p.B * p.T, p.Hqk, p.Hv, p.V, o);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status run_recurrent(const gdn_problem& p, const void* q, const void* k, const void* v, const float* a,
                         const float* b, const float* A_log, const float* dt_bias, float scale, float* state,
                         const int32_t* state_indices, int state_slots, const int32_t* cu, void* o,
                         cudaStream_t s) {
  if (p.N == 0 || p.Hv == 0) return GDN_OK;
  if (p.dt == GDN_F32)
    return launch_recurrent<float>(p, (const float*)q, (const float*)k, (const float*)v, a, b, A_log, dt_bias, scale,
                                   state, state_indices, state_slots, cu, (float*)o, s);
  using T = __nv_bfloat16;
  return launch_recurrent<T>(p, (const T*)q, (const T*)k, (const T*)v, a, b, A_log, dt_bias, scale, state,
                             state_indices, state_slots, cu, (T*)o, s);
}

}  // namespace gdn
