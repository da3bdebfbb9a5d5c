// gdn_conv1d.cu -- causal depthwise convolution with a carried state
// (TileLang x xLLM page, causal_conv1d: every output token depends on the
// current and earlier inputs of its own sequence; the last W-1 inputs of each
// sequence are kept in a state pool, the slot chosen by cache_indices, so
// that decode continues where prefill stopped).
//
// For a sequence with inputs x_0..x_{L-1}, ext = [W-1 initial inputs ;
// x_0..x_{L-1}] and, per channel d,
//     y_p[d]    = act(bias[d] + sum_{w<W} weight[d][w] ext_{p+w}[d])
//     new state = ext_L .. ext_{L+W-2}
//
// The operation is bound by HBM traffic (one read of x, one write of y).  A
// thread owns 8 consecutive channels (one 16-byte vector of bf16) over a run
// of kTok tokens; a warp reads and writes 512 contiguous bytes per token.  The
// W-1 previous inputs stay in registers as raw vectors (a sliding window), so
// x is read once plus a W-1 token halo per run; the loads of the next
// kUnroll tokens are issued before the arithmetic of the current ones, so
// that the memory stream overlaps the activation.  The state pool is rewritten by a second launch,
// after the first has read every old state.
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;   // channel vectors per CTA
// tokens per thread run: long runs spread the per-run start (weights, bias and
// the W-1 token halo) over more tokens (64: 1.31 ms, 128: 1.21, 256: 1.17, 512:
// 1.19 ms for 16 x 8192 tokens, D = 12288)
constexpr int kTok = 256;
constexpr int kUnroll = 4;          // tokens a batch (the next batch loaded ahead)

template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  uint4 raw;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { raw = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = raw; }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    raw = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ void zero() { raw = make_uint4(0u, 0u, 0u, 0u); }
};

template <>
struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = a;
    reinterpret_cast<float4*>(p)[1] = b;
  }
  __device__ __forceinline__ void to_float(float (&f)[8]) const {
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
  }
  __device__ __forceinline__ void from_float(const float (&f)[8]) {
    a = make_float4(f[0], f[1], f[2], f[3]);
    b = make_float4(f[4], f[5], f[6], f[7]);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
};

struct ConvArgs {
  const void* x;
  const float* weight;
  const float* bias;
  void* state;
  const int32_t* idx;
  const int32_t* init;
  const int32_t* cu;
  void* y;
  int64_t Ttot;
  int N, Tseq, D, slots;
};

// Sequence n's token range [s, e); false for malformed cu_seqlens entries.
__device__ __forceinline__ bool seq_bounds(const ConvArgs& a, int n, int64_t& s, int64_t& e) {
  if (a.cu) {
    s = a.cu[n];
    e = a.cu[n + 1];
  } else {
    s = (int64_t)n * a.Tseq;
    e = s + a.Tseq;
  }
  return 0 <= s && s <= e && e <= a.Ttot;
}

// Sequence n's state slot, or -1 when it has none.
__device__ __forceinline__ int seq_slot(const ConvArgs& a, int n) {
  if (!a.state) return -1;
  const int slot = a.idx ? a.idx[n] : n;
  return (slot >= 0 && slot < a.slots) ? slot : -1;
}

// 1/y on the MUFU unit (rcp.approx.ftz.f32: about 1 ulp; 1/+inf = +0).
__device__ __forceinline__ float rcp_approx(float y) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// SiLU u sigmoid(u) = u / (1 + e^{-u}) is evaluated in emit below with two
// MUFU operations per value (ex2 of -u log2 e, then rcp) instead of an IEEE
// division; for very negative u, e^{-u} overflows to +inf and the result is
// -0.  The multiplies, adds and the convolution's FMAs run on pairs of
// channels (the packed fp32 instructions of sm_100+, the same IEEE rounding
// per value as the scalar ones).

template <typename T, int W, bool SILU>
__global__ void __launch_bounds__(kConvThreads, sizeof(T) == 2 ? 4 : 2) conv1d_kernel(const ConvArgs a) {
  const int c0 = 8 * (blockIdx.y * kConvThreads + threadIdx.x);
  if (c0 >= a.D) return;
  const int64_t t0 = (int64_t)blockIdx.x * kTok;
  const int64_t t1 = t0 + kTok < a.Ttot ? t0 + kTok : a.Ttot;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ y = static_cast<T*>(a.y);
  const T* st = static_cast<const T*>(a.state);
  const int64_t D = a.D;

  float wt[W][8], bs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int w = 0; w < W; ++w) wt[w][j] = __ldg(a.weight + (int64_t)(c0 + j) * W + w);
    bs[j] = a.bias ? __ldg(a.bias + c0 + j) : 0.f;
  }

  // first sequence that can hold t0: the last n whose start is <= t0
  int n;
  if (a.cu) {
    int lo = 0, hi = a.N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu[mid] <= t0) lo = mid; else hi = mid - 1;
    }
    n = lo;
  } else {
    n = (int)(t0 / a.Tseq);
  }

  int64_t t = t0;
  while (t < t1 && n < a.N) {
    int64_t s, e;
    if (!seq_bounds(a, n, s, e) || e <= t) {   // malformed, empty or already passed
      ++n;
      continue;
    }
    if (s > t) {   // tokens that no sequence covers stay unwritten
      t = s;
      continue;
    }
    const int64_t end = e < t1 ? e : t1;
    const int slot = seq_slot(a, n);
    const bool has = slot >= 0 && (a.init ? a.init[n] != 0 : true);
    // win[i] = ext_{p - (W-1) + i} for the token at position p = t - s
    Vec8<T> win[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
      const int64_t pos = (t - s) - (W - 1) + i;
      if (pos >= 0) win[i].load(x + (s + pos) * D + c0);
      else if (has) win[i].load(st + ((int64_t)slot * (W - 1) + (W - 1) + pos) * D + c0);
      else win[i].zero();
    }
    auto emit = [&](const Vec8<T>& xin, int64_t tt) {
      float acc[8], f[8];
      float2 a2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) a2[j] = make_float2(bs[2 * j], bs[2 * j + 1]);
#pragma unroll
      for (int w = 0; w < W; ++w) {
        if (w < W - 1) win[w].to_float(f);
        else xin.to_float(f);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          a2[j] = __ffma2_rn(make_float2(wt[w][2 * j], wt[w][2 * j + 1]), make_float2(f[2 * j], f[2 * j + 1]), a2[j]);
      }
      if (SILU) {
        const float2 nl = make_float2(-sm100::kLog2e, -sm100::kLog2e), one = make_float2(1.f, 1.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 t = __fmul2_rn(a2[j], nl);
          const float2 d = __fadd2_rn(make_float2(sm100::ex2_fast(t.x), sm100::ex2_fast(t.y)), one);
          a2[j] = __fmul2_rn(a2[j], make_float2(rcp_approx(d.x), rcp_approx(d.y)));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[2 * j] = a2[j].x, acc[2 * j + 1] = a2[j].y;
#pragma unroll
      for (int w = 0; w + 1 < W - 1; ++w) win[w] = win[w + 1];
      if (W > 1) win[W > 1 ? W - 2 : 0] = xin;
      Vec8<T> o;
      o.from_float(acc);
      o.store(y + tt * D + c0);
    };
    // batches of kUnroll tokens, the next batch's loads issued before this
    // batch's arithmetic so that they overlap it
    if (t + kUnroll <= end) {
      Vec8<T> v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u].load(x + (t + u) * D + c0);
      for (;;) {
        const bool more = t + 2 * kUnroll <= end;
        Vec8<T> nv[kUnroll];
        if (more) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) nv[u].load(x + (t + kUnroll + u) * D + c0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) emit(v[u], t + u);
        t += kUnroll;
        if (!more) break;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = nv[u];
      }
    }
    for (; t < end; ++t) {
      Vec8<T> v;
      v.load(x + t * D + c0);
      emit(v, t);
    }
  }
}

// New state of sequence n = its last W-1 ext entries (raw copies: exact).
// One thread per (sequence, channel vector) reads every entry it needs from
// the old state before it writes any, so the in-place update is safe.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads) conv1d_state_kernel(const ConvArgs a) {
  const int n = blockIdx.x;
  const int c0 = 8 * (blockIdx.y * kConvThreads + threadIdx.x);
  if (c0 >= a.D) return;
  const int slot = seq_slot(a, n);
  if (slot < 0) return;
  int64_t s, e;
  if (!seq_bounds(a, n, s, e)) return;
  const int64_t L = e - s, D = a.D;
  const bool has = a.init ? a.init[n] != 0 : true;
  const T* x = static_cast<const T*>(a.x);
  T* st = static_cast<T*>(a.state) + (int64_t)slot * (W - 1) * D;
  Vec8<T> v[W - 1];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t pos = L - (W - 1) + j;
    if (pos >= 0) v[j].load(x + (s + pos) * D + c0);
    else if (has) v[j].load(st + ((W - 1) + pos) * D + c0);   // an older entry of the same slot
    else v[j].zero();
  }
#pragma unroll
  for (int j = 0; j < W - 1; ++j) v[j].store(st + j * D + c0);
}

template <typename T, int W>
gdn_status launch_conv(const ConvArgs& a, bool silu_act, cudaStream_t s) {
  const int cvb = (a.D / 8 + kConvThreads - 1) / kConvThreads;
  if (a.Ttot > 0) {
    const dim3 grid((unsigned)((a.Ttot + kTok - 1) / kTok), cvb);
    if (silu_act) conv1d_kernel<T, W, true><<<grid, kConvThreads, 0, s>>>(a);
    else conv1d_kernel<T, W, false><<<grid, kConvThreads, 0, s>>>(a);
  }
  if constexpr (W > 1) {
    if (a.state && a.N > 0) conv1d_state_kernel<T, W><<<dim3(a.N, cvb), kConvThreads, 0, s>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
gdn_status dispatch_w(const ConvArgs& a, int W, bool silu_act, cudaStream_t s) {
  switch (W) {
    case 1: return launch_conv<T, 1>(a, silu_act, s);
    case 2: return launch_conv<T, 2>(a, silu_act, s);
    case 3: return launch_conv<T, 3>(a, silu_act, s);
    default: return launch_conv<T, 4>(a, silu_act, s);
  }
}

}  // namespace

gdn_status run_causal_conv1d(const void* x, const float* weight, const float* bias, int W, void* conv_state,
                             int state_slots, const int32_t* cache_indices, const int32_t* has_initial_state,
                             const int32_t* cu_seqlens, int N, int B, int T, int D, gdn_dtype dt, bool silu_act,
                             void* y, cudaStream_t s) {
  ConvArgs a;
  a.x = x;
  a.weight = weight;
  a.bias = bias;
  a.state = W > 1 ? conv_state : nullptr;
  a.idx = cache_indices;
  a.init = has_initial_state;
  a.cu = cu_seqlens;
  a.y = y;
  a.Ttot = (int64_t)B * T;
  a.N = N;
  a.Tseq = T;
  a.D = D;
  a.slots = state_slots;
  if (dt == GDN_F32) return dispatch_w<float>(a, W, silu_act, s);
  return dispatch_w<__nv_bfloat16>(a, W, silu_act, s);
}

}  // namespace gdn
