// gdn_cp.cu -- chunk-parallel forward pass for problems with few
// (sequence, value head) chains: each sequence is cut into segments of whole
// 64-token chunks that run on separate SMs (the "AutoCP" intra-sequence chunk
// parallelism of the FlashQLA notes, sections 8.3 and 9.2).
//
// The chunk recurrence is affine in the state: a segment maps its initial
// state S to M S + B, with M (K x K) the product of its chunks' transitions and
// B its final state from S = 0.  Three steps:
//   1. one states-only launch of the fused kernel over all segments x heads
//      computes B (zero initial state) and M (initial state I, v = 0);
//   2. a small kernel chains the segments of each (sequence, head):
//      S_{j+1} = M_j S_j + B_j, starting from h0 (tcgen05 products in three
//      bf16 terms); it records every segment's initial state S_j and writes
//      the sequence's final state (ht);
//   3. the fused kernel reruns every segment from its S_j and writes o.
// Work is about three times that of the serial pass, spread over
// (segments x heads) CTAs instead of (sequences x heads).
#include "gdn_internal.h"
#include "gdn_solve64.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kPrepThreads = 1024;

struct CpLayout {
  size_t status, seg_cu, seq_seg, bst, mst, h0s, total;
  int ns_max;
};

CpLayout cp_layout(const gdn_problem& p, int seg_len) {
  CpLayout L;
  const int64_t Ttot = (int64_t)p.B * p.T;
  L.ns_max = (int)((Ttot + seg_len - 1) / seg_len) + p.N;
  const size_t st = sizeof(float) * (size_t)L.ns_max * p.Hv * kD * kD;
  size_t off = 0;
  L.status = off;
  off += kAlign;
  L.seg_cu = off;
  off = align_up(off + sizeof(int32_t) * (L.ns_max + 1));
  L.seq_seg = off;
  off = align_up(off + sizeof(int32_t) * (p.N + 1));
  L.bst = off;
  off = align_up(off + st);
  L.mst = off;
  off = align_up(off + st);
  L.h0s = off;
  off = align_up(off + st);
  L.total = off;
  return L;
}

// Segment tables from the sequence bounds (single CTA).  Sequence n gets
// ceil(L_n / seg_len) segments of seg_len tokens (the last may be shorter);
// seq_seg[n] is its first segment, seg_cu the segments' token offsets, padded
// to ns_max segments with empty ones at the end.  Malformed cu_seqlens: status
// is set and every table entry is 0, so that the launches that follow reject
// the segment table and no sequence has a segment.
__global__ void __launch_bounds__(kPrepThreads) cp_prepare_kernel(const int32_t* __restrict__ cu, int N, int Tseq,
                                                                  int64_t Ttot, int seg_len, int ns_max,
                                                                  int32_t* __restrict__ seg_cu,
                                                                  int32_t* __restrict__ seq_seg, int32_t* status) {
  __shared__ int bad;
  __shared__ int carry;
  __shared__ int part[kPrepThreads];
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = 0;
    carry = 0;
  }
  __syncthreads();
  auto start = [&](int n) -> int64_t { return cu ? (int64_t)cu[n] : (int64_t)n * Tseq; };
  if (cu) {
    for (int n = tid; n < N; n += kPrepThreads)
      if (cu[n] > cu[n + 1]) bad = 1;
    if (tid == 0 && (cu[0] != 0 || cu[N] != Ttot)) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) atomicExch(status, GDN_DEV_BAD_CU_SEQLENS);
    for (int i = tid; i <= ns_max; i += kPrepThreads) seg_cu[i] = 0;
    for (int i = tid; i <= N; i += kPrepThreads) seq_seg[i] = 0;
    return;
  }
  // exclusive prefix sum of the segment counts, kPrepThreads sequences at a time
  for (int base = 0; base < N; base += kPrepThreads) {
    const int n = base + tid;
    int cnt = 0;
    if (n < N) cnt = (int)((start(n + 1) - start(n) + seg_len - 1) / seg_len);
    part[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < kPrepThreads; off <<= 1) {
      const int x = tid >= off ? part[tid - off] : 0;
      __syncthreads();
      part[tid] += x;
      __syncthreads();
    }
    const int first = carry + part[tid] - cnt;
    if (n < N) {
      seq_seg[n] = first;
      for (int j = 0; j < cnt; ++j) seg_cu[first + j] = (int32_t)(start(n) + (int64_t)j * seg_len);
    }
    __syncthreads();
    if (tid == kPrepThreads - 1) carry += part[tid];
    __syncthreads();
  }
  const int total = carry;
  if (tid == 0) seq_seg[N] = total;
  for (int i = total + tid; i <= ns_max; i += kPrepThreads) seg_cu[i] = (int32_t)Ttot;
}

// Chain the segments of (sequence n, value head h) for 64 state columns
// [e0, e0 + 64): H0s[j] = S_j, S_{j+1} = M_j S_j + B_j from S_0 = h0, ht = the
// last S.  One CTA of 128 threads per (sequence, head, column half); thread d
// owns row d of the state slice (TMEM lane d).  Each step's product runs on the
// tensor cores (tcgen05, fp32 accumulation in TMEM) in three bf16 terms: with
// x = hi + lo (hi = x rounded to bf16, lo = the rest rounded to bf16),
// M S = Mh Sh + Mh Sl + Ml Sh up to the dropped Ml Sl and the rounding of the
// lo parts, about 2^-17 of each product.  While a step's product runs, M_{j+1}
// and the slice of B_j are staged in shared memory by coalesced cp.async.
//   A = M_j [d][d'] (K-major, 128-byte swizzle): Mh, Ml, 2 atoms of 16 KB each
//   B = S_j [d'][e] (MN-major, one 64-wide group): Sh, Sl, 16 KB each
constexpr uint32_t kCbMH = 0, kCbML = 32768, kCbSH = 65536, kCbSL = 81920;
constexpr uint32_t kCbMst = 98304;              // M_{j+1} fp32 [128][128], row-major
constexpr uint32_t kCbBst = 163840;             // B_j fp32 [128][64], rows of 68 floats
constexpr uint32_t kCbBld = 68;
constexpr uint32_t kCbBar = kCbBst + 128 * kCbBld * 4;
constexpr uint32_t kCbSmem = kCbBar + 64 + 1024;   // + alignment slack

// Eight floats split into bf16 hi / lo halves, one 16-byte chunk each.
__device__ __forceinline__ void split8_store(const float* x, uint8_t* hi, uint8_t* lo) {
  float h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
    l[i] = x[i] - h[i];
  }
  solve64::store8_bf16(hi, h);
  solve64::store8_bf16(lo, l);
}

__global__ void __launch_bounds__(128) cp_combine_kernel(const int32_t* __restrict__ seq_seg, int Hv,
                                                         const float* __restrict__ h0, const float* __restrict__ Bst,
                                                         const float* __restrict__ Mst, float* __restrict__ H0s,
                                                         float* __restrict__ ht, int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kCbBar);
  volatile uint32_t* flags = reinterpret_cast<volatile uint32_t*>(sm + kCbBar + 8);
  const float* mst = reinterpret_cast<const float*>(sm + kCbMst);
  const float* bst = reinterpret_cast<const float*>(sm + kCbBst);
  const int n = blockIdx.x, h = blockIdx.y, e0 = 64 * blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, d = tid;
  const size_t mat = (size_t)kD * kD;
  const int j0 = seq_seg[n], j1 = seq_seg[n + 1];
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
    flags[1] = 0;
  }
  if (warp == 0) tmem_alloc(const_cast<uint32_t*>(flags), 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = flags[0];
  const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
  const uint32_t s4 = (smem_u32(sm) & 0x3FFFFu) >> 4;
  auto mat_of = [&](const float* base, int j) { return base + ((size_t)j * Hv + h) * mat; };
  // cp.async of M_j (all of it) and of B_j's column slice
  auto stage_m = [&](int j) {
    const float* src = mat_of(Mst, j);
    for (int i = tid; i < kD * kD / 4; i += 128) cp_async16(sm + kCbMst + 16 * i, src + 4 * i);
  };
  auto stage_b = [&](int j) {
    const float* src = mat_of(Bst, j) + e0;
    for (int i = tid; i < kD * 16; i += 128) {
      const int r = i >> 4, q = i & 15;
      cp_async16(sm + kCbBst + (r * kCbBld + 4 * q) * 4, src + (size_t)r * kD + 4 * q);
    }
  };
  // M (staged) -> Mh, Ml: warp w splits rows 32w..32w+31, lane l columns 4l..4l+3
  auto split_m = [&]() {
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * warp + i;
      const float4 v = *reinterpret_cast<const float4*>(mst + r * kD + 4 * lane);
      const float x[4] = {v.x, v.y, v.z, v.w};
      uint32_t hw[2], lw[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float h0f = __bfloat162float(__float2bfloat16_rn(x[2 * u]));
        const float h1f = __bfloat162float(__float2bfloat16_rn(x[2 * u + 1]));
        hw[u] = pack_bf16(h0f, h1f);
        lw[u] = pack_bf16(x[2 * u] - h0f, x[2 * u + 1] - h1f);
      }
      const int c = 4 * lane;
      const uint32_t off = (c >> 6) * 16384u + sw128_chunk(r, (c & 63) >> 3) + (c & 7) * 2;
      *reinterpret_cast<uint2*>(sm + kCbMH + off) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(sm + kCbML + off) = make_uint2(lw[0], lw[1]);
    }
  };
  // row d of a state slice -> its record (H0s or ht) and, when another step
  // follows, Sh / Sl
  auto emit_row = [&](const float (&x)[64], float* dst, bool split) {
    if (dst) {
#pragma unroll
      for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    }
    if (split) {
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) split8_store(x + 8 * cc, sm + kCbSH + sw128_chunk(d, cc), sm + kCbSL + sw128_chunk(d, cc));
    }
  };
  auto rec = [&](int j) -> float* {   // where S_j's row d is recorded
    if (j < j1) return H0s + ((size_t)j * Hv + h) * mat + (size_t)d * kD + e0;
    return ht ? ht + ((size_t)n * Hv + h) * mat + (size_t)d * kD + e0 : nullptr;
  };

  if (j1 > j0) {
    stage_m(j0);
    cp_async_commit();
  }
  {
    const float* h0p = h0 ? h0 + ((size_t)n * Hv + h) * mat + (size_t)d * kD + e0 : nullptr;
    float x[64];
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      const float4 v = h0p ? *reinterpret_cast<const float4*>(h0p + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[i] = v.x, x[i + 1] = v.y, x[i + 2] = v.z, x[i + 3] = v.w;
    }
    emit_row(x, rec(j0), j1 > j0);
  }
  if (j1 > j0) {
    cp_async_wait_all();
    __syncthreads();
    split_m();
  }
  uint32_t ph = 0;
#pragma unroll 1
  for (int j = j0; j < j1; ++j) {
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();   // Mh, Ml, Sh, Sl complete; the staging buffers read
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64, 0, 1, 0);
      const uint32_t a_off[3] = {kCbMH, kCbMH, kCbML}, b_off[3] = {kCbSH, kCbSL, kCbSH};
#pragma unroll
      for (int t = 0; t < 3; ++t)
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_bf16(tmem, solve64::dsw(s4, a_off[t] + (s >> 2) * 16384 + (s & 3) * 32, 16),
                   solve64::dsw(s4, b_off[t] + s * 2048, 16384), id, (t | s) ? 1u : 0u);
      mma_commit(bar);
    }
    stage_b(j);
    if (j + 1 < j1) stage_m(j + 1);
    cp_async_commit();
    if (!mbar_wait(bar, ph, status)) flags[1] = 1;
    ph ^= 1;
    cp_async_wait_all();
    __syncwarp();
    tc_fence_after();
    __syncthreads();   // the staged B_j and M_{j+1} are visible to every thread
    if (flags[1]) break;
    // S_{j+1} row d = D row d + B_j row d
    {
      float x[64], y[32];
      tmem_ld32(tmem + lane_off, y);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = y[i];
      tmem_ld32(tmem + lane_off + 32, y);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[32 + i] = y[i];
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(bst + d * kCbBld + i);
        x[i] += v.x, x[i + 1] += v.y, x[i + 2] += v.z, x[i + 3] += v.w;
      }
      emit_row(x, rec(j + 1), j + 1 < j1);
    }
    if (j + 1 < j1) split_m();
    tc_fence_before();
  }
  if (tid == 0 && flags[1]) mbar_wait(bar, ph, status, 100000000ull);
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 148;
  return n > 0 ? n : 148;
}

// Segment length (a multiple of the 64-token chunk, at least 512 tokens): aim
// for about two (segment, head) chains per SM in the final pass, from the mean
// sequence length (the host does not read cu_seqlens).
int cp_segment_length(const gdn_problem& p) {
  const int64_t Ttot = (int64_t)p.B * p.T;
  const int64_t chains = (int64_t)p.N * p.Hv;
  if (Ttot <= 0 || chains <= 0) return 64;
  const int64_t per_seq = (Ttot + p.N - 1) / p.N;
  const int64_t want = 2LL * sm_count();
  const int64_t segs = want / chains > 1 ? want / chains : 1;
  int64_t len = (per_seq + segs - 1) / segs;
  len = (len + 63) / 64 * 64;
  // at least 8 chunks a segment: shorter ones leave the launches and the
  // serial combine step to dominate
  return (int)(len < 512 ? 512 : (len > (1 << 30) ? (1 << 30) : len));
}

size_t cp_workspace_bytes(const gdn_problem& p) { return cp_layout(p, cp_segment_length(p)).total; }

// Fewer chains than half the SMs and sequences of at least 2048 tokens on
// average: the serial pass would leave most SMs idle for many chunks.
bool cp_preferred(const gdn_problem& p) {
  const int64_t Ttot = (int64_t)p.B * p.T;
  const int64_t chains = (int64_t)p.N * p.Hv;
  if (chains <= 0 || Ttot <= 0 || !fused128_supported(p)) return false;
  return 2 * chains <= sm_count() && Ttot / p.N >= 2048;
}

gdn_status run_cp(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                  const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht, void* ws,
                  size_t ws_bytes, cudaStream_t s) {
  if (!fused128_supported(p)) return GDN_ERR_UNSUPPORTED;
  const int seg_len = cp_segment_length(p);
  const CpLayout L = cp_layout(p, seg_len);
  if (ws_bytes < L.total) return GDN_ERR_INVALID_ARG;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w + L.status);
  int32_t* seg_cu = reinterpret_cast<int32_t*>(w + L.seg_cu);
  int32_t* seq_seg = reinterpret_cast<int32_t*>(w + L.seq_seg);
  float* Bst = reinterpret_cast<float*>(w + L.bst);
  float* Mst = reinterpret_cast<float*>(w + L.mst);
  float* H0s = reinterpret_cast<float*>(w + L.h0s);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  const int64_t Ttot = (int64_t)p.B * p.T;
  if (Ttot == 0 || (int64_t)p.N * p.Hv == 0) {
    if (ht) {
      const size_t bytes = sizeof(float) * (size_t)p.N * p.Hv * p.K * p.V;
      cudaError_t e = h0 ? cudaMemcpyAsync(ht, h0, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(ht, 0, bytes, s);
      if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
  }
  cp_prepare_kernel<<<1, kPrepThreads, 0, s>>>(p.varlen ? cu : nullptr, p.N, p.T, Ttot, seg_len, L.ns_max, seg_cu,
                                               seq_seg, status);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  // the segments as a packed batch of ns_max sequences
  gdn_problem ps = p;
  ps.B = 1;
  ps.T = (int)Ttot;
  ps.N = L.ns_max;
  ps.varlen = 1;
  gdn_status st = run_fused_states(ps, k, v, g, beta, seg_cu, Bst, Mst, status, s);
  if (st != GDN_OK) return st;
  if (cudaFuncSetAttribute(cp_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCbSmem) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  cp_combine_kernel<<<dim3(p.N, p.Hv, 2), 128, kCbSmem, s>>>(seq_seg, p.Hv, h0, Bst, Mst, H0s, ht, status);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  return launch_fused(ps, 0, q, k, v, g, beta, scale, H0s, seg_cu, o, nullptr, nullptr, status, s);
}

}  // namespace gdn
