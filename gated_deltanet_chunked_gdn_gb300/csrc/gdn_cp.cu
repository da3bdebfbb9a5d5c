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
//   2. a small fp32 kernel chains the segments of each (sequence, head):
//      S_{j+1} = M_j S_j + B_j, starting from h0; it records every segment's
//      initial state S_j and writes the sequence's final state (ht);
//   3. the fused kernel reruns every segment from its S_j and writes o.
// Work is about three times that of the serial pass, spread over
// (segments x heads) CTAs instead of (sequences x heads).
#include "gdn_internal.h"
#include "gdn_sm100.cuh"

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

// Chain the segments of (sequence n, value head h) for 16 state columns:
// H0s[j] = S_j, S_{j+1} = M_j S_j + B_j from S_0 = h0, ht = the last S.
// 128 threads, thread t owning rows t/4 + 32 r (r < 4) and 4 columns of the
// 128 x 16 slice.  M_j is row-major in 32-column k-blocks, staged into a
// double-buffered shared tile by cp.async one block ahead of the FMAs; a
// step of the inner product reads four rows of M and four rows of S as
// 16-byte loads for 64 FMAs (row stride 36 floats: the eight rows a warp
// reads fall on distinct banks).
constexpr int kCSlice = 16;
constexpr int kKb = 32;
constexpr int kMld = kKb + 4;

__global__ void __launch_bounds__(128) cp_combine_kernel(const int32_t* __restrict__ seq_seg, int Hv,
                                                         const float* __restrict__ h0, const float* __restrict__ Bst,
                                                         const float* __restrict__ Mst, float* __restrict__ H0s,
                                                         float* __restrict__ ht) {
  __shared__ __align__(16) float S[kD][kCSlice];
  __shared__ __align__(16) float Mb[2][kD][kMld];
  const int n = blockIdx.x, h = blockIdx.y, e0 = kCSlice * blockIdx.z;
  const int tid = threadIdx.x, t = tid >> 2, c0 = 4 * (tid & 3);
  const size_t mat = (size_t)kD * kD;
  const float* h0p = h0 ? h0 + ((size_t)n * Hv + h) * mat : nullptr;
  for (int i = tid; i < kD * kCSlice; i += 128) {
    const int r = i / kCSlice, c = i % kCSlice;
    S[r][c] = h0p ? h0p[(size_t)r * kD + e0 + c] : 0.f;
  }
  const int j0 = seq_seg[n], j1 = seq_seg[n + 1];
  const int nb = (j1 - j0) * (kD / kKb);   // k-blocks of all the segments, in order
  auto stage = [&](int blk) {
    const float* src = Mst + ((size_t)(j0 + blk / (kD / kKb)) * Hv + h) * mat + (blk % (kD / kKb)) * kKb;
    float* dst = &Mb[blk & 1][0][0];
    for (int i = tid; i < kD * (kKb / 4); i += 128) {
      const int d = i / (kKb / 4), q = i % (kKb / 4);
      cp_async16(dst + d * kMld + 4 * q, src + (size_t)d * kD + 4 * q);
    }
    cp_async_commit();
  };
  if (nb > 0) stage(0);
  __syncthreads();
  float acc[4][4];
  for (int blk = 0; blk < nb; ++blk) {
    const int j = j0 + blk / (kD / kKb), kbi = blk % (kD / kKb), kb = kbi * kKb;
    const size_t base = ((size_t)j * Hv + h) * mat;
    if (kbi == 0) {
      // segment start: record S_j, start from B_j
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = t + 32 * r;
        const float4 sv = *reinterpret_cast<const float4*>(&S[d][c0]);
        *reinterpret_cast<float4*>(H0s + base + (size_t)d * kD + e0 + c0) = sv;
        const float4 bv = *reinterpret_cast<const float4*>(Bst + base + (size_t)d * kD + e0 + c0);
        acc[r][0] = bv.x, acc[r][1] = bv.y, acc[r][2] = bv.z, acc[r][3] = bv.w;
      }
    }
    if (blk + 1 < nb) {
      stage(blk + 1);
      cp_async_wait_prev();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();   // block blk is in shared memory
    const float* Mk = &Mb[blk & 1][0][0];
#pragma unroll 2
    for (int g = 0; g < kKb / 4; ++g) {
      float m[4][4], x[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(Mk + (t + 32 * r) * kMld + 4 * g);
        m[r][0] = v.x, m[r][1] = v.y, m[r][2] = v.z, m[r][3] = v.w;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 v = *reinterpret_cast<const float4*>(&S[kb + 4 * g + u][c0]);
        x[u][0] = v.x, x[u][1] = v.y, x[u][2] = v.z, x[u][3] = v.w;
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(m[r][u], x[u][c], acc[r][c]);
    }
    __syncthreads();   // this buffer and S read: the next stage and S's update may go ahead
    if (kbi == kD / kKb - 1) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4*>(&S[t + 32 * r][c0]) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      __syncthreads();
    }
  }
  if (ht) {
    float* htp = ht + ((size_t)n * Hv + h) * mat;
    for (int i = tid; i < kD * kCSlice; i += 128) {
      const int r = i / kCSlice, c = i % kCSlice;
      htp[(size_t)r * kD + e0 + c] = S[r][c];
    }
  }
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
  cp_combine_kernel<<<dim3(p.N, p.Hv, kD / kCSlice), 128, 0, s>>>(seq_seg, p.Hv, h0, Bst, Mst, H0s, ht);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  return launch_fused(ps, 0, q, k, v, g, beta, scale, H0s, seg_cu, o, nullptr, nullptr, status, s);
}

}  // namespace gdn
