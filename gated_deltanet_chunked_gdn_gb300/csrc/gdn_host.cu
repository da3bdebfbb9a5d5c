// gdn_host.cu -- the forward pass on host-resident tensors: the batch is cut
// into sub-batches of whole sequences that flow through the GPU in a
// pipeline, sub-batch i's inputs copied in while sub-batch i - 1 computes and
// sub-batch i - 2's outputs are copied back (three library-owned streams, two
// sets of device buffers).  Each sub-batch runs the device-buffer forward
// (gdn_chunk_fwd) unchanged.
#include <mutex>
#include <vector>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kMaxDev = 64;

struct HostPipe {
  cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, ev_in[2] = {}, ev_cmp[2] = {}, ev_out[2] = {};
};

std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDev];

// The current device's streams and events, created on first use.
gdn_status pipe_for_device(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return GDN_ERR_UNSUPPORTED;
  HostPipe& h = g_pipe[dev];
  if (!h.in) {
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&h.in, sf) != cudaSuccess || cudaStreamCreateWithFlags(&h.cmp, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h.out, sf) != cudaSuccess || cudaEventCreateWithFlags(&h.start, ef) != cudaSuccess)
      return GDN_ERR_CUDA;
    for (int i = 0; i < 2; ++i)
      if (cudaEventCreateWithFlags(&h.ev_in[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&h.ev_cmp[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&h.ev_out[i], ef) != cudaSuccess)
        return GDN_ERR_CUDA;
  }
  *out = &h;
  return GDN_OK;
}

// Keeps the first non-zero status of the sub-batches.
__global__ void status_keep(int32_t* outer, const int32_t* inner) {
  if (*outer == 0) *outer = *inner;
}

// dst[i] = src[i] - base, i < n: a sub-batch's offsets from the whole batch's.
__global__ void rebase_offsets(int32_t* dst, const int32_t* src, int n, int32_t base) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i] - base;
}

size_t up(size_t b) { return ((b + kAlign - 1) / kAlign) * kAlign; }

// One sub-batch: sequences [s0, s1), tokens [t0, t1) of the packed stream.
struct Sub {
  int s0, s1;
  int64_t t0, t1;
};

// Sub-batches of whole sequences with about equal token counts (fixed
// length: equal sequence counts).
std::vector<Sub> split(const gdn_problem& p, const int32_t* cu, int nsplit) {
  std::vector<Sub> subs;
  const int N = p.N;
  if (nsplit > N) nsplit = N;
  if (nsplit < 1) nsplit = 1;
  const int64_t T = p.varlen ? (int64_t)cu[N] : (int64_t)p.B * p.T;
  int s = 0;
  for (int i = 0; i < nsplit && s < N; ++i) {
    int e;
    if (!p.varlen) {
      e = (int)(((int64_t)N * (i + 1)) / nsplit);
    } else {
      const int64_t goal = (T * (i + 1)) / nsplit;
      e = s + 1;
      while (e < N && cu[e] < goal) ++e;
      if (i == nsplit - 1) e = N;
    }
    if (e <= s) continue;
    const int64_t t0 = p.varlen ? (int64_t)cu[s] : (int64_t)s * p.T;
    const int64_t t1 = p.varlen ? (int64_t)cu[e] : (int64_t)e * p.T;
    subs.push_back({s, e, t0, t1});
    s = e;
  }
  return subs;
}

// The device-buffer problem of one sub-batch.
gdn_problem sub_problem(const gdn_problem& p, const Sub& b) {
  gdn_problem q = p;
  q.N = b.s1 - b.s0;
  if (p.varlen) {
    q.B = 1;
    q.T = (int)(b.t1 - b.t0);
  } else {
    q.B = q.N;
  }
  return q;
}

// Byte layout of the device workspace: the outer status word, the whole
// batch's offsets (packed sequences), the inner forward's workspace, then two
// buffer sets (q, k, v, g, beta, h0, cu, o, ht) sized for the largest
// sub-batch.
struct HostLayout {
  size_t cu_all = 0, inner = 0, inner_bytes = 0, set = 0, set_bytes = 0, total = 0;
  size_t q = 0, k = 0, v = 0, g = 0, beta = 0, h0 = 0, cu = 0, o = 0, ht = 0;
};

HostLayout host_layout(const gdn_problem& p, const std::vector<Sub>& subs, gdn_path path) {
  HostLayout L;
  int64_t tok = 0, seq = 0;
  size_t inner = 0;
  for (const Sub& b : subs) {
    tok = b.t1 - b.t0 > tok ? b.t1 - b.t0 : tok;
    seq = b.s1 - b.s0 > seq ? b.s1 - b.s0 : seq;
    const gdn_problem q = sub_problem(p, b);
    const size_t w = gdn_chunk_fwd_workspace_size(&q, path);
    inner = w > inner ? w : inner;
  }
  const size_t e = p.dt == GDN_BF16 ? 2 : 4;
  L.cu_all = kAlign;
  L.inner = L.cu_all + (p.varlen ? up((size_t)(p.N + 1) * 4) : 0);
  L.inner_bytes = up(inner);
  size_t o = 0;
  L.q = o;
  o += up((size_t)tok * p.Hqk * p.K * e);
  L.k = o;
  o += up((size_t)tok * p.Hqk * p.K * e);
  L.v = o;
  o += up((size_t)tok * p.Hv * p.V * e);
  L.g = o;
  o += up((size_t)tok * p.Hv * 4);
  L.beta = o;
  o += up((size_t)tok * p.Hv * 4);
  L.h0 = o;
  o += up((size_t)seq * p.Hv * p.K * p.V * 4);
  L.cu = o;
  o += up((size_t)(seq + 1) * 4);
  L.o = o;
  o += up((size_t)tok * p.Hv * p.V * e);
  L.ht = o;
  o += up((size_t)seq * p.Hv * p.K * p.V * 4);
  L.set_bytes = o;
  L.set = L.inner + L.inner_bytes;
  L.total = L.set + 2 * L.set_bytes;
  return L;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_chunk_fwd_host_workspace_size(const gdn_problem* p, const int32_t* cu_seqlens, int nsplit, gdn_path path) {
  if (!p || nsplit < 1 || (p->varlen && !cu_seqlens)) return 0;
  if (p->N <= 0 || (int64_t)p->B * p->T <= 0) return kAlign;
  const std::vector<Sub> subs = split(*p, cu_seqlens, nsplit);
  for (const Sub& b : subs) {
    const gdn_problem q = sub_problem(*p, b);
    if (gdn_chunk_fwd_workspace_size(&q, path) == 0) return 0;
  }
  return host_layout(*p, subs, path).total;
}

gdn_status gdn_chunk_fwd_host(const gdn_problem* pp, gdn_path path, int nsplit, const void* q, const void* k,
                              const void* v, const float* g, const float* beta, float scale, const float* h0,
                              const int32_t* cu_seqlens, void* o, float* ht, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!pp || nsplit < 1 || !workspace) return GDN_ERR_INVALID_ARG;
  const gdn_problem p = *pp;
  if (p.varlen != (cu_seqlens != nullptr)) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_chunk_fwd_host_workspace_size(&p, cu_seqlens, nsplit, path);
  if (need == 0 || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % kAlign) return GDN_ERR_INVALID_ARG;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* outer = reinterpret_cast<int32_t*>(ws);
  if (p.N <= 0 || (int64_t)p.B * p.T <= 0)
    return cudaMemsetAsync(outer, 0, sizeof(int32_t), user) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  if (p.varlen) {   // host-side check of the offsets (the device checks again per sub-batch)
    if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[p.N] != (int64_t)p.T) return GDN_ERR_INVALID_ARG;
    for (int n = 0; n < p.N; ++n)
      if (cu_seqlens[n + 1] < cu_seqlens[n]) return GDN_ERR_INVALID_ARG;
  }
  const std::vector<Sub> subs = split(p, cu_seqlens, nsplit);
  const HostLayout L = host_layout(p, subs, path);
  const size_t e = p.dt == GDN_BF16 ? 2 : 4;
  const size_t kv = (size_t)p.K * p.V * 4;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  gdn_status st = pipe_for_device(&hp);
  if (st != GDN_OK) return st;
  auto ok = [](cudaError_t r) { return r == cudaSuccess; };
  if (!ok(cudaEventRecord(hp->start, user)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->cmp, hp->start, 0)) || !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)) ||
      !ok(cudaMemsetAsync(outer, 0, sizeof(int32_t), hp->cmp)))
    return GDN_ERR_CUDA;
  int32_t* cu_all = reinterpret_cast<int32_t*>(ws + L.cu_all);
  if (p.varlen && !ok(cudaMemcpyAsync(cu_all, cu_seqlens, (size_t)(p.N + 1) * 4, cudaMemcpyHostToDevice, hp->in)))
    return GDN_ERR_CUDA;
  for (size_t i = 0; i < subs.size(); ++i) {
    const Sub& b = subs[i];
    const int set = (int)(i & 1);
    uint8_t* base = ws + L.set + set * L.set_bytes;
    const gdn_problem sp = sub_problem(p, b);
    const int64_t nt = b.t1 - b.t0, ns = b.s1 - b.s0;
    // copy-in, once the compute two sub-batches back has read this set
    if (i >= 2 && !ok(cudaStreamWaitEvent(hp->in, hp->ev_cmp[set], 0))) return GDN_ERR_CUDA;
    auto h2d = [&](size_t off, const void* src, size_t bytes) {
      return bytes == 0 || ok(cudaMemcpyAsync(base + off, src, bytes, cudaMemcpyHostToDevice, hp->in));
    };
    const uint8_t* q8 = static_cast<const uint8_t*>(q);
    const uint8_t* k8 = static_cast<const uint8_t*>(k);
    const uint8_t* v8 = static_cast<const uint8_t*>(v);
    if (!h2d(L.q, q8 + (size_t)b.t0 * p.Hqk * p.K * e, (size_t)nt * p.Hqk * p.K * e) ||
        !h2d(L.k, k8 + (size_t)b.t0 * p.Hqk * p.K * e, (size_t)nt * p.Hqk * p.K * e) ||
        !h2d(L.v, v8 + (size_t)b.t0 * p.Hv * p.V * e, (size_t)nt * p.Hv * p.V * e) ||
        !h2d(L.g, g + (size_t)b.t0 * p.Hv, (size_t)nt * p.Hv * 4) ||
        !h2d(L.beta, beta + (size_t)b.t0 * p.Hv, (size_t)nt * p.Hv * 4) ||
        (h0 && !h2d(L.h0, h0 + (size_t)b.s0 * p.Hv * p.K * p.V, (size_t)ns * p.Hv * kv)))
      return GDN_ERR_CUDA;
    if (p.varlen) {
      rebase_offsets<<<1, 256, 0, hp->in>>>(reinterpret_cast<int32_t*>(base + L.cu), cu_all + b.s0, (int)ns + 1,
                                            (int32_t)b.t0);
      if (!ok(cudaGetLastError())) return GDN_ERR_CUDA;
    }
    if (!ok(cudaEventRecord(hp->ev_in[set], hp->in))) return GDN_ERR_CUDA;
    // compute, once this set's inputs are in and its outputs two sub-batches
    // back are out
    if (!ok(cudaStreamWaitEvent(hp->cmp, hp->ev_in[set], 0))) return GDN_ERR_CUDA;
    if (i >= 2 && !ok(cudaStreamWaitEvent(hp->cmp, hp->ev_out[set], 0))) return GDN_ERR_CUDA;
    st = gdn_chunk_fwd(&sp, path, base + L.q, base + L.k, base + L.v, reinterpret_cast<const float*>(base + L.g),
                       reinterpret_cast<const float*>(base + L.beta), scale,
                       h0 ? reinterpret_cast<const float*>(base + L.h0) : nullptr,
                       p.varlen ? reinterpret_cast<const int32_t*>(base + L.cu) : nullptr, base + L.o,
                       ht ? reinterpret_cast<float*>(base + L.ht) : nullptr, ws + L.inner, L.inner_bytes, hp->cmp);
    if (st != GDN_OK) return st;
    status_keep<<<1, 1, 0, hp->cmp>>>(outer, reinterpret_cast<const int32_t*>(ws + L.inner + fwd_status_offset(sp, path)));
    if (!ok(cudaGetLastError()) || !ok(cudaEventRecord(hp->ev_cmp[set], hp->cmp))) return GDN_ERR_CUDA;
    // copy-out
    if (!ok(cudaStreamWaitEvent(hp->out, hp->ev_cmp[set], 0))) return GDN_ERR_CUDA;
    uint8_t* o8 = static_cast<uint8_t*>(o);
    if (!ok(cudaMemcpyAsync(o8 + (size_t)b.t0 * p.Hv * p.V * e, base + L.o, (size_t)nt * p.Hv * p.V * e,
                            cudaMemcpyDeviceToHost, hp->out)))
      return GDN_ERR_CUDA;
    if (ht && !ok(cudaMemcpyAsync(ht + (size_t)b.s0 * p.Hv * p.K * p.V, base + L.ht, (size_t)ns * p.Hv * kv,
                                  cudaMemcpyDeviceToHost, hp->out)))
      return GDN_ERR_CUDA;
    if (!ok(cudaEventRecord(hp->ev_out[set], hp->out))) return GDN_ERR_CUDA;
  }
  // the caller's stream resumes once every output is back
  const int last = (int)((subs.size() - 1) & 1);
  if (!ok(cudaStreamWaitEvent(user, hp->ev_out[last], 0)) ||
      (subs.size() > 1 && !ok(cudaStreamWaitEvent(user, hp->ev_out[last ^ 1], 0))))
    return GDN_ERR_CUDA;
  return GDN_OK;
}

gdn_status gdn_chunk_fwd_host_get_device_status(void* workspace, void* stream, int* dev_status) {
  if (!workspace || !dev_status) return GDN_ERR_INVALID_ARG;
  int32_t host = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpy(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(int32_t)) != cudaSuccess) return GDN_ERR_CUDA;
  *dev_status = host;
  return GDN_OK;
}

}  // extern "C"
