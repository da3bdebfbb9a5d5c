// gdn_api.cu -- the C ABI of libgdn.so (declared in include/gdn.h): host-side
// validation, workspace sizing, path selection and the device status word.
#include <string.h>

#include "gdn_internal.h"

using namespace gdn;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

// Shape checks that need no pointer.  Also normalises N for fixed length.
bool problem_ok(const gdn_problem* pp, gdn_problem* out) {
  if (!pp) return false;
  gdn_problem p = *pp;
  if (p.dt != GDN_F32 && p.dt != GDN_BF16) return false;
  if (p.Hqk <= 0 || p.Hv <= 0 || p.Hv % p.Hqk != 0 || p.Hv > 1024) return false;
  if (!dim_ok(p.K) || !dim_ok(p.V)) return false;
  if (p.C != 64 && p.C != 128) return false;
  if (p.varlen) {
    if (p.B != 1 || p.N <= 0 || p.T < 0) return false;
  } else {
    if (p.B <= 0 || p.T <= 0) return false;
    p.N = p.B;
  }
  // Token indices are int32 inside the kernels; element offsets are int64.
  if ((int64_t)p.B * p.T >= ((int64_t)1 << 31)) return false;
  if ((int64_t)p.N * p.Hv >= ((int64_t)1 << 31)) return false;
  *out = p;
  return true;
}

gdn_path resolve(const gdn_problem& p, gdn_path path) {
  if (path == GDN_PATH_AUTO) {
    if (!fused_supported(p) && !fused1_supported(p)) return GDN_PATH_STAGED;
    if (!fused128_supported(p)) return GDN_PATH_FUSED1;
    if (cp_preferred(p)) return GDN_PATH_CP;
    return fused1_preferred(p) ? GDN_PATH_FUSED1 : GDN_PATH_FUSED;
  }
  return path;
}

bool path_ok(gdn_path path) {
  return path == GDN_PATH_AUTO || path == GDN_PATH_STAGED || path == GDN_PATH_FUSED || path == GDN_PATH_CP ||
         path == GDN_PATH_FUSED1;
}

bool path_supported(const gdn_problem& p, gdn_path path) {
  if (path == GDN_PATH_FUSED) return fused_supported(p);
  if (path == GDN_PATH_FUSED1) return fused1_supported(p);
  if (path == GDN_PATH_CP) return fused128_supported(p);
  return true;
}

size_t workspace_for(const gdn_problem& p, gdn_path path) {
  if (path == GDN_PATH_FUSED1) return fused1_workspace_bytes(p);
  if (path == GDN_PATH_FUSED) return fused_workspace_bytes(p);
  if (path == GDN_PATH_CP) return cp_workspace_bytes(p);
  gdn_staged_layout_t L;
  staged_layout(p, &L);
  return L.total;
}

size_t status_offset(const gdn_problem& p, gdn_path path) {
  if (path == GDN_PATH_FUSED || path == GDN_PATH_FUSED1) return fused_status_offset(p);
  if (path == GDN_PATH_CP) return 0;
  gdn_staged_layout_t L;
  staged_layout(p, &L);
  return L.status;
}

gdn_status check_call(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const float* h0, const int32_t* cu, const void* o, const float* ht,
                      const void* ws, size_t ws_bytes, size_t need) {
  const bool any_tokens = (int64_t)p.B * p.T > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
  if (p.varlen && !cu) return GDN_ERR_INVALID_ARG;
  if (!p.varlen && cu) return GDN_ERR_INVALID_ARG;
  if (!ws || ws_bytes < need || !aligned(ws, kAlign)) return GDN_ERR_INVALID_ARG;
  const void* a16[] = {q, k, v, o};
  for (const void* x : a16)
    if (x && !aligned(x, 16)) return GDN_ERR_INVALID_ARG;
  const void* a4[] = {g, beta, h0, ht, cu};
  for (const void* x : a4)
    if (x && !aligned(x, 4)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // namespace

size_t gdn::fwd_status_offset(const gdn_problem& p, gdn_path path) { return status_offset(p, resolve(p, path)); }

extern "C" {

size_t gdn_chunk_fwd_workspace_size(const gdn_problem* pp, gdn_path path) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return 0;
  if (!path_ok(path)) return 0;
  path = resolve(p, path);
  if (!path_supported(p, path)) return 0;
  return workspace_for(p, path);
}

gdn_path gdn_resolve_path(const gdn_problem* pp) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_PATH_STAGED;
  return resolve(p, GDN_PATH_AUTO);
}

gdn_status gdn_chunk_fwd(const gdn_problem* pp, gdn_path path, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, float scale, const float* h0,
                         const int32_t* cu_seqlens, void* o, float* ht, void* workspace, size_t workspace_bytes,
                         void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_ERR_INVALID_ARG;
  if (!path_ok(path)) return GDN_ERR_INVALID_ARG;
  path = resolve(p, path);
  if (!path_supported(p, path)) return GDN_ERR_UNSUPPORTED;
  gdn_status st = check_call(p, q, k, v, g, beta, h0, cu_seqlens, o, ht, workspace, workspace_bytes,
                             workspace_for(p, path));
  if (st != GDN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == GDN_PATH_FUSED) return run_fused(p, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, workspace, s);
  if (path == GDN_PATH_FUSED1) return run_fused1(p, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, workspace, s);
  if (path == GDN_PATH_CP)
    return run_cp(p, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, workspace, workspace_bytes, s);
  return run_staged(p, 6, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, workspace, s);
}

gdn_status gdn_chunk_fwd_staged(const gdn_problem* pp, int stop_after, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, float scale, const float* h0,
                                const int32_t* cu_seqlens, void* o, float* ht, void* workspace,
                                size_t workspace_bytes, void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_ERR_INVALID_ARG;
  if (stop_after < 0 || stop_after > 6) return GDN_ERR_INVALID_ARG;
  gdn_status st = check_call(p, q, k, v, g, beta, h0, cu_seqlens, o, ht, workspace, workspace_bytes,
                             workspace_for(p, GDN_PATH_STAGED));
  if (st != GDN_OK) return st;
  return run_staged(p, stop_after, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, workspace,
                    static_cast<cudaStream_t>(stream));
}

gdn_status gdn_staged_layout(const gdn_problem* pp, gdn_staged_layout_t* out) {
  gdn_problem p;
  if (!problem_ok(pp, &p) || !out) return GDN_ERR_INVALID_ARG;
  return staged_layout(p, out);
}

gdn_status gdn_get_device_status(const gdn_problem* pp, gdn_path path, void* workspace, void* stream,
                                 int* dev_status) {
  gdn_problem p;
  if (!problem_ok(pp, &p) || !workspace || !dev_status) return GDN_ERR_INVALID_ARG;
  if (!path_ok(path)) return GDN_ERR_INVALID_ARG;
  path = resolve(p, path);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* word = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + status_offset(p, path));
  int32_t host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpy(&host, word, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemset(word, 0, sizeof(int32_t)) != cudaSuccess) return GDN_ERR_CUDA;
  *dev_status = host;
  return GDN_OK;
}

gdn_status gdn_selftest_handover_timeout(const gdn_problem* pp, gdn_path path, const void* q, const void* k,
                                         const void* v,
                                         const float* g, const float* beta, float scale, const float* h0, void* o,
                                         float* ht, void* workspace, size_t workspace_bytes, int drop_window,
                                         long long wait_ns, void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p) || p.varlen || wait_ns <= 0) return GDN_ERR_INVALID_ARG;
  if (path != GDN_PATH_FUSED && path != GDN_PATH_FUSED1) return GDN_ERR_INVALID_ARG;
  const bool one = path == GDN_PATH_FUSED1;
  if (!(one ? fused1_supported(p) && fused1_handover_window(p, drop_window) : fused_handover_window(p, drop_window)))
    return GDN_ERR_UNSUPPORTED;
  gdn_status st = check_call(p, q, k, v, g, beta, h0, nullptr, o, ht, workspace, workspace_bytes,
                             workspace_for(p, path));
  if (st != GDN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned long long lim = static_cast<unsigned long long>(wait_ns);
  return one ? run_fused1(p, q, k, v, g, beta, scale, h0, nullptr, o, ht, workspace, s, drop_window, lim)
             : run_fused(p, q, k, v, g, beta, scale, h0, nullptr, o, ht, workspace, s, drop_window, lim);
}

gdn_status gdn_recurrent_fwd(const gdn_problem* pp, const void* q, const void* k, const void* v, const float* a,
                             const float* b, const float* A_log, const float* dt_bias, float scale, float* state,
                             const int32_t* state_indices, int state_slots, const int32_t* cu_seqlens, void* o,
                             void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_ERR_INVALID_ARG;
  if (p.V % 64 != 0 || state_slots <= 0 || !state || !A_log) return GDN_ERR_INVALID_ARG;
  if (!state_indices && state_slots < p.N) return GDN_ERR_INVALID_ARG;
  const bool any_tokens = (int64_t)p.B * p.T > 0;
  if (any_tokens && (!q || !k || !v || !a || !b || !o)) return GDN_ERR_INVALID_ARG;
  if (p.varlen != (cu_seqlens != nullptr)) return GDN_ERR_INVALID_ARG;
  const void* a16[] = {q, k, v, o, state};
  for (const void* x : a16)
    if (x && !aligned(x, 16)) return GDN_ERR_INVALID_ARG;
  const void* a4[] = {a, b, A_log, dt_bias, state_indices, cu_seqlens};
  for (const void* x : a4)
    if (x && !aligned(x, 4)) return GDN_ERR_INVALID_ARG;
  return run_recurrent(p, q, k, v, a, b, A_log, dt_bias, scale, state, state_indices, state_slots, cu_seqlens, o,
                       static_cast<cudaStream_t>(stream));
}

gdn_status gdn_causal_conv1d_fwd(const void* x, const float* weight, const float* bias, int W, void* conv_state,
                                 int state_slots, const int32_t* cache_indices, const int32_t* has_initial_state,
                                 const int32_t* cu_seqlens, int N, int B, int T, int D, gdn_dtype dt,
                                 gdn_activation act, void* y, void* stream) {
  if (W < 1 || W > 4 || D <= 0 || D % 8 != 0 || B < 0 || T < 0 || N < 0) return GDN_ERR_INVALID_ARG;
  if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (act != GDN_ACT_NONE && act != GDN_ACT_SILU) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens ? B != 1 : N != B) return GDN_ERR_INVALID_ARG;
  if ((int64_t)B * T > 0 && (!x || !y)) return GDN_ERR_INVALID_ARG;
  if (!weight) return GDN_ERR_INVALID_ARG;
  if (W > 1 && conv_state && (state_slots <= 0 || (!cache_indices && state_slots < N))) return GDN_ERR_INVALID_ARG;
  const void* a16[] = {x, y, W > 1 ? conv_state : nullptr};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return GDN_ERR_INVALID_ARG;
  const void* a4[] = {weight, bias, cache_indices, has_initial_state, cu_seqlens};
  for (const void* p : a4)
    if (p && !aligned(p, 4)) return GDN_ERR_INVALID_ARG;
  return run_causal_conv1d(x, weight, bias, W, conv_state, state_slots, cache_indices, has_initial_state, cu_seqlens,
                           N, B, T, D, dt, act == GDN_ACT_SILU, y, static_cast<cudaStream_t>(stream));
}

size_t gdn_chunk_bwd_workspace_size(const gdn_problem* pp) {
  gdn_problem p;
  if (!problem_ok(pp, &p) || !bwd_supported(p)) return 0;
  // the chunked form also needs 16-byte aligned q, k, v and dout, which the
  // query cannot see: size for whichever form the call takes
  const size_t token = bwd_workspace_bytes(p);
  if (!bwdc_supported(p)) return token;
  const size_t chunked = bwdc_workspace_bytes(p);
  return chunked > token ? chunked : token;
}

gdn_status gdn_chunk_bwd(const gdn_problem* pp, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, float scale, const float* h0, const int32_t* cu_seqlens,
                         const void* dout, const float* dht, float* dq, float* dk, float* dv, float* dg,
                         float* dbeta, float* dh0, void* workspace, size_t workspace_bytes, void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_ERR_INVALID_ARG;
  if (!bwd_supported(p)) return GDN_ERR_UNSUPPORTED;
  const bool any_tokens = (int64_t)p.B * p.T > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_INVALID_ARG;
  if (p.varlen != (cu_seqlens != nullptr)) return GDN_ERR_INVALID_ARG;
  // the chunked backward reads q, k, v and dout in 16-byte vectors
  const bool chunked = bwdc_supported(p) && (int64_t)p.N * p.Hv > 0 && aligned(q, 16) && aligned(k, 16) &&
                       aligned(v, 16) && aligned(dout, 16);
  const size_t need = chunked ? bwdc_workspace_bytes(p) : bwd_workspace_bytes(p);
  if (!workspace || workspace_bytes < need || !aligned(workspace, kAlign)) return GDN_ERR_INVALID_ARG;
  const void* a16[] = {dh0, dht, h0};
  for (const void* x : a16)
    if (x && !aligned(x, 16)) return GDN_ERR_INVALID_ARG;
  const void* a4[] = {q, k, v, g, beta, cu_seqlens, dout, dq, dk, dv, dg, dbeta};
  for (const void* x : a4)
    if (x && !aligned(x, 4)) return GDN_ERR_INVALID_ARG;
  if (chunked)
    return run_bwdc(p, q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                    static_cast<cudaStream_t>(stream));
  return run_bwd(p, q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                 static_cast<cudaStream_t>(stream));
}

gdn_status gdn_chunk_bwd_get_device_status(void* workspace, void* stream, int* dev_status) {
  if (!workspace || !dev_status) return GDN_ERR_INVALID_ARG;
  int32_t* word = static_cast<int32_t*>(workspace);
  int32_t host = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpy(&host, word, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemset(word, 0, sizeof(int32_t)) != cudaSuccess) return GDN_ERR_CUDA;
  *dev_status = host;
  return GDN_OK;
}

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported problem for this path";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_DEVICE: return "device reported an error";
    case GDN_ERR_SCRATCH_LIMIT: return "problem needs more than the built-in 32 MiB static scratch";
  }
  return "unknown status";
}

const char* gdn_version(void) { return "gdn 0.1 sm_103a"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward pass without any caller-provided or library-allocated device memory
// beyond the caller's inputs and outputs.
//
// Some callers cannot allocate device memory in the call path: an op embedded
// in a host framework that owns every device buffer and hands the op only its
// inputs and outputs (no workspace), or a caller that cannot afford the
// implicit device-wide synchronisation of cudaMalloc/cudaFree between its
// launches.  For them the forward pass runs with its workspace in one
// file-scope device array, kStaticScratchBytes (32 MiB) per GPU, which every
// GPU that loads this library holds until the process exits: the fused
// kernels whenever their workspace fits (a status word, the order table of a
// packed batch, or the window schedule's hand-over states: about 20 MB on 152
// SMs), else the staged path when its intermediates fit.  The first kAlign
// bytes of the array hold the status word of the last call (copied there from
// the workspace, which starts right after it), so that
// gdn_chunk_fwd_noalloc_get_device_status can read it without the problem.
#include <cudaTypedefs.h>
#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr size_t kStaticStagedBytes = kStaticScratchBytes - kAlign;   // after the status slot
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};
unsigned long long g_static_ctx[kMaxDevices] = {};   // context the cached address belongs to

// Unique id of the current CUDA context (0 when the driver cannot tell), through
// the driver entry points that the runtime hands out.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_scratch on the current device.  The host-side
// name of the array is only a stand-in, so the address is fetched with
// cudaGetSymbolAddress (with that device current) once per device and
// context, and cached: a device reset that replaces the context makes the
// next call look the address up again.
gdn_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  // 0 before the runtime has made the device's context current: then the
  // look-up below creates it, and the id is read again afterwards
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev] || ctx == 0 || g_static_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_static_ptr[dev] = p;
    g_static_ctx[dev] = current_context_id();
  }
  *out = g_static_ptr[dev];
  return GDN_OK;
}

// The path of a gdn_chunk_fwd_noalloc call: AUTO's choice, with the fused
// kernel in place of the chunk-parallel path (whose per-segment states do
// not fit the array), when its workspace fits; else the staged path when its
// intermediates fit; GDN_PATH_AUTO when neither does.
gdn_path noalloc_path(const gdn_problem& p) {
  gdn_path path = resolve(p, GDN_PATH_AUTO);
  if (path == GDN_PATH_CP) path = GDN_PATH_FUSED;
  if (path != GDN_PATH_STAGED && workspace_for(p, path) <= kStaticStagedBytes) return path;
  if (workspace_for(p, GDN_PATH_STAGED) <= kStaticStagedBytes) return GDN_PATH_STAGED;
  return GDN_PATH_AUTO;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(const gdn_problem* pp, const void* q, const void* k, const void* v,
                                            const float* g, const float* beta, float scale, const float* h0,
                                            const int32_t* cu_seqlens, void* o, float* ht, void* stream) {
  gdn_problem p;
  if (!problem_ok(pp, &p)) return GDN_ERR_INVALID_ARG;
  const gdn_path path = noalloc_path(p);
  if (path == GDN_PATH_AUTO) return GDN_ERR_SCRATCH_LIMIT;
  const size_t need = workspace_for(p, path);
  void* scratch = nullptr;
  gdn_status st = static_scratch(&scratch);
  if (st != GDN_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(scratch) + kAlign;
  st = check_call(p, q, k, v, g, beta, h0, cu_seqlens, o, ht, ws, kStaticStagedBytes, need);
  if (st != GDN_OK) return st;
  // each path clears the status word (and the window flags) it uses; every
  // other intermediate is rewritten before it is read, so stale contents of
  // earlier calls are harmless.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == GDN_PATH_FUSED) st = run_fused(p, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, ws, s);
  else if (path == GDN_PATH_FUSED1) st = run_fused1(p, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, ws, s);
  else st = run_staged(p, 6, q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, ws, s);
  if (st != GDN_OK) return st;
  // the call's status word goes to the fixed slot at the array's start
  if (cudaMemcpyAsync(scratch, ws + status_offset(p, path), sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

extern "C" gdn_status gdn_chunk_fwd_noalloc_get_device_status(void* stream, int* dev_status) {
  if (!dev_status) return GDN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  gdn_status st = static_scratch(&scratch);
  if (st != GDN_OK) return st;
  int32_t host = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpy(&host, scratch, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemset(scratch, 0, sizeof(int32_t)) != cudaSuccess) return GDN_ERR_CUDA;
  *dev_status = host;
  return GDN_OK;
}
