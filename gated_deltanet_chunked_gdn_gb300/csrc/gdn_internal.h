// gdn_internal.h -- shared host/device helpers of libgdn (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr size_t kAlign = 256;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Chunk tables written by the prepare kernel (layout documented in gdn.h,
// gdn_staged_layout_t::tables).  nc < 0 marks malformed cu_seqlens.
struct Tables {
  int32_t* seq_chunk0;  // [N + 1]
  int32_t* chunk_seq;   // [nc_max]
  int32_t* chunk_tok0;  // [nc_max]
  int32_t* chunk_len;   // [nc_max]
  int32_t* nc;          // [1]
};

inline Tables tables_at(void* base, int N, int nc_max) {
  int32_t* p = reinterpret_cast<int32_t*>(base);
  Tables t;
  t.seq_chunk0 = p;
  t.chunk_seq = p + (N + 1);
  t.chunk_tok0 = t.chunk_seq + nc_max;
  t.chunk_len = t.chunk_tok0 + nc_max;
  t.nc = t.chunk_len + nc_max;
  return t;
}

inline size_t tables_bytes(int N, int nc_max) { return sizeof(int32_t) * ((size_t)N + 1 + 3 * (size_t)nc_max + 1); }

inline int nc_max_of(const gdn_problem& p, int C) {
  return p.varlen ? (int)(ceil_div(p.T, C) + p.N) : (int)(p.B * ceil_div(p.T, C));
}

// Launch the prepare kernel: chunk tables for chunk length C, validation of
// cu_seqlens (status word + nc = -1 on error).
cudaError_t launch_prepare(const gdn_problem& p, int C, const int32_t* cu_seqlens, Tables t, int nc_max,
                           int32_t* status, cudaStream_t s);

// TMA tensor map over a bf16 tensor, 128-byte swizzle, zero fill out of
// bounds (gdn_tmap.cu).  dims / box innermost first; strides_bytes has
// rank - 1 entries (dims 1..rank-1).
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// Staged path (gdn_staged.cu).
gdn_status staged_layout(const gdn_problem& p, gdn_staged_layout_t* out);
gdn_status run_staged(const gdn_problem& p, int stop_after, const void* q, const void* k, const void* v,
                      const float* g, const float* beta, float scale, const float* h0, const int32_t* cu,
                      void* o, float* ht, void* ws, cudaStream_t s);

// Fused recurrent (decode) step (gdn_decode.cu).
gdn_status run_causal_conv1d(const void* x, const float* weight, const float* bias, int W, void* conv_state,
                             int state_slots, const int32_t* cache_indices, const int32_t* has_initial_state,
                             const int32_t* cu_seqlens, int N, int B, int T, int D, gdn_dtype dt, bool silu_act,
                             void* y, cudaStream_t s);

gdn_status run_recurrent(const gdn_problem& p, const void* q, const void* k, const void* v, const float* a,
                         const float* b, const float* A_log, const float* dt_bias, float scale, float* state,
                         const int32_t* state_indices, int state_slots, const int32_t* cu, void* o,
                         cudaStream_t s);

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // default limit of the hand-over wait

// Longest-first order of a packed batch (gdn_fused.cu): order[r] is the
// sequence of rank r by chunk count, descending, equal counts by index, so
// that a launch of one chain per CTA starts its longest chains first (the
// hardware hands out CTAs in index order).  Computed on the device from
// cu_seqlens (any int32 values: lengths below one token count as empty).
// varlen_order_bytes: the workspace the table takes (0 when p is not packed or
// has more than kOrderMaxN sequences: those keep the index order).
constexpr int kOrderMaxN = 16384;
size_t varlen_order_bytes(const gdn_problem& p);
gdn_status launch_varlen_order(const int32_t* cu, int N, int32_t* order, cudaStream_t s);

// Fused paths.  gdn_fused.cu: the two-CTA-per-SM kernel, K = V = 128
// (GDN_PATH_FUSED).  gdn_fused1.cu: the one-CTA-per-SM kernel, K = 128 or 256,
// V = 128 or 256 in value slices of 128 columns (GDN_PATH_FUSED1; also what
// GDN_PATH_FUSED runs for K = 256).  fused_supported: the problems
// GDN_PATH_FUSED accepts.  fused1_preferred: AUTO's choice between the two
// kernels for K = V = 128.
bool fused_supported(const gdn_problem& p);
bool fused128_supported(const gdn_problem& p);
bool fused1_supported(const gdn_problem& p);
bool fused1_preferred(const gdn_problem& p);
size_t fused1_workspace_bytes(const gdn_problem& p);
bool fused1_handover_window(const gdn_problem& p, int window);
gdn_status run_fused1(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                      void* ws, cudaStream_t s, int drop_flag = -1, unsigned long long wait_ns = kWaitLimitNs);
size_t fused_workspace_bytes(const gdn_problem& p);
size_t fused_status_offset(const gdn_problem& p);
// drop_flag / wait_ns: test hook of the window schedule -- the hand-over flag
// of window drop_flag is never raised, and a window waits at most wait_ns for
// its flag (then records GDN_DEV_WAIT_TIMEOUT and stops).
gdn_status run_fused(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                     const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                     void* ws, cudaStream_t s, int drop_flag = -1, unsigned long long wait_ns = kWaitLimitNs);
// True when the fused pass over p cuts a chain at the start of window
// `window` (so window - 1 waits for the hand-over flag of `window`).
bool fused_handover_window(const gdn_problem& p, int window);
// States-only launch over the chains of p (p.varlen with cu): chains started
// from a zero state write their final states to ht_zero, the same chains
// started from the identity with v = 0 write their transition matrices to
// ht_trans.
gdn_status run_fused_states(const gdn_problem& p, const void* k, const void* v, const float* g, const float* beta,
                            const int32_t* cu, float* ht_zero, float* ht_trans, int32_t* status, cudaStream_t s);

// Backward pass (gdn_bwd.cu).
bool bwd_supported(const gdn_problem& p);
size_t bwd_workspace_bytes(const gdn_problem& p);
gdn_status run_bwd(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                   const float* beta, float scale, const float* h0, const int32_t* cu, const void* dout,
                   const float* dht, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws,
                   cudaStream_t s);

// Chunked backward (gdn_bwdc.cu): K = V = 128; equal-length batches in
// sequence groups, packed sequences in one group (bounded workspace, tables
// built on the device from cu_seqlens); the token-recurrence backward above
// covers the rest.
bool bwdc_supported(const gdn_problem& p);
size_t bwdc_workspace_bytes(const gdn_problem& p);
gdn_status run_bwdc(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                    const float* beta, float scale, const float* h0, const int32_t* cu_seqlens, const void* dout,
                    const float* dht, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws,
                    cudaStream_t s);

// Chunk-parallel path (gdn_cp.cu): sequences cut into segments run in parallel.
size_t cp_workspace_bytes(const gdn_problem& p);
gdn_status run_cp(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                  const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht, void* ws,
                  size_t ws_bytes, cudaStream_t s);
int cp_segment_length(const gdn_problem& p);
// AUTO takes the chunk-parallel path for long sequences with few chains.
bool cp_preferred(const gdn_problem& p);
// One fused-kernel launch (mode 0: the full pass; 1: final states only).
// sched / hand / nwin / W: the window schedule of an equal-length full pass
// (sched null: one chain per CTA).  order: the longest-first table of a
// packed full pass (null: index order).
gdn_status launch_fused(const gdn_problem& p, int mode, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                        float* ht2, int32_t* status, cudaStream_t s, int* sched = nullptr, float* hand = nullptr,
                        int64_t nwin = 0, int64_t W = 0, int drop_flag = -1,
                        unsigned long long wait_ns = kWaitLimitNs, const int32_t* order = nullptr);
// Streaming multiprocessors of the current device (148 when none can be queried).
int sm_count();
// Byte offset of the device status word inside a forward workspace for `path`
// (AUTO resolved as gdn_chunk_fwd resolves it).
size_t fwd_status_offset(const gdn_problem& p, gdn_path path);

}  // namespace gdn
