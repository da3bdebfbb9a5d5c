/*
 * gdn.h -- C ABI of libgdn.so: the Gated DeltaNet chunked forward pass on one
 * GB300 (sm_103a).
 *
 * Operator (MegaGDN-PTO walkthrough, section 1.1, the seven-stage chunk
 * pipeline; TileLang x xLLM page, Step 1, chunk_gated_delta_rule_fwd_h):
 *
 *   S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T     (S is [K][V])
 *   o_t = scale * S_t^T q_t
 *
 * evaluated chunk-wise (cumsum -> scaled_dot_kkt -> solve_tril -> wy_fast ->
 * chunk_h -> chunk_o).  Inputs with GQA: value head h reads q/k head
 * h / (Hv / Hqk) (MegaGDN-PTO walkthrough, section 5.2).  Packed variable-length
 * batches use cu_seqlens (section 5.3).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *    owned by the caller; the library allocates nothing.
 *  - q, k, v and o must be 16-byte aligned (they are read/written by TMA).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Host-side argument checks run before any launch; a
 *    failed check returns an error and launches nothing.  Errors found on the
 *    device (malformed cu_seqlens, a bounded wait that timed out) are written
 *    to a status word inside the workspace; read it with
 *    gdn_get_device_status().
 *  - No exception or C++ type crosses this boundary.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or workspace too small */
  GDN_ERR_UNSUPPORTED = 2,   /* valid request that this build does not implement */
  GDN_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute, ...) */
  GDN_ERR_DEVICE = 4,        /* the device reported an error through the status word */
  GDN_ERR_SCRATCH_LIMIT = 5  /* gdn_chunk_fwd_noalloc: problem larger than its static scratch */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Device status word values (read by gdn_get_device_status). */
#define GDN_DEV_OK 0
#define GDN_DEV_BAD_CU_SEQLENS 1   /* cu[0] != 0, decreasing, or cu[N] != T */
#define GDN_DEV_WAIT_TIMEOUT 2     /* a bounded spin-wait inside a kernel gave up */

/* Execution path. */
typedef enum {
  GDN_PATH_AUTO = 0,    /* cp or fused when supported, else staged */
  GDN_PATH_STAGED = 1,  /* one kernel per stage, intermediates in the workspace */
  GDN_PATH_FUSED = 2,   /* single persistent tcgen05 kernel: two CTAs per SM for bf16 K = V = 128
                           (the throughput form), the one-CTA-per-SM kernel for bf16 K = V = 256 */
  GDN_PATH_CP = 3,      /* chunk-parallel: each sequence cut into segments run on separate SMs
                           (bf16, K = V = 128); AUTO takes it for sequences of >= 2048 tokens
                           when the (sequence, value head) chains number at most half the SMs */
  GDN_PATH_FUSED1 = 4   /* single tcgen05 kernel with one CTA per SM and the value dimension in
                           slices of 128 columns (bf16, K in {128, 256}, V in {128, 256}); AUTO
                           takes it for K = 256, and for K = V = 128 when the (sequence, value
                           head) chains number at most the SMs or a packed batch is small enough
                           (ceil(T / 64) + N chunks a value head, times Hv, at most 256 x SMs)
                           that its longest sequence bounds the step */
} gdn_path;

/*
 * Problem description.
 *   B, T      : fixed-length batch [B, T] (cu_seqlens == NULL, N = B), or the
 *               packed batch [1, T] of N sequences (cu_seqlens != NULL, B = 1,
 *               T = total tokens, may be 0).
 *   Hqk, Hv   : q/k heads and value heads; Hv % Hqk == 0.
 *   K, V      : key and value head dims, each in {64, 128, 256}.
 *   C         : chunk length, 64 or 128.
 *   dt        : dtype of q, k, v and o (fp32 or bf16); g, beta, h0, ht are fp32.
 */
typedef struct {
  int B, T, N, Hqk, Hv, K, V, C;
  gdn_dtype dt;
  int varlen;   /* 1 when cu_seqlens is given */
} gdn_problem;

/*
 * Bytes of workspace that gdn_chunk_fwd needs for `path` (AUTO resolves as in
 * gdn_chunk_fwd).  Returns 0 for an invalid problem.  The varlen bound assumes
 * at most ceil(T / C) + N chunks, so cu_seqlens need not be read on the host.
 * The fused path over equal-length sequences spreads the (sequence, head)
 * chains' chunks evenly over the CTAs the current device holds at once (two
 * per SM), cutting a chain in two where a share ends; its workspace then holds
 * one K x V fp32 hand-over state per CTA (about 20 MB on 152 SMs), so query
 * the size with the device that will run the call current.  On packed
 * sequences (2 to 16384 of them) the fused paths also keep a table of N int32
 * there: a launch before the pass ranks the sequences by length so that the
 * longest chains start first.
 */
size_t gdn_chunk_fwd_workspace_size(const gdn_problem* p, gdn_path path);

/*
 * The chunked forward pass.
 *   q, k    : [B, T, Hqk, K]  dtype p->dt
 *   v       : [B, T, Hv, V]   dtype p->dt
 *   g       : [B, T, Hv] fp32, log-decay (used as given; no activation)
 *   beta    : [B, T, Hv] fp32
 *   scale   : multiplies o only (never the state); callers usually pass K^-0.5
 *   h0      : [N, Hv, K, V] fp32 initial state, or NULL for zeros
 *   cu_seqlens : [N + 1] int32 device array of token offsets, or NULL
 *   o       : out [B, T, Hv, V] dtype p->dt (round-to-nearest-even for bf16)
 *   ht      : out [N, Hv, K, V] fp32 final state, or NULL to skip it
 *   workspace / workspace_bytes : device scratch of at least
 *             gdn_chunk_fwd_workspace_size(p, path) bytes, 256-byte aligned
 * Returns GDN_OK once everything is enqueued on `stream`.
 */
gdn_status gdn_chunk_fwd(const gdn_problem* p, gdn_path path,
                         const void* q, const void* k, const void* v,
                         const float* g, const float* beta, float scale,
                         const float* h0, const int32_t* cu_seqlens,
                         void* o, float* ht,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Staged path with a stop point (the pages' staged mode and MEGA_STOP_AFTER_*
 * hooks, MegaGDN-PTO walkthrough, section 7.4).  Runs stages 0..stop_after:
 *   0 prepare (chunk tables), 1 cumsum, 2 scaled_dot_kkt, 3 solve_tril,
 *   4 wy_fast, 5 chunk_h, 6 chunk_o (6 = full forward; o/ht written only by
 *   stages 6 and 5 respectively).
 * Intermediates stay in the workspace at the offsets of gdn_staged_layout.
 */
gdn_status gdn_chunk_fwd_staged(const gdn_problem* p, int stop_after,
                                 const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, float scale,
                                 const float* h0, const int32_t* cu_seqlens,
                                 void* o, float* ht,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Byte offsets of the staged path's intermediates inside its workspace.
 * nc_max = B * ceil(T / C) (fixed length) or ceil(T / C) + N (varlen).
 *   tables : int32 seq_chunk0[N + 1] | chunk_seq[nc_max] | chunk_tok0[nc_max] |
 *            chunk_len[nc_max] | nc[1]   (chunk c of the packed token stream
 *            covers tokens chunk_tok0[c] .. + chunk_len[c] of sequence chunk_seq[c])
 *   status : int32 device status word
 *   gamma  : f32 [nc_max][Hv][C]      in-chunk cumsum of g
 *   A      : f32 [nc_max][Hv][C][C]   strictly lower, beta_i exp(g_i - g_j) k_i.k_j
 *   Tinv   : f32 [nc_max][Hv][C][C]   (I + A)^{-1}
 *   W, U   : f32 [nc_max][Hv][C][K] and [nc_max][Hv][C][V]
 *   S0     : f32 [nc_max][Hv][K][V]   state at each chunk's start
 *   Vn     : f32 [nc_max][Hv][C][V]   v_new = U - W S0
 * Rows past a chunk's length hold zeros, except Tinv, which holds the
 * identity there (the inverse of I + A with A zero-padded).
 */
typedef struct {
  size_t tables, status, gamma, A, Tinv, W, U, S0, Vn, total;
  int nc_max;
} gdn_staged_layout_t;

gdn_status gdn_staged_layout(const gdn_problem* p, gdn_staged_layout_t* out);

/*
 * Waits for `stream`, then reads the device status word that the last call
 * using `workspace` left (GDN_DEV_*) into *dev_status and clears it.
 * `path` must be the path that call ran with (it locates the status word).
 * Returns GDN_ERR_CUDA if the synchronisation or the copy fails.
 */
gdn_status gdn_get_device_status(const gdn_problem* p, gdn_path path, void* workspace,
                                 void* stream, int* dev_status);

/*
 * The forward pass on HOST tensors (no counterpart on the pages: the
 * streaming form of gdn_chunk_fwd for callers whose q, k, v, g, beta, h0 and
 * outputs live in host memory).  Same shapes and meaning as gdn_chunk_fwd,
 * but q, k, v, g, beta, h0, cu_seqlens, o and ht are HOST pointers; page-locked
 * memory (cudaHostAlloc) is needed for the copies to overlap the compute
 * (pageable memory is copied synchronously by the driver, still correctly).
 * The batch is cut into at most `nsplit` sub-batches of whole sequences (about
 * equal token counts); sub-batch i's inputs are copied to the device while
 * sub-batch i - 1 runs gdn_chunk_fwd(path) and sub-batch i - 2's o and ht are
 * copied back, on three streams that the library creates once per device and
 * orders after `stream`; `stream` resumes once every output is in host memory.
 * Calls from several host threads are enqueued one at a time.
 *   workspace : DEVICE memory of gdn_chunk_fwd_host_workspace_size(p,
 *               cu_seqlens, nsplit, path) bytes, 256-byte aligned: two sets
 *               of device buffers for the largest sub-batch and the inner
 *               forward's workspace.
 * Host-side checks: the ones of gdn_chunk_fwd and, for packed sequences,
 * cu_seqlens[0] == 0, cu_seqlens[N] == T and non-decreasing offsets
 * (GDN_ERR_INVALID_ARG otherwise, nothing enqueued).  Device-side errors of
 * any sub-batch (the first one kept) are read with
 * gdn_chunk_fwd_host_get_device_status.  The host buffers must stay valid and
 * unmodified until `stream` has passed the call.
 */
size_t gdn_chunk_fwd_host_workspace_size(const gdn_problem* p, const int32_t* cu_seqlens, int nsplit,
                                         gdn_path path);
gdn_status gdn_chunk_fwd_host(const gdn_problem* p, gdn_path path, int nsplit,
                              const void* q, const void* k, const void* v,
                              const float* g, const float* beta, float scale,
                              const float* h0, const int32_t* cu_seqlens,
                              void* o, float* ht,
                              void* workspace, size_t workspace_bytes, void* stream);
/* Waits for `stream`, reads and clears the status word of a
 * gdn_chunk_fwd_host workspace (GDN_DEV_*). */
gdn_status gdn_chunk_fwd_host_get_device_status(void* workspace, void* stream, int* dev_status);

/*
 * Self-test of the tensor-core operand layouts used by the fused kernel (no
 * counterpart on the pages; a test hook).  Computes D = A B (or -A B) with one
 * CTA through tcgen05.mma over 128-byte-swizzled shared-memory tiles.
 *   A : bf16 [128][Kd] row-major, B : bf16 [Kd][N] row-major, D : fp32 [128][N]
 *   variant bits: 1 = A staged MN-major (else K-major), 2 = B staged MN-major,
 *                 4 = N 128 (else 64), 8 = Kd 128 (else 64), 16 = negate A,
 *                 32 = stage A with a TMA tiled load (needs bit 1 clear,
 *                 A 16-byte aligned)
 *   workspace : >= 4 bytes of device memory for the status word
 */
gdn_status gdn_selftest_umma(int variant, const void* A, const void* B, float* D, void* workspace,
                             void* stream);

/*
 * Test hook of the fused paths' bounded waits (no counterpart on the pages).
 * Runs gdn_chunk_fwd(p, path, ...) (path GDN_PATH_FUSED or GDN_PATH_FUSED1)
 * on an equal-length batch whose chains the fused kernel deals out as windows
 * that hand a cut chain's state over from one CTA to another, except that
 * window `drop_window` never raises its hand-over flag and every window waits
 * at most `wait_ns` nanoseconds for the flag it needs.  The window that would
 * continue that chain (drop_window - 1 for GDN_PATH_FUSED; for
 * GDN_PATH_FUSED1, whose windows come in groups of G x V / 128, the window one
 * group below) therefore gives up: it records GDN_DEV_WAIT_TIMEOUT in the
 * workspace's status word (read it with gdn_get_device_status with the same
 * path) and stops, leaving the o rows and the final state of the chain it was
 * waiting for unwritten; every other window completes and the launch ends.
 * The failure is made on purpose in a wait that has a limit: nothing faults
 * and nothing hangs.
 *   Arguments as gdn_chunk_fwd (no cu_seqlens).  Returns GDN_ERR_UNSUPPORTED
 *   when the fused pass over p hands no chain over at the start of window
 *   drop_window (then nothing is launched).
 */
gdn_status gdn_selftest_handover_timeout(const gdn_problem* p, gdn_path path,
                                         const void* q, const void* k, const void* v,
                                         const float* g, const float* beta, float scale,
                                         const float* h0, void* o, float* ht,
                                         void* workspace, size_t workspace_bytes,
                                         int drop_window, long long wait_ns, void* stream);

/*
 * Forward pass for callers that cannot allocate device memory (no counterpart
 * on the pages).  Some callers cannot call cudaMalloc in their call path: an
 * op inside a host framework that owns every device buffer and passes the op
 * only its inputs and outputs, or a caller that cannot accept the implicit
 * device-wide synchronisation of cudaMalloc/cudaFree.  This entry point
 * allocates nothing and takes no workspace: it runs the forward pass with its
 * workspace in a file-scope device array of 32 MiB that every GPU which
 * loads libgdn.so holds until the process exits.  Path: AUTO's choice, with
 * GDN_PATH_FUSED in place of GDN_PATH_CP, when that path's workspace
 * (gdn_chunk_fwd_workspace_size) fits 32 MiB - 256 bytes (the array's first
 * 256 bytes hold the status word) -- the fused kernels need at most about 20
 * MB -- else GDN_PATH_STAGED when its workspace fits.
 *   Arguments as gdn_chunk_fwd (the caller still passes inputs and outputs).
 *   Returns GDN_ERR_SCRATCH_LIMIT, launching nothing, when neither fits (the
 *   staged path for problems no fused kernel takes, such as fp32 inputs).
 *   The first call on a device (and the first after a device reset replaced
 *   its context) looks up the array's device address with
 *   cudaGetSymbolAddress, with that device current; make that first call
 *   before any stream capture.
 *   All calls share the one array: calls whose executions overlap on the GPU
 *   (other streams, other host threads) race on it and must be serialised by
 *   the caller.
 *   Errors found on the device (malformed cu_seqlens) leave o and ht
 *   incomplete and are recorded in the array's status word, which
 *   gdn_chunk_fwd_noalloc_get_device_status reads: it waits for `stream`,
 *   then returns the status (GDN_DEV_*) of the last gdn_chunk_fwd_noalloc call
 *   on the current device in *dev_status and clears it.  It allocates
 *   nothing either.
 */
gdn_status gdn_chunk_fwd_noalloc(const gdn_problem* p,
                                 const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, float scale,
                                 const float* h0, const int32_t* cu_seqlens,
                                 void* o, float* ht, void* stream);
gdn_status gdn_chunk_fwd_noalloc_get_device_status(void* stream, int* dev_status);

/*
 * Fused recurrent (decode) step with sigmoid gating (TileLang x xLLM page,
 * fused_sigmoid_gating_delta_rule: the decode-phase operator that fuses the
 * sigmoid activation, the gate computation from the decay rate A_log and the
 * delta-rule update of the fp32 state, with per-sequence state offsets).
 * For every token t of every sequence, value head h:
 *     g_t    = -exp(A_log[h]) * softplus(a_t + dt_bias[h])
 *     beta_t = sigmoid(b_t)
 *     S <- e^{g_t} (I - beta_t k_t k_t^T) S + beta_t k_t v_t^T,   o_t = scale * S^T q_t
 * Tokens of a sequence are processed in order (one token per sequence is the
 * decode case; several run the plain recurrence).
 *   p           : as for gdn_chunk_fwd (C is ignored; V a multiple of 64)
 *   q, k        : [B, T, Hqk, K];  v : [B, T, Hv, V];  o : out [B, T, Hv, V]  (dtype p->dt)
 *   a, b        : [B, T, Hv] fp32 gate and beta pre-activations
 *   A_log       : [Hv] fp32;  dt_bias : [Hv] fp32 or NULL (= 0)
 *   state       : [state_slots, Hv, K, V] fp32 pool, read and updated in place
 *   state_indices : [N] int32 slot of each sequence, or NULL (slot n); a
 *                 sequence whose slot is negative or >= state_slots gets zero
 *                 outputs and no state update
 *   cu_seqlens  : [N + 1] int32 or NULL, as for gdn_chunk_fwd; sequences whose
 *                 offsets fall outside [0, T] are skipped
 * No workspace; asynchronous on `stream`.
 */
gdn_status gdn_recurrent_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* a, const float* b, const float* A_log, const float* dt_bias,
                             float scale, float* state, const int32_t* state_indices, int state_slots,
                             const int32_t* cu_seqlens, void* o, void* stream);

/*
 * Backward pass of gdn_chunk_fwd (the FlashQLA notes list a backward of the
 * chunk kernel among its variants, section 4.3): for upstream gradients
 * dout = dL/do and dht = dL/dht, the gradients of L with respect to q, k, v,
 * g, beta and h0, by reverse mode of the token recurrence
 *     G <- G + scale q_t dout_t^T;  dq_t = scale S_t dout_t
 *     u = S_{t-1}^T k_t, w = G^T k_t;  dv_t = beta_t w
 *     dg_t = e^{g_t} (<G, S_{t-1}> - beta_t w.u);  dbeta_t = -e^{g_t} w.u + w.v_t
 *     dk_t = -e^{g_t} beta_t (G u + S_{t-1} w) + beta_t G v_t
 *     G <- e^{g_t} (G - beta_t k_t w^T)
 * from G = dht down to dh0 = G (S_t the state after token t, S_0 = h0).
 * With K = V = 128 (and q, k, v, dout 16-byte aligned) the chunked form of
 * the same reverse mode runs (64-token chunks: batched products for
 * everything but the chunk-to-chunk state and adjoint recurrences, on the
 * tensor cores as tf32 in three terms, about 2^-19 of each product; about
 * 0.8 MB of workspace per (chunk, value head)): equal-length batches in
 * sequence groups within 16 GiB; packed sequences in one group sized for
 * ceil(T / 64) + N chunks a value head, with the chunk tables built on the
 * device from cu_seqlens (packed batches whose bound exceeds 32 GiB take the
 * token recurrence).  Other problems recompute the states in fp32 from
 * checkpoints at every 64th token.  Both keep fp32 accuracy.
 *   p, q, k, v, g, beta, scale, h0, cu_seqlens : as for gdn_chunk_fwd (K in
 *                 {64, 128}, V a multiple of 16; any C)
 *   dout        : [B, T, Hv, V], dtype p->dt;  dht : [N, Hv, K, V] fp32 or NULL (= 0)
 *   dq, dk      : out [B, T, Hqk, K] fp32 (summed over the value heads of each
 *                 q/k head);  dv : out [B, T, Hv, V] fp32
 *   dg, dbeta   : out [B, T, Hv] fp32;  dh0 : out [N, Hv, K, V] fp32 or NULL
 *   workspace   : gdn_chunk_bwd_workspace_size(p) bytes, 256-byte aligned
 *                 (the device status word and the per-chunk intermediates;
 *                 the size covers either form, since the choice also depends
 *                 on the alignment of q, k, v and dout)
 * dq and dk (and, for packed sequences or K = 64, dg and dbeta) are sums of
 * fp32 atomic additions across value heads or column slices (their rounding
 * may differ between runs).  Malformed cu_seqlens set the status word (read it
 * with gdn_chunk_bwd_get_device_status) and leave the gradients incomplete.
 * Asynchronous on `stream`.
 */
size_t gdn_chunk_bwd_workspace_size(const gdn_problem* p);
gdn_status gdn_chunk_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, float scale, const float* h0,
                         const int32_t* cu_seqlens, const void* dout, const float* dht,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dh0,
                         void* workspace, size_t workspace_bytes, void* stream);
/* Status word of a gdn_chunk_bwd workspace (synchronises `stream`, then
 * clears the word).  GDN_DEV_OK or GDN_DEV_BAD_CU_SEQLENS. */
gdn_status gdn_chunk_bwd_get_device_status(void* workspace, void* stream, int* dev_status);

/* Activation applied after the convolution of gdn_causal_conv1d_fwd. */
typedef enum { GDN_ACT_NONE = 0, GDN_ACT_SILU = 1 } gdn_activation;

/*
 * Causal depthwise convolution with a carried state (TileLang x xLLM page,
 * causal_conv1d: each output token depends on the current and earlier inputs
 * of its own sequence only; the convolution state keeps the last W-1 inputs of
 * every sequence for incremental decode, in the state-pool slot that
 * cache_indices gives it).  For a sequence with inputs x_0..x_{L-1}, let
 * ext = [the W-1 initial inputs ; x_0 .. x_{L-1}]; then for every channel d
 *     y_p[d]    = act(bias[d] + sum_{w<W} weight[d*W + w] * ext_{p+w}[d])
 *     new state = ext_L .. ext_{L+W-2}
 * so weight[d*W + W-1] multiplies the current token.  act is the identity or
 * SiLU, u * sigmoid(u).  The initial inputs are the slot's state, or zeros
 * when the sequence has no slot or has_initial_state[n] == 0.
 *   x, y        : [B, T, D] of dtype dt, 16-byte aligned, D % 8 == 0; with
 *                 cu_seqlens, B == 1 and T is the packed total.  y must not
 *                 overlap x or conv_state.
 *   weight      : [D, W] fp32, 1 <= W <= 4;  bias : [D] fp32 or NULL (= 0)
 *   conv_state  : [state_slots, W-1, D] of dtype dt (16-byte aligned), or NULL
 *                 (zero initial inputs, nothing kept).  Read by the
 *                 convolution, then rewritten in place with the new state.
 *                 Ignored when W == 1.
 *   cache_indices : [N] int32 slot per sequence, or NULL (slot n; then
 *                 state_slots >= N).  A slot outside [0, state_slots) means
 *                 "no state": zero initial inputs, nothing written.  Distinct
 *                 sequences must use distinct slots.
 *   has_initial_state : [N] int32 or NULL (all 1); 0 starts the sequence from
 *                 zeros but still writes its slot.
 *   cu_seqlens  : [N + 1] int32 or NULL (then N == B and sequence n is row n
 *                 of x).  A sequence whose offsets fall outside [0, T] or
 *                 decrease is skipped (outputs and state); tokens that no
 *                 well-formed sequence covers are not written.
 * States are exact copies of inputs.  Two launches (convolution, then state
 * update), asynchronous on `stream`; no workspace.  Returns
 * GDN_ERR_INVALID_ARG for a failed host-side check (nothing launched).
 */
gdn_status gdn_causal_conv1d_fwd(const void* x, const float* weight, const float* bias, int W,
                                 void* conv_state, int state_slots, const int32_t* cache_indices,
                                 const int32_t* has_initial_state, const int32_t* cu_seqlens, int N,
                                 int B, int T, int D, gdn_dtype dt, gdn_activation act, void* y,
                                 void* stream);

/*
 * Test hook (no counterpart on the pages): y[i] = e^{x[i]} computed the way
 * the fused kernel computes its decay factors (2^{x log2 e} on the MUFU ex2
 * unit), so tests can bound its error against CUDA's expf.  x, y device
 * arrays of n floats.
 */
gdn_status gdn_selftest_exp(const float* x, float* y, int n, void* stream);

/* Path that GDN_PATH_AUTO selects for this problem (STAGED, FUSED or CP). */
gdn_path gdn_resolve_path(const gdn_problem* p);

/* Human-readable name of a status code (static string). */
const char* gdn_status_string(gdn_status s);

/* Library version string, e.g. "gdn 0.1 sm_103a". */
const char* gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
