// gdn_fused.cu -- the fused path: the whole chunk pipeline (cumsum,
// scaled_dot_kkt, solve_tril, wy_fast, chunk_h, chunk_o; MegaGDN-PTO
// walkthrough, sections 1.1 and 4.5) in ONE sm_103a launch.
//
// A CTA walks a (sequence, value head) chain's chunks in order; the fp32
// state stays on the SM (TMEM) between chunks, and no intermediate goes
// through HBM.  Two CTAs share an SM (their shared memory and TMEM halves), so
// one chain's SIMT phases overlap the other's tensor phases.  With more chains
// than CTA slots, equal-length chains are dealt out as windows of an equal
// number of chunks (one slot each, so the last wave leaves no SM half idle):
// a chain cut at a window boundary hands its state over once through HBM.  Chunks are 64 tokens; a C = 128 request is processed as two
// 64-token chunks (the chunked form is exact for any chunk length).
//
// Layout: everything is transposed so that every tcgen05.mma has M = 128 on
// the key/value dimension (TMEM lane = value column e or key column d):
//
//   M1  [K;Q] K^T          D[0:64]   = K K^T, D[64:128] = Q K^T   (M128 N64 K128)
//   S1  A = strict-lower(beta_i e^{g_i - g_j} K K^T)  -> smem fp32
//       P = lower(e^{g_i - g_j} Q K^T)                 -> smem bf16
//   S2  T = (I + A)^{-1}: 16x16 diagonal blocks by forward substitution, then
//       merges T21 = -T22 A21 T11 (MegaGDN-PTO walkthrough, section 4.4)
//   M2  W^T = K^T (T diag(beta e^g))^T,  U^T = V^T (T diag(beta))^T (section 4.3)
//   S4  S^T (fp32, TMEM) -> bf16 operand; S^T *= e^{g_last}
//   M3  V'^T = U^T - S^T W^T;  OQ^T = S^T Q^T      (chunk_h first half)
//   S5  V'^T -> bf16, V''^T = V'^T diag(e^{g_last - g}) -> bf16
//   M4  OP^T = V'^T P^T;  S^T += V''^T K          (chunk_h second half)
//   S6  o_i = scale e^{g_i} OQ_i + OP_i           (chunk_o; P carries scale)
//
// Rows past a sequence's end (tail chunk) get beta = 0 and g = 0, which zeroes
// their rows of A, W, U and V' exactly; they are never stored.
#include <string.h>

#include "gdn_solve64.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace solve64;

constexpr int kD = 128;         // K = V
constexpr int kTmemCols = 256;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;         // [k rows 0..63 ; q rows 64..127] x 128 d, 2 atom columns of 16 KB
constexpr uint32_t OFF_V = 32768;      // v rows 0..63 x 128 e, 2 atom columns of 8 KB
constexpr uint32_t OFF_Y = 49152;      // T diag(beta) | T diag(beta e^g)  (8 KB each), then W^T, then V''^T (16 KB)
constexpr uint32_t OFF_TB = OFF_Y;
constexpr uint32_t OFF_TBE = OFF_Y + 8192;
constexpr uint32_t OFF_W = OFF_Y;
constexpr uint32_t OFF_P = 65536;      // P [i][j] bf16, 8 KB
constexpr uint32_t OFF_X = 73728;      // 32 KB, reused: A/T fp32 + scratch | S^T bf16 | V'^T | o staging
constexpr uint32_t OFF_AS = OFF_X;     // fp32 [64][68]
constexpr uint32_t OFF_TMP = OFF_X + 64 * 68 * 4;  // fp32 scratch for the solve merges (32 x 40 floats)
constexpr uint32_t OFF_ST = OFF_X;     // S^T bf16 [e][d], 2 atom columns of 16 KB
constexpr uint32_t OFF_VP = OFF_X;     // V'^T bf16 [e][j], 16 KB (the S^T half that M3 reads first)
constexpr uint32_t OFF_VPP = OFF_Y;    // V''^T bf16 [e][j], 16 KB (W^T is dead once V' is complete)
constexpr uint32_t OFF_OS = OFF_X;     // o staging bf16: 2 boxes [64 rows][64], 128-byte swizzle (TMA store)
constexpr uint32_t OFF_MISC = 106496;
constexpr uint32_t OFF_GAM = OFF_MISC;         // float[64] gamma (in-chunk cumsum of g)
constexpr uint32_t OFF_BET = OFF_MISC + 256;   // float[64] beta (0 past the end)
constexpr uint32_t OFF_BE = OFF_MISC + 512;    // float[64] beta e^gamma
constexpr uint32_t OFF_DL = OFF_MISC + 768;    // float[64] e^{gamma_last - gamma}
constexpr uint32_t OFF_EG = OFF_MISC + 1024;   // float[64] e^gamma
constexpr uint32_t OFF_BAR = OFF_MISC + 1280;    // 5 mbarriers: k/q tiles, v tile, three MMA commit groups
constexpr uint32_t OFF_FLAGS = OFF_MISC + 1320;  // [0] tmem base, [1] abort, [2] window
constexpr uint32_t OFF_BAR1 = OFF_MISC + 1336;   // sixth mbarrier: first half of S^T Q^T
constexpr uint32_t OFF_GRAW = OFF_MISC + 1344;   // float[2][2][64]: raw g, beta of two chunks
constexpr uint32_t kSmemUsed = OFF_MISC + 2368;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // + alignment slack

static_assert(OFF_TMP + 32 * 40 * 4 <= OFF_X + 32768, "solve scratch overflows region X");
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs must fit one SM");

struct FusedParams {
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;
  __nv_bfloat16* o;
  float* ht;
  int32_t* status;
  int N, Tseq, Ttot, Hqk, Hv, varlen;
  float scale;
  // packed batches, full pass: block b runs head b % Hv of sequence
  // order[b / Hv] (longest first); null: sequence b / Hv
  const int32_t* order;
  // kStates launches only: blocks [0, split) are the chains of a problem started
  // from a zero state (final state -> ht); blocks [split, 2 split) the same
  // chains started from the identity with v = 0 (final state = the chain's
  // state-transition matrix -> ht2)
  float* ht2;
  int split;
  // Window schedule (kFull, equal-length sequences; null sched = one chain per
  // CTA).  The chains' chunks are laid end to end, each chain's in reverse
  // order, and cut into nwin windows of W chunks; a CTA claims windows from
  // the last down (sched[0] counts the claims) and runs a window's pieces in
  // order.  A window starts with a prefix of a chain (or a whole chain) and
  // ends with a suffix of one: a chain cut at a window boundary has its prefix
  // run first thing by window m + 1, which hands its state over in slot m + 1
  // of `hand` ([K][V] fp32 per slot) and sets sched[1 + m + 1]; window m waits
  // for that flag before it runs the suffix, as its last piece.  W is at
  // least the chunks of one chain, so no chain spans more than two windows.
  int* sched;
  float* hand;
  int nwin, W;
  // limit of the wait for a hand-over flag, and a window whose flag is never
  // raised (-1: none; a test hook that makes one wait run out)
  unsigned long long wait_ns;
  int drop_flag;
};

// Kernel modes: the full forward pass, or final states only (no q, no o).
constexpr int kFull = 0;
constexpr int kStates = 1;

// WIN: the window schedule (kFull only); a separate instantiation, so that the
// one-chain-per-CTA code carries none of its state through the chunk loop.
template <int MODE, bool WIN>
__global__ void __launch_bounds__(kThreads, 2) gdn_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_k,
                                                                const __grid_constant__ CUtensorMap tm_v,
                                                                const __grid_constant__ CUtensorMap tm_o,
                                                                const FusedParams prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the __shared__
  // array so that every access below stays a shared-memory access
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  float* As = reinterpret_cast<float*>(sm + OFF_AS);
  float* tmp = reinterpret_cast<float*>(sm + OFF_TMP);
  float* gam = reinterpret_cast<float*>(sm + OFF_GAM);
  float* bet = reinterpret_cast<float*>(sm + OFF_BET);
  float* be = reinterpret_cast<float*>(sm + OFF_BE);
  float* dl = reinterpret_cast<float*>(sm + OFF_DL);
  float* eg = reinterpret_cast<float*>(sm + OFF_EG);
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_v = bar_kq + 1;
  // MMA commit groups.  Every commit is waited for (by every thread, in
  // order) before the next commit to the same barrier, so a waiter can never
  // miss a phase.
  uint64_t* bar_mma = bar_kq + 2;   // M1, M2, then the S^T Q^T product of M3
  uint64_t* bar_x = bar_kq + 3;     // V' (M3), then the state update (M4)
  uint64_t* bar_q = bar_kq + 4;     // V'^T P^T (M4)
  uint64_t* bar_o1 = reinterpret_cast<uint64_t*>(sm + OFF_BAR1);   // first half of S^T Q^T (M3)
  volatile uint32_t* flags = reinterpret_cast<volatile uint32_t*>(sm + OFF_FLAGS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hf = warp >> 2;   // TMEM lane quadrant, column half
  constexpr bool windowed = MODE == kFull && WIN;
  // kStates: the upper half of the grid computes transition matrices
  const bool trans = MODE == kStates && (int)blockIdx.x >= prm.split;
  // the chain of the current piece: sequence n, value head h, its qk head,
  // first token, length and chunks
  int n = 0, h = 0, hq = 0, nchunks = 0;
  int64_t tok0 = 0, L = 0;

  // one chain per CTA: sequence bounds (validated: a malformed cu_seqlens
  // touches no memory)
  if (!windowed) {
    int chain = trans ? (int)blockIdx.x - prm.split : (int)blockIdx.x;
    if (prm.order && !trans) chain = prm.order[chain / prm.Hv] * prm.Hv + chain % prm.Hv;
    n = chain / prm.Hv;
    h = chain % prm.Hv;
    hq = h / (prm.Hv / prm.Hqk);
    if (prm.varlen) {
      const int64_t a = prm.cu[n], b = prm.cu[n + 1];
      bool ok = (0 <= a) && (a <= b) && (b <= prm.Ttot);
      if (chain == 0 && (prm.cu[0] != 0 || prm.cu[prm.N] != prm.Ttot)) ok = false;
      if (!ok) {
        if (tid == 0) atomicExch(prm.status, GDN_DEV_BAD_CU_SEQLENS);
        return;
      }
      tok0 = a;
      L = b - a;
    } else {
      tok0 = (int64_t)n * prm.Tseq;
      L = prm.Tseq;
    }
    nchunks = (int)((L + kChunk - 1) / kChunk);
  }

  if (tid == 0) {
    flags[2] = windowed ? prm.nwin - 1 - atomicAdd(prm.sched, 1) : 0;
    mbar_init(bar_kq, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_q, 1);
    mbar_init(bar_o1, 1);
    mbar_fence_init();
    flags[1] = 0;
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  if (warp == 0) tmem_alloc(const_cast<uint32_t*>(flags), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = flags[0];
  const uint32_t R_S = tmem, R_a = tmem + 128, R_b = tmem + 192;
  const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
  const int row = 32 * qd + lane;   // this thread's TMEM lane (e or d or chunk row)

  uint32_t ph_kq = 0, ph_v = 0, ph_mma = 0, ph_x = 0, ph_q = 0, ph_o1 = 0;
  bool kq_pending = false, v_pending = false;   // meaningful in thread 0
  int mma_pending = 0, x_pending = 0, q_pending = 0, o1_pending = 0;   // commits not yet waited for (thread 0)
  auto issue_kq = [&](int c) {
    const int t = (int)(tok0 + (int64_t)kChunk * c);
    // kStates needs no q: its rows of the [k; q] tile are left as they are
    // (their products are computed but never used)
    mbar_arrive_expect_tx(bar_kq, MODE == kFull ? 32768 : 16384);
    tma_load_3d(sm + OFF_KQ, &tm_k, bar_kq, 0, hq, t);
    tma_load_3d(sm + OFF_KQ + 16384, &tm_k, bar_kq, 64, hq, t);
    if (MODE == kFull) {
      tma_load_3d(sm + OFF_KQ + 8192, &tm_q, bar_kq, 0, hq, t);
      tma_load_3d(sm + OFF_KQ + 24576, &tm_q, bar_kq, 64, hq, t);
    }
    kq_pending = true;
  };
  auto issue_v = [&](int c) {
    const int t = (int)(tok0 + (int64_t)kChunk * c);
    mbar_arrive_expect_tx(bar_v, 16384);
    tma_load_3d(sm + OFF_V, &tm_v, bar_v, 0, h, t);
    tma_load_3d(sm + OFF_V + 8192, &tm_v, bar_v, 64, h, t);
    v_pending = true;
  };
  // Every thread waits for every MMA commit, in commit order, so that all
  // threads track the same barrier phases.  A wait that times out raises the
  // abort flag; sync_ok() makes the flag visible to all threads.
  auto wait_commit = [&](uint64_t* bar, uint32_t& ph, int& pending) {
    if (!mbar_wait(bar, ph, prm.status)) flags[1] = 1;
    ph ^= 1;
    if (tid == 0) --pending;
  };
  auto sync_ok = [&]() -> bool {
    __syncthreads();
    tc_fence_after();
    return flags[1] == 0;
  };
  auto wait_mma = [&]() -> bool {
    wait_commit(bar_mma, ph_mma, mma_pending);
    return sync_ok();
  };
  const uint32_t s4 = (sbase & 0x3FFFFu) >> 4;   // descriptor address field of the tile base

  // warp 1 stages chunk cc's g and beta rows in graw[cc & 1] (lane l: rows
  // 2 l and 2 l + 1, zeros past the sequence) with asynchronous copies
  float* graw = reinterpret_cast<float*>(sm + OFF_GRAW);
  auto fetch_gb = [&](int cc) {
    float* dst = graw + (cc & 1) * 128;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int rr = 2 * lane + r;
      const int64_t tn = tok0 + (int64_t)kChunk * cc + rr;
      if (tn < tok0 + L) {
        cp_async4(dst + rr, prm.g + tn * prm.Hv + h);
        cp_async4(dst + 64 + rr, prm.beta + tn * prm.Hv + h);
      } else {
        dst[rr] = 0.f;
        dst[64 + rr] = 0.f;
      }
    }
    cp_async_commit();
  };
  // this CTA's window: positions [wpos, wend) of the reversed chunk order
  const int nch = (prm.Tseq + kChunk - 1) / kChunk;   // chunks per chain (window schedule)
  const int win = (int)flags[2];
  int64_t wpos = 0, wend = 0;
  if (windowed) {
    const int64_t U = (int64_t)prm.N * prm.Hv * nch;
    wpos = (int64_t)win * prm.W;
    wend = wpos + prm.W < U ? wpos + prm.W : U;
  }
  int* hflag = windowed ? prm.sched + 1 : nullptr;   // hflag[m]: slot m of `hand` is ready

#pragma unroll 1
  for (bool first = true;; first = false) {
    // ---- the next piece: chunks [c_begin, c_end) of one chain
    int c_begin = 0, c_end = nchunks;
    bool from_hand = false, to_hand = false;
    if (windowed) {
      if (wpos >= wend) break;
      const int64_t j = wpos / nch, off = wpos - j * nch;
      const int64_t len = (wend < (j + 1) * nch ? wend : (j + 1) * nch) - wpos;
      n = (int)(j / prm.Hv);
      h = (int)(j % prm.Hv);
      hq = h / (prm.Hv / prm.Hqk);
      tok0 = (int64_t)n * prm.Tseq;
      L = prm.Tseq;
      nchunks = nch;
      c_begin = (int)(nch - off - len);
      c_end = (int)(nch - off);
      from_hand = c_begin > 0;   // the suffix of a chain whose prefix window win + 1 ran
      to_hand = c_end < nch;     // the prefix of a chain whose suffix window win - 1 runs
      wpos += len;
    } else if (!first) {
      break;
    }
    if (from_hand) {
      if (tid == 0 && !flag_wait(hflag + win + 1, prm.status, prm.wait_ns)) flags[1] = 1;
      __syncthreads();
      if (flags[1]) break;
    }

    // state S^T[e][d] = h0[d][e] (the identity for a transition chain; the
    // handed-over state for a chain's suffix, read past L1)
    {
      const float* h0p = from_hand ? prm.hand + (int64_t)(win + 1) * kD * kD
                                   : (prm.h0 ? prm.h0 + ((int64_t)n * prm.Hv + h) * kD * kD : nullptr);
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[32];
        const int d0 = 64 * hf + 32 * half;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int64_t at = (int64_t)(d0 + i) * kD + row;
          v[i] = trans ? (d0 + i == row ? 1.f : 0.f) : (!h0p ? 0.f : (from_hand ? __ldcg(h0p + at) : h0p[at]));
        }
        tmem_st32(R_S + lane_off + d0, v);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && c_begin < c_end) {
      issue_kq(c_begin);
      if (!trans) issue_v(c_begin);   // a transition chain has v = 0: U = 0 and no v tile
    }
    if (warp == 1 && c_begin < c_end) fetch_gb(c_begin);

#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int64_t t0 = tok0 + (int64_t)kChunk * c;
      const int Lc = (int)((L - (int64_t)kChunk * c) < kChunk ? (L - (int64_t)kChunk * c) : kChunk);

      // ---- S0 (warp 1, while thread 0 issues M1): gamma = in-chunk cumsum of g,
      // from the g / beta rows copied to shared memory one chunk ahead (lane l
      // copied and reads rows 2l and 2l + 1); the next sync comes before any
      // other reader.
      if (warp == 1) {
        cp_async_wait_all();   // this lane's copies of chunk c (issued one chunk ago)
        const float* cur = graw + (c & 1) * 128;
        const float ga = cur[2 * lane], gb = cur[2 * lane + 1], ba = cur[64 + 2 * lane], bb = cur[64 + 2 * lane + 1];
        if (c + 1 < c_end) fetch_gb(c + 1);
        float sum = ga + gb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, sum, off);
          if (lane >= off) sum += t;
        }
        // gam <- log2(e) * cumsum: e^{gamma_i - gamma_j} is then one subtraction and one ex2
        const float g0 = (sum - gb) * kLog2e, g1 = sum * kLog2e;
        const float gl = __shfl_sync(0xffffffffu, sum, 31) * kLog2e;
        *reinterpret_cast<float2*>(gam + 2 * lane) = make_float2(g0, g1);
        *reinterpret_cast<float2*>(bet + 2 * lane) = make_float2(ba, bb);
        *reinterpret_cast<float2*>(be + 2 * lane) = make_float2(ba * ex2_fast(g0), bb * ex2_fast(g1));
        *reinterpret_cast<float2*>(dl + 2 * lane) = make_float2(ex2_fast(gl - g0), ex2_fast(gl - g1));
        *reinterpret_cast<float2*>(eg + 2 * lane) = make_float2(prm.scale * ex2_fast(g0), prm.scale * ex2_fast(g1));
      }

      // ---- M1: [K;Q] K^T -> R_a
      if (tid == 0) {
        // the next chunk's k / q boxes go to L2 now; their TMA load (issued
        // once M4 frees the tile) then waits on L2 instead of HBM
        if (!mbar_wait(bar_kq, ph_kq, prm.status)) {
          flags[1] = 1;
        } else {
          ph_kq ^= 1;
          kq_pending = false;
          tc_fence_after();
          const uint32_t id = idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint32_t a = OFF_KQ + (s >> 2) * 16384 + (s & 3) * 32;
            mma_bf16(R_a, dsw(s4, a, 16), dsw(s4, a, 16), id, s > 0);
          }
          mma_commit(bar_mma);
          ++mma_pending;
        }
        if (c + 1 < c_end) {
          const int tn = (int)(t0 + kChunk);
          tma_prefetch_3d(&tm_k, 0, hq, tn);
          tma_prefetch_3d(&tm_k, 64, hq, tn);
          if (MODE == kFull) {
            tma_prefetch_3d(&tm_q, 0, hq, tn);
            tma_prefetch_3d(&tm_q, 64, hq, tn);
          }
        }
        bulk_wait_read();   // the previous chunk's o staging (region X) has been read by its TMA store
      }
      if (!wait_mma()) break;

      // ---- S1: A rows (lanes 0..63) and P rows (lanes 64..127)
      {
        float v[32];
        // warps whose whole 32x32 block lies above the diagonal only write zeros
        const bool upper = (qd & 1) == 0 && hf == 1;
        const int i = qd < 2 ? row : row - 64;
        if (upper) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[jj] = 0.f;
        } else {
          tmem_ld32(R_a + lane_off + 32 * hf, v);
          const float ri = qd < 2 ? bet[i] : prm.scale;   // P carries the output scale: OP = scale V'^T P^T
          const float gi = gam[i];
          const int lim = qd < 2 ? i : i + 1;              // A: j < i (strict); P: j <= i
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 gj = *reinterpret_cast<const float4*>(gam + 32 * hf + 4 * k4);
            const float gjs[4] = {gj.x, gj.y, gj.z, gj.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = 32 * hf + 4 * k4 + u;
              v[4 * k4 + u] = j < lim ? ri * ex2_fast(gi - gjs[u]) * v[4 * k4 + u] : 0.f;
            }
          }
        }
        if (qd < 2) {
          float4* dst = reinterpret_cast<float4*>(As + i * kAsLd + 32 * hf);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + OFF_P + sw128_chunk(i, 4 * hf + cc), v + 8 * cc);
        }
      }

      // ---- S2: solve_tril in place; T diag(beta) and T diag(beta e^g) go out as
      // bf16 operands.  Warps 0 and 5 wrote rows 0..31 x cols 0..31 and rows
      // 32..63 x cols 32..63 of A: each solves its two diagonal 16x16 blocks,
      // then merges them into its 32x32 diagonal block of T together with a
      // partner warp (2 for 0, 7 for 5: other SM sub-partitions) that takes
      // the second column tile; the other warps meanwhile zero the upper 16x16
      // blocks of both operands (one 16-byte chunk per thread and operand).
      if (warp == 0 || warp == 5) {
        const int o = warp == 5 ? 32 : 0;
        __syncwarp();
        diag_pair(As, o, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);
        if (warp == 5) {   // the partner warp may read this block's T11, T22 and A21
          named_bar64<2>();
          merge16_half<2>(As, tmp + 16 * 24, o, 0, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);
        } else {
          named_bar64<1>();
          merge16_half<1>(As, tmp, o, 0, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);
        }
      } else {
        const int u = 32 * (warp - 1 - (warp > 5 ? 1 : 0)) + lane;   // 0..191 over warps 1-4, 6, 7
        const int blk = u >> 5, r = (u >> 1) & 15, half = u & 1;
        const int rb = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int cb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const uint32_t off = sw128_chunk(16 * rb + r, 2 * cb + half);
        *reinterpret_cast<uint4*>(sm + OFF_TB + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm + OFF_TBE + off) = make_uint4(0u, 0u, 0u, 0u);
        if (warp == 2 || warp == 7) {
          if (warp == 7) {
            named_bar64<2>();
            merge16_half<2>(As, tmp + 16 * 24, 32, 1, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);
          } else {
            named_bar64<1>();
            merge16_half<1>(As, tmp, 0, 1, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      merge_level<32>(As, tmp, warp, lane, sm + OFF_TB, sm + OFF_TBE, bet, be);

      // ---- M2: W^T = K^T (T diag(beta e^g))^T -> R_a ; U^T = V^T (T diag(beta))^T -> R_b
      if (tid == 0) {
        if (!trans && !mbar_wait(bar_v, ph_v, prm.status)) {
          flags[1] = 1;
        } else {
          if (!trans) {
            ph_v ^= 1;
            v_pending = false;
          }
          tc_fence_after();
          const uint32_t id = idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_bf16(R_a, dsw(s4, OFF_KQ + s * 2048, 16384), dsw(s4, OFF_TBE + s * 32, 16), id, s > 0);
          if (!trans) {
#pragma unroll
            for (int s = 0; s < 4; ++s)
              mma_bf16(R_b, dsw(s4, OFF_V + s * 2048, 8192), dsw(s4, OFF_TB + s * 32, 16), id, s > 0);
          }
          mma_commit(bar_mma);
          ++mma_pending;
        }
      }
      // ---- S4 (while M2 runs): S^T -> bf16 [e][d] (K-major A), S^T *= e^{g_last}
      {
        float v[32];
        const float dec = ex2_fast(gam[kChunk - 1]);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          const uint32_t col = 64 * hf + 32 * half;
          tmem_ld32(R_S + lane_off + col, v);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            store8_bf16(sm + OFF_ST + hf * 16384 + sw128_chunk(row, 4 * half + cc), v + 8 * cc);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= dec;
          tmem_st32(R_S + lane_off + col, v);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      if (!wait_mma()) break;
      if (tid == 0 && c + 1 < c_end && !trans) issue_v(c + 1);   // v tile consumed

      // ---- S3: W^T -> bf16 [d][i] (MN-major B)
      {
        float v[32];
        tmem_ld32(R_a + lane_off + 32 * hf, v);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + OFF_W + sw128_chunk(row, 4 * hf + cc), v + 8 * cc);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- M3: V'^T = U^T - S^T W^T (R_b) ; OQ^T = S^T Q^T (R_a).  S5 overwrites
      // the first half of S^T (k-steps 0..3) with V'^T: the S^T Q^T k-steps that
      // read it commit to bar_o1, which S5 waits for before that store.
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idv = idesc_bf16(128, 64, 0, 1, 1);
        const uint32_t ido = idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t a = OFF_ST + (s >> 2) * 16384 + (s & 3) * 32;
          mma_bf16(R_b, dsw(s4, a, 16), dsw(s4, OFF_W + s * 2048, 16384), idv, (trans && s == 0) ? 0u : 1u);
        }
        mma_commit(bar_x);    // V' ready: S5 starts while Q S runs
        ++x_pending;
#pragma unroll
        for (int s = 0; s < (MODE == kFull ? 8 : 0); ++s) {
          const uint32_t a = OFF_ST + (s >> 2) * 16384 + (s & 3) * 32;
          const uint32_t b = OFF_KQ + 8192 + (s >> 2) * 16384 + (s & 3) * 32;
          mma_bf16(R_a, dsw(s4, a, 16), dsw(s4, b, 16), ido, s > 0);
          if (s == 3) {
            mma_commit(bar_o1);   // S^T's first half read
            ++o1_pending;
          }
        }
        if (MODE == kFull) {
          mma_commit(bar_mma);
          ++mma_pending;
        }
      }
      wait_commit(bar_x, ph_x, x_pending);
      if (!sync_ok()) break;

      // ---- S5: V'^T -> bf16 [e][j] ; V''^T = V'^T diag(e^{g_last - g}) -> bf16
      {
        float v[32], w[32];
        tmem_ld32(R_b + lane_off + 32 * hf, v);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) w[jj] = v[jj] * dl[32 * hf + jj];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + OFF_VPP + sw128_chunk(row, 4 * hf + cc), w + 8 * cc);
        if (MODE == kFull) wait_commit(bar_o1, ph_o1, o1_pending);   // S^T Q^T no longer reads the first half of S^T
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + OFF_VP + sw128_chunk(row, 4 * hf + cc), v + 8 * cc);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- M4: OP^T = V'^T P^T (R_b) ; S^T += V''^T K (R_S)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idp = idesc_bf16(128, 64, 0, 0, 0);
        const uint32_t ids = idesc_bf16(128, 128, 0, 1, 0);
        if (MODE == kFull) {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_bf16(R_b, dsw(s4, OFF_VP + s * 32, 16), dsw(s4, OFF_P + s * 32, 16), idp, s > 0);
          mma_commit(bar_q);
          ++q_pending;
        }
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_bf16(R_S, dsw(s4, OFF_VPP + s * 32, 16), dsw(s4, OFF_KQ + s * 2048, 16384), ids, 1);
        mma_commit(bar_x);    // state updated: the k / q tiles are free
        ++x_pending;
      }
      if (MODE == kStates) {
        // final states only: wait for the state update, release the k tile
        wait_commit(bar_x, ph_x, x_pending);
        if (tid == 0 && c + 1 < c_end && !flags[1]) issue_kq(c + 1);
        if (!sync_ok()) break;
        continue;
      }
      wait_commit(bar_mma, ph_mma, mma_pending);   // S^T Q^T (committed in M3)
      if (!sync_ok()) break;

      // ---- S6: o_i = scale (e^{g_i} OQ_i + OP_i) -> staging -> global
      {
        // this thread holds column e = row of o for 32 rows i; neighbouring
        // lanes exchange values so that each writes bf16 pairs (e, e + 1)
        // staging row i, bf16 pair (e, e + 1): byte i*128 + ((e/8 ^ i%8) << 4) + (e%8)*2.
        // With i = col + 2 pp + odd (col a multiple of 16), i%8 = (2 pp)%8 | odd.
        const int ecol = (row & 63) & ~1;
        const bool odd = lane & 1;
        uint8_t* lbase = sm + OFF_OS + (row >> 6) * 8192 + (odd ? 128 : 0) + (ecol & 7) * 2;
        const uint32_t xsw = (static_cast<uint32_t>((ecol >> 3) ^ (odd ? 1 : 0))) << 4;
        // OQ while V'^T P^T is still in the tensor pipe, then OP
        float oq[2][16];
        tmem_ld16(R_a + lane_off + 32 * hf, oq[0]);
        tmem_ld16(R_a + lane_off + 32 * hf + 16, oq[1]);
        wait_commit(bar_q, ph_q, q_pending);   // V'^T P^T
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float b[16];
          const float* a = oq[q];
          const uint32_t col = 32 * hf + 16 * q;
          tmem_ld16(R_b + lane_off + col, b);
          float e[16];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float4 x = *reinterpret_cast<const float4*>(eg + col + 4 * k4);
            e[4 * k4] = x.x, e[4 * k4 + 1] = x.y, e[4 * k4 + 2] = x.z, e[4 * k4 + 3] = x.w;
          }
          uint8_t* qb = lbase + col * 128;
#pragma unroll
          for (int pp = 0; pp < 8; ++pp) {
            const float v0 = fmaf(e[2 * pp], a[2 * pp], b[2 * pp]);
            const float v1 = fmaf(e[2 * pp + 1], a[2 * pp + 1], b[2 * pp + 1]);
            const float other = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
            const uint32_t word = odd ? pack_bf16(other, v1) : pack_bf16(v0, other);
            const uint32_t off = (2 * pp) * 128 + (xsw ^ (static_cast<uint32_t>((2 * pp) & 7) << 4));
            *reinterpret_cast<uint32_t*>(qb + off) = word;
          }
        }
      }
      // the state update ran under S6; its completion frees the k / q tile
      wait_commit(bar_x, ph_x, x_pending);
      if (tid == 0 && c + 1 < c_end && !flags[1]) issue_kq(c + 1);
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (Lc == kChunk) {
        if (tid == 0) {
          tma_store_3d(&tm_o, sm + OFF_OS, 0, h, (int)t0);
          tma_store_3d(&tm_o, sm + OFF_OS + 8192, 64, h, (int)t0);
          bulk_commit();
        }
      } else {
        // tail chunk: only rows of this sequence are stored
        for (int u = tid; u < kChunk * 16; u += kThreads) {
          const int i = u >> 4, cc = u & 15;
          if (i < Lc) {
            const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_OS + (cc >> 3) * 8192 + sw128_chunk(i, cc & 7));
            *reinterpret_cast<uint4*>(prm.o + ((t0 + i) * prm.Hv + h) * kD + cc * 8) = val;
          }
        }
        __syncthreads();
      }
    }
    if (flags[1]) break;
    if (to_hand || (trans ? prm.ht2 != nullptr : prm.ht != nullptr)) {
      // final state ht[d][e] = S^T[e][d] (or the hand-over slot of this window)
      float* htp = to_hand ? prm.hand + (int64_t)win * kD * kD
                           : (trans ? prm.ht2 : prm.ht) + ((int64_t)n * prm.Hv + h) * kD * kD;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[32];
        const int d0 = 64 * hf + 32 * half;
        tmem_ld32(R_S + lane_off + d0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) htp[(int64_t)(d0 + i) * kD + row] = v[i];
      }
    }
    if (to_hand) {
      // every thread's part of the slot is written before the flag is raised
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        if (win != prm.drop_flag) atomicExch(hflag + win, 1);
      }
    }
  }   // pieces

  if (tid == 0) bulk_wait_read();   // staging reads done before shared memory is released
  if (warp == 1) cp_async_wait_all();   // g / beta copies of a chunk the loop did not reach

  if (flags[1]) {
    // abort: let copies and MMAs already in flight finish (bounded) before
    // the shared memory and TMEM are released
    if (tid == 0) {
      if (kq_pending) mbar_wait(bar_kq, ph_kq, prm.status, 100000000ull);
      if (v_pending) mbar_wait(bar_v, ph_v, prm.status, 100000000ull);
      for (; mma_pending > 0; --mma_pending, ph_mma ^= 1) mbar_wait(bar_mma, ph_mma, prm.status, 100000000ull);
      for (; x_pending > 0; --x_pending, ph_x ^= 1) mbar_wait(bar_x, ph_x, prm.status, 100000000ull);
      for (; q_pending > 0; --q_pending, ph_q ^= 1) mbar_wait(bar_q, ph_q, prm.status, 100000000ull);
      for (; o1_pending > 0; --o1_pending, ph_o1 ^= 1) mbar_wait(bar_o1, ph_o1, prm.status, 100000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool fused128_supported(const gdn_problem& p) {
  return p.dt == GDN_BF16 && p.K == kD && p.V == kD && (p.C == 64 || p.C == 128);
}

bool fused_supported(const gdn_problem& p) { return fused128_supported(p) || (fused1_supported(p) && p.K == 256); }



namespace {

constexpr int kOrderThreads = 256;

// Rank of each sequence by chunk count (descending, then by index), one thread
// per sequence against every sequence's count, tile by tile through shared
// memory.  The ranks are a permutation of 0..N-1 whatever cu holds.
__global__ void __launch_bounds__(kOrderThreads) varlen_order_kernel(const int32_t* __restrict__ cu, int N,
                                                                     int32_t* __restrict__ order) {
  __shared__ int tile[kOrderThreads];
  auto chunks = [&](int m) -> int {
    const int64_t len = (int64_t)cu[m + 1] - cu[m];
    return len > 0 ? (int)((len + kChunk - 1) / kChunk) : 0;
  };
  const int n = blockIdx.x * kOrderThreads + threadIdx.x;
  const int mine = n < N ? chunks(n) : 0;
  int rank = 0;
  for (int base = 0; base < N; base += kOrderThreads) {
    __syncthreads();
    const int m = base + threadIdx.x;
    tile[threadIdx.x] = m < N ? chunks(m) : -1;
    __syncthreads();
    const int cnt = N - base < kOrderThreads ? N - base : kOrderThreads;
    for (int j = 0; j < cnt; ++j) rank += tile[j] > mine || (tile[j] == mine && base + j < n);
  }
  if (n < N) order[rank] = n;
}

}  // namespace

size_t varlen_order_bytes(const gdn_problem& p) {
  if (!p.varlen || p.N <= 1 || p.N > kOrderMaxN) return 0;
  return ((sizeof(int32_t) * (size_t)p.N + kAlign - 1) / kAlign) * kAlign;
}

gdn_status launch_varlen_order(const int32_t* cu, int N, int32_t* order, cudaStream_t s) {
  varlen_order_kernel<<<(N + kOrderThreads - 1) / kOrderThreads, kOrderThreads, 0, s>>>(cu, N, order);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

namespace {

constexpr int kCtasPerSm = 2;   // resident fused CTAs per SM (shared memory and TMEM halves)

// Window schedule of the full pass over equal-length sequences: W chunks per
// window, at least one chain's chunks and about an equal share of the U chunks
// for each of the CTAs the GPU holds at once; nwin = 0: one chain per CTA
// (varying lengths).
struct Windows {
  int64_t W = 0, nwin = 0;
  bool handover() const { return nwin > 0; }
};

Windows fused_windows(const gdn_problem& p) {
  Windows w;
  if (p.varlen) return w;
  const int64_t nch = ((int64_t)p.T + kChunk - 1) / kChunk;
  const int64_t U = (int64_t)p.N * p.Hv * nch;
  if (U == 0) return w;
  const int64_t G = (int64_t)kCtasPerSm * sm_count();
  w.W = (U + G - 1) / G;
  if (w.W < nch) w.W = nch;
  w.nwin = (U + w.W - 1) / w.W;
  return w;
}

// Workspace: [status, claim counter, nwin hand-over flags] (int32), then, when
// a window boundary can cut a chain (W above one chain's chunks), nwin state
// slots of K x V fp32.
size_t sched_bytes(const Windows& w) { return ((sizeof(int32_t) * (2 + w.nwin) + kAlign - 1) / kAlign) * kAlign; }

bool cuts_chains(const gdn_problem& p, const Windows& w) {
  return w.nwin > 0 && w.W != ((int64_t)p.T + kChunk - 1) / kChunk;
}

}  // namespace

// K = V = 128: the one-CTA-per-SM kernel when the chains do not fill the SMs
// (each chain has an SM to itself either way, and its chunks are about twice as
// fast there), and for packed batches small enough (at most 128 chunks a CTA
// slot of the two-CTA kernel, counting ceil(T / 64) + N chunks a value head)
// that their longest sequence, not their total work, is what bounds the step.
bool fused1_preferred(const gdn_problem& p) {
  if (!fused1_supported(p) || p.K != 128) return false;
  const int64_t chains = (int64_t)p.N * p.Hv;
  if (chains <= sm_count()) return true;
  if (!p.varlen) return false;
  const int64_t chunk_heads = (((int64_t)p.T + kChunk - 1) / kChunk + p.N) * p.Hv;
  return chunk_heads <= (int64_t)kCtasPerSm * sm_count() * 128;
}

size_t fused_workspace_bytes(const gdn_problem& p) {
  if (!fused128_supported(p)) return fused1_workspace_bytes(p);
  const Windows w = fused_windows(p);
  if (!w.handover()) return kAlign + varlen_order_bytes(p);   // the status word (and the order table)
  return sched_bytes(w) + (cuts_chains(p, w) ? (size_t)w.nwin * kD * kD * sizeof(float) : 0);
}
size_t fused_status_offset(const gdn_problem&) { return 0; }

// One launch of the fused kernel over the chains of `p` (N x Hv, or twice
// that for kStates).  status: the device status word.
gdn_status launch_fused(const gdn_problem& p, int mode, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                        float* ht2, int32_t* status, cudaStream_t s, int* sched, float* hand, int64_t nwin,
                        int64_t W, int drop_flag, unsigned long long wait_ns, const int32_t* order) {
  const int64_t Ttot = (int64_t)p.B * p.T;
  CUtensorMap tq, tk, tv, to;
  memset(&to, 0, sizeof(to));
  memset(&tq, 0, sizeof(tq));
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  const uint32_t box[3] = {64, 1, kChunk};
  {
    const uint64_t dims[3] = {(uint64_t)p.K, (uint64_t)p.Hqk, (uint64_t)Ttot};
    const uint64_t str[2] = {(uint64_t)p.K * 2, (uint64_t)p.Hqk * p.K * 2};
    if (!make_tmap_bf16(&tq, q, 3, dims, str, box) || !make_tmap_bf16(&tk, k, 3, dims, str, box)) return GDN_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.V, (uint64_t)p.Hv, (uint64_t)Ttot};
    const uint64_t str[2] = {(uint64_t)p.V * 2, (uint64_t)p.Hv * p.V * 2};
    if (!make_tmap_bf16(&tv, v, 3, dims, str, box)) return GDN_ERR_CUDA;
    if (!make_tmap_bf16(&to, o, 3, dims, str, box)) return GDN_ERR_CUDA;
  }
  FusedParams prm;
  prm.g = g;
  prm.beta = beta;
  prm.h0 = h0;
  prm.cu = p.varlen ? cu : nullptr;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.ht = ht;
  prm.status = status;
  prm.N = p.N;
  prm.Tseq = p.T;
  prm.Ttot = (int)Ttot;
  prm.Hqk = p.Hqk;
  prm.Hv = p.Hv;
  prm.varlen = p.varlen;
  prm.scale = scale;
  prm.ht2 = ht2;
  prm.split = p.N * p.Hv;
  prm.sched = mode == kFull ? sched : nullptr;
  prm.hand = hand;
  prm.nwin = (int)nwin;
  prm.W = (int)W;
  prm.wait_ns = wait_ns;
  prm.drop_flag = drop_flag;
  prm.order = mode == kFull && p.varlen ? order : nullptr;
  const unsigned chains = (unsigned)((int64_t)p.N * p.Hv);
  auto kernel = mode == kStates ? gdn_fused_kernel<kStates, false>
               : (prm.sched ? gdn_fused_kernel<kFull, true> : gdn_fused_kernel<kFull, false>);
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return GDN_ERR_CUDA;
  const unsigned grid = mode == kStates ? 2 * chains : (prm.sched ? (unsigned)nwin : chains);
  kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status run_fused(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                     const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                     void* ws, cudaStream_t s, int drop_flag, unsigned long long wait_ns) {
  if (!fused128_supported(p)) {
    if (!fused_supported(p)) return GDN_ERR_UNSUPPORTED;
    return run_fused1(p, q, k, v, g, beta, scale, h0, cu, o, ht, ws, s, drop_flag, wait_ns);
  }
  int32_t* status = static_cast<int32_t*>(ws);
  const Windows w = fused_windows(p);
  if (cudaMemsetAsync(status, 0, w.handover() ? sizeof(int32_t) * (2 + w.nwin) : sizeof(int32_t), s) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int64_t Ttot = (int64_t)p.B * p.T;
  if (Ttot == 0 || (int64_t)p.N * p.Hv == 0) {
    // no tokens: ht = h0 (or zeros)
    if (ht) {
      const size_t bytes = sizeof(float) * (size_t)p.N * p.Hv * p.K * p.V;
      cudaError_t e = h0 ? cudaMemcpyAsync(ht, h0, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(ht, 0, bytes, s);
      if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
  }
  if (!w.handover()) {
    int32_t* order = nullptr;
    if (varlen_order_bytes(p) > 0) {
      order = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kAlign);
      const gdn_status st = launch_varlen_order(cu, p.N, order, s);
      if (st != GDN_OK) return st;
    }
    return launch_fused(p, kFull, q, k, v, g, beta, scale, h0, cu, o, ht, nullptr, status, s, nullptr, nullptr, 0, 0,
                        -1, kWaitLimitNs, order);
  }
  float* hand = cuts_chains(p, w) ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sched_bytes(w)) : nullptr;
  return launch_fused(p, kFull, q, k, v, g, beta, scale, h0, cu, o, ht, nullptr, status, s, status + 1, hand, w.nwin,
                      w.W, drop_flag, wait_ns);
}

bool fused_handover_window(const gdn_problem& p, int window) {
  if (!fused128_supported(p)) return fused_supported(p) && fused1_handover_window(p, window);
  const Windows w = fused_windows(p);
  if (!cuts_chains(p, w) || window < 1 || window >= w.nwin) return false;
  // window - 1 ends with the suffix of a chain whose prefix `window` runs
  const int64_t nch = ((int64_t)p.T + kChunk - 1) / kChunk;
  return ((int64_t)window * w.W) % nch != 0;
}

gdn_status run_fused_states(const gdn_problem& p, const void* k, const void* v, const float* g, const float* beta,
                            const int32_t* cu, float* ht_zero, float* ht_trans, int32_t* status, cudaStream_t s) {
  // q and o are never touched in this mode; k / v stand in for their maps
  return launch_fused(p, kStates, k, k, v, g, beta, 1.f, nullptr, cu, const_cast<void*>(v), ht_zero, ht_trans,
                      status, s);
}

}  // namespace gdn
