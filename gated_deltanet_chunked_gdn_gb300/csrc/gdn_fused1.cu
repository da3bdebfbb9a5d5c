// gdn_fused1.cu -- the fused forward pass with ONE CTA per SM (all 512 TMEM
// columns): the whole chunk pipeline (cumsum, scaled_dot_kkt, solve_tril,
// wy_fast, chunk_h, chunk_o; MegaGDN-PTO walkthrough, sections 1.1 and 4.5) in
// one sm_103a launch, for key dimension DK = 256 (the large-head-dim shapes the
// pages specialise for: TileLang x xLLM page, the build-specialisation step, H
// = 32 value heads on 8 qk groups, D = 256) and DK = 128 (the latency form of
// the K = V = 128 pass: for chains that do not share an SM, its chunks take
// about half the time of the two-CTA kernel's).
//
// The value dimension is cut into slices of 128 columns (a 256 x 256 fp32
// state is all of an SM's tensor memory): a CTA owns one slice of one
// (sequence, value head) chain -- its DK x 128 fp32 state slice S^T[e][d]
// lives in TMEM for the whole chain -- and walks the chain's 64-token chunks
// in order.  Everything of a chunk that does not depend on V (K K^T, Q K^T,
// gating, the triangular solve) is recomputed by each slice of a chain; v, Y,
// U, V', o and the state are the slice's own.  Equal-length problems deal the
// chunks out as windows of equal length over the SMs, handing a cut unit's
// state slice over through the workspace as the two-CTA kernel does, but
// group-aligned: the G value heads x V / 128 slices of one qk head (UG units
// that read the same q and k) run in lockstep on UG CTAs, window w taking unit
// w % UG of every qk head in its group's range, so each q / k chunk comes from
// DRAM once and from L2 for the others.
//
// Products (M = 128 on the slice's value columns e, or on the 64 k rows
// stacked over the 64 q rows).  The WY term is applied to the state through
// Y = K S (Y[j][e] = k_j . S[:, e], the state's current value for key j):
// V' = U - T diag(beta e^g) K S = U - (T diag(beta e^g)) Y, so no W = T diag(beta
// e^g) K is formed, and Y comes out of the same product as the query term:
//
//   M1  [K;Q] K^T                  -> R_A   (M128 N64, DK / 16 k-steps over d)
//   S1  A = strict-lower(beta_i e^{g_i - g_j} K K^T) -> smem fp32, P -> smem bf16
//   S2  T = (I + A)^{-1}; T diag(beta), T diag(beta e^g) -> bf16       (warps 0, 2, 5, 7, then all)
//   S4  S^T (fp32, TMEM) -> bf16 [e][d]; S^T *= e^{g_last}            (warps 1, 3, 4, 6, beside S2)
//   M3a [Y^T | OQ^T] = S^T [K;Q]^T -> R_Y   (M128 N128, DK / 16 k-steps; runs under the solve's merges)
//   S3  Y^T -> bf16 [e][j]
//   M3b V'^T = V^T (T diag(beta))^T - Y^T (T diag(beta e^g))^T -> R_B  (8 k-steps)
//   S5  V'^T -> bf16, V''^T = V'^T diag(e^{g_last - g}) -> bf16
//   M4  OP^T = V'^T P^T -> R_B;  S^T += V''^T K (N = DK) -> R_S
//   S6  o_i = scale e^{g_i} OQ_i + OP_i -> staging -> TMA store
//
// The k rows are double-buffered inside the [k; q] tile (per 64-column atom:
// k of even chunks, q, k of odd chunks), so the next chunk's k is loaded while
// this chunk runs and its q as soon as M3a has read this chunk's q: the next
// M1 no longer waits for the whole tile, loaded at the end of the chunk.  Odd
// chunks read the stacked operand as [q; k]: their M1 rows and M3a columns
// come out in the other order.
#include <string.h>

#include "gdn_solve64.cuh"

namespace gdn {
namespace {

using namespace sm100;
using namespace solve64;

constexpr int kVS = 128;         // value columns of one slice
constexpr int kTmemCols = 512;
constexpr uint32_t kAtomKQ = 24576;     // one 64-column atom of the [k even ; q ; k odd] tile
constexpr uint32_t kRowsQ = 8192;       // byte offset of the q rows in an atom (k of odd chunks: 2 kRowsQ)

__host__ __device__ constexpr uint32_t up1024(uint32_t x) { return (x + 1023u) / 1024u * 1024u; }

// Shared-memory map (bytes from a 1024-aligned base) and TMEM columns of the
// kernel for key dimension DK (128 or 256).
template <int DK>
struct Map {
  static constexpr int NA = DK / 64;                      // 64-column atoms of the key dimension
  static constexpr uint32_t KQ = 0;                       // NA atoms of [k even ; q ; k odd]
  static constexpr uint32_t V = NA * kAtomKQ;             // v slice rows 0..63 x 128 e, 2 atoms of 8 KB
  static constexpr uint32_t TB = V + 16384;               // T diag(beta) [i][j] bf16, 8 KB
  static constexpr uint32_t TBE = TB + 8192;              // T diag(beta e^g) [i][j] bf16, 8 KB
  static constexpr uint32_t P = TBE + 8192;               // P [i][j] bf16, 8 KB
  static constexpr uint32_t AS = P + 8192;                // A / T fp32 [64][68] and the merges' scratch
  static constexpr uint32_t TMP = AS + 64 * 68 * 4;
  static constexpr uint32_t ST = up1024(TMP + 32 * 40 * 4);   // S^T bf16 [e][d], NA atoms of 16 KB; after M3a:
  static constexpr uint32_t YT = ST;                      //   Y^T bf16 [e][j]
  static constexpr uint32_t VP = ST + 16384;              //   V'^T bf16 [e][j]
  static constexpr uint32_t VPP = ST + 32768;             //   V''^T bf16 [e][j]
  static constexpr uint32_t OS = ST + 49152;              //   o staging bf16: 2 boxes [64 rows][64 e]
  static constexpr uint32_t MISC = ST + (NA * 16384 > 65536 ? NA * 16384 : 65536);
  static constexpr uint32_t GAM = MISC, BET = MISC + 256, BE = MISC + 512, DL = MISC + 768, EG = MISC + 1024;
  static constexpr uint32_t BAR = MISC + 1280;            // 6 mbarriers: k/q, v, M1, M3a, M3b / M4 state, OP
  static constexpr uint32_t FLAGS = MISC + 1328;          // [0] tmem base, [1] abort, [2] window
  static constexpr uint32_t GRAW = MISC + 1344;           // float[2][2][64]: raw g, beta of two chunks
  static constexpr uint32_t SMEM = MISC + 2368 + 1024;    // + alignment slack
  // TMEM columns (lane = slice column e, or chunk row)
  static constexpr uint32_t R_S = 0;                      // S^T[e][d], d = 0..DK-1
  static constexpr uint32_t R_A = DK;                     // [K;Q] K^T (even chunks) or [Q;K] K^T (odd)
  static constexpr uint32_t R_Y = DK + 64;                // [Y^T | OQ^T] (even) or [OQ^T | Y^T] (odd)
  static constexpr uint32_t R_B = DK + 192;               // V'^T[e][i] -> OP^T
  static_assert(SMEM <= 232448, "one CTA must fit an SM");
  static_assert(R_B + 64 <= kTmemCols, "TMEM");
  static_assert(V % 1024 == 0 && TB % 1024 == 0 && P % 1024 == 0 && ST % 1024 == 0, "atom alignment");
};

struct Params {
  const float* g;
  const float* beta;
  const float* h0;
  const int32_t* cu;
  __nv_bfloat16* o;
  float* ht;
  int32_t* status;
  int N, Tseq, Ttot, Hqk, Hv, V, NS, varlen;   // NS = V / kVS slices per chain
  float scale;
  // packed batches: block b runs unit b % (Hv NS) of sequence order[b / (Hv NS)]
  // (longest first); null: of sequence b / (Hv NS)
  const int32_t* order;
  // group-aligned window schedule (null sched: one unit per CTA): nwin = UG x
  // window groups; group m covers positions [m W, (m + 1) W) of the qk heads'
  // chunks laid end to end (each head's in reverse), window w = UG m + k runs
  // unit k of those heads; a unit cut between groups m + 1 and m hands its
  // state from window w + UG to window w
  int* sched;
  float* hand;   // nwin slots of K x kVS fp32
  int nwin, W, UG;
  unsigned long long wait_ns;
  int drop_flag;
};

template <int DK, bool WIN>
__global__ void __launch_bounds__(kThreads, 1) gdn_fused1_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                   const __grid_constant__ CUtensorMap tm_k,
                                                                   const __grid_constant__ CUtensorMap tm_v,
                                                                   const __grid_constant__ CUtensorMap tm_o,
                                                                   const Params prm) {
  using M = Map<DK>;
  constexpr int NA = M::NA;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  float* As = reinterpret_cast<float*>(sm + M::AS);
  float* tmp = reinterpret_cast<float*>(sm + M::TMP);
  float* gam = reinterpret_cast<float*>(sm + M::GAM);
  float* bet = reinterpret_cast<float*>(sm + M::BET);
  float* be = reinterpret_cast<float*>(sm + M::BE);
  float* dl = reinterpret_cast<float*>(sm + M::DL);
  float* eg = reinterpret_cast<float*>(sm + M::EG);
  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + M::BAR);
  uint64_t* bar_v = bar_kq + 1;
  // MMA commit groups; every thread waits for every commit, in order, so all
  // threads track the same phases
  uint64_t* bar_mma = bar_kq + 2;   // M1
  uint64_t* bar_y = bar_kq + 3;     // M3a (issued by thread kYIssuer)
  uint64_t* bar_x = bar_kq + 4;     // M3b, then the state update (M4)
  uint64_t* bar_q = bar_kq + 5;     // OP^T (M4)
  volatile uint32_t* flags = reinterpret_cast<volatile uint32_t*>(sm + M::FLAGS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hf = warp >> 2;   // TMEM lane quadrant, column half
  constexpr int kYIssuer = 32;               // warp 1, lane 0: issues M3a after S4
  const int G = prm.Hv / prm.Hqk;
  // the unit of the current piece: sequence n, value head h, qk head hq, value
  // columns [e0, e0 + 128), first token, length and chunks
  int n = 0, h = 0, hq = 0, e0 = 0, nchunks = 0;
  int64_t tok0 = 0, L = 0;

  if (!WIN) {
    const int unit = (int)blockIdx.x;
    int chain = unit / prm.NS;
    if (prm.order) chain = prm.order[unit / (prm.Hv * prm.NS)] * prm.Hv + chain % prm.Hv;
    e0 = (unit % prm.NS) * kVS;
    n = chain / prm.Hv;
    h = chain % prm.Hv;
    hq = h / G;
    if (prm.varlen) {
      const int64_t a = prm.cu[n], b = prm.cu[n + 1];
      bool ok = (0 <= a) && (a <= b) && (b <= prm.Ttot);
      if (unit == 0 && (prm.cu[0] != 0 || prm.cu[prm.N] != prm.Ttot)) ok = false;
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
    flags[2] = WIN ? prm.nwin - 1 - atomicAdd(prm.sched, 1) : 0;
    mbar_init(bar_kq, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_y, 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_q, 1);
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
  const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
  const int row = 32 * qd + lane;   // this thread's TMEM lane

  const uint32_t s4 = (sbase & 0x3FFFFu) >> 4;
  uint32_t ph_kq = 0, ph_v = 0, ph_mma = 0, ph_y = 0, ph_x = 0, ph_q = 0;
  bool kq_pending = false, v_pending = false;          // thread 0
  bool q_owed = false;                                 // thread 0: k issued without its q
  int mma_pending = 0, x_pending = 0, q_pending = 0;   // commits of thread 0 not yet waited for
  int y_pending = 0;                                   // commits of kYIssuer not yet waited for
  // k rows of chunk c into buffer c & 1: raises the phase's byte count only
  // (the arrive comes with the q rows), so the phase completes once both are in
  auto issue_k = [&](int c) {
    const int t = (int)(tok0 + (int64_t)kChunk * c);
    mbar_expect_tx(bar_kq, NA * 8192);
#pragma unroll
    for (int a = 0; a < NA; ++a)
      tma_load_3d(sm + M::KQ + a * kAtomKQ + (c & 1) * 2 * kRowsQ, &tm_k, bar_kq, 64 * a, hq, t);
    kq_pending = true;
    q_owed = true;
  };
  auto issue_q = [&](int c) {
    const int t = (int)(tok0 + (int64_t)kChunk * c);
    mbar_arrive_expect_tx(bar_kq, NA * 8192);
#pragma unroll
    for (int a = 0; a < NA; ++a) tma_load_3d(sm + M::KQ + a * kAtomKQ + kRowsQ, &tm_q, bar_kq, 64 * a, hq, t);
    q_owed = false;
  };
  // M1 of chunk c: [K;Q] K^T (even c) or [Q;K] K^T (odd c) -> R_A; false if its
  // tiles never arrived
  auto issue_m1 = [&](int c) -> bool {
    if (!mbar_wait(bar_kq, ph_kq, prm.status)) return false;
    ph_kq ^= 1;
    kq_pending = false;
    tc_fence_after();
    const uint32_t id = idesc_bf16(128, 64, 0, 0, 0);
    const uint32_t sb = (c & 1) * kRowsQ, kb = (c & 1) * 2 * kRowsQ;
#pragma unroll
    for (int s = 0; s < DK / 16; ++s) {
      const uint32_t at = M::KQ + (s >> 2) * kAtomKQ + (s & 3) * 32;
      mma_bf16(tmem + M::R_A, dsw(s4, at + sb, 16), dsw(s4, at + kb, 16), id, s > 0);
    }
    mma_commit(bar_mma);
    ++mma_pending;
    return true;
  };
  auto issue_v = [&](int c) {
    const int t = (int)(tok0 + (int64_t)kChunk * c);
    mbar_arrive_expect_tx(bar_v, 16384);
    tma_load_3d(sm + M::V, &tm_v, bar_v, e0, h, t);
    tma_load_3d(sm + M::V + 8192, &tm_v, bar_v, e0 + 64, h, t);
    v_pending = true;
  };
  auto wait_commit = [&](uint64_t* bar, uint32_t& ph, int& pending, int owner) {
    if (!mbar_wait(bar, ph, prm.status)) flags[1] = 1;
    ph ^= 1;
    if (tid == owner) --pending;
  };
  auto sync_ok = [&]() -> bool {
    __syncthreads();
    tc_fence_after();
    return flags[1] == 0;
  };

  float* graw = reinterpret_cast<float*>(sm + M::GRAW);
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
  const int nch = (prm.Tseq + kChunk - 1) / kChunk;   // chunks per unit (window schedule)
  const int win = (int)flags[2];
  const int wunit = WIN ? win % prm.UG : 0;             // this window's unit within each qk head
  int64_t wpos = 0, wend = 0;
  if (WIN) {
    const int64_t U = (int64_t)prm.N * prm.Hqk * nch;
    wpos = (int64_t)(win / prm.UG) * prm.W;
    wend = wpos + prm.W < U ? wpos + prm.W : U;
  }
  int* hflag = WIN ? prm.sched + 1 : nullptr;
  constexpr int64_t kSlot = (int64_t)DK * kVS;   // floats of one hand-over slot

#pragma unroll 1
  for (bool first = true;; first = false) {
    int c_begin = 0, c_end = nchunks;
    bool from_hand = false, to_hand = false;
    if (WIN) {
      if (wpos >= wend) break;
      const int64_t j = wpos / nch, off = wpos - j * nch;   // j: qk head of the sequences' heads
      const int64_t len = (wend < (j + 1) * nch ? wend : (j + 1) * nch) - wpos;
      n = (int)(j / prm.Hqk);
      hq = (int)(j % prm.Hqk);
      h = hq * G + wunit / prm.NS;
      e0 = (wunit % prm.NS) * kVS;
      tok0 = (int64_t)n * prm.Tseq;
      L = prm.Tseq;
      nchunks = nch;
      c_begin = (int)(nch - off - len);
      c_end = (int)(nch - off);
      from_hand = c_begin > 0;
      to_hand = c_end < nch;
      wpos += len;
    } else if (!first) {
      break;
    }
    if (from_hand) {
      if (tid == 0 && !flag_wait(hflag + win + prm.UG, prm.status, prm.wait_ns)) flags[1] = 1;
      __syncthreads();
      if (flags[1]) break;
    }

    // state slice S^T[e][d] = h0[d][e0 + e] (or the handed-over slot [d][e])
    {
      const float* h0p = from_hand ? prm.hand + (int64_t)(win + prm.UG) * kSlot
                                   : (prm.h0 ? prm.h0 + ((int64_t)n * prm.Hv + h) * DK * prm.V + e0 : nullptr);
      const int64_t ld = from_hand ? kVS : prm.V;
#pragma unroll 1
      for (int q4 = 0; q4 < DK / 64; ++q4) {
        float v[32];
        const int d0 = (DK / 2) * hf + 32 * q4;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int64_t at = (int64_t)(d0 + i) * ld + row;
          v[i] = !h0p ? 0.f : (from_hand ? __ldcg(h0p + at) : h0p[at]);
        }
        tmem_st32(tmem + M::R_S + lane_off + d0, v);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && c_begin < c_end) {
      issue_k(c_begin);
      issue_q(c_begin);
      issue_v(c_begin);
    }
    if (warp == 1 && c_begin < c_end) fetch_gb(c_begin);

#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int64_t t0 = tok0 + (int64_t)kChunk * c;
      const int Lc = (int)((L - (int64_t)kChunk * c) < kChunk ? (L - (int64_t)kChunk * c) : kChunk);

      // ---- S0 (warp 1): gamma, beta and the decay factors of this chunk
      if (warp == 1) {
        cp_async_wait_all();
        const float* cur = graw + (c & 1) * 128;
        const float ga = cur[2 * lane], gb = cur[2 * lane + 1], ba = cur[64 + 2 * lane], bb = cur[64 + 2 * lane + 1];
        if (c + 1 < c_end) fetch_gb(c + 1);
        float sum = ga + gb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, sum, off);
          if (lane >= off) sum += t;
        }
        const float g0 = (sum - gb) * kLog2e, g1 = sum * kLog2e;
        const float gl = __shfl_sync(0xffffffffu, sum, 31) * kLog2e;
        *reinterpret_cast<float2*>(gam + 2 * lane) = make_float2(g0, g1);
        *reinterpret_cast<float2*>(bet + 2 * lane) = make_float2(ba, bb);
        *reinterpret_cast<float2*>(be + 2 * lane) = make_float2(ba * ex2_fast(g0), bb * ex2_fast(g1));
        *reinterpret_cast<float2*>(dl + 2 * lane) = make_float2(ex2_fast(gl - g0), ex2_fast(gl - g1));
        *reinterpret_cast<float2*>(eg + 2 * lane) = make_float2(prm.scale * ex2_fast(g0), prm.scale * ex2_fast(g1));
      }

      // ---- M1; then the next chunk's k into the other buffer (its last
      // reader, the previous chunk's state update, is complete)
      if (tid == 0) {
        if (!issue_m1(c)) flags[1] = 1;
        if (c + 1 < c_end && !flags[1]) issue_k(c + 1);
        const int tn = (int)(t0 + kChunk);
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          if (c + 1 < c_end) tma_prefetch_3d(&tm_q, 64 * a, hq, tn);
          if (c + 2 < c_end) tma_prefetch_3d(&tm_k, 64 * a, hq, tn + kChunk);
        }
        bulk_wait_read();   // the previous chunk's o staging has been read by its TMA store
      }
      wait_commit(bar_mma, ph_mma, mma_pending, 0);
      if (!sync_ok()) break;

      // ---- S1: A rows (lanes 0..63) and P rows (lanes 64..127)
      {
        float v[32];
        const bool upper = (qd & 1) == 0 && hf == 1;
        const bool isA = (qd < 2) != static_cast<bool>(c & 1);   // lanes of K K^T
        const int i = row & 63;
        if (upper) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[jj] = 0.f;
        } else {
          tmem_ld32(tmem + M::R_A + lane_off + 32 * hf, v);
          const float ri = isA ? bet[i] : prm.scale;
          const float gi = gam[i];
          const int lim = isA ? i : i + 1;
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
        if (isA) {
          float4* dst = reinterpret_cast<float4*>(As + i * kAsLd + 32 * hf);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + M::P + sw128_chunk(i, 4 * hf + cc), v + 8 * cc);
        }
      }

      // ---- S2 beside S4 and M3a.  The two warps that wrote the 32 x 32
      // diagonal blocks of A in S1 (warps 0 and 5 for even chunks, 2 and 7 for
      // odd ones, whose A rows sit in the other TMEM lanes) solve their 16 x 16
      // diagonal blocks and merge them with a partner warp (2 and 7, or 0 and
      // 5); warps 1, 3, 4 and 6 convert the state (S4), and kYIssuer then
      // issues M3a.
      const bool oddc = c & 1;
      const int w_sa = oddc ? 2 : 0, w_sb = oddc ? 7 : 5, w_pa = oddc ? 0 : 2, w_pb = oddc ? 5 : 7;
      if (warp == w_sa || warp == w_sb) {
        const int o = warp == w_sb ? 32 : 0;
        __syncwarp();
        diag_pair(As, o, lane, sm + M::TB, sm + M::TBE, bet, be);
        if (warp == w_sb) {
          named_bar64<2>();
          merge16_half<2>(As, tmp + 16 * 24, o, 0, lane, sm + M::TB, sm + M::TBE, bet, be);
        } else {
          named_bar64<1>();
          merge16_half<1>(As, tmp, o, 0, lane, sm + M::TB, sm + M::TBE, bet, be);
        }
      } else {
        // the six other warps zero the upper 16 x 16 blocks of both operands
        const int z = oddc ? warp - (warp > 2 ? 1 : 0) : warp - 1 - (warp > 5 ? 1 : 0);
        const int u = 32 * z + lane;
        const int blk = u >> 5, r = (u >> 1) & 15, half = u & 1;
        const int rb = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int cb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const uint32_t off = sw128_chunk(16 * rb + r, 2 * cb + half);
        *reinterpret_cast<uint4*>(sm + M::TB + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sm + M::TBE + off) = make_uint4(0u, 0u, 0u, 0u);
        if (warp == w_pa || warp == w_pb) {
          if (warp == w_pb) {
            named_bar64<2>();
            merge16_half<2>(As, tmp + 16 * 24, 32, 1, lane, sm + M::TB, sm + M::TBE, bet, be);
          } else {
            named_bar64<1>();
            merge16_half<1>(As, tmp, 0, 1, lane, sm + M::TB, sm + M::TBE, bet, be);
          }
        } else {
          // S4: S^T -> bf16 [e][d] (K-major A of M3a), S^T *= e^{g_last}; this
          // warp's lane quadrant, all 256 columns
          float v[32];
          const float dec = ex2_fast(gam[kChunk - 1]);
#pragma unroll 1
          for (int q8 = 0; q8 < DK / 32; ++q8) {
            const uint32_t col = 32 * q8;
            tmem_ld32(tmem + M::R_S + lane_off + col, v);
            uint8_t* atom = sm + M::ST + (col >> 6) * 16384;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) store8_bf16(atom + sw128_chunk(row, 4 * (q8 & 1) + cc), v + 8 * cc);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= dec;
            tmem_st32(tmem + M::R_S + lane_off + col, v);
          }
          tmem_wait_st();
          fence_proxy_async();   // S^T bf16 feeds tcgen05.mma
          tc_fence_before();
          named_bar128<3>();     // the four S4 warps are done
          // ---- M3a: [Y^T | OQ^T] = S^T [K;Q]^T -> R_Y (M128 N128)
          if (tid == kYIssuer) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, 0, 0, 0);
#pragma unroll
            for (int s = 0; s < DK / 16; ++s) {
              const uint32_t a = M::ST + (s >> 2) * 16384 + (s & 3) * 32;
              const uint32_t b = M::KQ + (s >> 2) * kAtomKQ + (c & 1) * kRowsQ + (s & 3) * 32;
              mma_bf16(tmem + M::R_Y, dsw(s4, a, 16), dsw(s4, b, 16), id, s > 0);
            }
            mma_commit(bar_y);
            ++y_pending;
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      merge_level<32>(As, tmp, warp, lane, sm + M::TB, sm + M::TBE, bet, be);

      // ---- S3: Y^T -> bf16 [e][j] (K-major A of M3b), over S^T's first atom
      wait_commit(bar_y, ph_y, y_pending, kYIssuer);
      tc_fence_after();
      if (tid == 0 && c + 1 < c_end && !flags[1]) issue_q(c + 1);   // this chunk's q has been read
      __syncwarp();
      const uint32_t col_y = (c & 1) ? 64 : 0, col_oq = 64 - col_y;
      {
        float v[32];
        tmem_ld32(tmem + M::R_Y + col_y + lane_off + 32 * hf, v);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + M::YT + sw128_chunk(row, 4 * hf + cc), v + 8 * cc);
      }
      fence_proxy_async();
      tc_fence_before();
      if (!sync_ok()) break;

      // ---- M3b: V'^T = V^T (T diag(beta))^T - Y^T (T diag(beta e^g))^T -> R_B
      if (tid == 0) {
        if (!mbar_wait(bar_v, ph_v, prm.status)) {
          flags[1] = 1;
        } else {
          ph_v ^= 1;
          v_pending = false;
          tc_fence_after();
          const uint32_t idu = idesc_bf16(128, 64, 1, 0, 0);
          const uint32_t idy = idesc_bf16(128, 64, 0, 0, 1);
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_bf16(tmem + M::R_B, dsw(s4, M::V + s * 2048, 8192), dsw(s4, M::TB + s * 32, 16), idu, s > 0);
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_bf16(tmem + M::R_B, dsw(s4, M::YT + s * 32, 16), dsw(s4, M::TBE + s * 32, 16), idy, 1u);
          mma_commit(bar_x);
          ++x_pending;
        }
      }
      wait_commit(bar_x, ph_x, x_pending, 0);
      if (!sync_ok()) break;
      if (tid == 0 && c + 1 < c_end) issue_v(c + 1);   // v tile consumed
      __syncwarp();

      // ---- S5: V'^T -> bf16 [e][j] ; V''^T = V'^T diag(e^{g_last - g}) -> bf16
      {
        float v[32], w[32];
        tmem_ld32(tmem + M::R_B + lane_off + 32 * hf, v);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) w[jj] = v[jj] * dl[32 * hf + jj];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + M::VPP + sw128_chunk(row, 4 * hf + cc), w + 8 * cc);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) store8_bf16(sm + M::VP + sw128_chunk(row, 4 * hf + cc), v + 8 * cc);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- M4: OP^T = V'^T P^T (R_B) ; S^T += V''^T K (R_S, N = DK)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idp = idesc_bf16(128, 64, 0, 0, 0);
        const uint32_t ids = idesc_bf16(128, DK, 0, 1, 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + M::R_B, dsw(s4, M::VP + s * 32, 16), dsw(s4, M::P + s * 32, 16), idp, s > 0);
        mma_commit(bar_q);
        ++q_pending;
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_bf16(tmem + M::R_S, dsw(s4, M::VPP + s * 32, 16),
                   dsw(s4, M::KQ + (c & 1) * 2 * kRowsQ + s * 2048, kAtomKQ), ids, 1);
        mma_commit(bar_x);
        ++x_pending;
      }
      __syncwarp();   // warp 0 reconverges before the warp-collective TMEM loads

      // ---- S6: o_i = scale (e^{g_i} OQ_i + OP_i) -> staging -> global
      {
        const int ecol = (row & 63) & ~1;
        const bool odd = lane & 1;
        uint8_t* lbase = sm + M::OS + (row >> 6) * 8192 + (odd ? 128 : 0) + (ecol & 7) * 2;
        const uint32_t xsw = (static_cast<uint32_t>((ecol >> 3) ^ (odd ? 1 : 0))) << 4;
        float oq[2][16];
        tmem_ld16(tmem + M::R_Y + col_oq + lane_off + 32 * hf, oq[0]);
        tmem_ld16(tmem + M::R_Y + col_oq + lane_off + 32 * hf + 16, oq[1]);
        wait_commit(bar_q, ph_q, q_pending, 0);   // OP^T
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float b[16];
          const float* a = oq[q];
          const uint32_t col = 32 * hf + 16 * q;
          tmem_ld16(tmem + M::R_B + lane_off + col, b);
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
      wait_commit(bar_x, ph_x, x_pending, 0);
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (Lc == kChunk) {
        if (tid == 0) {
          tma_store_3d(&tm_o, sm + M::OS, e0, h, (int)t0);
          tma_store_3d(&tm_o, sm + M::OS + 8192, e0 + 64, h, (int)t0);
          bulk_commit();
        }
      } else {
        for (int u = tid; u < kChunk * 16; u += kThreads) {
          const int i = u >> 4, cc = u & 15;
          if (i < Lc) {
            const uint4 val = *reinterpret_cast<const uint4*>(sm + M::OS + (cc >> 3) * 8192 + sw128_chunk(i, cc & 7));
            *reinterpret_cast<uint4*>(prm.o + ((t0 + i) * prm.Hv + h) * prm.V + e0 + cc * 8) = val;
          }
        }
        __syncthreads();
      }
    }
    if (flags[1]) break;
    if (to_hand || prm.ht != nullptr) {
      // final state slice ht[d][e0 + e] = S^T[e][d] (or the hand-over slot [d][e])
      float* htp = to_hand ? prm.hand + (int64_t)win * kSlot : prm.ht + ((int64_t)n * prm.Hv + h) * DK * prm.V + e0;
      const int64_t ld = to_hand ? kVS : prm.V;
#pragma unroll 1
      for (int q4 = 0; q4 < DK / 64; ++q4) {
        float v[32];
        const int d0 = (DK / 2) * hf + 32 * q4;
        tmem_ld32(tmem + M::R_S + lane_off + d0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) htp[(int64_t)(d0 + i) * ld + row] = v[i];
      }
    }
    if (to_hand) {
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        if (win != prm.drop_flag) atomicExch(hflag + win, 1);
      }
    }
  }   // pieces

  if (tid == 0) bulk_wait_read();
  if (warp == 1) cp_async_wait_all();

  if (flags[1]) {
    // abort: copies and MMAs already in flight finish (bounded) before the
    // shared memory and TMEM are released; each issuing thread waits for its own
    if (tid == 0) {
      if (q_owed) mbar_arrive_expect_tx(bar_kq, 0);   // the phase's arrive, so that it can complete
      if (kq_pending) mbar_wait(bar_kq, ph_kq, prm.status, 100000000ull);
      if (v_pending) mbar_wait(bar_v, ph_v, prm.status, 100000000ull);
      for (; mma_pending > 0; --mma_pending, ph_mma ^= 1) mbar_wait(bar_mma, ph_mma, prm.status, 100000000ull);
      for (; x_pending > 0; --x_pending, ph_x ^= 1) mbar_wait(bar_x, ph_x, prm.status, 100000000ull);
      for (; q_pending > 0; --q_pending, ph_q ^= 1) mbar_wait(bar_q, ph_q, prm.status, 100000000ull);
    }
    if (tid == kYIssuer)
      for (; y_pending > 0; --y_pending, ph_y ^= 1) mbar_wait(bar_y, ph_y, prm.status, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Group-aligned window schedule of an equal-length problem: UG = G x V / 128
// units per qk head, as many groups of UG windows as the SMs hold (at least
// one), W chunks of the qk heads' chunk order per group (at least one unit's).
struct Windows {
  int64_t W = 0, nwin = 0, UG = 0;
};

Windows windows_of(const gdn_problem& p) {
  Windows w;
  if (p.varlen) return w;
  const int64_t nch = ((int64_t)p.T + kChunk - 1) / kChunk;
  const int64_t U = (int64_t)p.N * p.Hqk * nch;
  if (U == 0) return w;
  w.UG = (int64_t)(p.Hv / p.Hqk) * (p.V / kVS);
  int64_t groups = sm_count() / w.UG;
  if (groups < 1) groups = 1;
  w.W = (U + groups - 1) / groups;
  if (w.W < nch) w.W = nch;
  w.nwin = w.UG * ((U + w.W - 1) / w.W);
  return w;
}

size_t sched_bytes(const Windows& w) { return ((sizeof(int32_t) * (2 + w.nwin) + kAlign - 1) / kAlign) * kAlign; }

bool cuts_units(const gdn_problem& p, const Windows& w) {
  return w.nwin > 0 && w.W != ((int64_t)p.T + kChunk - 1) / kChunk;
}

}  // namespace

bool fused1_supported(const gdn_problem& p) {
  return p.dt == GDN_BF16 && (p.K == 128 || p.K == 256) && p.V % kVS == 0 && p.V <= 256 &&
         (p.C == 64 || p.C == 128);
}

size_t fused1_workspace_bytes(const gdn_problem& p) {
  const Windows w = windows_of(p);
  if (w.nwin == 0) return kAlign + varlen_order_bytes(p);   // the status word (and the order table)
  return sched_bytes(w) + (cuts_units(p, w) ? (size_t)w.nwin * p.K * kVS * sizeof(float) : 0);
}

bool fused1_handover_window(const gdn_problem& p, int window) {
  if (!fused1_supported(p)) return false;
  const Windows w = windows_of(p);
  if (!cuts_units(p, w) || window < w.UG || window >= w.nwin) return false;
  // window - UG ends with the suffix of a unit whose prefix `window` runs
  const int64_t nch = ((int64_t)p.T + kChunk - 1) / kChunk;
  return ((int64_t)(window / w.UG) * w.W) % nch != 0;
}

namespace {

template <int DK>
gdn_status launch_fused1(const Params& prm, unsigned grid, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t s) {
  auto kernel = prm.sched ? gdn_fused1_kernel<DK, true> : gdn_fused1_kernel<DK, false>;
  const int smem = (int)Map<DK>::SMEM;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  kernel<<<grid, kThreads, smem, s>>>(tq, tk, tv, to, prm);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status run_fused1(const gdn_problem& p, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const float* h0, const int32_t* cu, void* o, float* ht,
                      void* ws, cudaStream_t s, int drop_flag, unsigned long long wait_ns) {
  if (!fused1_supported(p)) return GDN_ERR_UNSUPPORTED;
  int32_t* status = static_cast<int32_t*>(ws);
  const Windows w = windows_of(p);
  if (cudaMemsetAsync(status, 0, w.nwin > 0 ? sizeof(int32_t) * (2 + w.nwin) : sizeof(int32_t), s) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int64_t Ttot = (int64_t)p.B * p.T;
  if (Ttot == 0 || (int64_t)p.N * p.Hv == 0) {
    if (ht) {
      const size_t bytes = sizeof(float) * (size_t)p.N * p.Hv * p.K * p.V;
      cudaError_t e = h0 ? cudaMemcpyAsync(ht, h0, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(ht, 0, bytes, s);
      if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
  }
  CUtensorMap tq, tk, tv, to;
  memset(&tq, 0, sizeof(tq));
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  memset(&to, 0, sizeof(to));
  const uint32_t box[3] = {64, 1, kChunk};
  {
    const uint64_t dims[3] = {(uint64_t)p.K, (uint64_t)p.Hqk, (uint64_t)Ttot};
    const uint64_t str[2] = {(uint64_t)p.K * 2, (uint64_t)p.Hqk * p.K * 2};
    if (!make_tmap_bf16(&tq, q, 3, dims, str, box) || !make_tmap_bf16(&tk, k, 3, dims, str, box)) return GDN_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.V, (uint64_t)p.Hv, (uint64_t)Ttot};
    const uint64_t str[2] = {(uint64_t)p.V * 2, (uint64_t)p.Hv * p.V * 2};
    if (!make_tmap_bf16(&tv, v, 3, dims, str, box) || !make_tmap_bf16(&to, o, 3, dims, str, box)) return GDN_ERR_CUDA;
  }
  Params prm;
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
  prm.V = p.V;
  prm.NS = p.V / kVS;
  prm.varlen = p.varlen;
  prm.scale = scale;
  prm.sched = w.nwin > 0 ? status + 1 : nullptr;
  prm.hand = cuts_units(p, w) ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sched_bytes(w)) : nullptr;
  prm.nwin = (int)w.nwin;
  prm.W = (int)w.W;
  prm.UG = (int)w.UG;
  prm.wait_ns = wait_ns;
  prm.drop_flag = drop_flag;
  prm.order = nullptr;
  if (w.nwin == 0 && varlen_order_bytes(p) > 0) {
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kAlign);
    const gdn_status st = launch_varlen_order(cu, p.N, order, s);
    if (st != GDN_OK) return st;
    prm.order = order;
  }
  const unsigned grid = prm.sched ? (unsigned)w.nwin : (unsigned)((int64_t)p.N * p.Hv * prm.NS);
  return p.K == 256 ? launch_fused1<256>(prm, grid, tq, tk, tv, to, s) : launch_fused1<128>(prm, grid, tq, tk, tv, to, s);
}

}  // namespace gdn
