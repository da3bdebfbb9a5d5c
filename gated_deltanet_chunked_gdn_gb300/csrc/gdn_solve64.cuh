// gdn_solve64.cuh -- per-chunk pieces shared by the fused kernels (64-token
// chunks, 256 threads): the triangular solve T = (I + A)^{-1} (MegaGDN-PTO
// walkthrough, section 4.4, solve_tril), shared-memory descriptor arithmetic
// for 128-byte-swizzled operand tiles, and bf16 packing.
#pragma once

#include "gdn_sm100.cuh"

namespace gdn {
namespace solve64 {

using namespace sm100;

constexpr int kChunk = 64;      // tokens per chunk
constexpr int kThreads = 256;   // threads of a fused CTA (eight warps)
constexpr int kAsLd = 68;       // leading dimension of the fp32 A / T tile

// T = (I + A)^{-1} for a 64x64 strictly lower A held in place in As (fp32,
// leading dimension kAsLd, zeros on and above the diagonal).
//  1. Diagonal 16x16 blocks by forward substitution: a half-warp per block,
//     lane l keeps column l of the block's inverse in registers.
//  2. Merge neighbouring blocks, [[T11, 0], [A21, T22]] -> T21 = -T22 (A21 T11),
//     first the 16-blocks (two pairs; each pair's diagonal blocks are solved
//     by the warp that wrote that 32x32 diagonal block of A in the gating
//     step, which then merges one column tile while a partner warp merges
//     the other, joined by a named barrier instead of a block barrier), then
//     the 32-blocks (one pair, all warps).  The
//     merge products run on the tensor cores (mma.sync m16n8k8, tf32 inputs,
//     fp32 accumulation); the upper triangles hold zeros, so they are plain
//     square products.  The fp32 values enter the tf32 MMA unrounded (the unit
//     reads their upper 19 bits, i.e. truncates to tf32: at most 2^-10
//     relative per operand); measured end to end against the fp64 oracle,
//     this leaves the error of o and ht where rounding to tf32 puts it, far
//     below the bf16 rounding T receives as an MMA operand afterwards.
//     Rounding the operands first (cvt.rna, or an integer round-half-away of
//     the bit pattern) lengthens this serial phase enough to cost 7 % (3 %)
//     of the whole step at 16 x 8192, 32 heads.

// d[16x8] += A[16 x KK] B[KK x 8]; A(r, c) = A[r * lda + c], B(r, c) = B[r * ldb + c]
// (shared memory).  A's fragments come from one ldmatrix.x4 per k-step (four
// 8 x 4 fp32 sub-tiles, rows 16-byte aligned); the fp32 values go to the tf32
// MMA as they are (the unit reads their upper 19 bits).
template <int KK>
__device__ __forceinline__ void tile_mma_tf32(float (&d)[4], const float* A, int lda, const float* B, int ldb,
                                              int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t pa = smem_u32(A + ((lane & 7) + 8 * ((lane >> 3) & 1)) * lda + 4 * (lane >> 4));
#pragma unroll
  for (int k0 = 0; k0 < KK; k0 += 8) {
    uint32_t a0, a1, a2, a3;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(pa + 4u * k0));
    const uint32_t b0 = __float_as_uint(B[(k0 + t) * ldb + g]), b1 = __float_as_uint(B[(k0 + t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Store a 16x8 accumulator tile (times `sign`) at D(r, c) = D[r * ldd + c].
__device__ __forceinline__ void tile_store(const float (&d)[4], float* D, int ldd, int lane, float sign) {
  const int g = lane >> 2, t = lane & 3;
  D[g * ldd + 2 * t] = sign * d[0];
  D[g * ldd + 2 * t + 1] = sign * d[1];
  D[(g + 8) * ldd + 2 * t] = sign * d[2];
  D[(g + 8) * ldd + 2 * t + 1] = sign * d[3];
}

// One merge level: pairs of S x S blocks along the diagonal of the 64x64 tile.
// Output tiles (pair, 16-row tile, 8-column tile) are dealt to warps.  The
// final T21 tiles also go out as the two bf16 MMA operands T diag(beta) and
// T diag(beta e^g) (tb, tbe: 64 x 64 K-major tiles, 128-byte swizzle).
template <int S>
__device__ __forceinline__ void merge_level(float* As, float* tmp, int warp, int lane, uint8_t* tb, uint8_t* tbe,
                                            const float* bet, const float* be) {
  constexpr int NP = kChunk / (2 * S);
  constexpr int MT = S / 16, NT = S / 8;
  constexpr int TLD = S + 8;                  // padded leading dimension of tmp (no bank conflicts)
  constexpr int TILES = NP * MT * NT;
  // tmp_p = A21 T11
  for (int tile = warp; tile < TILES; tile += kThreads / 32) {
    const int p = tile / (MT * NT), mt = (tile / NT) % MT, nt = tile % NT;
    const int o = 2 * S * p;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma_tf32<S>(d, As + (o + S + 16 * mt) * kAsLd + o, kAsLd, As + o * kAsLd + o + 8 * nt, kAsLd, lane);
    tile_store(d, tmp + p * S * TLD + 16 * mt * TLD + 8 * nt, TLD, lane, 1.f);
  }
  __syncthreads();
  // T21 = -T22 tmp_p
  const int g = lane >> 2, t = lane & 3;
  for (int tile = warp; tile < TILES; tile += kThreads / 32) {
    const int p = tile / (MT * NT), mt = (tile / NT) % MT, nt = tile % NT;
    const int o = 2 * S * p;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma_tf32<S>(d, As + (o + S + 16 * mt) * kAsLd + o + S, kAsLd, tmp + p * S * TLD + 8 * nt, TLD, lane);
    const int r0 = o + S + 16 * mt, c0 = o + 8 * nt + 2 * t;
    tile_store(d, As + r0 * kAsLd + o + 8 * nt, kAsLd, lane, -1.f);
    const float b0 = bet[c0], b1 = bet[c0 + 1], e0 = be[c0], e1 = be[c0 + 1];
    *reinterpret_cast<uint32_t*>(tb + sw128_offset(r0 + g, c0)) = pack_bf16(-d[0] * b0, -d[1] * b1);
    *reinterpret_cast<uint32_t*>(tb + sw128_offset(r0 + g + 8, c0)) = pack_bf16(-d[2] * b0, -d[3] * b1);
    *reinterpret_cast<uint32_t*>(tbe + sw128_offset(r0 + g, c0)) = pack_bf16(-d[0] * e0, -d[1] * e1);
    *reinterpret_cast<uint32_t*>(tbe + sw128_offset(r0 + g + 8, c0)) = pack_bf16(-d[2] * e0, -d[3] * e1);
  }
  fence_proxy_async();   // the bf16 tiles feed tcgen05.mma
  __syncthreads();
}

// Shared-memory descriptor of the 128-byte-swizzled tile at byte offset `off`
// from the 1024-aligned base whose shared address / 16 is s4 (the same fields
// as desc_sw128 with SBO = 1024; no carry out of the address field, the
// shared window being below 256 KB): one add per descriptor in the issue loops.
__device__ __forceinline__ uint64_t dsw(uint32_t s4, uint32_t off, uint32_t lbo) {
  constexpr uint32_t hi = (1024u >> 4) | (1u << 14) | (2u << 29);
  return (static_cast<uint64_t>(hi) << 32) | (s4 + ((off >> 4) + ((lbo >> 4) << 16)));
}

// Diagonal 16x16 blocks b and b + 16 of T = (I + A)^{-1} by forward
// substitution, one half-warp per block (lane l keeps column l of the block's
// inverse), written to As (fp32) and to tb / tbe (bf16, times beta and beta e^g).
__device__ __forceinline__ void diag_pair(float* As, int b0, int lane, uint8_t* tb, uint8_t* tbe, const float* bet,
                                          const float* be) {
  const int b = b0 + 16 * (lane >> 4);
  const int l = lane & 15;
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float* arow = As + (b + i) * kAsLd + b;
    float x = (i == l) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < i; ++j) x = fmaf(-arow[j], t[j], x);
    t[i] = x;
  }
  __syncwarp();
  const float bl = bet[b + l], el = be[b + l];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    As[(b + i) * kAsLd + b + l] = t[i];
    *reinterpret_cast<__nv_bfloat16*>(tb + sw128_offset(b + i, b + l)) = __float2bfloat16_rn(t[i] * bl);
    *reinterpret_cast<__nv_bfloat16*>(tbe + sw128_offset(b + i, b + l)) = __float2bfloat16_rn(t[i] * el);
  }
}

// Named barrier ID over 64 threads (two warps).
template <int ID>
__device__ __forceinline__ void named_bar64() {
  asm volatile("bar.sync %0, 64;" :: "n"(ID) : "memory");
}

// Named barrier ID over 128 threads (four warps).
template <int ID>
__device__ __forceinline__ void named_bar128() {
  asm volatile("bar.sync %0, 128;" :: "n"(ID) : "memory");
}

// 16-level merge of the 32x32 diagonal block at o, T21 = -T22 (A21 T11),
// split over two warps: this one computes the 8-column tile nt of T21, the
// product A21 T11 passing through the pair's scratch (16 x 16, leading
// dimension 24; each warp touches only its own columns).  Named barrier BAR
// joins the pair between the two products, before A21 is overwritten by T21.
template <int BAR>
__device__ __forceinline__ void merge16_half(float* As, float* scr, int o, int nt, int lane, uint8_t* tb,
                                             uint8_t* tbe, const float* bet, const float* be) {
  constexpr int SLD = 24;
  const int g = lane >> 2, t = lane & 3;
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma_tf32<16>(d, As + (o + 16) * kAsLd + o, kAsLd, As + o * kAsLd + o + 8 * nt, kAsLd, lane);
    tile_store(d, scr + 8 * nt, SLD, lane, 1.f);
  }
  named_bar64<BAR>();   // both column tiles' A21 T11 done: A21 may be overwritten
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma_tf32<16>(d, As + (o + 16) * kAsLd + o + 16, kAsLd, scr + 8 * nt, SLD, lane);
    const int r0 = o + 16, c0 = o + 8 * nt + 2 * t;
    tile_store(d, As + r0 * kAsLd + o + 8 * nt, kAsLd, lane, -1.f);
    const float b0 = bet[c0], b1 = bet[c0 + 1], e0 = be[c0], e1 = be[c0 + 1];
    *reinterpret_cast<uint32_t*>(tb + sw128_offset(r0 + g, c0)) = pack_bf16(-d[0] * b0, -d[1] * b1);
    *reinterpret_cast<uint32_t*>(tb + sw128_offset(r0 + g + 8, c0)) = pack_bf16(-d[2] * b0, -d[3] * b1);
    *reinterpret_cast<uint32_t*>(tbe + sw128_offset(r0 + g, c0)) = pack_bf16(-d[0] * e0, -d[1] * e1);
    *reinterpret_cast<uint32_t*>(tbe + sw128_offset(r0 + g + 8, c0)) = pack_bf16(-d[2] * e0, -d[3] * e1);
  }
}

// Eight floats as bf16 into one 16-byte chunk of shared memory.
__device__ __forceinline__ void store8_bf16(uint8_t* p, const float* v) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

}  // namespace solve64
}  // namespace gdn
