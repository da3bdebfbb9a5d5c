// gdn_selftest.cu -- self-test of the tensor-core operand layouts the fused
// kernel relies on: one tcgen05.mma chain D = (+/-) A B over operands staged
// in 128-byte-swizzled shared memory as K-major or MN-major tiles (written by
// threads with the same addressing helpers as the fused kernel, or by a TMA
// tiled load), accumulator read back from TMEM.  Exposed through
// gdn_selftest_umma so tests can compare it with a host matmul.
#include <string.h>

#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kSelftestSmem = 1024 + 2 * 32768 + 64;

__global__ void __launch_bounds__(128) umma_selftest_kernel(const __nv_bfloat16* __restrict__ A,
                                                            const __nv_bfloat16* __restrict__ B,
                                                            float* __restrict__ D, int variant,
                                                            const __grid_constant__ CUtensorMap tmapA,
                                                            int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* As = base;
  uint8_t* Bs = base + 32768;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 65536);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 65536 + 16);
  const int a_mn = variant & 1, b_mn = (variant >> 1) & 1;
  const int N = (variant & 4) ? 128 : 64, Kd = (variant & 8) ? 128 : 64;
  const int neg = (variant >> 4) & 1, via_tma = (variant >> 5) & 1;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  // operands
  if (!via_tma) {
    for (int idx = tid; idx < 128 * Kd; idx += blockDim.x) {
      const int m = idx / Kd, k = idx % Kd;
      uint32_t off = a_mn ? (m / 64) * (Kd * 128) + sw128_offset(k, m % 64)
                          : (k / 64) * 16384 + sw128_offset(m, k % 64);
      *reinterpret_cast<__nv_bfloat16*>(As + off) = A[idx];
    }
  }
  for (int idx = tid; idx < Kd * N; idx += blockDim.x) {
    const int k = idx / N, n = idx % N;
    uint32_t off = b_mn ? (n / 64) * (Kd * 128) + sw128_offset(k, n % 64)
                        : (k / 64) * (N * 128) + sw128_offset(n, k % 64);
    *reinterpret_cast<__nv_bfloat16*>(Bs + off) = B[idx];
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (tid == 0) {
    if (via_tma) {
      mbar_arrive_expect_tx(&bar[0], 128 * Kd * 2);
      for (int a = 0; a < Kd / 64; ++a) tma_load_2d(As + a * 16384, &tmapA, &bar[0], 64 * a, 0);
      ok = mbar_wait(&bar[0], 0, status);
    }
    if (ok) {
      const uint32_t idesc = idesc_bf16(128, N, a_mn, b_mn, neg);
      for (int s = 0; s < Kd / 16; ++s) {
        const uint32_t aa = a_mn ? smem_u32(As) + s * 2048 : smem_u32(As) + (s / 4) * 16384 + (s % 4) * 32;
        const uint32_t bb = b_mn ? smem_u32(Bs) + s * 2048 : smem_u32(Bs) + (s / 4) * (N * 128) + (s % 4) * 32;
        mma_bf16(tmem, desc_sw128(aa, Kd * 128, 1024), desc_sw128(bb, Kd * 128, 1024), idesc, s > 0);
      }
      mma_commit(&bar[1]);
    }
  }
  __syncthreads();
  ok = mbar_wait(&bar[1], 0, status);
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
      for (int i = 0; i < 32; ++i) D[(32 * warp + lane) * N + c0 + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

__global__ void exp_selftest_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = exp_fast(x[i]);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_selftest_exp(const float* x, float* y, int n, void* stream) {
  if (!x || !y || n < 0) return GDN_ERR_INVALID_ARG;
  if (n == 0) return GDN_OK;
  exp_selftest_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_umma(int variant, const void* A, const void* B, float* D, void* workspace,
                                        void* stream) {
  if (!A || !B || !D || !workspace || variant < 0 || variant >= 64) return GDN_ERR_INVALID_ARG;
  const int a_mn = variant & 1;
  if ((variant >> 5) & 1) {
    if (a_mn) return GDN_ERR_INVALID_ARG;   // the TMA variant stages a K-major A
    if (reinterpret_cast<uintptr_t>(A) % 16) return GDN_ERR_INVALID_ARG;
  }
  const int Kd = (variant & 8) ? 128 : 64;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if ((variant >> 5) & 1) {
    const uint64_t dims[2] = {(uint64_t)Kd, 128};
    const uint64_t strides[1] = {(uint64_t)Kd * 2};
    const uint32_t box[2] = {64, 128};
    if (!make_tmap_bf16(&map, A, 2, dims, strides, box)) return GDN_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelftestSmem) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  umma_selftest_kernel<<<1, 128, kSelftestSmem, s>>>(static_cast<const __nv_bfloat16*>(A),
                                                     static_cast<const __nv_bfloat16*>(B), D, variant, map, status);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
