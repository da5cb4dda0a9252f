// Test-only kernel: one CTA computes D[128][N] = A[128][K] * sum_s B_s[N][K]^T
// with the library's tcgen05 helpers (dt_umma.cuh): operands written in the
// library's K-major no-swizzle layout, MMAs into tensor memory, mbarrier
// completion, tcgen05.ld readout. The test compares D with a float64 product.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../conditional_draft_tree_gb300/csrc/dt_umma.cuh"

using namespace dt;

__global__ void umma_selftest_kernel(const uint16_t *A, const uint16_t *B, float *D, int N, int K,
                                     int nsplit, uint32_t ncols, int *status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ uint32_t tmem_base;
  __shared__ __align__(8) uint64_t mbar;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char *sA = sm;
  unsigned char *sB = sm + 128 * K * 2;
  for (int i = tid; i < 128 * K; i += blockDim.x)
    *reinterpret_cast<uint16_t *>(sA + umma_offset(i / K, i % K, K)) = A[i];
  for (int s = 0; s < nsplit; ++s)
    for (int i = tid; i < N * K; i += blockDim.x)
      *reinterpret_cast<uint16_t *>(sB + s * N * K * 2 + umma_offset(i / K, i % K, K)) =
          B[static_cast<size_t>(s) * N * K + i];
  if (warp == 0) tmem_alloc(&tmem_base, ncols);
  if (tid == 0) mbar_init(&mbar, 1);
  fence_async_smem();
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t taddr = tmem_base;
  if (tid == 0) {
    const uint32_t idesc = umma_idesc_bf16(128, N);
    for (int kb = 0; kb < K / 16; ++kb) {
      const uint64_t ad = umma_desc(smem_u32(sA) + kb * 256, 128, 16 * K);
      for (int s = 0; s < nsplit; ++s) {
        const uint64_t bd = umma_desc(smem_u32(sB + s * N * K * 2) + kb * 256, 128, 16 * K);
        umma_bf16(taddr, ad, bd, idesc, kb > 0 || s > 0);
      }
    }
    umma_commit(&mbar);
  }
  bool ok = mbar_wait(&mbar, 0, 1000000000ull);
  if (!ok) ok = mbar_wait(&mbar, 0, 1000000000ull) && false;
  tmem_fence_after();
  if (warp < 4) {
    const int row = 32 * warp + lane;
    for (int c = 0; c < N; c += 8) {
      float v[8];
      tmem_ld8(taddr + (static_cast<uint32_t>(32 * warp) << 16) + c, v);
      tmem_wait_ld();
      for (int j = 0; j < 8; ++j) D[row * N + c + j] = v[j];
    }
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, ncols);
  if (tid == 0) *status = ok ? 0 : -5;
}

extern "C" int umma_selftest(const uint16_t *A, const uint16_t *B, float *D, int N, int K,
                             int nsplit, int *status) {
  if (N < 16 || N > 256 || N % 16 || K < 16 || K % 16 || nsplit < 1 || nsplit > 3) return -1;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(N)) ncols <<= 1;
  const int smem = 128 * K * 2 + nsplit * N * K * 2;
  if (smem > 200 * 1024) return -1;
  if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -3;
  umma_selftest_kernel<<<1, 128, smem>>>(A, B, D, N, K, nsplit, ncols, status);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
