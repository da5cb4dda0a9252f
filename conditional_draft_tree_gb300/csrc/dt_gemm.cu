// dt_gemm.cu -- fp32-accumulating CUDA-core GEMM C = A B^T (+ bias) for the
// path-independent projections:
//   * U[b][j][:] = W1[:, :d] H_j       (per round; the path-independent half of
//     the Domino correction W1 [H_i; S_{i-1}], shared by every node of depth j:
//     "Riassunto Tecnico: DominoTree", Componenti Core 1, H_i shared)
//   * G[v][:]    = W_ih E[v] + b_ih    (once per set of weights; the input half of
//     the GRU gates for every vocabulary token)
// Operands are fp32 (H) or bf16 weights decoded to fp32 on load; accumulation is
// fp32 FMA. Tile 128 x 128 x 16, 256 threads, 8 x 8 outputs per thread.
#include <cstdint>

#include "dt_common.cuh"
#include "dt_internal.h"

namespace dt {

namespace {

constexpr int BM = 128, BN = 128, BK = 16, kThreads = 256;

template <int DT>
__device__ __forceinline__ void load_tile_row8(const void *base, size_t ld, int row, int nrows,
                                               int k, int K, float f[8]) {
  if (row >= nrows) {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = 0.f;
    return;
  }
  const size_t off = static_cast<size_t>(row) * ld + k;
  if (k + 8 <= K) {
    load8<DT>(base, off, f);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (k + i < K) ? load1<DT>(base, off + i) : 0.f;
  }
}

// Split K: blockIdx.z takes one K chunk; with ksplit > 1 every block writes its
// partial tile and the last block of the tile (atomic ticket, no waiting) adds
// the partials in chunk order, so the result does not depend on timing.
template <int ADT, int BDT>
__global__ void __launch_bounds__(kThreads)
gemm_nt_kernel(int M, int N, int K, const void *__restrict__ A, size_t lda,
               const void *__restrict__ B, size_t ldb, const float *__restrict__ bias,
               float *__restrict__ C, size_t ldc, int ksplit, float *__restrict__ partial,
               unsigned *__restrict__ tickets) {
  __shared__ int s_last;
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int lr = tid >> 1, lk = (tid & 1) * 8;  // loader: row, k offset within the tile

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int kchunk = ((K + ksplit - 1) / ksplit + BK - 1) / BK * BK;
  const int kbeg = blockIdx.z * kchunk, kend = min(K, kbeg + kchunk);
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    float fa[8], fb[8];
    load_tile_row8<ADT>(A, lda, m0 + lr, M, k0 + lk, kend, fa);
    load_tile_row8<BDT>(B, ldb, n0 + lr, N, k0 + lk, kend, fb);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      As[lk + i][lr] = fa[i];
      Bs[lk + i][lr] = fb[i];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[8];
      float4 a0 = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
      float4 a1 = *reinterpret_cast<const float4 *>(&As[kk][64 + ty * 4]);
      float4 b0 = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
      float4 b1 = *reinterpret_cast<const float4 *>(&Bs[kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  if (ksplit == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
      if (m >= M) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
        if (n < N) C[static_cast<size_t>(m) * ldc + n] = acc[i][j] + (bias ? bias[n] : 0.f);
      }
    }
    return;
  }
  const size_t plane = static_cast<size_t>(M) * N;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n < N) partial[blockIdx.z * plane + static_cast<size_t>(m) * N + n] = acc[i][j];
    }
  }
  __threadfence();
  __syncthreads();
  const unsigned tile = blockIdx.y * gridDim.x + blockIdx.x;
  if (threadIdx.x == 0) s_last = atomicAdd(tickets + tile, 1u) == static_cast<unsigned>(ksplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n >= N) continue;
      float sum = 0.f;
      for (int z = 0; z < ksplit; ++z)
        sum += __ldcg(partial + z * plane + static_cast<size_t>(m) * N + n);
      C[static_cast<size_t>(m) * ldc + n] = sum + (bias ? bias[n] : 0.f);
    }
  }
  if (threadIdx.x == 0) tickets[tile] = 0u;
}

}  // namespace

cudaError_t launch_gemm_nt(int M, int N, int K, const void *A, int a_dtype, size_t lda,
                           const void *B, int b_dtype, size_t ldb, const float *bias, float *C,
                           size_t ldc, int ksplit, float *partial, unsigned *tickets,
                           cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (ksplit < 1) ksplit = 1;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM, ksplit);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
#define DT_GEMM_ARGS M, N, K, A, lda, B, ldb, bias, C, ldc, ksplit, partial, tickets
  if (a_dtype == DT_F32 && b_dtype == DT_F32)
    gemm_nt_kernel<0, 0><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else if (a_dtype == DT_F32 && b_dtype == DT_BF16)
    gemm_nt_kernel<0, 1><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else if (a_dtype == DT_BF16 && b_dtype == DT_F32)
    gemm_nt_kernel<1, 0><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else
    gemm_nt_kernel<1, 1><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
#undef DT_GEMM_ARGS
  return cudaGetLastError();
}

int gemm_tiles(int M, int N) { return ((N + BN - 1) / BN) * ((M + BM - 1) / BM); }

}  // namespace dt
