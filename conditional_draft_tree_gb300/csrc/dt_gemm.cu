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

// Split K: blockIdx.z takes one K chunk. With ksplit == 1 the block writes C;
// otherwise it writes its partial tile and splitk_reduce_kernel adds the
// partials in chunk order (deterministic). The next K tile is loaded into
// registers while the current one is multiplied (double-buffered tiles).
template <int ADT, int BDT>
__global__ void __launch_bounds__(kThreads)
gemm_nt_kernel(int M, int N, int K, const void *__restrict__ A, size_t lda,
               const void *__restrict__ B, size_t ldb, const float *__restrict__ bias,
               float *__restrict__ C, size_t ldc, int ksplit, float *__restrict__ partial) {
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
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
  float fa[8], fb[8];
  if (kbeg < kend) {
    load_tile_row8<ADT>(A, lda, m0 + lr, M, kbeg + lk, kend, fa);
    load_tile_row8<BDT>(B, ldb, n0 + lr, N, kbeg + lk, kend, fb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      As[0][lk + i][lr] = fa[i];
      Bs[0][lk + i][lr] = fb[i];
    }
  }
  __syncthreads();
  int buf = 0;
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) {
      load_tile_row8<ADT>(A, lda, m0 + lr, M, k0 + BK + lk, kend, fa);
      load_tile_row8<BDT>(B, ldb, n0 + lr, N, k0 + BK + lk, kend, fb);
    }
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[8];
      float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
      float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + ty * 4]);
      float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
      float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        As[buf ^ 1][lk + i][lr] = fa[i];
        Bs[buf ^ 1][lk + i][lr] = fb[i];
      }
    }
    __syncthreads();
    buf ^= 1;
  }
  float *out = C;
  size_t ldo = ldc;
  if (ksplit > 1) {
    out = partial + blockIdx.z * static_cast<size_t>(M) * N;
    ldo = N;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (n < N)
        out[static_cast<size_t>(m) * ldo + n] =
            acc[i][j] + ((ksplit == 1 && bias) ? bias[n] : 0.f);
    }
  }
}

// C = sum_z partial[z] (+ bias). Four lanes per four outputs (a float4):
// lane q sums the planes q, q + 4, q + 8, ... (its loads in flight together),
// then the four sums are combined by two exchanges, (s0 + s1) + (s2 + s3): a
// fixed order, so the result is deterministic. Blocks of 128 threads with at
// most 32 registers each (4 K registers) fit beside three top-M blocks on an
// SM, so the reduction of the projection does not wait for the top-M.
constexpr int kReduceThreads = 128;

__global__ void __launch_bounds__(kReduceThreads, 16) splitk_reduce_kernel(const float *__restrict__ partial, int ksplit, int M, int N,
                                     const float *__restrict__ bias, float *__restrict__ C,
                                     size_t ldc) {
  const size_t plane = static_cast<size_t>(M) * N;
  const size_t gid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t i4 = (gid >> 2) * 4;
  const int q = static_cast<int>(gid & 3);
  const bool valid = i4 < plane;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {
#pragma unroll 8
    for (int z = q; z < ksplit; z += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(partial + z * plane + i4));
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    s.x += __shfl_xor_sync(0xffffffffu, s.x, m);
    s.y += __shfl_xor_sync(0xffffffffu, s.y, m);
    s.z += __shfl_xor_sync(0xffffffffu, s.z, m);
    s.w += __shfl_xor_sync(0xffffffffu, s.w, m);
  }
  if (!valid || q != 0) return;
  const int m = static_cast<int>(i4 / N), n = static_cast<int>(i4 % N);
  if (bias) { s.x += bias[n]; s.y += bias[n + 1]; s.z += bias[n + 2]; s.w += bias[n + 3]; }
  float *c = C + static_cast<size_t>(m) * ldc + n;
  c[0] = s.x; c[1] = s.y; c[2] = s.z; c[3] = s.w;
}

}  // namespace

cudaError_t launch_gemm_nt(int M, int N, int K, const void *A, int a_dtype, size_t lda,
                           const void *B, int b_dtype, size_t ldb, const float *bias, float *C,
                           size_t ldc, int ksplit, float *partial, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (ksplit < 1 || N % 4) ksplit = 1;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM, ksplit);
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
#define DT_GEMM_ARGS M, N, K, A, lda, B, ldb, bias, C, ldc, ksplit, partial
  if (a_dtype == DT_F32 && b_dtype == DT_F32)
    gemm_nt_kernel<0, 0><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else if (a_dtype == DT_F32 && b_dtype == DT_BF16)
    gemm_nt_kernel<0, 1><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else if (a_dtype == DT_BF16 && b_dtype == DT_F32)
    gemm_nt_kernel<1, 0><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
  else
    gemm_nt_kernel<1, 1><<<grid, kThreads, 0, st>>>(DT_GEMM_ARGS);
#undef DT_GEMM_ARGS
  if (ksplit > 1) return launch_splitk_reduce(partial, ksplit, M, N, bias, C, ldc, st);
  return cudaGetLastError();
}

int gemm_tiles(int M, int N) { return ((N + BN - 1) / BN) * ((M + BM - 1) / BM); }

cudaError_t launch_splitk_reduce(const float *partial, int ksplit, int M, int N, const float *bias,
                                 float *C, size_t ldc, cudaStream_t st) {
  const size_t threads = (static_cast<size_t>(M) * N + 3) / 4 * 4;   // four lanes per float4
  splitk_reduce_kernel<<<static_cast<unsigned>((threads + kReduceThreads - 1) / kReduceThreads),
                         kReduceThreads, 0, st>>>(partial, ksplit, M, N, bias, C, ldc);
  return cudaGetLastError();
}

}  // namespace dt
