// dt_proj.cu -- the path-independent projection U = H W1[:, :d]^T on the
// tcgen05 tensor cores (bf16 weights).
//
// "Riassunto Tecnico: DominoTree", Componenti Core 1: the hidden state H_i of
// draft position i is shared by every node of depth i, so its half of the
// correction, W1[:, :d] H_i, is computed once per (request, depth) before the
// search; the released Domino decoder needs the same product per position.
// U[n][m] = sum_k H[n][k] W1[m][k] for the rows n = (request, depth) and the
// r output features m.
//
// Mapping: the MMA's M side is 128 rows of W1 (exact in bf16), its N side up
// to 256 rows of H; H is fp32 and enters as three bf16 terms (hi, mid, lo),
// three MMAs per K step, so the product keeps fp32 accuracy. A block owns one
// (W1 tile, H tile, K chunk of at most 128); its stages of 32 K values are
// all in flight from the start in a ring of raw copies (cp.async, 16 bytes a
// thread). Each thread converts the rows it copied into the K-major no-swizzle
// operand layout (H split into its three terms), one thread issues the
// stage's 6 MMAs and commits them, and the commit frees the operand buffer for
// the next stage. The fp32 accumulator (128 x 256) lives in TMEM and is written
// out as the K chunk's partial; split_k > 1 adds a deterministic reduction
// kernel (a fixed order over the chunks).
//
// The tensor cores' fp32 accumulation loses a little more than a sequential
// FMA chain over a long K (its error grows with the chunk length), hence the
// short chunks: every block covers at most 128 K values, so the plan takes
// about one block per SM and more K chunks than tiles.
#include <cstdint>

#include <cuda_bf16.h>

#include "dt_common.cuh"
#include "dt_internal.h"
#include "dt_umma.cuh"

namespace dt {

namespace {

constexpr int kPThreads = 512;                    // two per H row of a tile
constexpr int kPKc = 32;                          // K values per stage
constexpr int kPN = 256;                          // H rows per tile (MMA N, at most)
constexpr int kPABytes = 128 * kPKc * 2;          // W1 operand tile of a stage: 8 KB
constexpr int kPBTerm = kPN * kPKc * 2;           // one bf16 term of the H tile: 16 KB
constexpr int kPStage = kPABytes + 3 * kPBTerm;   // operand buffer: 56 KB
constexpr int kPRawH = kPN * kPKc * 4;            // raw H rows of a stage: 32 KB
constexpr int kPRawW = 128 * kPKc * 2;            // raw W1 rows of a stage: 8 KB
constexpr int kPRaw = kPRawH + kPRawW;
constexpr int kPBufs = 2;                         // operand buffers
constexpr int kPRing = 2;                         // raw stages in flight
constexpr int kPSmem = kPBufs * kPStage + kPRing * kPRaw + 64;   // 192 KB + barriers
constexpr int kPMaxChunk = 128;                   // K values per block, at most
constexpr unsigned long long kPLimitNs = 2000000000ull;   // per bounded wait

struct ProjParams {
  const float *H;      // [rows][ldh] fp32, 16-byte aligned, ldh % 4 == 0
  const uint16_t *W;   // [r][ldw] bf16, 16-byte aligned, ldw % 8 == 0
  float *out;          // [rows][r]: U (split_k == 1) or the partials [split_k][rows][r]
  int rows, r, K, ldh, ldw, kchunk;
  int *fail;           // set to 1 when a bounded wait runs out
};

// Raw copies of stage k0 into a ring slot: thread tid copies half hh = tid >> 8
// (16 fp32) of H row n0 + (tid & 255) (if that row < nn) and 8 bf16 (k group
// tid >> 7) of W1 row m0 + (tid & 127) (if < r); one commit group per call,
// also when it copies nothing.
__device__ __forceinline__ void issue_raw(const ProjParams &p, unsigned char *raw, int n0, int nn,
                                          int m0, int k0) {
  const int tid = threadIdx.x, row = tid & 255, hh = tid >> 8;
  if (row < nn) {
    const float *src = p.H + static_cast<size_t>(n0 + row) * p.ldh + k0 + 16 * hh;
    unsigned char *dst = raw + row * (kPKc * 4) + 64 * hh;
#pragma unroll
    for (int j = 0; j < 4; ++j) cp_async16(dst + 16 * j, src + 4 * j, 16);
  }
  const int m = m0 + (tid & 127);
  if (m < p.r)
    cp_async16(raw + kPRawH + (tid & 127) * (kPKc * 2) + (tid >> 7) * 16,
               p.W + static_cast<size_t>(m) * p.ldw + k0 + (tid >> 7) * 8, 16);
  cp_async_commit();
}

// This thread's raw rows -> the operand tiles (H split into three terms; rows
// of H in [nn, npad) and W1 rows past r are zero; rows past npad are not read
// by the MMA and not written).
__device__ __forceinline__ void convert(const ProjParams &p, const unsigned char *raw,
                                       unsigned char *opnd, int nn, int npad, int m0) {
  const int tid = threadIdx.x, row = tid & 255, hh = tid >> 8;
  const int m = m0 + (tid & 127);
  *reinterpret_cast<uint4 *>(opnd + umma_offset(tid & 127, (tid >> 7) * 8, kPKc)) =
      m < p.r ? *reinterpret_cast<const uint4 *>(raw + kPRawH + (tid & 127) * (kPKc * 2) +
                                                 (tid >> 7) * 16)
              : make_uint4(0u, 0u, 0u, 0u);
  if (row >= npad) return;
  const float4 *h = reinterpret_cast<const float4 *>(raw + row * (kPKc * 4) + 64 * hh);
  unsigned char *sB = opnd + kPABytes;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int kg = 2 * hh + g;
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
    if (row < nn) {
      x0 = h[2 * g];
      x1 = h[2 * g + 1];
    }
    const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint16_t t[3][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) split3(v[j], t[0][j], t[1][j], t[2][j]);
#pragma unroll
    for (int term = 0; term < 3; ++term) {
      uint4 q;
      q.x = t[term][0] | (static_cast<uint32_t>(t[term][1]) << 16);
      q.y = t[term][2] | (static_cast<uint32_t>(t[term][3]) << 16);
      q.z = t[term][4] | (static_cast<uint32_t>(t[term][5]) << 16);
      q.w = t[term][6] | (static_cast<uint32_t>(t[term][7]) << 16);
      *reinterpret_cast<uint4 *>(sB + term * kPBTerm + umma_offset(row, kg * 8, kPKc)) = q;
    }
  }
}

// grid (H tiles, W1 tiles, K chunks); K chunk z covers [z kchunk, (z+1) kchunk)
// (kchunk and K multiples of 32; every chunk is non-empty). At most 48
// registers a thread (24 K a block), so that two top-M blocks fit beside it.
__global__ void __maxnreg__(48) proj_umma_kernel(const ProjParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *opnd0 = smem;                              // kPBufs operand buffers
  unsigned char *raw0 = smem + kPBufs * kPStage;            // kPRing raw slots
  uint64_t *mbar = reinterpret_cast<uint64_t *>(raw0 + kPRing * kPRaw);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(mbar + kPBufs);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kPN, m0 = blockIdx.y * 128, kz = blockIdx.z;
  const int nn = min(kPN, p.rows - n0);
  const int npad = (nn + 15) & ~15;
  const int kbeg = kz * p.kchunk, kend = min(p.K, kbeg + p.kchunk);
  const int nst = (kend - kbeg) / kPKc;
  if (warp == 0) tmem_alloc(s_tmem, 256);
  if (tid == 0)
    for (int i = 0; i < kPBufs; ++i) mbar_init(&mbar[i], 1);
  for (int i = 0; i < kPRing; ++i) {
    if (i < nst) issue_raw(p, raw0 + i * kPRaw, n0, nn, m0, kbeg + i * kPKc);
    else cp_async_commit();
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t idesc = umma_idesc_bf16(128, npad);

  bool ok = true;
  int i = 0;
  for (; i < nst; ++i) {
    const int b = i % kPBufs;
    unsigned char *opnd = opnd0 + b * kPStage;
    unsigned char *raw = raw0 + (i % kPRing) * kPRaw;
    // the MMAs of stage i - kPBufs must have read this operand buffer
    if (i >= kPBufs && !mbar_wait(&mbar[b], ((i / kPBufs) - 1) & 1u, kPLimitNs)) ok = false;
    if (!__syncthreads_and(ok)) break;
    cp_async_wait_group<kPRing - 1>();   // this thread's copies of stage i have landed
    convert(p, raw, opnd, nn, npad, m0);
    // the raw slot is free again (only this thread reads its rows)
    if (i + kPRing < nst) issue_raw(p, raw, n0, nn, m0, kbeg + (i + kPRing) * kPKc);
    else cp_async_commit();
    fence_async_smem();   // generic writes -> the tensor cores' operand reads
    __syncthreads();
    if (tid == 0) {
      tmem_fence_after();
      const uint32_t a0 = smem_u32(opnd), b0 = a0 + kPABytes;
#pragma unroll
      for (int s = 0; s < kPKc / 16; ++s)
#pragma unroll
        for (int term = 0; term < 3; ++term)
          umma_bf16(tmem, umma_desc(a0 + s * 256, 128, 16 * kPKc),
                    umma_desc(b0 + term * kPBTerm + s * 256, 128, 16 * kPKc), idesc,
                    i > 0 || s > 0 || term > 0);
      umma_commit(&mbar[b]);
    }
  }
  cp_async_wait_all();   // no copy may still be landing when the block ends
  // commits complete in order: the last issued stage covers every MMA (waited
  // for once more, with the limit, after a failure above)
  if (i > 0) {
    const int last = i - 1;
    if (!mbar_wait(&mbar[last % kPBufs], (last / kPBufs) & 1u, kPLimitNs)) ok = false;
  }
  ok = __syncthreads_and(ok);
  tmem_fence_after();
  if (ok) {
    // TMEM lane = W1 row of the tile (warps w, w + 4, w + 8, w + 12 share a
    // lane quarter), column = H row; 8 columns per load (few registers)
    const int quarter = warp & 3;
    const int m = m0 + quarter * 32 + lane;
    float *dst = p.out + static_cast<size_t>(kz) * p.rows * p.r;
    for (int c0 = (warp >> 2) * 8; c0 < npad; c0 += 8 * (kPThreads / 128)) {
      float v[8];
      tmem_ld8(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
      tmem_wait_ld();
      if (m < p.r) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < nn) dst[static_cast<size_t>(n0 + c0 + j) * p.r + m] = v[j];
      }
    }
  } else if (tid == 0) {
    atomicExch(p.fail, 1);
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

bool proj_umma_supported(const dt_dims &d, int wdtype) {
  return wdtype == DT_BF16 && d.d % kPKc == 0 && d.r % 4 == 0 &&
         (static_cast<long long>(d.d) + d.d_s) % 8 == 0;
}

// K split of the projection: about target_blocks blocks, every chunk a
// multiple of 32, at most kPMaxChunk long and non-empty; 1 when r is not a
// multiple of 4 (the reduction reads float4) and K fits one chunk.
int proj_umma_split(int rows, int r, int K, int target_blocks) {
  const int tiles = ((rows + kPN - 1) / kPN) * ((r + 127) / 128);
  const int kmax = K / kPKc;
  int ks = target_blocks / tiles;
  const int ks_min = (K + kPMaxChunk - 1) / kPMaxChunk;
  if (ks < ks_min) ks = ks_min;
  if (ks > kmax) ks = kmax;
  if (ks < 1) ks = 1;
  const int kchunk = (kmax + ks - 1) / ks * kPKc;
  return (K + kchunk - 1) / kchunk;
}

cudaError_t launch_proj_umma(int rows, int r, int K, const float *H, int ldh, const void *W1,
                             int ldw, float *U, int split_k, float *partial, int *fail,
                             cudaStream_t st) {
  if (rows <= 0 || r <= 0) return cudaSuccess;
  const int kmax = K / kPKc;
  const int kchunk = (kmax + split_k - 1) / split_k * kPKc;
  ProjParams p;
  p.H = H;
  p.W = static_cast<const uint16_t *>(W1);
  p.out = split_k > 1 ? partial : U;
  p.rows = rows;
  p.r = r;
  p.K = K;
  p.ldh = ldh;
  p.ldw = ldw;
  p.kchunk = kchunk;
  p.fail = fail;
  cudaError_t e = cudaFuncSetAttribute(proj_umma_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((rows + kPN - 1) / kPN, (r + 127) / 128, split_k);
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidConfiguration;
  proj_umma_kernel<<<grid, kPThreads, kPSmem, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || split_k == 1) return e;
  return launch_splitk_reduce(partial, split_k, rows, r, nullptr, U, r, st);
}

}  // namespace dt
