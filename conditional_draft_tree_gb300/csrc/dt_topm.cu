// dt_topm.cu -- per-depth top-M selection over the base-logit rows.
//
// "Riassunto Tecnico: DominoTree", Componenti Core 2: the correction is only
// evaluated on the top-M marginal candidates of each depth. For every row
// (request b, depth j) this kernel returns the M token ids with the largest
// base logit, ordered by (logit desc, id asc).
//
// The rows are 151936 fp32 wide and read once. Each row is cut into pieces,
// one block each, filtered by the block-level selection of dt_topm_block.cuh;
// the last block of a row (atomic ticket, no waiting) merges the piece lists
// and writes the row's result. It serves dt_build_trees (before the search),
// the marginal-score mode and dt_select_topm_noalloc.
#include <cstdint>

#include "dt_common.cuh"
#include "dt_internal.h"
#include "dt_topm_block.cuh"

namespace dt {

namespace {

// The result of one piece of a row: written directly when the piece is the
// whole row; otherwise published as list `slot` of the row, and the last of
// the row's `npieces` pieces to arrive (atomic ticket, no waiting) merges them
// and writes the row.
template <int SLOTS>
__device__ void finish_piece(int row, int slot, int npieces, int M, const float *rowp,
                             uint64_t *lists, uint64_t *partial, int maxpieces, unsigned *ticket,
                             int32_t *cand_id, float *cand_val, int32_t *topm_out) {
  constexpr int MP = SLOTS * 32;
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (npieces > 1) {
    for (int i = threadIdx.x; i < M; i += kTopmThreads)
      partial[(static_cast<size_t>(row) * maxpieces + slot) * M + i] = lists[i];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      s_last = (atomicAdd(ticket + row, 1u) == static_cast<unsigned>(npieces - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    WarpList<SLOTS> acc;
    acc.clear();
    for (int s = warp; s < npieces; s += kTopmWarps) {
      WarpList<SLOTS> b;
      b.load(partial + (static_cast<size_t>(row) * maxpieces + s) * M, M, lane, true);
      acc.merge(b, lane);
    }
    __syncwarp();
    acc.store(lists + warp * MP, lane);
    block_merge_lists<SLOTS>(lists, warp, lane);
    if (threadIdx.x == 0) ticket[row] = 0u;
  }
  for (int i = threadIdx.x; i < M; i += kTopmThreads) {
    const uint64_t k = lists[i];
    const size_t o = static_cast<size_t>(row) * M + i;
    // key 0 only survives when the row holds fewer than M non-NaN values; the
    // request is then flagged non-finite and never searched
    const int32_t id = (k != 0ull) ? static_cast<int32_t>(key_id(k)) : -1;
    cand_id[o] = id;
    cand_val[o] = (id >= 0) ? __ldg(rowp + id) : -__int_as_float(0x7f800000);
    if (topm_out) topm_out[o] = id;
  }
  __syncthreads();   // lists are reused by the block's next piece
}

// Two launch shapes.
//  * nblk == 0: row blockIdx.y in `maxpieces` equal segments, one per block.
//  * nblk > 0 (rows of a multiple of 4 floats, 16-byte aligned): the rows'
//    float4 units, concatenated, in nblk equal contiguous ranges, one per
//    block; a range covers pieces of one or two rows (rarely more). A block
//    thus streams about rows / nblk of a row with one threshold, instead of
//    one segment, and the grid is one wave of resident blocks.
template <int SLOTS>
__global__ void __launch_bounds__(kTopmThreads, 3)
topm_kernel(const float *__restrict__ logits, int V, int D, int M, int maxpieces, int nblk,
            int rows, uint64_t *__restrict__ partial, unsigned *__restrict__ ticket,
            int *__restrict__ req_flags, int32_t *__restrict__ cand_id,
            float *__restrict__ cand_val, int32_t *__restrict__ topm_out) {
  constexpr int MP = SLOTS * 32;
  __shared__ uint64_t lists[kTopmWarps * MP];
  __shared__ uint64_t bufs[kTopmWarps * kBuf];
  __shared__ unsigned long long s_tau;
  __shared__ unsigned long long s_wq[kTopmWarps];
  if (nblk == 0) {
    const int row = blockIdx.y, split = blockIdx.x;
    const size_t row_base = static_cast<size_t>(row) * V;
    const float *rowp = logits + row_base;
    // vector part [a0, a0 + 4 nv) is 16-byte aligned; scalar head [0, a0), tail
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(rowp) >> 2) & 3u);
    const int a0 = min(V, (4 - mis) & 3);
    const int nv = (V - a0) >> 2;
    const int u0 = static_cast<int>(static_cast<long long>(split) * nv / maxpieces);
    const int u1 = static_cast<int>(static_cast<long long>(split + 1) * nv / maxpieces);
    block_topm<SLOTS, 4>(rowp, V, M, a0, nv, u0, u1, split == 0, split == maxpieces - 1, lists,
                      bufs, &s_tau, s_wq, req_flags + row / D);
    finish_piece<SLOTS>(row, split, maxpieces, M, rowp, lists, partial, maxpieces, ticket,
                        cand_id, cand_val, topm_out);
    return;
  }
  const int nv = V >> 2;
  const long long TU = static_cast<long long>(rows) * nv;
  auto bound = [&](long long b) { return b * TU / nblk; };   // first unit of block b
  auto block_of = [&](long long x) {                         // block holding unit x
    long long b = x * nblk / TU;
    while (b + 1 < nblk && bound(b + 1) <= x) ++b;
    while (b > 0 && bound(b) > x) --b;
    return b;
  };
  const long long g0 = bound(blockIdx.x), g1 = bound(blockIdx.x + 1);
  for (long long r = g0 / nv; r * nv < g1; ++r) {
    const int row = static_cast<int>(r);
    const long long rb = r * nv;
    const int u0 = static_cast<int>((g0 > rb ? g0 : rb) - rb);
    const int u1 = static_cast<int>((g1 < rb + nv ? g1 : rb + nv) - rb);
    const float *rowp = logits + static_cast<size_t>(row) * V;
    block_topm<SLOTS, 4>(rowp, V, M, 0, nv, u0, u1, false, false, lists, bufs, &s_tau, s_wq,
                      req_flags + row / D);
    const long long fb = block_of(rb), lb = block_of(rb + nv - 1);
    finish_piece<SLOTS>(row, static_cast<int>(blockIdx.x - fb), static_cast<int>(lb - fb + 1), M,
                        rowp, lists, partial, maxpieces, ticket, cand_id, cand_val, topm_out);
  }
}

}  // namespace

// The same kernel on explicit scratch pointers (used by the allocation-free
// entry point, whose scratch is a static device array).
cudaError_t launch_topm_raw(const float *base_logits, int batch, int D, int V, int M, int nsplit,
                            int nblk, uint64_t *partial, unsigned *ticket, int *req_flags,
                            int32_t *cand_id, float *cand_val, int32_t *topm_out, cudaStream_t st) {
  const int rows = batch * D;
  dim3 grid = nblk > 0 ? dim3(nblk, 1) : dim3(nsplit, rows);
  const int mp = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  switch (mp) {
    case 32:
      topm_kernel<1><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, nblk, rows,
                                                   partial, ticket, req_flags, cand_id, cand_val,
                                                   topm_out);
      break;
    case 64:
      topm_kernel<2><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, nblk, rows,
                                                   partial, ticket, req_flags, cand_id, cand_val,
                                                   topm_out);
      break;
    case 128:
      topm_kernel<4><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, nblk, rows,
                                                   partial, ticket, req_flags, cand_id, cand_val,
                                                   topm_out);
      break;
    default:
      topm_kernel<8><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, nblk, rows,
                                                   partial, ticket, req_flags, cand_id, cand_val,
                                                   topm_out);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_topm(const Plan &p, const float *base_logits, void *ws, int32_t *topm_out,
                        cudaStream_t st) {
  char *w = static_cast<char *>(ws);
  const dt_dims &d = p.dims;
  unsigned *ticket = reinterpret_cast<unsigned *>(w + p.off_ctrl + kCtrlHeader);
  int *req_flags = reinterpret_cast<int *>(ticket + static_cast<size_t>(d.batch) * d.D);
  uint64_t *partial = reinterpret_cast<uint64_t *>(w + p.off_part);
  int32_t *cid = reinterpret_cast<int32_t *>(w + p.off_cand_id);
  float *cval = reinterpret_cast<float *>(w + p.off_cand_val);
  const int rows = d.batch * d.D, nblk = p.topm_blocks;
  dim3 grid = nblk > 0 ? dim3(nblk, 1) : dim3(p.nsplit, rows);
  const int mp = d.M <= 32 ? 32 : d.M <= 64 ? 64 : d.M <= 128 ? 128 : 256;
  switch (mp) {
    case 32:
      topm_kernel<1><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, nblk,
                                                   rows, partial, ticket, req_flags, cid, cval,
                                                   topm_out);
      break;
    case 64:
      topm_kernel<2><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, nblk,
                                                   rows, partial, ticket, req_flags, cid, cval,
                                                   topm_out);
      break;
    case 128:
      topm_kernel<4><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, nblk,
                                                   rows, partial, ticket, req_flags, cid, cval,
                                                   topm_out);
      break;
    default:
      topm_kernel<8><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, nblk,
                                                   rows, partial, ticket, req_flags, cid, cval,
                                                   topm_out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace dt
