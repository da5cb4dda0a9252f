// dt_topm.cu -- per-depth top-M selection over the base-logit rows.
//
// "Riassunto Tecnico: DominoTree", Componenti Core 2: the correction is only
// evaluated on the top-M marginal candidates of each depth. For every row
// (request b, depth j) this kernel returns the M token ids with the largest
// base logit, ordered by (logit desc, id asc).
//
// The rows are 151936 fp32 wide and read once: the kernel is HBM bound. Each
// row is cut into `nsplit` segments, one block each. Every warp streams its
// part of the segment with 128-bit loads and keeps a sorted top-M list of
// 64-bit (order(value), ~id) keys in registers; a candidate touches the list
// only when it beats the current M-th key, which after the first few hundred
// elements is rare. The eight warp lists of a block are combined with bitonic
// merges; the last block of a row (atomic ticket, no waiting) merges the
// segment lists and writes the row's result.
#include <cstdint>

#include "dt_common.cuh"
#include "dt_internal.h"

namespace dt {

namespace {

constexpr int kTopmThreads = 256;
constexpr int kTopmWarps = kTopmThreads / 32;
constexpr int kQ = 4;                          // float4 loads per lane per iteration
constexpr int kBuf = 32 + 4 * 32;              // per-warp candidate buffer (keys)

// Sorted (descending) list of 32*SLOTS keys spread over a warp: element
// i = s*32 + lane lives in register v[s] of `lane`.
template <int SLOTS>
struct WarpList {
  uint64_t v[SLOTS];

  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) v[s] = 0;
  }
  // element i (warp-uniform i); every slot is shuffled so that no register is
  // selected by a runtime index
  __device__ __forceinline__ uint64_t at(int i) const {
    uint64_t x = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const uint64_t y = shfl64(v[s], i & 31);
      x = (s == (i >> 5)) ? y : x;
    }
    return x;
  }
  // compare-exchange of registers s and s + DS (lower index keeps the max)
  template <int DS>
  __device__ __forceinline__ void cmpx_slots() {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      if ((s & DS) == 0 && s + DS < SLOTS) {
        const uint64_t a = v[s], b = v[s + DS];
        v[s] = a > b ? a : b;
        v[s + DS] = a > b ? b : a;
      }
    }
  }
  // this <- top 32*SLOTS of (this U other), both sorted descending
  __device__ __forceinline__ void merge(const WarpList &o, int lane) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const uint64_t rev = shfl64(o.v[SLOTS - 1 - s], 31 - lane);
      v[s] = v[s] > rev ? v[s] : rev;  // bitonic sequence holding the top elements
    }
    if (SLOTS >= 8) cmpx_slots<4>();
    if (SLOTS >= 4) cmpx_slots<2>();
    if (SLOTS >= 2) cmpx_slots<1>();
#pragma unroll
    for (int stride = 16; stride >= 1; stride >>= 1) {
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const uint64_t o2 = shfl64_xor(v[s], stride);
        const bool low = (lane & stride) == 0;
        const uint64_t mx = v[s] > o2 ? v[s] : o2, mn = v[s] > o2 ? o2 : v[s];
        v[s] = low ? mx : mn;
      }
    }
  }
  __device__ __forceinline__ void store(uint64_t *dst, int lane) const {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) dst[s * 32 + lane] = v[s];
  }
  // load `n` keys (n <= 32*SLOTS), padding with 0
  __device__ __forceinline__ void load(const uint64_t *src, int n, int lane, bool bypass_l1) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      int i = s * 32 + lane;
      v[s] = (i < n) ? (bypass_l1 ? __ldcg(reinterpret_cast<const unsigned long long *>(src) + i)
                                  : src[i])
                     : 0ull;
    }
  }
};

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// element `bit` (0..15) of four float4 registers, without local memory
__device__ __forceinline__ float pick16(const float4 c[kQ], int bit) {
  const float4 a = (bit & 8) ? ((bit & 4) ? c[3] : c[2]) : ((bit & 4) ? c[1] : c[0]);
  return (bit & 2) ? ((bit & 1) ? a.w : a.z) : ((bit & 1) ? a.y : a.x);
}

// The (k+1)-th largest of the 32 lane values (k < 32; NaN lanes count as -inf).
__device__ __forceinline__ float warp_kth_largest(float v, int k, int lane) {
  if (k >= 32) return -__int_as_float(0x7f800000);
  v = (v == v) ? v : -__int_as_float(0x7f800000);
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride >= 1; stride >>= 1) {
      const float o = __shfl_xor_sync(kFull, v, stride);
      const bool desc = (lane & size) == 0 || size == 32;
      const bool low = (lane & stride) == 0;
      const float mx = fmaxf(v, o), mn = fminf(v, o);
      v = (low == desc) ? mx : mn;
    }
  }
  return __shfl_sync(kFull, v, k);
}

// Descending bitonic sort of one key per lane.
__device__ __forceinline__ uint64_t sort32_desc(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride >= 1; stride >>= 1) {
      const uint64_t o = shfl64_xor(v, stride);
      const bool desc = (lane & size) == 0 || size == 32;
      const bool low = (lane & stride) == 0;
      const uint64_t mx = v > o ? v : o, mn = v > o ? o : v;
      v = (low == desc) ? mx : mn;
    }
  }
  return v;
}

// Streaming top-M of one warp. Candidates above the current threshold are
// appended to a per-warp shared-memory buffer; every 32 buffered keys are
// sorted and merged into the register-resident list in one bitonic merge.
//
// Threshold: any value below the M-th largest key seen so far by the whole
// block can be dropped. Two lower bounds of that key are kept in a block-shared
// maximum: each warp's own M-th key, and the smallest of the warps' q-th keys,
// q = ceil(M / warps) (every warp holds at least q keys at or above it, so the
// block holds at least M). The second tracks the block's M-th key about as if
// one warp had seen the whole segment, so few elements pass after a short start.
template <int SLOTS>
struct Select {
  WarpList<SLOTS> L;
  uint64_t tau;
  float tau_v;
  uint64_t *buf;                 // [kBuf] per warp
  unsigned long long *s_tau;     // block-wide threshold
  unsigned long long *s_wq;      // [warps] each warp's q-th key
  int cnt, M, qi, lane, warp;
  bool bad;

  __device__ __forceinline__ void set_tau(uint64_t t) {
    tau = t;
    tau_v = (t == 0ull) ? -__int_as_float(0x7f800000) : key_value(t);
  }
  __device__ __forceinline__ void sync_tau() {
    const uint64_t sh = *reinterpret_cast<volatile unsigned long long *>(s_tau);
    if (sh > tau) set_tau(sh);
  }
  __device__ __forceinline__ void merge_batch(uint64_t k) {
    WarpList<SLOTS> b;
    b.clear();
    b.v[0] = sort32_desc(k, lane);
    L.merge(b, lane);
    const uint64_t own = L.at(M - 1);
    const uint64_t qk = L.at(qi);
    if (lane == 0) reinterpret_cast<volatile unsigned long long *>(s_wq)[warp] = qk;
    __syncwarp();
    uint64_t mn = (lane < kTopmWarps) ? reinterpret_cast<volatile unsigned long long *>(s_wq)[lane]
                                      : ~0ull;
#pragma unroll
    for (int o = 4; o; o >>= 1) {
      const uint64_t y = shfl64_xor(mn, o);
      mn = y < mn ? y : mn;
    }
    mn = shfl64(mn, 0);
    const uint64_t best = own > mn ? own : mn;
    if (best != 0ull) {
      if (lane == 0) atomicMax(s_tau, static_cast<unsigned long long>(best));
      if (best > tau) set_tau(best);
    }
  }
  // one candidate per lane: keys above the threshold are appended to the
  // buffer; the merges happen in drain(), after every four pushes (keeping the
  // merge code out of the per-element path keeps the kernel small enough for
  // the instruction cache)
  __device__ __forceinline__ void push(float v, uint32_t id, bool valid) {
    bad |= valid && !(v < __int_as_float(0x7f800000));
    const uint64_t key = make_key(v, id);
    const bool pass = valid && (v >= tau_v) && key > tau;
    const unsigned m = __ballot_sync(kFull, pass);
    if (pass) buf[cnt + __popc(m & ((1u << lane) - 1u))] = key;
    cnt += __popc(m);
  }
  // merge full batches of 32, taken from the end of the buffer
  __device__ __forceinline__ void drain() {
    __syncwarp();
    while (cnt >= 32) {
      const uint64_t k = buf[cnt - 32 + lane];
      cnt -= 32;
      __syncwarp();
      merge_batch(k);
    }
  }
  __device__ __forceinline__ void flush() {
    __syncwarp();
    if (cnt > 0) {
      const uint64_t k = (lane < cnt) ? buf[lane] : 0ull;
      cnt = 0;
      __syncwarp();
      merge_batch(k);
    }
  }
};

template <int SLOTS>
__device__ void block_merge_lists(uint64_t *lists /* [8][MP] */, int warp, int lane) {
  constexpr int MP = SLOTS * 32;
  for (int step = 1; step < kTopmWarps; step <<= 1) {
    __syncthreads();
    if ((warp % (2 * step)) == 0) {
      WarpList<SLOTS> a, b;
      a.load(lists + warp * MP, MP, lane, false);
      b.load(lists + (warp + step) * MP, MP, lane, false);
      a.merge(b, lane);
      __syncwarp();
      a.store(lists + warp * MP, lane);
    }
  }
  __syncthreads();
}

// Top-M keys of float4 units [u0, u1) of a row's aligned part (element
// a0 + 4u + c), plus the scalar head [0, a0) when `head` and the tail
// [a0 + 4 nv, V) when `tail`, by all warps of the block. The block's M best
// keys end in lists[0, M) (sorted, 0 past the end); a NaN or +inf sets
// kReqFlagNonfinite in *flag.
template <int SLOTS>
__device__ void block_topm(const float *rowp, int V, int M, int a0, int nv, int u0, int u1,
                           bool head, bool tail, uint64_t *lists, uint64_t *bufs,
                           unsigned long long *s_tau_p, unsigned long long *s_wq, int *flag) {
  constexpr int MP = SLOTS * 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long &s_tau = *s_tau_p;
  if (threadIdx.x == 0) s_tau = 0ull;
  if (threadIdx.x < kTopmWarps) s_wq[threadIdx.x] = 0ull;
  __syncthreads();
  const int cnt = u1 - u0;
  const int w0 = u0 + static_cast<int>(static_cast<long long>(warp) * cnt / kTopmWarps);
  const int w1 = u0 + static_cast<int>(static_cast<long long>(warp + 1) * cnt / kTopmWarps);

  Select<SLOTS> st;
  st.L.clear();
  st.M = M;
  st.qi = (M + kTopmWarps - 1) / kTopmWarps - 1;
  st.lane = lane;
  st.warp = warp;
  st.s_wq = s_wq;
  st.bad = false;
  st.cnt = 0;
  st.buf = bufs + warp * kBuf;
  st.s_tau = &s_tau;
  st.set_tau(0ull);

  // kQ float4 per lane per tile; two register tiles alternate so that the next
  // tile's loads are in flight while this one is filtered
  const float4 *vec = reinterpret_cast<const float4 *>(rowp + a0);
  auto load_tile = [&](float4 (&dst)[kQ], int b) {
    if (b + kQ * 32 <= w1) {                     // warp-uniform: a full tile
#pragma unroll
      for (int q = 0; q < kQ; ++q) dst[q] = __ldcs(vec + b + q * 32 + lane);
    } else {
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int u = b + q * 32 + lane;
        dst[q] = (u < w1) ? __ldcs(vec + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  auto filter_tile = [&](const float4 (&c)[kQ], int b) {
    const bool full = b + kQ * 32 <= w1;
    st.sync_tau();
    // NaN-propagating maximum: a NaN (or +inf) forces the slow path, where
    // push() flags it; -inf is an ordinary (masked) value
    bool any = false;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const bool ok = full || b + q * 32 + lane < w1;
      const float m4 = fmax_nan(fmax_nan(c[q].x, c[q].y), fmax_nan(c[q].z, c[q].w));
      any |= ok && !(m4 < st.tau_v);
    }
    if (__any_sync(kFull, any)) {
      // only the elements at or above the threshold (or NaN): one push round
      // per element of the busiest lane, usually one or two
      uint32_t mask = 0u;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        if (full || b + q * 32 + lane < w1) {
          mask |= (!(c[q].x < st.tau_v) ? 1u : 0u) << (4 * q + 0);
          mask |= (!(c[q].y < st.tau_v) ? 1u : 0u) << (4 * q + 1);
          mask |= (!(c[q].z < st.tau_v) ? 1u : 0u) << (4 * q + 2);
          mask |= (!(c[q].w < st.tau_v) ? 1u : 0u) << (4 * q + 3);
        }
      }
      while (__any_sync(kFull, mask != 0u)) {
        const bool has = mask != 0u;
        const int bit = has ? __ffs(mask) - 1 : 0;
        mask &= mask - 1u;
        const int u = b + (bit >> 2) * 32 + lane;
        st.push(pick16(c, bit), static_cast<uint32_t>(a0 + 4 * u + (bit & 3)), has);
        if (st.cnt > kBuf - 32) st.drain();
      }
      st.drain();
    }
  };
  float4 ta[kQ], tb[kQ];
  load_tile(ta, w0);
  // starting threshold from the first tile of every warp: the q-th largest of
  // a warp's lane maxima is a value that at least q of its elements reach, so
  // the smallest such value over the warps is reached by at least M elements
  // of the block and nothing below it can be among the block's top M
  {
    const float ninf = -__int_as_float(0x7f800000);
    float lm = ninf;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      if (w0 + q * 32 + lane < w1)
        lm = fmaxf(lm, fmaxf(fmaxf(ta[q].x, ta[q].y), fmaxf(ta[q].z, ta[q].w)));
    }
    const float t = warp_kth_largest(lm, st.qi, lane);
    if (lane == 0) s_wq[warp] = static_cast<unsigned long long>(__float_as_uint(t));
    __syncthreads();
    float t0 = __uint_as_float(static_cast<uint32_t>(s_wq[0]));
#pragma unroll
    for (int w = 1; w < kTopmWarps; ++w)
      t0 = fminf(t0, __uint_as_float(static_cast<uint32_t>(s_wq[w])));
    __syncthreads();
    if (threadIdx.x < kTopmWarps) s_wq[threadIdx.x] = 0ull;
    // key of (t0, largest id): every element of value t0 or more passes
    if (t0 > ninf && st.qi < 32) st.set_tau(make_key(t0, 0xffffffffu));
    __syncthreads();
  }
  for (int base = w0; base < w1; base += 2 * kQ * 32) {
    const int b2 = base + kQ * 32;
    if (b2 < w1) load_tile(tb, b2);
    filter_tile(ta, base);
    if (b2 >= w1) break;
    if (b2 + kQ * 32 < w1) load_tile(ta, b2 + kQ * 32);
    filter_tile(tb, b2);
  }
  // scalar head and tail, warp 0
  if (warp == 0) {
    if (head && a0 > 0) {
      bool ok = lane < a0;
      st.push(ok ? __ldg(rowp + lane) : 0.f, static_cast<uint32_t>(lane), ok);
    }
    const int t0 = a0 + 4 * nv;
    if (tail && t0 < V) {
      bool ok = t0 + lane < V;
      st.push(ok ? __ldg(rowp + t0 + lane) : 0.f, static_cast<uint32_t>(t0 + lane), ok);
    }
    st.drain();
  }
  st.flush();
  if (__any_sync(kFull, st.bad) && lane == 0) atomicOr(flag, kReqFlagNonfinite);

  st.L.store(lists + warp * MP, lane);
  block_merge_lists<SLOTS>(lists, warp, lane);
}

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
    const int a0 = min(V, static_cast<int>((4 - (row_base & 3)) & 3));
    const int nv = (V - a0) >> 2;
    const int u0 = static_cast<int>(static_cast<long long>(split) * nv / maxpieces);
    const int u1 = static_cast<int>(static_cast<long long>(split + 1) * nv / maxpieces);
    block_topm<SLOTS>(rowp, V, M, a0, nv, u0, u1, split == 0, split == maxpieces - 1, lists,
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
    block_topm<SLOTS>(rowp, V, M, 0, nv, u0, u1, false, false, lists, bufs, &s_tau, s_wq,
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
