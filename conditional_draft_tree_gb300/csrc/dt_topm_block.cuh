// dt_topm_block.cuh -- block-level top-M selection over a range of one row
// (the top-M kernel of dt_topm.cu), in building blocks: a warp's streaming
// selection, the starting threshold, the tile filter and the block merge.
//
// "Riassunto Tecnico: DominoTree", Componenti Core 2: the correction is only
// evaluated on the top-M marginal candidates of each depth, the M token ids of
// largest base logit, ordered (logit desc, id asc). Every warp streams its
// part of the range with 128-bit loads and keeps a sorted top-M list of 64-bit
// (order(value), ~id) keys in registers; a candidate touches the list only when
// it beats the current threshold, which after the first few hundred elements
// is rare. The eight warp lists of a block are combined with bitonic merges.
#pragma once

#include <cstdint>

#include "dt_common.cuh"
#include "dt_internal.h"

namespace dt {
namespace {

constexpr int kTopmThreads = 256;
constexpr int kTopmWarps = kTopmThreads / 32;
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

// element `bit` (0..4Q-1) of Q float4 registers (Q = 4 or 8), without local memory
template <int Q>
__device__ __forceinline__ float pick_elem(const float4 (&c)[Q], int bit) {
  float4 a;
  if constexpr (Q == 4) {
    a = (bit & 8) ? ((bit & 4) ? c[3] : c[2]) : ((bit & 4) ? c[1] : c[0]);
  } else {
    static_assert(Q == 8, "tiles of 4 or 8 float4 per lane");
    const float4 lo = (bit & 8) ? ((bit & 4) ? c[3] : c[2]) : ((bit & 4) ? c[1] : c[0]);
    const float4 hi = (bit & 8) ? ((bit & 4) ? c[7] : c[6]) : ((bit & 4) ? c[5] : c[4]);
    a = (bit & 16) ? hi : lo;
  }
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

// ------------------------------------------------- block-level building blocks
// All warps of a block take part; each keeps a Select whose list the block
// merges at the end.

// A Select for this warp, threshold tau0 (0: none); s_tau / s_wq zeroed.
template <int SLOTS>
__device__ __forceinline__ void select_begin(Select<SLOTS> &st, int M, uint64_t *bufs,
                                             unsigned long long *s_tau,
                                             unsigned long long *s_wq, uint64_t tau0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) *s_tau = tau0;
  if (threadIdx.x < kTopmWarps) s_wq[threadIdx.x] = 0ull;
  __syncthreads();
  st.L.clear();
  st.M = M;
  st.qi = (M + kTopmWarps - 1) / kTopmWarps - 1;
  st.lane = lane;
  st.warp = warp;
  st.s_wq = s_wq;
  st.bad = false;
  st.cnt = 0;
  st.buf = bufs + warp * kBuf;
  st.s_tau = s_tau;
  st.set_tau(tau0);
}

// This lane's maximum over a tile's elements (units b + q*32 + lane < end;
// NaN ignored), folded into lm.
template <int Q>
__device__ __forceinline__ void tile_max(float &lm, const float4 (&c)[Q], int b, int end,
                                         int lane) {
#pragma unroll
  for (int q = 0; q < Q; ++q)
    if (b + q * 32 + lane < end)
      lm = fmaxf(lm, fmaxf(fmaxf(c[q].x, c[q].y), fmaxf(c[q].z, c[q].w)));
}

// Starting threshold from every lane's maximum lm over some of its elements:
// the q-th largest of a warp's lane maxima is a value that at least q of its
// elements reach, so the smallest such value over the warps is reached by at
// least M elements of the block and nothing below it can be among the block's
// top M. Block-wide.
template <int SLOTS>
__device__ __forceinline__ void start_threshold(Select<SLOTS> &st, float lm,
                                                unsigned long long *s_wq) {
  const float ninf = -__int_as_float(0x7f800000);
  const float t = warp_kth_largest(lm, st.qi, st.lane);
  if (st.lane == 0) s_wq[st.warp] = static_cast<unsigned long long>(__float_as_uint(t));
  __syncthreads();
  float t0 = __uint_as_float(static_cast<uint32_t>(s_wq[0]));
#pragma unroll
  for (int w = 1; w < kTopmWarps; ++w)
    t0 = fminf(t0, __uint_as_float(static_cast<uint32_t>(s_wq[w])));
  __syncthreads();
  if (threadIdx.x < kTopmWarps) s_wq[threadIdx.x] = 0ull;
  // key of (t0, largest id): every element of value t0 or more passes
  if (t0 > ninf && st.qi < 32) {
    const uint64_t k0 = make_key(t0, 0xffffffffu);
    if (k0 > st.tau) st.set_tau(k0);
  }
  __syncthreads();
}

// One tile of Q float4 per lane (units b + q*32 + lane, those < end; element
// ids a0 + 4u + c): the elements at or above the threshold are pushed. Warp-wide.
template <int SLOTS, int Q>
__device__ __forceinline__ void filter_tile(Select<SLOTS> &st, const float4 (&c)[Q], int b,
                                            int end, int a0) {
  const int lane = st.lane;
  const bool full = b + Q * 32 <= end;
  st.sync_tau();
  // NaN-propagating maximum: a NaN (or +inf) forces the slow path, where
  // push() flags it; -inf is an ordinary (masked) value. gm: the float4
  // groups of this lane with an element at or above the threshold.
  uint32_t gm = 0u;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const bool ok = full || b + q * 32 + lane < end;
    const float m4 = fmax_nan(fmax_nan(c[q].x, c[q].y), fmax_nan(c[q].z, c[q].w));
    gm |= (ok && !(m4 < st.tau_v)) ? (1u << q) : 0u;
  }
  const uint32_t gor = __reduce_or_sync(kFull, gm);
  if (gor == 0u) return;
  // only the elements at or above the threshold (or NaN): the element bits of
  // a group are formed only where some lane's group passes (a warp-uniform
  // branch), then one push round per element of the busiest lane, usually one
  // or two
  uint32_t mask = 0u;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if ((gor >> q) & 1u) {
      uint32_t e = 0u;
      e |= !(c[q].x < st.tau_v) ? 1u : 0u;
      e |= !(c[q].y < st.tau_v) ? 2u : 0u;
      e |= !(c[q].z < st.tau_v) ? 4u : 0u;
      e |= !(c[q].w < st.tau_v) ? 8u : 0u;
      mask |= ((gm >> q) & 1u) ? (e << (4 * q)) : 0u;
    }
  }
  while (__any_sync(kFull, mask != 0u)) {
    const bool has = mask != 0u;
    const int bit = has ? __ffs(mask) - 1 : 0;
    mask &= mask - 1u;
    const int u = b + (bit >> 2) * 32 + lane;
    st.push(pick_elem<Q>(c, bit), static_cast<uint32_t>(a0 + 4 * u + (bit & 3)), has);
    if (st.cnt > kBuf - 32) st.drain();
  }
  st.drain();
}

// The scalar head [0, a0) (if `head`) and tail [a0 + 4 nv, V) (if `tail`) by
// warp 0, the last merges, the non-finite flag, and the block merge: the M
// best keys end in lists[0, M). Block-wide.
template <int SLOTS>
__device__ __forceinline__ void select_finish(Select<SLOTS> &st, const float *rowp, int V,
                                              int a0, int nv, bool head, bool tail,
                                              uint64_t *lists, int *flag) {
  constexpr int MP = SLOTS * 32;
  const int lane = st.lane, warp = st.warp;
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

// Top-M keys of float4 units [u0, u1) of a row's aligned part (element
// a0 + 4u + c), plus the scalar head [0, a0) when `head` and the tail
// [a0 + 4 nv, V) when `tail`, by all warps of the block: each warp streams a
// contiguous share with Q float4 per lane per register tile, two tiles in
// flight. Keys at or below `tau0` (0: none; a lower bound of the row's M-th
// key known from elsewhere) are skipped. The block's M best keys above tau0
// end in lists[0, M) (sorted, 0 past the end); a NaN or +inf sets
// kReqFlagNonfinite in *flag.
template <int SLOTS, int Q>
__device__ void block_topm(const float *rowp, int V, int M, int a0, int nv, int u0, int u1,
                           bool head, bool tail, uint64_t *lists, uint64_t *bufs,
                           unsigned long long *s_tau, unsigned long long *s_wq, int *flag,
                           uint64_t tau0 = 0ull) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Select<SLOTS> st;
  select_begin(st, M, bufs, s_tau, s_wq, tau0);
  const int cnt = u1 - u0;
  const int w0 = u0 + static_cast<int>(static_cast<long long>(warp) * cnt / kTopmWarps);
  const int w1 = u0 + static_cast<int>(static_cast<long long>(warp + 1) * cnt / kTopmWarps);
  const float4 *vec = reinterpret_cast<const float4 *>(rowp + a0);
  auto load_tile = [&](float4 (&dst)[Q], int b) {
    if (b + Q * 32 <= w1) {                     // warp-uniform: a full tile
#pragma unroll
      for (int q = 0; q < Q; ++q) dst[q] = __ldcs(vec + b + q * 32 + lane);
    } else {
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int u = b + q * 32 + lane;
        dst[q] = (u < w1) ? __ldcs(vec + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  // the starting threshold is taken over the first two tiles of every warp
  // (both in registers before the loop; the second is not loaded again)
  float4 ta[Q], tb[Q];
  load_tile(ta, w0);
  float lm = -__int_as_float(0x7f800000);
  tile_max(lm, ta, w0, w1, lane);
  if (w0 + Q * 32 < w1) {
    load_tile(tb, w0 + Q * 32);
    tile_max(lm, tb, w0 + Q * 32, w1, lane);
  }
  start_threshold(st, lm, s_wq);
  for (int base = w0; base < w1; base += 2 * Q * 32) {
    const int b2 = base + Q * 32;
    if (b2 < w1 && base != w0) load_tile(tb, b2);
    filter_tile(st, ta, base, w1, a0);
    if (b2 >= w1) break;
    if (b2 + Q * 32 < w1) load_tile(ta, b2 + Q * 32);
    filter_tile(st, tb, b2, w1, a0);
  }
  select_finish(st, rowp, V, a0, nv, head, tail, lists, flag);
}

}  // namespace
}  // namespace dt
