// dt_common.cuh -- device helpers shared by the kernels of libdt.so.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dt {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- weights
// Weights arrive as fp32 or as raw bf16 bit patterns; both decode exactly to fp32.

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Eight consecutive weights starting at element `i` of row pointer `p` into f[8].
// Requires 16-byte alignment of p + i (bf16) or of p + i and p + i + 4 (fp32).
template <int WDT>
__device__ __forceinline__ void load8(const void *p, size_t i, float f[8]);

template <>
__device__ __forceinline__ void load8<0>(const void *p, size_t i, float f[8]) {
  const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
  float4 a = __ldg(q), b = __ldg(q + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<1>(const void *p, size_t i, float f[8]) {
  uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + i));
  f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xffff0000u);
}

template <int WDT>
__device__ __forceinline__ float load1(const void *p, size_t i) {
  if (WDT == 1) return bf16_bits_to_float(static_cast<const uint16_t *>(p)[i]);
  return static_cast<const float *>(p)[i];
}

// ------------------------------------------------------------ ordering keys
// 64-bit key whose unsigned order is (value desc, id asc) when sorted
// descending: high word = order-preserving image of the fp32 value (-0 folded
// onto +0), low word = ~id. Key 0 is below every real key.

__device__ __forceinline__ uint32_t float_order_bits(float v) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float order_bits_float(uint32_t o) {
  uint32_t b = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(b);
}

__device__ __forceinline__ uint64_t make_key(float v, uint32_t id) {
  return (static_cast<uint64_t>(float_order_bits(v)) << 32) | static_cast<uint64_t>(~id);
}
__device__ __forceinline__ uint32_t key_id(uint64_t k) { return ~static_cast<uint32_t>(k); }
__device__ __forceinline__ float key_value(uint64_t k) {
  return order_bits_float(static_cast<uint32_t>(k >> 32));
}

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src, unsigned mask = kFull) {
  uint32_t lo = __shfl_sync(mask, static_cast<uint32_t>(v), src);
  uint32_t hi = __shfl_sync(mask, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64_xor(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64_up(uint64_t v, int d) {
  uint32_t lo = __shfl_up_sync(kFull, static_cast<uint32_t>(v), d);
  uint32_t hi = __shfl_up_sync(kFull, static_cast<uint32_t>(v >> 32), d);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// ----------------------------------------------------------------- timing

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_acquire_s32(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_u32(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded grid-wide barrier for a cooperative launch of `nblocks` blocks. The
// counter only grows: barrier number i completes when it reaches i * nblocks
// (`target`, advanced by every call, wrap-safe). A block that failed locally
// (`fail`) raises *abort and does not arrive; a wait longer than `limit_ns`, or
// one that sees *abort, returns false. Never traps or spins forever.
// `skip_arrival` (failure-detection tests only) waits without arriving.
__device__ __forceinline__ bool grid_barrier(unsigned *count, int *abort, unsigned nblocks,
                                             uint64_t limit_ns, unsigned &target, bool fail,
                                             bool skip_arrival = false) {
  __shared__ int s_ok;
  target += nblocks;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (fail) {
      atomicExch(abort, 1);
      ok = 0;
    } else {
      if (!skip_arrival) red_release_add_u32(count, 1u);
      uint64_t t0 = 0;
      for (unsigned spins = 0;; ++spins) {
        if (static_cast<int>(ld_acquire_u32(count) - target) >= 0) break;
        if ((spins & 31u) == 31u) {
          if (ld_acquire_s32(abort)) { ok = 0; break; }
          const uint64_t now = global_ns();
          if (spins == 31u) {
            t0 = now;
          } else if (now - t0 > limit_ns) {
            atomicExch(abort, 1);
            ok = 0;
            break;
          }
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Asynchronous prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Full descending bitonic sort of 32*SLOTS keys held slot-major in a warp.
template <int SLOTS>
__device__ __forceinline__ void warp_sort_desc(uint64_t v[SLOTS], int lane) {
  constexpr int n = 32 * SLOTS;
#pragma unroll
  for (int size = 2; size <= n; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride >= 1; stride >>= 1) {
      if (stride >= 32) {
        const int ds = stride >> 5;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          if ((s & ds) == 0) {
            const int i = s * 32 + lane;
            const bool desc = (i & size) == 0;
            uint64_t a = v[s], b = v[s + ds];
            bool sw = desc ? (a < b) : (a > b);
            v[s] = sw ? b : a;
            v[s + ds] = sw ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
          const int i = s * 32 + lane;
          const bool desc = (i & size) == 0;
          uint64_t o = shfl64_xor(v[s], stride);
          const bool low = (lane & stride) == 0;
          // lower index keeps the larger key in a descending run
          const bool keep_max = (low == desc);
          uint64_t mx = v[s] > o ? v[s] : o, mn = v[s] > o ? o : v[s];
          v[s] = keep_max ? mx : mn;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ math

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

}  // namespace dt
