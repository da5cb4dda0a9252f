// dt_verify.cu -- verify-side consumption of a draft tree: position ids of
// the tree rows and tree attention under the ancestor mask.
//
// "Riassunto Tecnico: DominoTree", Componenti Core 5: the target model checks
// every drafted node in one forward pass with tree attention, each node seeing
// the verified prefix and its own ancestors, through the ancestor mask the
// builder emits. The target model is not part of this library; these kernels
// take its per-layer Q, K, V (synthetic in the tests and the benchmark).
//
// Positions: the prefix cache holds the prefix_len tokens before the anchor;
// the anchor is tree row 0 at position prefix_len and a node at depth j sits at
// prefix_len + j (empty rows: -1).
//
// Attention: one block per (request, query head), 8 warps; a warp owns up to
// kQW query rows of a pass. Keys stream in chunks of 32 (one per lane) through
// shared memory as fp32, the next chunk's global loads in flight while the
// current one is used. Scores are q . k over the head dimension (each lane one
// key), masked by visibility (prefix key p < prefix_len, tree key t iff
// mask[row][t]), then an online softmax per row (running max and sum, warp
// reductions) and the weighted sum of values (each lane 64/32 ... dh/32 output
// dims). bf16 Q/K/V, fp32 arithmetic and output. CUDA cores (FFMA): the work per
// request and layer is small and irregular (65 rows of a 64-node tree).
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "dt_common.cuh"
#include "dt_internal.h"

namespace dt {

namespace {

constexpr int kVThreads = 256;
constexpr int kQW = 9;                  // query rows per warp and pass (72 per pass)
constexpr int kRows = 8 * kQW;

struct TreeAttnArgs {
  const uint16_t *q, *k, *v;
  const uint8_t *mask;
  const int32_t *prefix_len;
  int H, Hkv, n1, P;
  float scale;
  float *out;
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 x, float *dst) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dst[2 * i] = __uint_as_float(w[i] << 16);
    dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// DPL consecutive floats at p (p is DPL * 4-byte aligned: float4 steps when
// DPL is a multiple of 4, one float2 when DPL is 2)
template <int DPL>
__device__ __forceinline__ void load_dpl(const float *p, float (&v)[DPL]) {
  static_assert(DPL == 2 || DPL % 4 == 0, "dims per lane");
  if constexpr (DPL == 2) {
    const float2 x = *reinterpret_cast<const float2 *>(p);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int e = 0; e < DPL; e += 4) {
      const float4 x = *reinterpret_cast<const float4 *>(p + e);
      v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
    }
  }
}
template <int DPL>
__device__ __forceinline__ void store_dpl(float *p, const float (&v)[DPL]) {
  static_assert(DPL == 2 || DPL % 4 == 0, "dims per lane");
  if constexpr (DPL == 2) {
    *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int e = 0; e < DPL; e += 4)
      *reinterpret_cast<float4 *>(p + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
  }
}

// this thread's share of the K and V rows [c0, c0 + 32) (zeros past L)
template <int U, int C8, int DH>
__device__ __forceinline__ void fetch_chunk(const uint16_t *kb, const uint16_t *vb, int c0, int L,
                                            uint4 (&pk)[U], uint4 (&pv)[U]) {
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const int u = threadIdx.x + j * kVThreads, key = u / C8, c8 = u - key * C8;
    const int jj = c0 + key;
    pk[j] = make_uint4(0u, 0u, 0u, 0u);
    pv[j] = make_uint4(0u, 0u, 0u, 0u);
    if (jj < L) {
      pk[j] = *reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(jj) * DH + c8 * 8);
      pv[j] = *reinterpret_cast<const uint4 *>(vb + static_cast<size_t>(jj) * DH + c8 * 8);
    }
  }
}

template <int DPL>
__global__ void __launch_bounds__(kVThreads) tree_attention_kernel(TreeAttnArgs a) {
  constexpr int DH = 32 * DPL;          // head dimension
  constexpr int KS = DH + 4;            // K row stride: conflict-free 16-byte reads by lane
  constexpr int C8 = DH / 8;            // 16-byte units per row
  constexpr int U = 32 * C8 / kVThreads;  // units per thread per chunk (K, and V)
  static_assert(U >= 1, "head dimension too small");
  extern __shared__ __align__(16) float sm[];
  float *sK = sm;                       // [32][KS]
  float *sV = sK + 32 * KS;             // [32][DH]
  float *sQ = sV + 32 * DH;             // [kRows][DH]
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = h / (a.H / a.Hkv);
  const int L = a.P + a.n1;
  const int plen = min(max(a.prefix_len[b], 0), a.P);
  const uint16_t *kb = a.k + (static_cast<size_t>(b) * a.Hkv + hk) * L * DH;
  const uint16_t *vb = a.v + (static_cast<size_t>(b) * a.Hkv + hk) * L * DH;
  const uint16_t *qb = a.q + (static_cast<size_t>(b) * a.H + h) * a.n1 * DH;
  float *ob = a.out + (static_cast<size_t>(b) * a.H + h) * a.n1 * DH;
  const uint8_t *mb = a.mask + static_cast<size_t>(b) * a.n1 * a.n1;
  const float ninf = -__int_as_float(0x7f800000);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

  for (int pass = 0; pass < a.n1; pass += kRows) {
    __syncthreads();   // the previous pass is done with sQ
    for (int u = threadIdx.x; u < kRows * C8; u += kVThreads) {
      const int row = u / C8, c8 = u - row * C8, r = pass + row;
      const uint4 x = r < a.n1 ? *reinterpret_cast<const uint4 *>(qb + static_cast<size_t>(r) * DH + c8 * 8)
                               : zero;
      bf16x8_to_f32(x, sQ + row * DH + c8 * 8);
    }
    float m[kQW], l[kQW], o[kQW][DPL];
#pragma unroll
    for (int qq = 0; qq < kQW; ++qq) {
      m[qq] = ninf;
      l[qq] = 0.0f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[qq][e] = 0.0f;
    }
    uint4 pk[U], pv[U];
    fetch_chunk<U, C8, DH>(kb, vb, 0, L, pk, pv);
    for (int c0 = 0; c0 < L; c0 += 32) {
      __syncthreads();   // the previous chunk is consumed (and sQ staged)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int u = threadIdx.x + j * kVThreads, key = u / C8, c8 = u - key * C8;
        bf16x8_to_f32(pk[j], sK + key * KS + c8 * 8);
        bf16x8_to_f32(pv[j], sV + key * DH + c8 * 8);
      }
      __syncthreads();
      if (c0 + 32 < L) fetch_chunk<U, C8, DH>(kb, vb, c0 + 32, L, pk, pv);
      // scores of key c0 + lane for the warp's rows
      float s[kQW];
#pragma unroll
      for (int qq = 0; qq < kQW; ++qq) s[qq] = 0.0f;
#pragma unroll 4
      for (int d = 0; d < DH; d += 4) {
        const float4 k4 = *reinterpret_cast<const float4 *>(sK + lane * KS + d);
#pragma unroll
        for (int qq = 0; qq < kQW; ++qq) {
          const float4 q4 = *reinterpret_cast<const float4 *>(sQ + (warp + 8 * qq) * DH + d);
          s[qq] = fmaf(q4.x, k4.x, s[qq]);
          s[qq] = fmaf(q4.y, k4.y, s[qq]);
          s[qq] = fmaf(q4.z, k4.z, s[qq]);
          s[qq] = fmaf(q4.w, k4.w, s[qq]);
        }
      }
      const int j = c0 + lane;
      float p[kQW];
#pragma unroll
      for (int qq = 0; qq < kQW; ++qq) {
        p[qq] = 0.0f;
        const int r = pass + warp + 8 * qq;
        if (r >= a.n1) continue;   // warp-uniform
        const bool vis = j < L && (j < a.P ? j < plen : mb[static_cast<size_t>(r) * a.n1 + (j - a.P)] != 0);
        const float x = vis ? s[qq] * a.scale : ninf;
        const float mc = warp_max(x);
        if (mc == ninf) continue;  // no visible key in this chunk (warp-uniform)
        const float mn = fmaxf(m[qq], mc);
        const float alpha = expf(m[qq] - mn);   // 0 while nothing was seen
        p[qq] = vis ? expf(x - mn) : 0.0f;
        l[qq] = l[qq] * alpha + warp_sum(p[qq]);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[qq][e] *= alpha;
        m[qq] = mn;
      }
      // weighted values: lane owns output dims [DPL lane, DPL lane + DPL)
#pragma unroll 4
      for (int kk = 0; kk < 32; ++kk) {
        float vv[DPL];
        load_dpl<DPL>(sV + kk * DH + lane * DPL, vv);
#pragma unroll
        for (int qq = 0; qq < kQW; ++qq) {
          const float w = __shfl_sync(kFull, p[qq], kk);
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[qq][e] = fmaf(w, vv[e], o[qq][e]);
        }
      }
    }
#pragma unroll
    for (int qq = 0; qq < kQW; ++qq) {
      const int r = pass + warp + 8 * qq;
      if (r >= a.n1) continue;
      const float inv = l[qq] > 0.0f ? 1.0f / l[qq] : 0.0f;
      float w[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) w[e] = o[qq][e] * inv;
      store_dpl<DPL>(ob + static_cast<size_t>(r) * DH + lane * DPL, w);
    }
  }
}

__global__ void tree_positions_kernel(const int32_t *depths, const int32_t *prefix_len,
                                      int batch, int n1, int32_t *pos) {
  const size_t total = static_cast<size_t>(batch) * n1;
  for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int d = depths[e];
    pos[e] = d >= 0 ? prefix_len[e / n1] + d : -1;
  }
}

template <int DPL>
size_t attn_smem() {
  constexpr int DH = 32 * DPL;
  return sizeof(float) * (32 * (DH + 4) + 32 * DH + kRows * DH);
}

template <int DPL>
cudaError_t launch_attn(const TreeAttnArgs &a, int batch, cudaStream_t st) {
  const size_t smem = attn_smem<DPL>();
  cudaError_t e = cudaFuncSetAttribute(tree_attention_kernel<DPL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  tree_attention_kernel<DPL><<<dim3(a.H, batch), kVThreads, smem, st>>>(a);
  return cudaGetLastError();
}

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

}  // namespace dt

extern "C" {

int dt_tree_positions(const int32_t *depths, const int32_t *prefix_len, int batch, int n1,
                      int32_t *positions, void *stream) {
  if (!depths || !prefix_len || !positions || batch < 1 || n1 < 1 || n1 > DT_MAX_N + 1 ||
      !dt::al4(depths) || !dt::al4(prefix_len) || !dt::al4(positions))
    return DT_ERR_INVALID_ARG;
  const size_t total = static_cast<size_t>(batch) * n1;
  const int grid = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  dt::tree_positions_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      depths, prefix_len, batch, n1, positions);
  return cudaGetLastError() == cudaSuccess ? DT_OK : DT_ERR_CUDA;
}

int dt_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const uint8_t *mask, const int32_t *prefix_len, int batch, int H, int Hkv,
                      int n1, int P, int dh, float scale, float *out, void *stream) {
  if (!q || !k || !v || !mask || !prefix_len || !out) return DT_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || H < 1 || Hkv < 1 || H % Hkv || n1 < 1 ||
      n1 > DT_MAX_N + 1 || P < 0 || P > (1 << 24) || !(dh == 64 || dh == 128 || dh == 256) ||
      !std::isfinite(scale))
    return DT_ERR_INVALID_ARG;
  if (!dt::al16(q) || !dt::al16(k) || !dt::al16(v) || !dt::al16(out) || !dt::al4(prefix_len))
    return DT_ERR_INVALID_ARG;
  dt::TreeAttnArgs a;
  a.q = q; a.k = k; a.v = v; a.mask = mask; a.prefix_len = prefix_len;
  a.H = H; a.Hkv = Hkv; a.n1 = n1; a.P = P; a.scale = scale; a.out = out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = dh == 64 ? dt::launch_attn<2>(a, batch, st)
                : dh == 128 ? dt::launch_attn<4>(a, batch, st)
                            : dt::launch_attn<8>(a, batch, st);
  return e == cudaSuccess ? DT_OK : DT_ERR_CUDA;
}

}  // extern "C"
