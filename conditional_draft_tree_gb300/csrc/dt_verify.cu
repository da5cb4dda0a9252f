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
// Attention on the tensor cores (tcgen05): one block of eight warps per
// (request, key/value head, tile of 128 query rows), where the rows of the
// H / Hkv query heads that share the key/value head are stacked (head-major),
// so K and V are staged once for all of them; TMEM lane t is query row t of
// the tile, and threads t and t + 128 own it, each for half of every chunk's
// keys (and half of the output columns): two threads per row double the
// resident warps at the same shared memory, the bound of this latency-bound
// kernel. Keys are taken in chunks of 64: the visible
// prefix [0, prefix_len) and the tree rows (prefix keys past prefix_len are
// never read). One pass over the chunks with an online softmax: S = Q K^T
// (bf16 operands, exact products, fp32 accumulation in TMEM); the row's
// reference maximum m follows the running maximum of x = scale S, moved only
// when the chunk maximum exceeds it by more than 8 (then O in TMEM and l are
// rescaled); e = exp(x - m) (0 where not visible) as two bf16 terms hi + lo
// (16 significant bits), O += e_hi V + e_lo V in TMEM, l += e; and out = O / l
// (0 for a row that sees no key). Operands are staged in
// shared memory in the K-major no-swizzle layout of dt_umma.cuh: Q and the
// key chunk as they are stored, V transposed (head dimension as rows). One
// thread issues the MMAs; completion is an mbarrier commit, every wait bounded.
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "dt_common.cuh"
#include "dt_internal.h"
#include "dt_umma.cuh"

namespace dt {

namespace {

constexpr int kAThreads = 256;         // two threads per query row of a tile
constexpr int kHalf = 32;               // keys of a chunk per thread
constexpr int kKeys = 64;               // keys per chunk (the S tile's N)
constexpr uint64_t kAttnLimitNs = 2000000000ull;

struct TreeAttnArgs {
  const uint16_t *q, *k, *v;
  const uint8_t *mask;
  const int32_t *prefix_len;
  int H, Hkv, n1, P;
  float scale;
  float *out;
};

// TMEM columns of the block: O (DH columns) at 0, S (kKeys) after it, rounded
// up to a power of two
template <int DH>
__host__ __device__ constexpr uint32_t attn_tmem_cols() {
  return DH + kKeys <= 128 ? 128u : (DH + kKeys <= 256 ? 256u : 512u);
}
template <int DH>
__host__ __device__ constexpr int attn_smem_bytes() {
  // Q tile, K chunk, V^T chunk, e in two terms
  return 128 * DH * 2 + kKeys * DH * 2 + DH * kKeys * 2 + 2 * 128 * kKeys * 2;
}

template <int DH>
__global__ void __launch_bounds__(kAThreads) tree_attention_kernel(TreeAttnArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ float s_ml[2][128];         // the key-half-1 threads' (m, l) per row
  unsigned char *sQ = sm;                              // [128 rows][DH], K-major
  unsigned char *sK = sQ + 128 * DH * 2;               // [kKeys rows][DH]
  unsigned char *sV = sK + kKeys * DH * 2;             // [DH rows][kKeys] (V^T)
  unsigned char *sE = sV + DH * kKeys * 2;             // 2 x [128 rows][kKeys]
  const int tid = threadIdx.x, warp = tid >> 5;
  const int row = tid & 127, half = tid >> 7;   // TMEM lane; keys [32 half, 32 half + 32)
  const int mt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int G = a.H / a.Hkv, rows = G * a.n1;
  const int L = a.P + a.n1;
  const int plen = min(max(a.prefix_len[b], 0), a.P);
  const uint16_t *kb = a.k + (static_cast<size_t>(b) * a.Hkv + hk) * L * DH;
  const uint16_t *vb = a.v + (static_cast<size_t>(b) * a.Hkv + hk) * L * DH;
  const uint8_t *mb = a.mask + static_cast<size_t>(b) * a.n1 * a.n1;
  // this thread's query row
  const int g = mt * 128 + row;
  const bool mine = g < rows;
  const int h = hk * G + (mine ? g / a.n1 : 0), qr = mine ? g % a.n1 : 0;
  const float ninf = -__int_as_float(0x7f800000);

  if (tid == 0) {
    mbar_init(&s_bar, 1);
    s_fail = 0;
  }
  if (warp == 0) tmem_alloc(&s_tmem, attn_tmem_cols<DH>());
  // Q tile: 16-byte pieces in place (rows past the group are zeros)
  constexpr int C8 = DH / 8;
  for (int u = tid; u < 128 * C8; u += kAThreads) {
    const int r = u / C8, c8 = u - r * C8, gr = mt * 128 + r;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (gr < rows) {
      const int hh = hk * G + gr / a.n1, rr = gr % a.n1;
      x = *reinterpret_cast<const uint4 *>(
          a.q + ((static_cast<size_t>(b) * a.H + hh) * a.n1 + rr) * DH + c8 * 8);
    }
    *reinterpret_cast<uint4 *>(sQ + umma_offset(r, c8 * 8, DH)) = x;
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t t_o = tmem, t_s = tmem + DH;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;   // lanes of row
  const uint32_t idesc_s = umma_idesc_bf16(128, kKeys), idesc_o = umma_idesc_bf16(128, DH);
  // chunks: the visible prefix, then the tree rows
  const int npre = (plen + kKeys - 1) / kKeys, ntree = (a.n1 + kKeys - 1) / kKeys;
  const int nch = npre + ntree;
  uint32_t phase = 0;
  auto chunk_first = [&](int c) { return c < npre ? c * kKeys : a.P + (c - npre) * kKeys; };
  auto chunk_end = [&](int c) { return c < npre ? plen : a.P + a.n1; };
  // visibility of key j (within [first, end)) for this thread's row
  auto visible = [&](int j) {
    return j < a.P ? j < plen : mb[static_cast<size_t>(qr) * a.n1 + (j - a.P)] != 0;
  };
  // key chunk c in registers: unit i of this thread is key 32 (warp & 1) + lane
  // of the chunk, 16-byte piece c8 = (warp >> 1) + NWP i (a warp covers 32
  // consecutive keys, so the transposed V stores of a warp spread over banks);
  // rows past the chunk's end are zeros
  constexpr int UPT = kKeys * C8 / kAThreads;   // pieces per thread: 4 (DH 128)
  constexpr int NWP = kAThreads / 64;           // warp pairs
  static_assert(kKeys == 64 && UPT * kAThreads == kKeys * C8, "piece mapping");
  uint4 pk[UPT], pv[UPT];
  const int my_key = 32 * (warp & 1) + (tid & 31);
  auto fetch = [&](int c, bool with_v) {
    const int j = chunk_first(c) + my_key;
    const bool in = j < chunk_end(c);
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      const int c8 = (warp >> 1) + NWP * i;
      pk[i] = in ? *reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(j) * DH + c8 * 8)
                 : make_uint4(0u, 0u, 0u, 0u);
      pv[i] = (in && with_v)
                  ? *reinterpret_cast<const uint4 *>(vb + static_cast<size_t>(j) * DH + c8 * 8)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // the fetched chunk into shared memory (K as is, V transposed)
  auto stage = [&](bool with_v) {
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      const int c8 = (warp >> 1) + NWP * i;
      *reinterpret_cast<uint4 *>(sK + umma_offset(my_key, c8 * 8, DH)) = pk[i];
      if (with_v) {
        const uint32_t w[4] = {pv[i].x, pv[i].y, pv[i].z, pv[i].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint16_t x = static_cast<uint16_t>((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu));
          *reinterpret_cast<uint16_t *>(sV + umma_offset(c8 * 8 + e, my_key, kKeys)) = x;
        }
      }
    }
    fence_async_smem();   // plain stores -> tensor-core reads
  };
  // one thread issues, everyone waits for the commit (bounded)
  auto mma_wait = [&]() {
    if (!mbar_wait(&s_bar, phase, kAttnLimitNs)) s_fail = 1;
    phase ^= 1u;
    tmem_fence_after();
  };
  auto issue_s = [&]() {
    if (tid == 0) {
      tmem_fence_after();
#pragma unroll
      for (int k = 0; k < DH / 16; ++k)
        umma_bf16(t_s, umma_desc(smem_u32(sQ) + k * 256, 128, 16 * DH),
                  umma_desc(smem_u32(sK) + k * 256, 128, 16 * DH), idesc_s, k > 0);
      umma_commit(&s_bar);
    }
  };
  // this thread's half of its row of S for chunk c, scaled, -inf where not visible
  auto row_scores = [&](int c, float (&x)[kHalf]) {
    tmem_ld32(t_s + lane_off + kHalf * half, x);
    tmem_wait_ld();
    const int j0 = chunk_first(c) + kHalf * half, j1 = chunk_end(c);
#pragma unroll
    for (int t = 0; t < kHalf; ++t) {
      const int j = j0 + t;
      x[t] = (mine && j < j1 && visible(j)) ? x[t] * a.scale : ninf;
    }
  };

  // One pass, online softmax. Per chunk: S = Q K_c^T; the row's chunk maximum
  // (the two half-row threads exchange theirs); when it exceeds the row's
  // reference maximum m by more than kRescale, O and l are rescaled to the new
  // maximum (O in TMEM by tcgen05.ld / st, after the previous chunk's O
  // product has completed), otherwise m stays and e stays below exp(kRescale);
  // e = exp(x - m) as two bf16 terms (hi + lo), O += e V_c. The first chunk's
  // product initialises O, so no row is ever rescaled from unwritten TMEM.
  constexpr float kRescale = 8.0f;
  float m = ninf, l = 0.0f;   // row reference maximum; this thread's half of l
  fetch(0, true);
  for (int c = 0; c < nch && !s_fail; ++c) {
    stage(true);   // sK, sV free: S and O of chunk c - 1 were waited for
    tmem_fence_before();
    __syncthreads();
    issue_s();
    if (c + 1 < nch) fetch(c + 1, true);
    mma_wait();    // S of chunk c (and O of chunk c - 1 before it)
    float x[kHalf];
    row_scores(c, x);
    float mc = ninf;
#pragma unroll
    for (int t = 0; t < kHalf; ++t) mc = fmaxf(mc, x[t]);
    s_ml[half][row] = mc;
    __syncthreads();
    mc = fmaxf(mc, s_ml[half ^ 1][row]);
    // both threads of a row take the same decision from the same values
    const bool grow = mc > m + kRescale || (m == ninf && mc != ninf);
    float f = 1.0f;
    if (grow) {
      f = (m == ninf) ? 0.0f : expf(m - mc);
      l *= f;
      m = mc;
    }
    // O follows (chunk 0's product has not written it yet); tcgen05.ld / st
    // are warp-wide, so a warp with one growing row rescales all its rows,
    // the others by 1
    if (c > 0 && __any_sync(kFull, grow)) {
#pragma unroll 1
      for (int c0 = (DH / 2) * half; c0 < (DH / 2) * (half + 1); c0 += 32) {
        float o[32];
        tmem_ld32(t_o + lane_off + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] *= f;
        tmem_st32(t_o + lane_off + c0, o);
      }
      tmem_wait_st();
    }
#pragma unroll
    for (int t0 = 0; t0 < kHalf; t0 += 8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float ev[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
          ev[z] = (x[t0 + e + z] == ninf) ? 0.0f : expf(x[t0 + e + z] - m);
          l += ev[z];
        }
        const __nv_bfloat16 h0 = __float2bfloat16_rn(ev[0]), h1 = __float2bfloat16_rn(ev[1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(ev[0] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(ev[1] - __bfloat162float(h1));
        hi[e >> 1] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                     (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lo[e >> 1] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                     (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
      }
      *reinterpret_cast<uint4 *>(sE + umma_offset(row, kHalf * half + t0, kKeys)) =
          make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(sE + 128 * kKeys * 2 + umma_offset(row, kHalf * half + t0, kKeys)) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_async_smem();
    tmem_fence_before();
    __syncthreads();   // e in sE, O rescaled, S read: O += e V
    if (tid == 0) {
      tmem_fence_after();
#pragma unroll
      for (int term = 0; term < 2; ++term)
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          umma_bf16(t_o,
                    umma_desc(smem_u32(sE) + term * 128 * kKeys * 2 + k * 256, 128, 16 * kKeys),
                    umma_desc(smem_u32(sV) + k * 256, 128, 16 * kKeys), idesc_o,
                    c > 0 || term > 0 || k > 0);
      umma_commit(&s_bar);
    }
    mma_wait();    // O of chunk c: sE, sV, sK free
  }
  // the row's l: the sum of its two halves (both taken against the same m)
  s_ml[half][row] = l;
  __syncthreads();
  l += s_ml[half ^ 1][row];
  // out = O / l
  if (!s_fail && nch > 0) {
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    float *ob = a.out + ((static_cast<size_t>(b) * a.H + h) * a.n1 + qr) * DH;
#pragma unroll 1
    for (int c0 = (DH / 2) * half; c0 < (DH / 2) * (half + 1); c0 += 32) {
      float o[32];
      tmem_ld32(t_o + lane_off + c0, o);
      tmem_wait_ld();
      if (mine) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4 *>(ob + c0 + e) =
              make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
      }
    }
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  if (warp == 0) tmem_dealloc(tmem, attn_tmem_cols<DH>());
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

template <int DH>
cudaError_t launch_attn(const TreeAttnArgs &a, int batch, cudaStream_t st) {
  constexpr int smem = attn_smem_bytes<DH>();
  cudaError_t e = cudaFuncSetAttribute(tree_attention_kernel<DH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = (a.H / a.Hkv) * a.n1;
  tree_attention_kernel<DH><<<dim3((rows + 127) / 128, a.Hkv, batch), kAThreads, smem, st>>>(a);
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
  cudaError_t e = dh == 64 ? dt::launch_attn<64>(a, batch, st)
                : dh == 128 ? dt::launch_attn<128>(a, batch, st)
                            : dt::launch_attn<256>(a, batch, st);
  return e == cudaSuccess ? DT_OK : DT_ERR_CUDA;
}

}  // extern "C"
