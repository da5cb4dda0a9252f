// dt_decode.cu -- Domino chain decoding: one draft token per position along a
// single path, with the GRU correction over the whole vocabulary.
//
// "Domino：在投机解码中将因果建模与自回归草稿解耦", method steps (inference): the
// parallel backbone gives the base logits L_base^i; the Domino head updates the
// causal state from the previously drawn draft token, forms the correction and
// draws each draft token from the corrected logits. Core method: S_{i-1} =
// GRU(E_{<=i-1}), dL_i = W2 SiLU(W1 [H_i; S_{i-1}]), L_i = L_base^i + dL_i.
// "Riassunto Tecnico: DominoTree", Definizione del Problema: the released Domino
// decoder follows this single chain. Readings shared with the tree builder: the
// root state is GRU(state0, E[anchor]); GRU gates r, z, n; the temperature
// divides the corrected logits. T = 0 takes the argmax (lowest id on ties);
// T > 0 draws by the inverse CDF of softmax(L / T) in token-id order at a
// uniform number the caller passes in.
//
// One persistent cooperative launch per wave of requests, one block per SM,
// grid barriers between phases. Per draft position i:
//   A. state GEMM y = [W_hh; W1_S] S_{i-1} on the tensor cores. A operand:
//      128-row weight tiles, prepared once in the operand layout (64-wide K
//      chunks of 16 KB); B operand: the fp32 states split into three bf16
//      terms (hi, mid, lo), so the products are those of the fp32 states.
//      Items = (row tile, 256-wide K range); partial sums per K range.
//   C. vocabulary GEMM W2 h over every token, same operand scheme (W2 tiles
//      streamed by bulk copies through a 4-stage ring, h's three terms as B),
//      two TMEM accumulators so that the epilogue of one tile overlaps the
//      MMAs of the next. The epilogue sums the three terms, adds L_base,
//      divides by T and reduces every 32-token group to (max, sum of exp,
//      first argmax); the logits themselves are not stored.
//   D. per request: combine the groups, take the token (argmax, or the group
//      where the CDF passes u Z and then the token in it, the group's 32
//      logits recomputed from h and their W2 rows), its log-probability, then
//      the GRU step S_i = GRU(S_{i-1}, E[d_i]) from the prepared input table G
//      and the recurrent half from A.
// Block roles: warps 0-7 build B operands, run epilogues, sampling and the GRU;
// warp 8 lane 0 issues the bulk copies, warp 9 lane 0 the MMAs. Every wait is
// bounded; a timeout aborts the launch with DT_ERR_TIMEOUT for its requests.
#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>

#include "dt_common.cuh"
#include "dt_internal.h"
#include "dt_umma.cuh"

namespace dt {

namespace {

constexpr int kDThreads = 320;
constexpr int kWork = 256;                          // threads of warps 0-7
constexpr int kProd = 256, kMma = 288;              // issuing threads
constexpr int kChunkK = 64;                         // K columns per A chunk
constexpr uint32_t kChunkBytes = 128 * kChunkK * 2; // 16 KB
// vocabulary epilogue: per work warp, x of 8 requests x 32 tokens (rows padded
// to 33 floats, so the transposed reads hit 32 different banks)
constexpr int kRedRow = 33;
constexpr int kRedBytes = (kWork / 32) * 8 * kRedRow * 4;
constexpr int kStages = 4;
constexpr int kRangeK = 256;                        // K columns of one state-GEMM item
constexpr int kMaxBpad = 80;                        // 3 terms x 80 = 240 accumulator columns
constexpr uint32_t kAccCols = 256;                  // TMEM columns per accumulator
constexpr uint64_t kLimitNs = 2000000000ull;        // 2 s per wait
constexpr int kKzBatch = 8;                         // K-range partials loaded together

struct DecodeParams {
  int V, d, d_s, r, D;
  int b0, nb, bpad, N;          // wave: requests [b0, b0 + nb), bpad rows per B term, N = 3 bpad
  int R;                        // 3 d_s + r
  int n_tA, nchA, n_kz;         // state GEMM: row tiles, K chunks per tile, K ranges
  int n_tV, nchV;               // vocabulary GEMM: tiles, K chunks per tile
  int kb;                       // K width of the B buffer layout
  int Gn;                       // 32-token groups (n_tV * 4)
  const unsigned char *wall, *w2;
  const float *G, *b_hh, *U, *base, *state0, *temperature, *uniforms;
  const int32_t *anchor;
  const uint16_t *W2;           // [V][r] bf16 bits, the caller's W2 (the sampled group's logits)
  float *ypart, *S, *st_m, *st_s;
  int32_t *st_a;
  int *flags;
  Ctrl *ctrl;
  int32_t *tokens;
  float *logprobs;
  int32_t *status;
};

// Counters of the copy ring and the accumulators. Every thread advances them
// identically, so each role knows the stage, buffer and parity of each item.
struct Pipe {
  uint32_t g;   // A chunks issued so far
  uint32_t q;   // items so far
};

__device__ __forceinline__ bool bad_temperature(float T) {
  return !(T >= 0.0f) || T == __int_as_float(0x7f800000);
}

// Writes 8 consecutive K values (k0 = 8 kg) of B row b in the three term
// blocks of the operand (term t at rows t * bpad + b), K-major layout of width kb.
__device__ __forceinline__ void put_b8(unsigned char *sB, const DecodeParams &p, int b, int kg,
                                       const float v[8]) {
  uint16_t t0[8], t1[8], t2[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) split3(v[j], t0[j], t1[j], t2[j]);
  const uint16_t *src[3] = {t0, t1, t2};
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    uint4 q;
    q.x = src[t][0] | (static_cast<uint32_t>(src[t][1]) << 16);
    q.y = src[t][2] | (static_cast<uint32_t>(src[t][3]) << 16);
    q.z = src[t][4] | (static_cast<uint32_t>(src[t][5]) << 16);
    q.w = src[t][6] | (static_cast<uint32_t>(src[t][7]) << 16);
    *reinterpret_cast<uint4 *>(sB + umma_offset(t * p.bpad + b, kg * 8, p.kb)) = q;
  }
}

// Copies and MMAs of one item: `nch` A chunks from `a_src` (contiguous 16 KB
// chunks) times B columns [0, 64 nch) into accumulator buffer q & 1.
__device__ void issue_item(const DecodeParams &p, const unsigned char *a_src, int nch,
                           unsigned char *ring, uint32_t sB_addr, uint64_t *full, uint64_t *empty,
                           uint64_t *accf, uint64_t *acce, uint32_t tmem, const Pipe &pp,
                           volatile int *fail) {
  if (threadIdx.x == kProd) {
    for (int c = 0; c < nch; ++c) {
      const uint32_t g = pp.g + c, s = g % kStages;
      if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) - 1) & 1u, kLimitNs)) {
        *fail = 1;
        break;
      }
      mbar_expect_tx(&full[s], kChunkBytes);
      bulk_g2s(ring + s * kChunkBytes, a_src + static_cast<size_t>(c) * kChunkBytes, kChunkBytes,
               &full[s]);
    }
  } else if (threadIdx.x == kMma) {
    const uint32_t buf = pp.q & 1u;
    if (pp.q >= 2 && !mbar_wait(&acce[buf], ((pp.q >> 1) - 1) & 1u, kLimitNs)) *fail = 1;
    tmem_fence_after();
    const uint32_t d_addr = tmem + buf * kAccCols;
    const uint32_t idesc = umma_idesc_bf16(128, p.N);
    for (int c = 0; c < nch && !*fail; ++c) {
      const uint32_t g = pp.g + c, s = g % kStages;
      if (!mbar_wait(&full[s], (g / kStages) & 1u, kLimitNs)) {
        *fail = 1;
        break;
      }
      tmem_fence_after();
      const uint32_t a0 = smem_u32(ring + s * kChunkBytes);
#pragma unroll
      for (int kk = 0; kk < kChunkK / 16; ++kk)
        umma_bf16(d_addr, umma_desc(a0 + kk * 256, 128, 16 * kChunkK),
                  umma_desc(sB_addr + (c * (kChunkK / 16) + kk) * 256, 128, 16u * p.kb), idesc,
                  c > 0 || kk > 0);
      umma_commit(&empty[s]);
    }
    umma_commit(&accf[buf]);
  }
}

// Epilogue entry: waits for the item's accumulator; false on timeout.
__device__ __forceinline__ bool wait_acc(uint64_t *accf, const Pipe &pp) {
  const bool ok = mbar_wait(&accf[pp.q & 1u], (pp.q >> 1) & 1u, kLimitNs);
  tmem_fence_after();
  return ok;
}

__device__ __forceinline__ void release_acc(uint64_t *acce, const Pipe &pp) {
  tmem_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&acce[pp.q & 1u]);
}

// --------------------------------------------------------- A. state GEMM

__device__ bool state_gemm(const DecodeParams &p, unsigned char *ring, unsigned char *sB,
                           uint64_t *full, uint64_t *empty, uint64_t *accf, uint64_t *acce,
                           uint32_t tmem, Pipe &pp, int *s_fail) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_tA * p.n_kz;
  bool ok = true;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int kz = it / p.n_tA, t = it - kz * p.n_tA;
    // B: the states' K range [256 kz, 256 kz + 256), zero past d_s and nb
    if (threadIdx.x < kWork) {
      constexpr int kU = 4;   // units of 8 K values per thread with loads in flight together
      const int units = p.bpad * (kRangeK / 8);
      for (int u0 = threadIdx.x; u0 < units; u0 += kU * kWork) {
        float4 x[kU][2];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          const int u = u0 + j * kWork;
          const int b = u / (kRangeK / 8), kg = u - b * (kRangeK / 8);
          const int k0 = kz * kRangeK + kg * 8;
          x[j][0] = x[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (u < units && b < p.nb && k0 < p.d_s) {
            const float4 *src =
                reinterpret_cast<const float4 *>(p.S + static_cast<size_t>(b) * p.d_s + k0);
            x[j][0] = __ldcg(src);
            x[j][1] = __ldcg(src + 1);
          }
        }
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          const int u = u0 + j * kWork;
          if (u >= units) break;
          const int b = u / (kRangeK / 8), kg = u - b * (kRangeK / 8);
          const float v[8] = {x[j][0].x, x[j][0].y, x[j][0].z, x[j][0].w,
                              x[j][1].x, x[j][1].y, x[j][1].z, x[j][1].w};
          put_b8(sB, p, b, kg, v);
        }
      }
    }
    fence_async_smem();
    __syncthreads();
    const int c0 = kz * (kRangeK / kChunkK);
    const int nch = min(kRangeK / kChunkK, p.nchA - c0);
    issue_item(p, p.wall + (static_cast<size_t>(t) * p.nchA + c0) * kChunkBytes, nch, ring,
               smem_u32(sB), full, empty, accf, acce, tmem, pp, s_fail);
    if (threadIdx.x < kWork) {
      ok &= wait_acc(accf, pp);
      const int quarter = warp & 3, half = warp >> 2, hb = p.bpad >> 1;
      const int row = t * 128 + quarter * 32 + lane;
      const uint32_t ta = tmem + ((quarter * 32u) << 16) + (pp.q & 1u) * kAccCols;
      for (int b0 = half * hb; b0 < (half + 1) * hb; b0 += 8) {
        float a[8], m[8], l[8];
        tmem_ld8(ta + b0, a);
        tmem_ld8(ta + p.bpad + b0, m);
        tmem_ld8(ta + 2 * p.bpad + b0, l);
        tmem_wait_ld();
        if (row < p.R) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (b0 + j < p.nb)
              p.ypart[(static_cast<size_t>(kz) * p.bpad + b0 + j) * p.R + row] = (a[j] + m[j]) + l[j];
        }
      }
      release_acc(acce, pp);
    }
    pp.g += nch;
    pp.q += 1;
    __syncthreads();   // the next item rebuilds B
  }
  return ok;
}

// ---------------------------------------------------- C. vocabulary GEMM

__device__ bool vocab_gemm(const DecodeParams &p, int i, unsigned char *ring, unsigned char *sB,
                           uint64_t *full, uint64_t *empty, uint64_t *accf, uint64_t *acce,
                           uint32_t tmem, Pipe &pp, int *s_fail, const float *s_T,
                           float *s_red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rp8 = p.nchV * (kChunkK / 8);
  // B: h = SiLU(U_i + W1_S S) in three terms, K padded with zeros to 64 nchV
  if (threadIdx.x < kWork) {
    for (int u = threadIdx.x; u < p.bpad * rp8; u += kWork) {
      const int b = u / rp8, kg = u - b * rp8, k0 = kg * 8;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
      if (b < p.nb && k0 < p.r) {
        const float4 *U = reinterpret_cast<const float4 *>(
            p.U + (static_cast<size_t>(p.b0 + b) * p.D + i) * p.r + k0);
        float acc[8];
        const float4 u0 = __ldg(U), u1 = __ldg(U + 1);
        acc[0] = u0.x; acc[1] = u0.y; acc[2] = u0.z; acc[3] = u0.w;
        acc[4] = u1.x; acc[5] = u1.y; acc[6] = u1.z; acc[7] = u1.w;
        // W1_S S: the K-range partial sums, in K-range order (kKzBatch loads in flight)
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int kz0 = 0; kz0 < p.n_kz; kz0 += kKzBatch) {
          float4 q[kKzBatch][2];
#pragma unroll
          for (int z = 0; z < kKzBatch; ++z) {
            if (kz0 + z < p.n_kz) {
              const float4 *src = reinterpret_cast<const float4 *>(
                  p.ypart + (static_cast<size_t>(kz0 + z) * p.bpad + b) * p.R + 3 * p.d_s + k0);
              q[z][0] = __ldcg(src);
              q[z][1] = __ldcg(src + 1);
            } else {
              q[z][0] = q[z][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int z = 0; z < kKzBatch; ++z) {
            if (kz0 + z >= p.n_kz) break;
            s[0] += q[z][0].x; s[1] += q[z][0].y; s[2] += q[z][0].z; s[3] += q[z][0].w;
            s[4] += q[z][1].x; s[5] += q[z][1].y; s[6] += q[z][1].z; s[7] += q[z][1].w;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = siluf_(acc[j] + s[j]);
      }
      put_b8(sB, p, b, kg, v);
    }
  }
  fence_async_smem();
  __syncthreads();
  bool ok = true;
  const float ninf = -__int_as_float(0x7f800000);
  // Each work warp owns 32 tokens of a tile (its TMEM lane quarter, one 32-token
  // group) and half of the requests. The base logits of a tile's requests are
  // loaded together, one tile ahead, so that their HBM latency overlaps the
  // previous tile. The group records are reduced transposed: the warp writes x
  // of 8 requests x 32 tokens to shared memory, then four lanes per request
  // scan 8 tokens each (maximum, sum of exp, first argmax) and combine by two
  // exchanges, instead of two 32-lane reductions per request.
  constexpr int kHalf = kMaxBpad / 2;
  const int quarter = warp & 3, half = warp >> 2, hb = p.bpad >> 1;
  const int my0 = half * hb;
  const int myn = max(0, min(hb, p.nb - my0));
  float pre[kHalf];
  auto load_base = [&](int tt) {
    const int v = tt * 128 + quarter * 32 + lane;
    const bool in = v < p.V;
    const float *src = p.base + (static_cast<size_t>(p.b0 + my0) * p.D + i) * p.V + v;
    const size_t step = static_cast<size_t>(p.D) * p.V;
#pragma unroll
    for (int j = 0; j < kHalf; ++j)
      pre[j] = (in && j < myn) ? __ldcs(src + j * step) : 0.0f;
  };
  if (threadIdx.x < kWork && blockIdx.x < p.n_tV) load_base(blockIdx.x);
  for (int t = blockIdx.x; t < p.n_tV; t += gridDim.x) {
    issue_item(p, p.w2 + static_cast<size_t>(t) * p.nchV * kChunkBytes, p.nchV, ring,
               smem_u32(sB), full, empty, accf, acce, tmem, pp, s_fail);
    if (threadIdx.x < kWork) {
      ok &= wait_acc(accf, pp);
      float cur[kHalf];
#pragma unroll
      for (int j = 0; j < kHalf; ++j) cur[j] = pre[j];
      if (t + static_cast<int>(gridDim.x) < p.n_tV) load_base(t + gridDim.x);
      const int v = t * 128 + quarter * 32 + lane;
      const int grp = t * 4 + quarter;
      const bool valid = v < p.V;
      const uint32_t ta = tmem + ((quarter * 32u) << 16) + (pp.q & 1u) * kAccCols;
      float *xr = s_red + warp * (8 * kRedRow);
      const int vg = t * 128 + quarter * 32;   // first token of the group
#pragma unroll
      for (int c = 0; c < kHalf; c += 8) {
        if (c >= myn) break;
        float a[8], m[8], l[8];
        tmem_ld8(ta + my0 + c, a);
        tmem_ld8(ta + p.bpad + my0 + c, m);
        tmem_ld8(ta + 2 * p.bpad + my0 + c, l);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = ninf;
          if (c + j < myn && valid) {
            const int b = my0 + c + j;
            const float bv = cur[c + j];
            if (bv != bv || bv == __int_as_float(0x7f800000)) atomicOr(&p.flags[b], 1);
            x = __fdiv_rn(bv + ((a[j] + m[j]) + l[j]), s_T[b]);
          }
          xr[j * kRedRow + lane] = x;
        }
        __syncwarp();
        // request c + jr: lanes 4 jr .. 4 jr + 3, tokens t0 .. t0 + 7 each
        const int jr = lane >> 2, t0 = (lane & 3) * 8;
        float xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) xv[u] = xr[jr * kRedRow + t0 + u];
        float mx = xv[0];
#pragma unroll
        for (int u = 1; u < 8; ++u) mx = fmaxf(mx, xv[u]);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        float sum = 0.0f;
        int first = 32;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sum += (xv[u] == ninf) ? 0.0f : expf(xv[u] - mx);
          if (first == 32 && vg + t0 + u < p.V && xv[u] == mx) first = t0 + u;
        }
        sum += __shfl_xor_sync(kFull, sum, 1);
        sum += __shfl_xor_sync(kFull, sum, 2);
        first = min(first, __shfl_xor_sync(kFull, first, 1));
        first = min(first, __shfl_xor_sync(kFull, first, 2));
        if ((lane & 3) == 0 && c + jr < myn) {
          const size_t o = static_cast<size_t>(my0 + c + jr) * p.Gn + grp;
          p.st_m[o] = mx;
          p.st_s[o] = sum;
          p.st_a[o] = first < 32 ? grp * 32 + first : -1;
        }
        __syncwarp();   // the rows are written again for the next 8 requests
      }
      release_acc(acce, pp);
    }
    pp.g += p.nchV;
    pp.q += 1;
  }
  __syncthreads();
  return ok;
}

// -------------------------------------------- D. token choice and GRU step

// GRU step of request b from token `tok`: gh = sum of the K-range partials + b_hh.
__device__ void gru_request(const DecodeParams &p, int b, int tok) {
  const int ds = p.d_s;
  const float *gi = p.G + static_cast<size_t>(tok) * 3 * ds;
  for (int k = threadIdx.x; k < ds; k += kWork) {
    const float gir = __ldg(gi + k), giz = __ldg(gi + ds + k), gin = __ldg(gi + 2 * ds + k);
    float *sp = p.S + static_cast<size_t>(b) * ds + k;
    const float old = __ldcg(sp);
    float gh[3] = {0.f, 0.f, 0.f};
    // the K-range partial sums of the three gates, in K-range order
    for (int kz0 = 0; kz0 < p.n_kz; kz0 += kKzBatch) {
      float q[kKzBatch][3];
#pragma unroll
      for (int z = 0; z < kKzBatch; ++z)
#pragma unroll
        for (int g = 0; g < 3; ++g)
          q[z][g] = kz0 + z < p.n_kz
                        ? __ldcg(p.ypart + (static_cast<size_t>(kz0 + z) * p.bpad + b) * p.R + g * ds + k)
                        : 0.0f;
#pragma unroll
      for (int z = 0; z < kKzBatch; ++z) {
        if (kz0 + z >= p.n_kz) break;
#pragma unroll
        for (int g = 0; g < 3; ++g) gh[g] += q[z][g];
      }
    }
#pragma unroll
    for (int g = 0; g < 3; ++g) gh[g] += p.b_hh ? p.b_hh[g * ds + k] : 0.0f;
    const float rr = sigmoidf_(gir + gh[0]);
    const float z = sigmoidf_(giz + gh[1]);
    const float n = tanhf(gin + rr * gh[2]);
    __stcg(sp, (1.0f - z) * n + z * old);
  }
}

// Token of position i for request b (one block), then its GRU step. The
// request's group records are first copied into `stage` (the W2 ring, idle in
// this phase) by coalesced loads when they fit, so that the passes below, in
// which every thread walks its own contiguous range of groups, read shared
// memory instead of strided global words.
__device__ void choose_token(const DecodeParams &p, int i, int b, float *stage) {
  __shared__ float s_red[32];
  __shared__ float s_f[4];
  __shared__ int s_i[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool work = tid < kWork;
  const float ninf = -__int_as_float(0x7f800000);
  const int gb = p.b0 + b;
  const bool bad = p.flags[b] != 0 || bad_temperature(p.temperature ? p.temperature[gb] : 1.0f);
  const bool greedy = (p.temperature ? p.temperature[gb] : 1.0f) == 0.0f;
  const float *m = p.st_m + static_cast<size_t>(b) * p.Gn;
  const float *sg = p.st_s + static_cast<size_t>(b) * p.Gn;
  const bool staged = 2 * p.Gn <= static_cast<int>(kStages * kChunkBytes / 4);
  float *sm_m = stage, *sm_s = stage + p.Gn;
  if (staged) {
    for (int u = tid; u < p.Gn; u += kDThreads) {
      sm_m[u] = __ldcg(m + u);
      sm_s[u] = __ldcg(sg + u);
    }
    __syncthreads();
  }
  // group record g (the records are rewritten at every position: global reads bypass L1)
  auto ld_m = [&](int g) { return staged ? sm_m[g] : __ldcg(m + g); };
  auto ld_s = [&](int g) { return staged ? sm_s[g] : __ldcg(sg + g); };
  const int cpt = (p.Gn + kWork - 1) / kWork;
  const int g0 = work ? min(p.Gn, tid * cpt) : p.Gn, g1 = min(p.Gn, g0 + cpt);
  // 1. maximum, its first group, the last group with mass
  // a thread's group records are loaded kG at a time, all in flight together
  constexpr int kG = 24;
  float mt = ninf;
  int gt = 0x7fffffff, lastpos = -1;
  for (int gb0 = g0; gb0 < g1; gb0 += kG) {
    float mv[kG], sv[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      mv[j] = gb0 + j < g1 ? ld_m(gb0 + j) : ninf;
      sv[j] = gb0 + j < g1 ? ld_s(gb0 + j) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      if (gb0 + j >= g1) break;
      if (gt == 0x7fffffff || mv[j] > mt) { mt = mv[j]; gt = gb0 + j; }   // first group of the maximum
      if (sv[j] > 0.0f) lastpos = gb0 + j;
    }
  }
  // reduce (max, first group) and last positive group over the block
  for (int o = 16; o; o >>= 1) {
    const float mo = __shfl_xor_sync(kFull, mt, o);
    const int go = __shfl_xor_sync(kFull, gt, o);
    if (mo > mt || (mo == mt && go < gt)) { mt = mo; gt = go; }
    lastpos = max(lastpos, __shfl_xor_sync(kFull, lastpos, o));
  }
  __shared__ float s_wm[kDThreads / 32];
  __shared__ int s_wg[kDThreads / 32], s_wl[kDThreads / 32];
  if (lane == 0) { s_wm[warp] = mt; s_wg[warp] = gt; s_wl[warp] = lastpos; }
  __syncthreads();
  if (tid == 0) {
    float M = s_wm[0];
    int gm = s_wg[0], lp = s_wl[0];
    for (int w = 1; w < kWork / 32; ++w) {
      if (s_wm[w] > M || (s_wm[w] == M && s_wg[w] < gm)) { M = s_wm[w]; gm = s_wg[w]; }
      lp = max(lp, s_wl[w]);
    }
    s_f[0] = M; s_i[0] = gm; s_i[1] = lp;
  }
  __syncthreads();
  const float M = s_f[0];
  const int gmax = s_i[0], glast = s_i[1];
  // 2. Z = sum over groups of s_g e^{m_g - M}, per thread then over the block
  float zt = 0.0f;
  if (M != ninf)
    for (int gb0 = g0; gb0 < g1; gb0 += kG) {
      float mv[kG], sv[kG];
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        mv[j] = gb0 + j < g1 ? ld_m(gb0 + j) : ninf;
        sv[j] = gb0 + j < g1 ? ld_s(gb0 + j) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kG; ++j)
        if (mv[j] != ninf) zt += sv[j] * expf(mv[j] - M);
    }
  // exclusive scan of the thread sums (id order) and the total
  float incl = zt;
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  float wbase = 0.0f, Z = 0.0f;
  for (int w = 0; w < kWork / 32; ++w) {
    if (w < warp) wbase += s_red[w];
    Z += s_red[w];
  }
  const float P = wbase + incl - zt;   // mass of the groups before this thread's range
  const float lse = (M == ninf) ? ninf : M + logf(Z);
  int tok = 0;
  float lp = ninf;
  if (bad) {
    tok = 0;
    lp = __int_as_float(0x7fc00000);
  } else if (M == ninf) {
    tok = 0;
  } else if (greedy) {
    tok = __ldcg(p.st_a + static_cast<size_t>(b) * p.Gn + gmax);
    lp = M - lse;
  } else {
    float u = p.uniforms ? p.uniforms[static_cast<size_t>(gb) * p.D + i] : 0.0f;
    u = (u >= 0.0f) ? (u < 1.0f ? u : __int_as_float(0x3f7fffff)) : 0.0f;
    const float target = u * Z;
    // the last thread whose range starts at or below the target walks its groups
    if (tid == 0) s_i[2] = 0;
    __syncthreads();
    if (work && P <= target) atomicMax(&s_i[2], tid);
    __syncthreads();
    if (tid == s_i[2]) {
      float cum = P;
      int gsel = -1;
      for (int gb0 = g0; gb0 < g1 && gsel < 0; gb0 += kG) {
        float mv[kG], sv[kG];
#pragma unroll
        for (int j = 0; j < kG; ++j) {
          mv[j] = gb0 + j < g1 ? ld_m(gb0 + j) : ninf;
          sv[j] = gb0 + j < g1 ? ld_s(gb0 + j) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kG; ++j) {
          const float w = (mv[j] == ninf) ? 0.0f : sv[j] * expf(mv[j] - M);
          if (gsel < 0 && gb0 + j < g1) {
            if (cum + w > target) gsel = gb0 + j;
            else cum += w;
          }
        }
      }
      s_i[3] = gsel >= 0 ? gsel : glast;
      s_f[1] = gsel >= 0 ? cum : __int_as_float(0x7f800000);   // +inf: take the last token with mass
    }
    __syncthreads();
    // the chosen group's 32 logits: (L_base + W2[v] . h) / T with h = SiLU(U_i
    // + W1_S S) of this request summed as the GEMM's B operand was (same
    // order), h in chunks of 256 in shared memory; fp32 products (the GEMM took
    // products of h's three bf16 terms: the same value to a few ulps, which
    // moves a choice only at a near tie)
    __shared__ float s_h[256];
    const int gsel = s_i[3];   // >= 0: the group holding the CDF crossing or the last one with mass
    const float before = s_f[1];
    const bool gok = gsel >= 0 && gsel < p.Gn;
    const int v = gok ? gsel * 32 + lane : p.V;   // (p.V: no token, nothing read)
    float dl = 0.0f;
    for (int k0 = 0; k0 < p.r; k0 += 256) {
      const int kn = min(256, p.r - k0);
      for (int k = tid; k < kn; k += kDThreads) {
        // the K-range partials in order, kKzBatch loads in flight
        const float *src = p.ypart + static_cast<size_t>(b) * p.R + 3 * p.d_s + k0 + k;
        const size_t zstep = static_cast<size_t>(p.bpad) * p.R;
        float acc = 0.0f;
        for (int kz0 = 0; kz0 < p.n_kz; kz0 += kKzBatch) {
          float q[kKzBatch];
#pragma unroll
          for (int z = 0; z < kKzBatch; ++z)
            q[z] = kz0 + z < p.n_kz ? __ldcg(src + (kz0 + z) * zstep) : 0.0f;
#pragma unroll
          for (int z = 0; z < kKzBatch; ++z)
            if (kz0 + z < p.n_kz) acc += q[z];
        }
        s_h[k] = siluf_(__ldg(p.U + (static_cast<size_t>(gb) * p.D + i) * p.r + k0 + k) + acc);
      }
      __syncthreads();
      if (warp == 0 && v < p.V) {
        const uint16_t *w = p.W2 + static_cast<size_t>(v) * p.r + k0;
#pragma unroll 4
        for (int k = 0; k < kn; k += 8) {
          const uint4 q = __ldg(reinterpret_cast<const uint4 *>(w + k));
          const uint32_t q4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            dl = fmaf(__uint_as_float(q4[t] << 16), s_h[k + 2 * t], dl);
            dl = fmaf(__uint_as_float(q4[t] & 0xffff0000u), s_h[k + 2 * t + 1], dl);
          }
        }
      }
      __syncthreads();
    }
    if (warp == 0) {
      float x = ninf;
      if (v < p.V) {
        const float bv = p.base[(static_cast<size_t>(gb) * p.D + i) * p.V + v];
        const float T = p.temperature ? p.temperature[gb] : 1.0f;
        x = __fdiv_rn(bv + dl, T);
      }
      const float e = (x == ninf) ? 0.0f : expf(x - M);
      float c = e;
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(kFull, c, o);
        if (lane >= o) c += y;
      }
      // before = +inf marks the fallback: the last token with mass
      const bool fallback = before == __int_as_float(0x7f800000);
      const unsigned crossing = __ballot_sync(kFull, before + c > target);
      const unsigned cross = fallback ? 0u : crossing;
      const unsigned pos = __ballot_sync(kFull, e > 0.0f);
      const int l = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
      const float xl = __shfl_sync(kFull, x, l);
      if (lane == 0) { s_i[3] = gsel * 32 + l; s_f[2] = xl - lse; }
    }
    __syncthreads();
    tok = s_i[3];
    lp = s_f[2];
  }
  if (tid == 0) {
    p.tokens[static_cast<size_t>(gb) * p.D + i] = tok;
    p.logprobs[static_cast<size_t>(gb) * p.D + i] = lp;
  }
  if (i + 1 < p.D && !bad && work) gru_request(p, b, tok);
  if (staged) fence_async_smem();   // the ring's generic writes -> its next bulk copies
  __syncthreads();
}

__global__ void __launch_bounds__(kDThreads, 1) decode_kernel(DecodeParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[2 * kStages + 4];
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ float s_T[kMaxBpad];
  uint64_t *full = bars, *empty = bars + kStages, *accf = bars + 2 * kStages, *acce = accf + 2;
  unsigned char *ring = smem;
  unsigned char *sB = smem + kStages * kChunkBytes;
  float *s_red = reinterpret_cast<float *>(sB + static_cast<size_t>(6) * p.bpad * p.kb);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&accf[s], 1);
      mbar_init(&acce[s], 8);
    }
    s_fail = 0;
  }
  for (int b = threadIdx.x; b < kMaxBpad; b += kDThreads) {
    float T = 1.0f;
    if (b < p.nb && p.temperature) {
      T = p.temperature[p.b0 + b];
      T = (T == 0.0f || bad_temperature(T)) ? 1.0f : T;   // greedy positions divide by 1
    }
    s_T[b] = T;
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = s_tmem;
  Ctrl *ctrl = p.ctrl;
  unsigned target = 0;
  Pipe pp{0u, 0u};
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  uint64_t tp = clock_me ? global_ns() : 0;
  auto lap = [&](int slot) {
    if (clock_me) {
      const uint64_t now = global_ns();
      ctrl->t_ns[slot] += now - tp;
      tp = now;
    }
  };
  auto barrier = [&](bool fail) {
    const bool r = grid_barrier(&ctrl->bar_count, &ctrl->abort, gridDim.x, kLimitNs, target, fail);
    lap(3);
    return r;
  };

  // the states start as state0; flags cleared
  for (size_t e = static_cast<size_t>(blockIdx.x) * kDThreads + threadIdx.x;
       e < static_cast<size_t>(p.nb) * p.d_s; e += static_cast<size_t>(gridDim.x) * kDThreads)
    p.S[e] = p.state0[static_cast<size_t>(p.b0) * p.d_s + e];
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < p.bpad; b += kDThreads) p.flags[b] = 0;
  bool ok = barrier(false);

  // root: S_0 = GRU(state0, E[anchor])
  if (ok) {
    const bool g = state_gemm(p, ring, sB, full, empty, accf, acce, tmem, pp, &s_fail);
    lap(0);
    ok = barrier(!g || s_fail);
  }
  if (ok) {
    for (int b = blockIdx.x; b < p.nb; b += gridDim.x) {
      const int gb = p.b0 + b;
      const bool bad = bad_temperature(p.temperature ? p.temperature[gb] : 1.0f);
      if (!bad && threadIdx.x < kWork) gru_request(p, b, p.anchor[gb]);
    }
    lap(2);
    ok = barrier(false);
  }
  for (int i = 0; i < p.D && ok; ++i) {
    bool g = state_gemm(p, ring, sB, full, empty, accf, acce, tmem, pp, &s_fail);
    lap(0);
    ok = barrier(!g || s_fail);
    if (!ok) break;
    g = vocab_gemm(p, i, ring, sB, full, empty, accf, acce, tmem, pp, &s_fail, s_T, s_red);
    lap(1);
    ok = barrier(!g || s_fail);
    if (!ok) break;
    for (int b = blockIdx.x; b < p.nb; b += gridDim.x)
      choose_token(p, i, b, reinterpret_cast<float *>(ring));
    lap(2);
    if (i + 1 < p.D) ok = barrier(false);
  }

  // statuses (the block of each request), then TMEM back
  for (int b = blockIdx.x; b < p.nb; b += gridDim.x) {
    const int gb = p.b0 + b;
    const float T = p.temperature ? p.temperature[gb] : 1.0f;
    int st = DT_OK;
    if (!ok) st = DT_ERR_TIMEOUT;
    else if (p.flags[b]) st = DT_ERR_NONFINITE;
    else if (bad_temperature(T)) st = DT_ERR_BAD_TEMPERATURE;
    if (st != DT_OK)
      for (int i = threadIdx.x; i < p.D; i += kDThreads) {
        p.tokens[static_cast<size_t>(gb) * p.D + i] = -1;
        p.logprobs[static_cast<size_t>(gb) * p.D + i] = __int_as_float(0x7fc00000);
      }
    if (threadIdx.x == 0) p.status[gb] = st;
  }
  // every issued MMA has completed once its accumulator was waited for; on a
  // failure, wait (bounded) for the last commit and the copies in flight
  if (!ok && threadIdx.x == kMma && pp.q > 0) {
    const uint32_t q = pp.q - 1;
    mbar_wait(&accf[q & 1u], (q >> 1) & 1u, kLimitNs);
  }
  if (!ok && threadIdx.x == kProd) {
    for (uint32_t g = pp.g > kStages ? pp.g - kStages : 0; g < pp.g; ++g)
      mbar_wait(&full[g % kStages], (g / kStages) & 1u, kLimitNs);
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void prep_tiles_kernel(const uint16_t *A, int rowsA, size_t ldA, int colA,
                                  const uint16_t *B, int rowsB, size_t ldB, int colB, int K,
                                  int nch, int ntiles, unsigned char *dst) {
  const size_t total = static_cast<size_t>(ntiles) * nch * 128 * 8;
  for (size_t u = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int kg = static_cast<int>(u & 7), row = static_cast<int>((u >> 3) & 127);
    const size_t tc = u >> 10;
    const int c = static_cast<int>(tc % nch), t = static_cast<int>(tc / nch);
    const int R = t * 128 + row, k0 = c * kChunkK + kg * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k0 < K) {
      if (R < rowsA)
        v = *reinterpret_cast<const uint4 *>(A + static_cast<size_t>(R) * ldA + colA + k0);
      else if (R < rowsA + rowsB)
        v = *reinterpret_cast<const uint4 *>(B + static_cast<size_t>(R - rowsA) * ldB + colB + k0);
    }
    *reinterpret_cast<uint4 *>(dst + tc * kChunkBytes + umma_offset(row, kg * 8, kChunkK)) = v;
  }
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

void decode_shape(const dt_dims &d, DecodePlan *p) {
  p->dims = d;
  p->R = 3 * d.d_s + d.r;
  p->n_tA = ceil_div(p->R, 128);
  p->nchA = ceil_div(d.d_s, kChunkK);
  p->n_kz = ceil_div(p->nchA * kChunkK, kRangeK);
  p->n_tV = ceil_div(d.V, 128);
  p->nchV = ceil_div(d.r, kChunkK);
  p->kb = p->nchV * kChunkK > kRangeK ? p->nchV * kChunkK : kRangeK;
}

size_t decode_prepared_bytes(const dt_dims &d) {
  DecodePlan p;
  decode_shape(d, &p);
  return (static_cast<size_t>(p.n_tA) * p.nchA + static_cast<size_t>(p.n_tV) * p.nchV) *
         kChunkBytes;
}

int decode_plan(const dt_dims &d, int num_sms, int smem_optin, DecodePlan *p) {
  decode_shape(d, p);
  p->num_sms = num_sms;
  p->grid = num_sms;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, decode_kernel) != cudaSuccess) return DT_ERR_CUDA;
  const long avail = static_cast<long>(smem_optin) - static_cast<long>(fa.sharedSizeBytes) -
                     static_cast<long>(kStages) * kChunkBytes - kRedBytes;
  int bpad = static_cast<int>(avail / (6L * p->kb)) / 16 * 16;
  if (bpad > kMaxBpad) bpad = kMaxBpad;
  if (bpad < 16) return DT_ERR_UNSUPPORTED;
  p->wave = bpad;
  p->smem = static_cast<size_t>(kStages) * kChunkBytes + static_cast<size_t>(6) * bpad * p->kb +
            kRedBytes;
  if (cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(p->smem)) != cudaSuccess)
    return DT_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel, kDThreads,
                                                    static_cast<int>(p->smem)) != cudaSuccess)
    return DT_ERR_CUDA;
  if (per_sm < 1) return DT_ERR_UNSUPPORTED;
  return DT_OK;
}

cudaError_t launch_decode_prepare(const dt_dims &d, const dt_weights *w, void *out,
                                  cudaStream_t st) {
  DecodePlan p;
  decode_shape(d, &p);
  unsigned char *dst = static_cast<unsigned char *>(out);
  const uint16_t *W_hh = static_cast<const uint16_t *>(w->W_hh);
  const uint16_t *W1 = static_cast<const uint16_t *>(w->W1);
  const uint16_t *W2 = static_cast<const uint16_t *>(w->W2);
  prep_tiles_kernel<<<1024, 256, 0, st>>>(W_hh, 3 * d.d_s, d.d_s, 0, W1, d.r,
                                          static_cast<size_t>(d.d) + d.d_s, d.d, d.d_s, p.nchA,
                                          p.n_tA, dst);
  prep_tiles_kernel<<<2048, 256, 0, st>>>(W2, d.V, d.r, 0, nullptr, 0, 0, 0, d.r, p.nchV, p.n_tV,
                                          dst + static_cast<size_t>(p.n_tA) * p.nchA * kChunkBytes);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodePlan &pl, const DecodeArgs &a, cudaStream_t st) {
  const dt_dims &d = pl.dims;
  DecodeParams p;
  p.V = d.V; p.d = d.d; p.d_s = d.d_s; p.r = d.r; p.D = d.D;
  p.b0 = a.b0; p.nb = a.nb;
  p.bpad = (a.nb + 15) / 16 * 16;
  p.N = 3 * p.bpad;
  p.R = pl.R;
  p.n_tA = pl.n_tA; p.nchA = pl.nchA; p.n_kz = pl.n_kz;
  p.n_tV = pl.n_tV; p.nchV = pl.nchV;
  p.kb = pl.kb;
  p.Gn = pl.n_tV * 4;
  p.wall = static_cast<const unsigned char *>(a.chain_prepared);
  p.w2 = p.wall + static_cast<size_t>(pl.n_tA) * pl.nchA * kChunkBytes;
  p.G = a.G; p.b_hh = a.b_hh; p.U = a.U; p.base = a.base; p.state0 = a.state0;
  p.temperature = a.temperature; p.uniforms = a.uniforms; p.anchor = a.anchor;
  p.ypart = a.ypart; p.S = a.S; p.st_m = a.st_m; p.st_s = a.st_s; p.st_a = a.st_a;
  p.W2 = a.W2;
  p.flags = a.flags; p.ctrl = a.ctrl;
  p.tokens = a.tokens; p.logprobs = a.logprobs; p.status = a.status;
  void *args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(decode_kernel), dim3(pl.grid),
                                     dim3(kDThreads), args, pl.smem, st);
}

}  // namespace dt
