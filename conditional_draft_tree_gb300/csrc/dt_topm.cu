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

// Sorted (descending) list of 32*SLOTS keys spread over a warp: element
// i = s*32 + lane lives in register v[s] of `lane`.
template <int SLOTS>
struct WarpList {
  uint64_t v[SLOTS];

  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) v[s] = 0;
  }
  // element i (warp-uniform i)
  __device__ __forceinline__ uint64_t at(int i) const {
    uint64_t x = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
      if (s == (i >> 5)) x = v[s];
    return shfl64(x, i & 31);
  }
  // insert warp-uniform key c (unique), dropping the smallest element
  __device__ __forceinline__ void insert(uint64_t c, int lane) {
    int p = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) p += __popc(__ballot_sync(kFull, v[s] > c));
    uint64_t carry = 0;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      uint64_t up = shfl64_up(v[s], 1);
      uint64_t last = shfl64(v[s], 31);
      if (lane == 0) up = carry;
      int i = s * 32 + lane;
      v[s] = (i < p) ? v[s] : (i == p ? c : up);
      carry = last;
    }
  }
  // this <- top 32*SLOTS of (this U other), both sorted descending
  __device__ __forceinline__ void merge(const WarpList &o, int lane) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      uint64_t rev = shfl64(o.v[SLOTS - 1 - s], 31 - lane);
      v[s] = v[s] > rev ? v[s] : rev;  // bitonic sequence holding the top elements
    }
#pragma unroll
    for (int stride = SLOTS * 16; stride >= 32; stride >>= 1) {
      const int ds = stride >> 5;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        if ((s & ds) == 0) {
          uint64_t a = v[s], b = v[s + ds];
          v[s] = a > b ? a : b;
          v[s + ds] = a > b ? b : a;
        }
      }
    }
#pragma unroll
    for (int stride = 16; stride >= 1; stride >>= 1) {
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        uint64_t o2 = shfl64_xor(v[s], stride);
        bool low = (lane & stride) == 0;
        uint64_t mx = v[s] > o2 ? v[s] : o2, mn = v[s] > o2 ? o2 : v[s];
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

template <int SLOTS>
struct Stream {
  WarpList<SLOTS> L;
  uint64_t tau;   // current M-th key
  float tau_v;
  uint32_t tau_id;
  int M, lane;
  bool bad;

  __device__ __forceinline__ void refresh() {
    tau = L.at(M - 1);
    tau_v = key_value(tau);
    tau_id = key_id(tau);
  }
  // offer one candidate per lane; lanes with valid == false offer nothing
  __device__ __forceinline__ void offer(float v, uint32_t id, bool valid) {
    bad |= valid && ((v != v) || v == __int_as_float(0x7f800000));
    const uint64_t key = make_key(v, id);
    bool pass = valid && (v == v) && key > tau;
    unsigned m = __ballot_sync(kFull, pass);
    while (m) {
      int src = __ffs(m) - 1;
      uint64_t c = shfl64(key, src);
      L.insert(c, lane);
      refresh();
      pass = pass && lane != src && key > tau;
      m = __ballot_sync(kFull, pass);
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

template <int SLOTS>
__global__ void __launch_bounds__(kTopmThreads)
topm_kernel(const float *__restrict__ logits, int V, int D, int M, int nsplit,
            uint64_t *__restrict__ partial, unsigned *__restrict__ ticket,
            int *__restrict__ req_flags, int32_t *__restrict__ cand_id,
            float *__restrict__ cand_val, int32_t *__restrict__ topm_out) {
  constexpr int MP = SLOTS * 32;
  __shared__ uint64_t lists[kTopmWarps * MP];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.y, split = blockIdx.x;
  const size_t row_base = static_cast<size_t>(row) * V;
  const float *rowp = logits + row_base;

  // vector part [a0, a0 + 4 nv) is 16-byte aligned; scalar head [0, a0), tail
  const int a0 = min(V, static_cast<int>((4 - (row_base & 3)) & 3));
  const int nv = (V - a0) >> 2;
  const int u0 = static_cast<int>(static_cast<long long>(split) * nv / nsplit);
  const int u1 = static_cast<int>(static_cast<long long>(split + 1) * nv / nsplit);
  const int cnt = u1 - u0;
  const int w0 = u0 + static_cast<int>(static_cast<long long>(warp) * cnt / kTopmWarps);
  const int w1 = u0 + static_cast<int>(static_cast<long long>(warp + 1) * cnt / kTopmWarps);

  Stream<SLOTS> st;
  st.L.clear();
  st.M = M;
  st.lane = lane;
  st.bad = false;
  st.refresh();

  const float4 *vec = reinterpret_cast<const float4 *>(rowp + a0);
  for (int u = w0 + lane; u - lane < w1; u += 32) {
    bool ok = u < w1;
    float4 x = ok ? __ldcs(vec + u) : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t id = static_cast<uint32_t>(a0 + 4 * u);
    bool any = ok && (x.x >= st.tau_v || x.y >= st.tau_v || x.z >= st.tau_v ||
                      x.w >= st.tau_v || st.tau == 0ull);
    bool nonfin = ok && ((x.x != x.x) || (x.y != x.y) || (x.z != x.z) || (x.w != x.w) ||
                         x.x == __int_as_float(0x7f800000) || x.y == __int_as_float(0x7f800000) ||
                         x.z == __int_as_float(0x7f800000) || x.w == __int_as_float(0x7f800000));
    st.bad |= nonfin;
    if (__any_sync(kFull, any)) {
      st.offer(x.x, id + 0, ok);
      st.offer(x.y, id + 1, ok);
      st.offer(x.z, id + 2, ok);
      st.offer(x.w, id + 3, ok);
    }
  }
  // scalar head (split 0) and tail (last split), warp 0
  if (warp == 0) {
    if (split == 0 && a0 > 0) {
      bool ok = lane < a0;
      st.offer(ok ? __ldg(rowp + lane) : 0.f, static_cast<uint32_t>(lane), ok);
    }
    const int t0 = a0 + 4 * nv;
    if (split == nsplit - 1 && t0 < V) {
      bool ok = t0 + lane < V;
      st.offer(ok ? __ldg(rowp + t0 + lane) : 0.f, static_cast<uint32_t>(t0 + lane), ok);
    }
  }
  if (__any_sync(kFull, st.bad) && lane == 0) atomicOr(req_flags + row / D, kReqFlagNonfinite);

  st.L.store(lists + warp * MP, lane);
  block_merge_lists<SLOTS>(lists, warp, lane);

  if (nsplit > 1) {
    // publish this segment's list; the last block of the row merges them all
    for (int i = threadIdx.x; i < M; i += kTopmThreads)
      partial[(static_cast<size_t>(row) * nsplit + split) * M + i] = lists[i];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(ticket + row, 1u) == static_cast<unsigned>(nsplit - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    WarpList<SLOTS> acc;
    acc.clear();
    for (int s = warp; s < nsplit; s += kTopmWarps) {
      WarpList<SLOTS> b;
      b.load(partial + (static_cast<size_t>(row) * nsplit + s) * M, M, lane, true);
      acc.merge(b, lane);
    }
    __syncwarp();
    acc.store(lists + warp * MP, lane);
    block_merge_lists<SLOTS>(lists, warp, lane);
    if (threadIdx.x == 0) ticket[row] = 0u;
  }
  for (int i = threadIdx.x; i < M; i += kTopmThreads) {
    uint64_t k = lists[i];
    size_t o = static_cast<size_t>(row) * M + i;
    // key 0 only survives when the row holds fewer than M non-NaN values; the
    // request is then flagged non-finite and never searched
    int32_t id = (k != 0ull) ? static_cast<int32_t>(key_id(k)) : -1;
    cand_id[o] = id;
    cand_val[o] = (id >= 0) ? __ldg(rowp + id) : -__int_as_float(0x7f800000);
    if (topm_out) topm_out[o] = id;
  }
}

}  // namespace

// The same kernel on explicit scratch pointers (used by the allocation-free
// entry point, whose scratch is a static device array).
cudaError_t launch_topm_raw(const float *base_logits, int batch, int D, int V, int M, int nsplit,
                            uint64_t *partial, unsigned *ticket, int *req_flags, int32_t *cand_id,
                            float *cand_val, int32_t *topm_out, cudaStream_t st) {
  dim3 grid(nsplit, batch * D);
  const int mp = M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  switch (mp) {
    case 32:
      topm_kernel<1><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, partial, ticket,
                                                   req_flags, cand_id, cand_val, topm_out);
      break;
    case 64:
      topm_kernel<2><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, partial, ticket,
                                                   req_flags, cand_id, cand_val, topm_out);
      break;
    case 128:
      topm_kernel<4><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, partial, ticket,
                                                   req_flags, cand_id, cand_val, topm_out);
      break;
    default:
      topm_kernel<8><<<grid, kTopmThreads, 0, st>>>(base_logits, V, D, M, nsplit, partial, ticket,
                                                   req_flags, cand_id, cand_val, topm_out);
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
  dim3 grid(p.nsplit, d.batch * d.D);
  const int mp = d.M <= 32 ? 32 : d.M <= 64 ? 64 : d.M <= 128 ? 128 : 256;
  switch (mp) {
    case 32:
      topm_kernel<1><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, partial,
                                                   ticket, req_flags, cid, cval, topm_out);
      break;
    case 64:
      topm_kernel<2><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, partial,
                                                   ticket, req_flags, cid, cval, topm_out);
      break;
    case 128:
      topm_kernel<4><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, partial,
                                                   ticket, req_flags, cid, cval, topm_out);
      break;
    default:
      topm_kernel<8><<<grid, kTopmThreads, 0, st>>>(base_logits, d.V, d.D, d.M, p.nsplit, partial,
                                                   ticket, req_flags, cid, cval, topm_out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace dt
