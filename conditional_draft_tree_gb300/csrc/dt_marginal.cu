// dt_marginal.cu -- draft trees with marginal (path-independent) scores.
//
// "Riassunto Tecnico: DominoTree", Risultati Sperimentali: the ablation of the
// conditional scores against marginal ones (a DDTree-style builder). Here the
// correction is left out: the children of every node at depth j - 1 are the k
// best of the depth's top-M candidates C_j under L_c = L_base^j[c] / T, with
// log-probabilities lp_c = L_c - logsumexp_{C_j} L (the same normalisation over
// the M candidates as the conditional builder), so a node's score is the sum of
// its path's per-depth lp. This is exactly the conditional builder with W2 = 0.
// The best-first order, the budget and the outputs are those of the conditional
// builder; no GRU state and no weight is needed.
//
// One block per request: warp j (of 8, looping) forms depth j's k children
// from the top-M kernel's sorted candidates; then warp 0 pops N nodes in
// (score desc, push order asc) order from the frontier of sorted runs (the
// children of each popped node, in rank order), as the conditional search does.
#include <cstdint>

#include "dt_common.cuh"
#include "dt_internal.h"

namespace dt {

namespace {

constexpr int kMThreads = 256;

struct MarginalArgs {
  int V, D, M, k, N, batch;
  const int32_t *cand_id;
  const float *cand_val;
  const int *req_flags;
  const int32_t *anchor;
  const float *temperature;
  int32_t *tokens, *parents, *depths;
  float *scores;
  uint8_t *mask;
  int32_t *status;
};

__device__ __forceinline__ uint32_t score_key(float s) {   // 0: exhausted (NaN)
  return s == s ? float_order_bits(s) : 0u;
}

template <int SLOTS>
__global__ void __launch_bounds__(kMThreads)
marginal_kernel(MarginalArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n1 = a.N + 1;
  // shared: lp [D][k], tok [D][k]; per run: parent score, head score, output
  // row of the parent, depth, next entry; par [N+1] (4-, then 2-, then 1-byte
  // arrays, so every array is aligned to its element)
  float *lp = reinterpret_cast<float *>(smem);
  int32_t *tok = reinterpret_cast<int32_t *>(lp + a.D * a.k);
  float *run_ps = reinterpret_cast<float *>(tok + a.D * a.k);
  float *run_hs = run_ps + n1;
  int16_t *run_pos = reinterpret_cast<int16_t *>(run_hs + n1);
  int16_t *par = run_pos + n1;
  int8_t *run_dep = reinterpret_cast<int8_t *>(par + n1);
  uint8_t *run_head = reinterpret_cast<uint8_t *>(run_dep + n1);
  __shared__ int s_status, s_count;
  const size_t orow = static_cast<size_t>(b) * n1;
  const float ninf = -__int_as_float(0x7f800000);

  float T = a.temperature ? a.temperature[b] : 1.0f;
  if (threadIdx.x == 0) {
    int st = DT_OK;
    if (a.req_flags[b] & kReqFlagNonfinite) st = DT_ERR_NONFINITE;
    else if (!(T >= 0.0f) || T == __int_as_float(0x7f800000)) st = DT_ERR_BAD_TEMPERATURE;
    s_status = st;
    s_count = 0;
  }
  T = (T == 0.0f) ? 1.0f : T;   // T = 0: greedy ordering, read as T = 1
  __syncthreads();
  const int status = s_status;

  // 1. per depth: L over the M candidates, log-sum-exp, and the k best by
  //    (L desc, id asc); the division by T can merge distinct values, so the
  //    order is taken after it, as the conditional builder does
  if (status == DT_OK) {
    for (int j = warp; j < a.D; j += kMThreads / 32) {
      const size_t row = (static_cast<size_t>(b) * a.D + j) * a.M;
      uint64_t key[SLOTS];
      float Lv[SLOTS];
      float mx = ninf;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int c = s * 32 + lane;
        key[s] = 0ull;
        Lv[s] = ninf;
        if (c < a.M) {
          const int32_t id = a.cand_id[row + c];
          if (id >= 0) {
            Lv[s] = __fdiv_rn(a.cand_val[row + c] + 0.0f, T);
            key[s] = make_key(Lv[s], static_cast<uint32_t>(id));
          }
        }
        mx = fmaxf(mx, Lv[s]);
      }
      mx = warp_max(mx);
      float sum = 0.f;
#pragma unroll
      for (int s = 0; s < SLOTS; ++s)
        if (s * 32 + lane < a.M) sum += expf(Lv[s] - mx);
      sum = warp_sum(sum);
      const float lse = (mx == ninf) ? ninf : mx + logf(sum);
      warp_sort_desc<SLOTS>(key, lane);
#pragma unroll
      for (int s = 0; s < SLOTS; ++s) {
        const int c = s * 32 + lane;
        if (c < a.k) {
          lp[j * a.k + c] = (lse == ninf) ? ninf : key_value(key[s]) - lse;
          tok[j * a.k + c] = static_cast<int32_t>(key_id(key[s]));
        }
      }
    }
  }
  __syncthreads();

  // 2. best-first over the runs (warp 0); run r holds the children of the
  //    node at output row run_pos[r], at depth run_dep[r], next entry run_head[r]
  if (status == DT_OK && warp == 0 && a.N > 0) {
    auto head_score = [&](int r, int h) {
      return h < a.k ? run_ps[r] + lp[(run_dep[r] - 1) * a.k + h] : __int_as_float(0x7fc00000);
    };
    int n_runs = 1, count = 0;
    if (lane == 0) {
      run_ps[0] = 0.0f; run_dep[0] = 1; run_head[0] = 0; run_pos[0] = 0;
      run_hs[0] = head_score(0, 0);
      par[0] = -1;
    }
    __syncwarp();
    uint32_t my_key = 0u;
    int my_run = -1;
    auto lane_scan = [&]() {
      my_key = 0u;
      my_run = -1;
      for (int r = lane; r < n_runs; r += 32) {
        const uint32_t kk = score_key(run_hs[r]);
        if (kk > my_key) { my_key = kk; my_run = r; }
      }
    };
    lane_scan();
    while (count < a.N) {
      const uint32_t kmax = __reduce_max_sync(kFull, my_key);
      if (kmax == 0u) break;   // every run exhausted
      const int r = static_cast<int>(
          __reduce_min_sync(kFull, my_key == kmax ? static_cast<uint32_t>(my_run) : 0xffffffffu));
      const int h = run_head[r], dep = run_dep[r], rpos = run_pos[r];
      const float sc = run_hs[r];
      const int pos = count + 1;
      if (lane == 0) {
        a.tokens[orow + pos] = tok[(dep - 1) * a.k + h];
        a.parents[orow + pos] = rpos;
        a.depths[orow + pos] = dep;
        a.scores[orow + pos] = sc;
        par[pos] = static_cast<int16_t>(rpos);
      }
      const bool expand = dep < a.D && pos < a.N;
      __syncwarp();
      if (lane == (r & 31)) {
        run_head[r] = static_cast<uint8_t>(h + 1);
        run_hs[r] = head_score(r, h + 1);
      }
      if (expand && lane == (n_runs & 31)) {
        run_ps[n_runs] = sc;
        run_dep[n_runs] = static_cast<int8_t>(dep + 1);
        run_head[n_runs] = 0;
        run_pos[n_runs] = static_cast<int16_t>(pos);
        run_hs[n_runs] = head_score(n_runs, 0);
      }
      n_runs += expand ? 1 : 0;
      count = pos;
      __syncwarp();
      if (lane == (r & 31) || (expand && lane == ((n_runs - 1) & 31))) lane_scan();
    }
    if (lane == 0) s_count = count;
  }
  __syncthreads();

  // 3. rows: the root, then empty rows past the last pop; mask; status
  const int count = s_count;
  const bool ok = status == DT_OK;
  if (threadIdx.x == 0) {
    a.tokens[orow] = ok ? a.anchor[b] : -1;
    a.parents[orow] = -1;
    a.depths[orow] = ok ? 0 : -1;
    a.scores[orow] = ok ? 0.0f : ninf;
    a.status[b] = status;
  }
  for (int i = (ok ? count + 1 : 1) + threadIdx.x; i <= a.N; i += kMThreads) {
    a.tokens[orow + i] = -1;
    a.parents[orow + i] = -1;
    a.depths[orow + i] = -1;
    a.scores[orow + i] = ninf;
  }
  if (a.mask) {
    uint8_t *mb = a.mask + static_cast<size_t>(b) * n1 * n1;
    for (size_t i = threadIdx.x; i < static_cast<size_t>(n1) * n1; i += kMThreads) mb[i] = 0;
    __syncthreads();
    if (ok) {
      if (threadIdx.x == 0) par[0] = -1;
      __syncthreads();
      for (int i = threadIdx.x; i <= count; i += kMThreads)
        for (int q = i; q >= 0; q = par[q]) mb[static_cast<size_t>(i) * n1 + q] = 1;
    }
  }
}

}  // namespace

size_t marginal_smem_bytes(const dt_dims &d) {
  const size_t n1 = static_cast<size_t>(d.N) + 1;
  return static_cast<size_t>(d.D) * d.k * 8 + n1 * (4 + 4 + 2 + 2 + 1 + 1);
}

cudaError_t launch_marginal(const dt_dims &d, const int32_t *cand_id, const float *cand_val,
                            const int *req_flags, const int32_t *anchor, const float *temperature,
                            const dt_tree_out *out, cudaStream_t st) {
  MarginalArgs a;
  a.V = d.V; a.D = d.D; a.M = d.M; a.k = d.k; a.N = d.N; a.batch = d.batch;
  a.cand_id = cand_id; a.cand_val = cand_val; a.req_flags = req_flags;
  a.anchor = anchor; a.temperature = temperature;
  a.tokens = out->tokens; a.parents = out->parents; a.depths = out->depths;
  a.scores = out->scores; a.mask = out->mask; a.status = out->status;
  const size_t smem = marginal_smem_bytes(d);
  const int mp = d.M <= 32 ? 1 : d.M <= 64 ? 2 : d.M <= 128 ? 4 : 8;
  const void *fn = mp == 1 ? reinterpret_cast<const void *>(&marginal_kernel<1>)
                 : mp == 2 ? reinterpret_cast<const void *>(&marginal_kernel<2>)
                 : mp == 4 ? reinterpret_cast<const void *>(&marginal_kernel<4>)
                           : reinterpret_cast<const void *>(&marginal_kernel<8>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  void *args[] = {&a};
  return cudaLaunchKernel(fn, dim3(d.batch), dim3(kMThreads), args, smem, st);
}

}  // namespace dt
