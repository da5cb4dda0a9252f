// dt_adaptive.cu -- cost-aware adaptive node budget (CondAdaptive).
//
// "Riassunto Tecnico: DominoTree", Componenti Core 4: the pages carry
// CaDDTree's cost-aware rule (stop growing the tree once the throughput gain
// fades) over to the conditional tree and find that it saturates at the
// maximum budget, because the corrected path probabilities overestimate
// acceptance. Reading: with the drafter's path probabilities the expected
// accepted length of an n-node tree is A(n) = 1 + sum_{i<=n} exp(score_i) and a
// round costs C(n) = c_fixed + c_node n; growth continues while A(n) / C(n)
// rises, i.e. node n is kept while exp(score_n) C(n-1) > A(n-1) c_node.
// Best-first pops come in non-increasing score order and a prefix of the pop
// order is a subtree, so the adaptive tree is the first rows of the
// fixed-budget tree: this kernel takes the decision (fp64, pop order) and
// empties the later rows in place.
#include <cmath>
#include <cstdint>

#include "dt_internal.h"

namespace dt {

namespace {

__global__ void adaptive_budget_kernel(int N, double c_fixed, double c_node, int32_t *tokens,
                                       int32_t *parents, int32_t *depths, float *scores,
                                       uint8_t *mask, int32_t *counts) {
  __shared__ int s_keep;
  const int b = blockIdx.x;
  const size_t n1 = static_cast<size_t>(N) + 1;
  const size_t row0 = static_cast<size_t>(b) * n1;
  if (threadIdx.x == 0) {
    double A = 1.0, C = c_fixed;
    int keep = 0;
    for (int n = 1; n <= N; ++n) {
      if (tokens[row0 + n] < 0) break;
      const double e = exp(static_cast<double>(scores[row0 + n]));
      if (!(e * C > A * c_node)) break;
      A += e;
      C += c_node;
      keep = n;
    }
    s_keep = keep;
    counts[b] = keep;
  }
  __syncthreads();
  const int keep = s_keep;
  for (size_t i = keep + 1 + threadIdx.x; i <= static_cast<size_t>(N); i += blockDim.x) {
    tokens[row0 + i] = -1;
    parents[row0 + i] = -1;
    depths[row0 + i] = -1;
    scores[row0 + i] = -INFINITY;
  }
  if (mask) {
    uint8_t *mb = mask + static_cast<size_t>(b) * n1 * n1;
    for (size_t e = (keep + 1) * n1 + threadIdx.x; e < n1 * n1; e += blockDim.x) mb[e] = 0;
  }
}

inline bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

}  // namespace dt

extern "C" int dt_adaptive_budget(const dt_tree_out *out, int batch, int N, double c_fixed,
                                  double c_node, int32_t *counts, void *stream) {
  if (!out || !out->tokens || !out->parents || !out->depths || !out->scores || !counts ||
      batch < 1 || batch > 65535 || N < 0 || N > DT_MAX_N || !std::isfinite(c_fixed) ||
      !std::isfinite(c_node) || !(c_fixed > 0.0) || !(c_node > 0.0) || !dt::al4(out->tokens) ||
      !dt::al4(out->parents) || !dt::al4(out->depths) || !dt::al4(out->scores) ||
      !dt::al4(counts))
    return DT_ERR_INVALID_ARG;
  dt::adaptive_budget_kernel<<<batch, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      N, c_fixed, c_node, out->tokens, out->parents, out->depths, out->scores, out->mask, counts);
  return cudaGetLastError() == cudaSuccess ? DT_OK : DT_ERR_CUDA;
}
