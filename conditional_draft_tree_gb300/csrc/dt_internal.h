// dt_internal.h -- declarations shared by the translation units of libdt.so.
// Host-side only: workspace layout, launch parameters and kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dt.h"

namespace dt {

// Sizes and pointers of one dt_build_trees call, resolved on the host.
struct Plan {
  dt_dims dims;
  int wdtype;          // DT_F32 / DT_BF16
  int spec;            // speculative expansions per request and step (P)
  int e_cap;           // expansion slots per request
  int nsplit;          // top-M row segments (pieces per row at most, with topm_blocks)
  int topm_blocks;     // > 0: top-M over contiguous unit ranges, this many blocks
  int proj_ksplit;     // K split of the projection GEMM
  int proj_umma;       // the projection on the tensor cores (dt_proj.cu)
  int umma;            // search GEMM on tcgen05 (bf16 weights)
  int n_mt, ks, kc;    // its 128-row tiles, K chunks and K chunk width
  int nbufs;           // its B slice buffers in flight (2..4)
  int test_timeout;    // DT_OPT_TEST_BARRIER_TIMEOUT
  int marginal;        // DT_OPT_MARGINAL: top-M, then the marginal tree kernel
  int num_sms;
  int chain_grid;      // co-resident blocks of the search kernel
  int wave;            // requests per search launch (<= chain_grid)
  size_t chain_smem;   // dynamic shared memory of the search kernel
  // workspace carve-up (byte offsets)
  size_t off_ctrl, off_part, off_cand_id, off_cand_val, off_U, off_S, off_gh, off_gin, off_p,
      off_colexp, off_colinfo, off_kids, off_ghflag, off_upart, off_partial, off_gin16, off_end;
  size_t off_gemm_tickets;  // inside the control region
};

// Control block at the start of the workspace; zeroed by every call.
struct Ctrl {
  unsigned int bar_count;  // grid barrier arrivals (monotonic within a launch)
  unsigned int red_next;   // column counter of the gh sums of even steps
  int abort;           // set when a bounded wait expired
  int active;          // requests of the current wave still searching
  unsigned int steps;      // lockstep steps of the last search launch
  unsigned int expansions; // expansions of the last search launch
  unsigned int red_next_odd;  // column counter of the gh sums of odd steps
  unsigned int pad;
  // block 0 of the last search launch, ns summed over steps: [0] GEMM phase,
  // [1] barrier after it; as request 0's leader: [2] scoring its nodes, [3]
  // waiting for and gathering the other members' children, [4] pops and
  // selection, [5] GRU cells (with the waits for the parents' gh); [6] gh
  // sums after the request phase, [7] barrier after the request phase, [8]
  // the part of [5] spent waiting for the parents' gh;
  // GEMM parts: [9] MMA loop, [10] epilogue, [12] waits for MMA completion;
  // scoring of block 0's nodes: [13] h, [14] candidate loop, [15] softmax +
  // sort + children; GEMM issuing thread, in SM cycles: [24] waits for free
  // buffers, [25] waits for landed copies, [26] copy issue, [27] MMA issue;
  // request 0's replay: [28] pop iterations, [29] their cycles, [30] selection
  // iterations, [31] their cycles
  unsigned long long t_ns[32];
  // followed by: unsigned row_ticket[batch * D]; int req_flags[batch]; gemm tickets
};

constexpr int kCtrlHeader = sizeof(Ctrl);
constexpr int kReqFlagNonfinite = 1;

int make_plan(const dt_dims *dims, int wdtype, const dt_options *opt, Plan *p);
int validate_dims(const dt_dims *dims);

// top-M over base logits -> candidate ids/values (+ optional user copy)
cudaError_t launch_topm(const Plan &p, const float *base_logits, void *ws, int32_t *topm_out,
                        cudaStream_t st);
cudaError_t launch_topm_raw(const float *base_logits, int batch, int D, int V, int M, int nsplit,
                            int nblk, uint64_t *partial, unsigned *ticket, int *req_flags,
                            int32_t *cand_id, float *cand_val, int32_t *topm_out, cudaStream_t st);

// C[m][n] = sum_k A[m][k] * B[n][k] (+ bias[n]); fp32 accumulation.
// a_dtype/b_dtype: DT_F32 or DT_BF16.
// ksplit > 1 splits K over blockIdx.z (partial: ksplit*M*N floats) and adds a
// reduction launch; requires N % 4 == 0 (else ksplit is forced to 1).
cudaError_t launch_gemm_nt(int M, int N, int K, const void *A, int a_dtype, size_t lda,
                           const void *B, int b_dtype, size_t ldb, const float *bias, float *C,
                           size_t ldc, int ksplit, float *partial, cudaStream_t st);
int gemm_tiles(int M, int N);
// C = sum of the ksplit planes [ksplit][M][N] (in order) + bias; N % 4 == 0
cudaError_t launch_splitk_reduce(const float *partial, int ksplit, int M, int N, const float *bias,
                                 float *C, size_t ldc, cudaStream_t st);

// U = H W1[:, :K]^T on the tensor cores (bf16 W1; dt_proj.cu): rows x r
// outputs, K split in split_k chunks (partials [split_k][rows][r] plus the
// reduction when split_k > 1); *fail = 1 when a bounded wait runs out.
bool proj_umma_supported(const dt_dims &d, int wdtype);
int proj_umma_split(int rows, int r, int K, int target_blocks);
cudaError_t launch_proj_umma(int rows, int r, int K, const float *H, int ldh, const void *W1,
                             int ldw, float *U, int split_k, float *partial, int *fail,
                             cudaStream_t st);

// The best-first search for requests [b0, b0 + nb).
struct ChainArgs {
  const dt_weights *w;
  const float *G;            // prepared [V][3 d_s]
  const float *state0;       // [batch][d_s]
  const int32_t *anchor;     // [batch]
  const float *temperature;  // [batch] or null
  const dt_tree_out *out;
  int b0, nb;
};
cudaError_t launch_chain(const Plan &p, const ChainArgs &a, void *ws, cudaStream_t st);

// Domino chain decoding (dt_decode.cu): sizes of the two tensor-core GEMMs,
// wave size (requests per launch) and the workspace carve-up.
struct DecodePlan {
  dt_dims dims;
  int num_sms, grid, wave;
  int R, n_tA, nchA, n_kz, n_tV, nchV, kb;
  size_t smem;
  int proj_ksplit;
  int proj_umma;        // the projection on the tensor cores (dt_proj.cu)
  size_t off_ctrl, off_U, off_upart, off_ypart, off_S, off_stm, off_sts, off_sta,
      off_flags, off_end;
};
struct DecodeArgs {
  const void *chain_prepared;  // dt_prepare_chain output
  const float *G;              // dt_prepare_weights output [V][3 d_s]
  const float *b_hh, *U, *base, *state0, *temperature, *uniforms;
  const int32_t *anchor;
  const uint16_t *W2;          // [V][r] bf16 bits
  float *ypart, *S, *st_m, *st_s;
  int32_t *st_a;
  int *flags;
  Ctrl *ctrl;
  int32_t *tokens;
  float *logprobs;
  int32_t *status;
  int b0, nb;
};
void decode_shape(const dt_dims &d, DecodePlan *p);
size_t decode_prepared_bytes(const dt_dims &d);
int decode_plan(const dt_dims &d, int num_sms, int smem_optin, DecodePlan *p);
cudaError_t launch_decode_prepare(const dt_dims &d, const dt_weights *w, void *out,
                                  cudaStream_t st);
cudaError_t launch_decode(const DecodePlan &pl, const DecodeArgs &a, cudaStream_t st);

// Marginal-score trees (DT_OPT_MARGINAL): one block per request over the top-M
// kernel's candidates (cand_id / cand_val [batch][D][M], req_flags [batch]).
size_t marginal_smem_bytes(const dt_dims &d);
cudaError_t launch_marginal(const dt_dims &d, const int32_t *cand_id, const float *cand_val,
                            const int *req_flags, const int32_t *anchor, const float *temperature,
                            const dt_tree_out *out, cudaStream_t st);

}  // namespace dt
