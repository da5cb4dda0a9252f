/*
 * dt.h -- C ABI of the GB300 (sm_103a) conditional draft-tree builder.
 *
 * One call of dt_build_trees() runs one drafting round of DominoTree for a batch
 * of independent requests: per-depth top-M candidate selection over the base
 * logits, then a best-first search whose node scores re-run the Domino GRU
 * correction along each root-to-node path, then the emission of the tree and
 * its ancestor attention mask.
 *
 * Sources (page title, section):
 *  - "Riassunto Tecnico: DominoTree" (gist.science/it/paper/2607.08642),
 *    Componenti Core 1 (best-first max-heap on cumulative path log-probability;
 *    children scored by re-running the GRU correction along the node's path;
 *    the backbone states H_i are shared and path independent), 2 (correction
 *    restricted to the top-M marginal candidates of each depth, then top-k
 *    children), 4 (fixed node budget), 5 (verification with an ancestor mask).
 *  - "Domino：在投机解码中将因果建模与自回归草稿解耦" (paper.rainbus.top/paper/2605.29707),
 *    core method (S_{i-1} = GRU(E_{<=i-1}); dL_i = W2 SiLU(W1 [H_i; S_{i-1}]);
 *    L_i = L_base^i + dL_i) and method steps (draft block of size B anchored on
 *    the last verified token; base logits for the B-1 future positions).
 *
 * Conventions used throughout:
 *  - All pointers passed to dt_build_trees / dt_prepare_weights are DEVICE
 *    pointers on the current CUDA device unless a comment says "host".
 *  - Arrays are dense and row-major. Float tensors are IEEE fp32. Weights are
 *    fp32 or bf16 (raw 16-bit patterns) as dt_weights.wdtype says.
 *  - The caller owns every buffer. No entry point allocates or frees device
 *    memory; scratch memory is the caller's `workspace`.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous. The host return value covers argument
 *    validation and launch errors only; conditions found on the device are
 *    written to out->status[b].
 *  - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef DT_H_
#define DT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DT_ABI_VERSION 1

/* ------------------------------------------------------------ status codes */
#define DT_OK 0
#define DT_ERR_INVALID_ARG (-1)   /* bad size, null pointer, misalignment, limit exceeded */
#define DT_ERR_UNSUPPORTED (-2)   /* no sm_103a device, or a shape beyond this library's kernels */
#define DT_ERR_CUDA (-3)          /* a CUDA runtime call or kernel launch failed */
#define DT_ERR_NONFINITE (-4)     /* device: a base logit of the request is NaN or +inf */
#define DT_ERR_TIMEOUT (-5)       /* device: a bounded inter-block wait expired; request output invalid */
#define DT_ERR_BAD_TEMPERATURE (-6) /* device: temperature < 0 or not finite */

/* Hard limits of this library (checked by every entry point). */
#define DT_MAX_M 256        /* candidates per depth */
#define DT_MAX_K 32         /* children per node */
#define DT_MAX_D 64         /* draft depths (block size - 1) */
#define DT_MAX_N 1024       /* node budget (non-root nodes) */
#define DT_MAX_DS 4096      /* GRU state width */
#define DT_MAX_R 1024       /* correction rank */
#define DT_MAX_SPEC 16      /* speculative expansions per request and step */

typedef enum { DT_F32 = 0, DT_BF16 = 1 } dt_dtype;

/* Problem sizes. Notation of the pages: V vocabulary, d backbone hidden size,
 * d_s GRU state size, r correction rank, D = B - 1 draft depths, M candidates per
 * depth, k children per expanded node, N node budget (non-root nodes). */
typedef struct {
  int V, d, d_s, r, D, M, k, N;
  int batch;          /* requests per call (>= 1) */
} dt_dims;

/* Domino head weights (device, read-only). Layouts:
 *   E    [V][d]          token embedding (the GRU input)
 *   W_ih [3 d_s][d]      GRU input weights, row blocks ordered r, z, n
 *   W_hh [3 d_s][d_s]    GRU recurrent weights, row blocks ordered r, z, n
 *   b_ih, b_hh [3 d_s]   fp32 GRU biases, or NULL for zero
 *   W1   [r][d + d_s]    columns 0..d-1 act on H_i, columns d.. on the GRU state
 *   W2   [V][r]          correction output rows (gathered for the M candidates)
 * Every pointer must be 16-byte aligned. */
typedef struct {
  const void *E, *W_ih, *W_hh;
  const float *b_ih, *b_hh;
  const void *W1, *W2;
  dt_dtype wdtype;
} dt_weights;

/* Per-request outputs (device, caller-owned). Row 0 of each tree is the root
 * (anchor token, parent -1, depth 0, score 0). Rows 1..N are nodes in best-first
 * pop order, so parents[i] < i and scores never increase with i. Rows after the
 * last node (when the candidate tree has fewer than N nodes) hold token, parent
 * and depth -1 and score -inf. */
typedef struct {
  int32_t *tokens;    /* [batch][N+1] */
  int32_t *parents;   /* [batch][N+1] */
  int32_t *depths;    /* [batch][N+1] */
  float *scores;      /* [batch][N+1] cumulative path log-probability */
  uint8_t *mask;      /* [batch][N+1][N+1]: mask[i][j] = 1 iff j is i or an ancestor of i; or NULL */
  int32_t *topm;      /* [batch][D][M]: candidate ids of each depth, (logit desc, id asc); or NULL */
  int32_t *status;    /* [batch]: DT_OK or a device-side DT_ERR_* code; required */
} dt_tree_out;

/* Optional tuning and instrumentation (may be NULL in every call). */
typedef struct {
  int spec_width;     /* speculative expansions per request and step, 1..DT_MAX_SPEC;
                         0 = library default. Any value yields the same trees. */
  void **phase_events;/* NULL, or DT_NUM_PHASE_EVENTS cudaEvent_t handles recorded on
                         the stream at phase boundaries (for timing) */
  int flags;          /* DT_OPT_* bits; 0 = defaults */
} dt_options;

/* dt_options.flags, test hook for failure detection: in the search launch the
 * last block skips its first grid-barrier arrival and every barrier wait is
 * limited to 2 ms, so the other blocks' bounded waits run out. Every request
 * then reports DT_ERR_TIMEOUT with empty rows; no fault, and the context stays
 * usable. */
#define DT_OPT_TEST_BARRIER_TIMEOUT 2

/* dt_options.flags: marginal scoring, the conditionality ablation of
 * "Riassunto Tecnico: DominoTree" (Risultati Sperimentali), a DDTree-style
 * builder. The children of a node at depth j - 1 are the k best of C_j (the
 * depth's top-M candidates) by L_c = L_base^j[c] / T alone, with
 * lp_c = L_c - logsumexp over C_j; no GRU state and no correction, so a node's
 * score is the sum of its path's per-depth lp and the result equals the
 * conditional build with W2 = 0. Best-first order, budget and outputs are those
 * of the conditional build. In this mode w, prepared, H and state0 are not read
 * and may be NULL; one small kernel replaces the projection and the search. */
#define DT_OPT_MARGINAL 8

/* dt_options.flags, dt_build_trees_host only: copy the base logits into the
 * workspace even when they are mapped page-locked memory (by default such
 * logits are read in place; see dt_build_trees_host). */
#define DT_OPT_STAGE_HOST_LOGITS 16


/* phase events: [0] start, [1] after the top-M, [2] after the projection
 * (which runs beside the top-M on a second stream: [2] marks the later of the
 * two), [3] after the search */
#define DT_NUM_PHASE_EVENTS 4

/* Bytes of the prepared-weights buffer for `dims`: the GRU input projection of
 * every vocabulary row, G[v] = W_ih E[v] + b_ih, as fp32 [V][3 d_s]. */
size_t dt_prepared_bytes(const dt_dims *dims);

/* Fill `prepared` (device, dt_prepared_bytes() bytes, 256-byte aligned) from the
 * weights. Run once per set of weights; every later dt_build_trees call with the
 * same weights reads it. The GRU gate input W_ih E[tok] depends only on the
 * weights, so computing it for the whole vocabulary once replaces a 3 d_s x d
 * mat-vec per tree node by a 3 d_s row gather. Returns a DT_ status. */
int dt_prepare_weights(const dt_dims *dims, const dt_weights *w, void *prepared,
                       size_t prepared_bytes, void *stream);

/* Scratch bytes dt_build_trees needs for `dims` and `opt` (may be NULL). */
size_t dt_workspace_bytes(const dt_dims *dims, const dt_options *opt);

/* Kernel launches one dt_build_trees call makes for `dims`, weight type
 * `wdtype` (DT_F32 / DT_BF16) and `opt` (may be NULL): top-M, projection (plus
 * its split-K sum when K is split), one search launch per wave of requests;
 * with DT_OPT_MARGINAL, top-M and the marginal tree kernel.
 * Memsets and event records are not counted. Returns 0 for invalid dims.
 * Host only; needs the device for its SM count. */
int dt_kernel_launches(const dt_dims *dims, int wdtype, const dt_options *opt);

/* Build one round of draft trees for dims->batch requests.
 *   base_logits [batch][D][V] fp32  base logits L_base^j of depths j = 1..D
 *   H           [batch][D][d] fp32  backbone states H_j of depths 1..D
 *   state0      [batch][d_s]  fp32  initial GRU state (zeros in the pages' setting)
 *   anchor_tok  [batch]       int32 last verified token x_t, in [0, V)
 *   temperature [batch]       fp32  per request; NULL = 1.0; 0.0 reads as 1.0
 *                                   (greedy ordering); < 0 or non-finite gives
 *                                   DT_ERR_BAD_TEMPERATURE for that request
 *   prepared    dt_prepare_weights() output for the same weights
 *   workspace   dt_workspace_bytes() bytes, 256-byte aligned, not shared by
 *               overlapping calls
 * Float inputs must be 16-byte aligned when their row length is a multiple of 4
 * floats. Returns DT_OK when the work was enqueued. Part of the work (the
 * projection U = W1[:, :d] H: on the tensor cores for bf16 weights when d is a
 * multiple of 32, r of 4 and d + d_s of 8, else on the CUDA cores) runs on a
 * library-owned stream of the current device, forked from and joined back into
 * `stream` with events, so every result is ordered on `stream` as usual. A
 * bounded wait of the tensor-core projection that runs out makes every request
 * of the call report DT_ERR_TIMEOUT. (The fork and join are events, as stream capture into a
 * CUDA graph requires; capture is not covered by a test yet.) */
int dt_build_trees(const dt_dims *dims, const dt_weights *w, const void *prepared,
                   const float *base_logits, const float *H, const float *state0,
                   const int32_t *anchor_tok, const float *temperature,
                   void *workspace, size_t workspace_bytes, const dt_tree_out *out,
                   const dt_options *opt, void *stream);

/* Same as dt_build_trees, but the per-round inputs and outputs are HOST buffers
 * (pinned memory gives asynchronous copies). The call copies the inputs into
 * the workspace, builds the trees and copies the outputs back, all on `stream`;
 * synchronise the stream before reading the outputs. The workspace must be
 * dt_host_workspace_bytes() bytes. The weights and `prepared` stay on the device.
 * Host output pointers follow dt_tree_out (mask and topm may be NULL).
 * Base logits in page-locked memory that the device maps (dt_mapped_host_pointer
 * returns non-NULL for the whole [batch][D][V] extent, at the alignment
 * dt_build_trees asks for) are not copied: the top-M scan, their only reader,
 * reads them in place over the host link. DT_OPT_STAGE_HOST_LOGITS turns this
 * off. Either way the host inputs must stay unchanged until `stream` has passed
 * the call, as for any asynchronous copy. */
size_t dt_host_workspace_bytes(const dt_dims *dims, const dt_options *opt);
int dt_build_trees_host(const dt_dims *dims, const dt_weights *w, const void *prepared,
                        const float *base_logits, const float *H, const float *state0,
                        const int32_t *anchor_tok, const float *temperature,
                        void *workspace, size_t workspace_bytes, const dt_tree_out *host_out,
                        const dt_options *opt, void *stream);

/* Device address through which kernels on the current device can read `bytes`
 * bytes of host memory starting at `host` in place, or NULL. Non-NULL only for
 * page-locked memory (cudaHostAlloc, cudaHostRegister) mapped for the current
 * device whose registration covers the whole extent, as the driver reports it;
 * pageable memory, device memory, a failed query or an extent past the end of
 * its registration give NULL. Host only; clears any CUDA error it provokes. */
const void *dt_mapped_host_pointer(const void *host, size_t bytes);

/* Allocation-free top-M selection (the pages have no counterpart: this entry
 * point exists for callers of this library that may not allocate device memory,
 * such as a serving runtime whose device memory is entirely pre-reserved for its
 * own pool, a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation, or a plug-in running inside a host framework that
 * owns every device allocation).
 *
 * Computes what dt_build_trees writes to out->topm: for every request b and
 * depth j, the M token ids of base_logits[b][j][:] with the largest values,
 * ordered by (value desc, id asc); status[b] = DT_OK or DT_ERR_NONFINITE (a
 * NaN or +inf logit; the ids of that request are then unspecified).
 *   base_logits [batch][D][V] fp32 device (16-byte aligned when V % 4 == 0)
 *   topm        [batch][D][M] int32 device output
 *   status      [batch]       int32 device output
 * No memory is allocated: the scratch is a static device array of
 * DT_NOALLOC_SCRATCH_BYTES bytes that every device loading the library holds
 * until the process exits. A call needs about batch*D*(4*M + 4) bytes of it
 * (plus 8*M bytes per extra row segment, which the call drops first when short
 * of room); shapes that do not fit return DT_ERR_INVALID_ARG. The first call on
 * a device resolves the array's address (cudaGetSymbolAddress) with that device
 * current; make it before any stream capture. The address is kept per device
 * number for the device's primary context (the one the CUDA runtime uses): it
 * does not follow a cudaDeviceReset or a caller that switches to another
 * driver-API context on the same device. All calls share the array, so calls
 * that overlap on the GPU race; serialise them. Asynchronous on `stream`. */
#define DT_NOALLOC_SCRATCH_BYTES (8u << 20)
int dt_select_topm_noalloc(const float *base_logits, int batch, int D, int V, int M,
                           int32_t *topm, int32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * Domino chain decoding: the released Domino decoder, a single draft chain per
 * request with the correction over the whole vocabulary ("Domino：在投机解码中将因果建模与自回归草稿解耦",
 * method steps, inference, and core method; "Riassunto Tecnico: DominoTree",
 * Definizione del Problema: the released decoder is chain-only). Per request:
 *   S_0 = GRU(state0, E[anchor])
 *   for i = 1..D:  h = SiLU(W1 [H_i; S_{i-1}])
 *                  x_v = (L_base^i[v] + W2[v,:] . h) / T       for every token v
 *                  T = 0: d_i = argmax_v x_v (lowest id on ties), x taken at T = 1
 *                  T > 0: d_i = the smallest v whose cumulative softmax(x) mass
 *                         in token-id order exceeds u_i (inverse CDF)
 *                  logprob_i = log softmax(x)[d_i]
 *                  S_i = GRU(S_{i-1}, E[d_i])
 * Weights must be bf16 (the two products run on the tensor cores with the fp32
 * states and h split into three bf16 terms each); f32 weights give
 * DT_ERR_UNSUPPORTED. dims->M, k and N are not used (any valid values).
 *
 * dt_prepare_chain: once per set of weights, [W_hh; W1[:, d:]] and W2 re-laid
 * out in 128-row tensor-core tiles (dt_chain_prepared_bytes bytes, 256-byte
 * aligned device buffer, caller-owned). The GRU input table comes from
 * dt_prepare_weights (`prepared`).
 *
 * dt_decode_chains: one decoding round for dims->batch requests (device
 * pointers; inputs as for dt_build_trees):
 *   uniforms   [batch][D] fp32 draws for T > 0 (u outside [0, 1) is clamped into
 *              it, NaN reads as 0; NULL reads as 0); unused where T = 0
 *   tokens     [batch][D] int32 output: d_1..d_D (-1 on a non-OK status)
 *   logprobs   [batch][D] fp32 output (NaN on a non-OK status)
 *   status     [batch] DT_OK, DT_ERR_NONFINITE, DT_ERR_BAD_TEMPERATURE or
 *              DT_ERR_TIMEOUT
 *   workspace  dt_chain_workspace_bytes bytes, 256-byte aligned
 * Asynchronous on `stream`; requests run in waves of up to 80 per launch.
 * dt_chain_kernel_launches gives the launches of one call (projection, its
 * split-K sum when K is split, one decoding launch per wave). */
size_t dt_chain_prepared_bytes(const dt_dims *dims);
int dt_prepare_chain(const dt_dims *dims, const dt_weights *w, void *chain_prepared,
                     size_t chain_prepared_bytes, void *stream);
size_t dt_chain_workspace_bytes(const dt_dims *dims);
int dt_chain_kernel_launches(const dt_dims *dims);
int dt_decode_chains(const dt_dims *dims, const dt_weights *w, const void *prepared,
                     const void *chain_prepared, const float *base_logits, const float *H,
                     const float *state0, const int32_t *anchor_tok, const float *temperature,
                     const float *uniforms, void *workspace, size_t workspace_bytes,
                     int32_t *tokens, float *logprobs, int32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * Verify-side consumption of a tree ("Riassunto Tecnico: DominoTree",
 * Componenti Core 5: the target model checks every node in one pass with tree
 * attention, each node seeing the verified prefix and its ancestors). The
 * target model is not part of this library; these calls take its tensors.
 *
 * dt_tree_positions: position ids of the tree rows. The prefix cache holds the
 * prefix_len[b] tokens before the anchor; the anchor (row 0) sits at position
 * prefix_len[b] and a row of depth j at prefix_len[b] + j; rows with depth -1
 * (empty) get -1.
 *   depths     [batch][n1] int32 (dt_tree_out.depths), device
 *   prefix_len [batch] int32, device
 *   positions  [batch][n1] int32 output, device
 *
 * dt_tree_attention: one attention layer over the tree rows (device pointers):
 *   q    [batch][H][n1][dh]        bf16 bits, 16-byte aligned
 *   k, v [batch][Hkv][P + n1][dh]  bf16 bits: keys 0..P-1 are the prefix cache
 *                                  (only p < prefix_len[b] are attended; the rest
 *                                  is padding), key P + t is tree row t
 *   mask [batch][n1][n1]           row i sees tree row t iff mask[i][t] != 0
 *                                  (dt_tree_out.mask)
 *   prefix_len [batch]             clamped into [0, P]
 *   out  [batch][H][n1][dh]        fp32 output, 16-byte aligned:
 *        out_i = sum_j softmax_j(scale q_i . k_j) v_j over the visible keys j,
 *        0 for a row that sees no key
 * Query head h reads key/value head h / (H / Hkv) (H % Hkv == 0). dh is 64, 128
 * or 256; n1 <= DT_MAX_N + 1. On the tensor cores: q.k as exact products of the
 * bf16 inputs accumulated in fp32, the softmax weights in two bf16 terms (16
 * significant bits) against the bf16 values, fp32 accumulation. Both calls
 * return DT_ERR_INVALID_ARG for bad sizes or pointers and are asynchronous on
 * `stream`. */
int dt_tree_positions(const int32_t *depths, const int32_t *prefix_len, int batch, int n1,
                      int32_t *positions, void *stream);
int dt_tree_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const uint8_t *mask, const int32_t *prefix_len, int batch, int H, int Hkv,
                      int n1, int P, int dh, float scale, float *out, void *stream);

/* ------------------------------------------------------------------------
 * CondAdaptive: the cost-aware adaptive node budget ("Riassunto Tecnico:
 * DominoTree", Componenti Core 4, reported there as a negative result: with
 * the corrected path probabilities the rule saturates at the maximum budget).
 * Applied in place to the trees of a dt_build_trees call (device pointers of
 * dt_tree_out; status is not read, mask may be NULL), N = the call's budget.
 * Expected accepted length A(n) = 1 + sum_{i<=n} exp(score_i) over the rows in
 * pop order, round cost C(n) = c_fixed + c_node n; row n is kept while
 * A(n) / C(n) rises, i.e. while exp(score_n) C(n-1) > A(n-1) c_node (fp64, pop
 * order), so the kept rows are a prefix of the tree (a subtree: every ancestor
 * has a lower index). Later rows become empty (token, parent, depth -1, score
 * -inf, mask rows 0); counts[b] = rows kept besides the root.
 * c_fixed, c_node > 0 and finite, else DT_ERR_INVALID_ARG. Asynchronous. */
int dt_adaptive_budget(const dt_tree_out *out, int batch, int N, double c_fixed, double c_node,
                       int32_t *counts, void *stream);

/* Static description of a status code. */
const char *dt_status_string(int code);

/* DT_ABI_VERSION of the loaded library. */
int dt_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DT_H_ */
