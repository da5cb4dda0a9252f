// dt_chain.cu -- the best-first conditional search, one persistent cooperative
// kernel for a wave of requests.
//
// What it computes ("Riassunto Tecnico: DominoTree", Componenti Core 1, 2, 4, 5;
// "Domino", core method): node 0 is the root (anchor token, score 0) with GRU
// state S_0 = GRU(state0, E[anchor]). Expanding a node x of depth j-1 scores the
// top-M candidates C_j of depth j with the correction along x's path,
//   h    = SiLU(U_j + W1_S S_x),    U_j = W1_H H_j precomputed per depth
//   L_c  = (L_base^j[c] + W2[c,:] h) / T,   lp_c = L_c - logsumexp_{C_j} L
// and offers its k best candidates (L desc, id asc) as children with score
// score(x) + lp_c. Nodes are popped best first, (score desc, push order asc),
// until N nodes are out; a popped node gets the state S = GRU(S_parent, E[tok])
// and is expanded unless it is at depth D or is the N-th pop.
//
// How (GB300 design): the requests advance in lockstep steps of two phases,
// each ended by a grid barrier:
//   GEMM phase    (tensor-core blocks): [gh_x; p_x] = [W_hh; W1_S] S_x for the
//                 nodes x of every request chosen at the last step, as partial
//                 products over K chunks;
//   request phase (block b = request b): score the children of its nodes from
//                 the p partials, pop as far as the exact best-first order
//                 allows, choose the next nodes to expand and run their GRU
//                 cells, writing the next GEMM's input columns. Meanwhile every
//                 other block sums the gh partials of the step's columns
//                 (+ b_hh) into the per-node store, one column at a time from a
//                 shared counter, and marks each column done; a request block
//                 that needs the gh of a parent expanded in this step waits for
//                 its mark and sums columns itself while it waits.
// The GRU input half W_ih E[tok] + b_ih is a row of the prepared table G, and
// the recurrent half gh of a node is produced by the GEMM of the step that
// expanded its parent, so the per-node GRU is elementwise.
//
// Exact speculative expansion: the order in which nodes are popped depends only
// on scores, so expanding a node earlier than the one-at-a-time builder would
// changes nothing but the time at which its children become known. The request
// phase replays the canonical best-first order over the discovered nodes and
// stops at the first popped node that still needs its children ("stall"). It
// then expands that node together with up to P-1 of the next best unexpanded
// frontier nodes (P = spec width). Each step therefore pops at least one node,
// the trees are identical for every P, and the number of lockstep steps drops
// from about N to about the depth of the tree when the tree is bushy.
//
// Frontier representation: the children of an expanded node are stored sorted
// (their scores are non-increasing in rank), so the frontier is a set of sorted
// runs, one per popped expanded node, created in pop order. The next pop is the
// best run head under (score desc, run index asc) -- run index order is the
// parents' pop order and rank order is push order, which is exactly the heap's
// (score desc, push sequence asc) key.
#include <cstdint>

#include <cuda_bf16.h>

#include "dt_common.cuh"
#include "dt_internal.h"
#include "dt_umma.cuh"

namespace dt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGemmCols = 8;     // columns per GEMM work unit (fp32 path)
constexpr int kGemmKC = 1024;    // K chunk staged in shared memory (fp32 path)
constexpr int kState0 = -2;      // column code: the state0 column of the first step
constexpr unsigned long long kEmptyKid = ~0ull;   // a child word not yet written

struct ChainParams {
  int V, d, d_s, r, D, M, k, N;
  int nb, b0, P, e_cap;
  const void *W_hh, *W1, *W2;
  const float *b_hh;
  const float *G;
  const float *state0;
  const int32_t *anchor;
  const float *temperature;
  const int32_t *cand_id;
  const float *cand_val;
  const float *U;
  float *S_store, *gh_store, *gin, *pbuf;
  int *col_count;
  // per GEMM column (slot = request * P + rank): its record (see col_record)
  // and, when a member of the request's group scored it, its k children as
  // 64-bit words (token << 32 | score bits); kEmptyKid until written
  int4 *col_rec;
  unsigned long long *kids;
  // marks (release / acquire, zeroed at launch): per request, step + 1 once
  // its selection is out; per (request, expansion), nonzero once the
  // expansion's gh is in gh_store
  unsigned *sel_mark, *gh_mark;
  int grp;             // blocks per request group (leader = member 0)
  // tensor-core GEMM path (bf16 weights): A tiles of 128 rows x kc K stay in
  // shared memory; the input columns arrive as three bf16 terms per state
  int umma, n_mt, ks, kc, cols_cap;
  int nbufs;           // B slice buffers (2..kMaxBufs)
  float *partial;      // [ks][cols_cap][R] per-K-chunk partial products, by slot
  uint16_t *gin16;     // B operand in tile layout (bcol_index)
  Ctrl *ctrl;
  const int *req_flags;
  int32_t *tokens, *parents, *depths;
  float *scores;
  uint8_t *mask;
  int32_t *status;
  unsigned long long limit_ns;
  int test_skip;       // failure-detection test: the last block skips its first arrival
  // dynamic shared memory carve-up (byte offsets)
  int sm_child_score, sm_child_tok, sm_child_exp, sm_exp_depth, sm_exp_parent, sm_exp_score,
      sm_exp_tok, sm_run_e, sm_run_head, sm_run_pos, sm_vhead, sm_par, sm_slots, sm_recs,
      sm_scratch, sm_total;
  int sm_A, sm_B, sm_mbar, sm_tmem, sm_run_hs, sm_vhs;
};

struct TailState {
  int count;      // nodes popped so far (root excluded)
  int n_runs;
  int e_count;    // expansions assigned
  int done;
  int n_sel;
  int spec_used;  // speculative (non-stall) expansions made so far
  int sel_e[DT_MAX_SPEC];    // expansions chosen at the last selection (the next GEMM's columns)
  float T;
  int status;
};

__device__ __forceinline__ float ldcg(const float *p) { return __ldcg(p); }

// ---------------------------------------------------------------- GEMM phase

// Record of one GEMM column: the expansion e it computes (kState0: the state0
// column of the first step), its parent expansion (-1: the root, whose input
// state is state0), the depth of its children, its token (the GRU input) and
// its path score. One 16-byte word so that a column's facts arrive together.
__device__ __forceinline__ int4 col_record(int e, int parent, int child_depth, int tok,
                                           float score) {
  return make_int4(e, (parent + 1) | (child_depth << 16), tok, __float_as_int(score));
}

// Sum of v[i] over the 32 lanes, scattered: lane l returns the total of v[l].
__device__ __forceinline__ float reduce_scatter32(float v[32], int lane) {
#pragma unroll
  for (int m = 16, n = 32; m >= 1; m >>= 1, n >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      float send = hi ? v[i] : v[i + n / 2];
      float keep = hi ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, m);
    }
  }
  return v[0];
}

// Active GEMM columns in (request, rank) order: slot ids written to `slots`,
// count returned. With `cl` also their records (taken before the request
// phase reassigns them) and, per request, the index of its first column and
// its column count. nb <= 256 requests per wave: one thread per request reads
// its count and, in the same round trip, the records of all its P slots; then
// a block-wide exclusive scan.
struct ColList {
  int4 *recs;        // [cols_cap] records of the listed columns
  int *req_first;    // [nb]
  int *req_cnt;      // [nb]
};

__device__ int compact_slots(const ChainParams &p, int *slots, const ColList *cl = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ int s_warp_sum[kWarps];
  __shared__ int s_total;
  const int b_me = threadIdx.x;
  const bool mine = b_me < p.nb;
  const int c_me = mine ? __ldcg(p.col_count + b_me) : 0;
  int4 r8[8];
  if (cl) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      r8[i] = (mine && i < p.P) ? __ldcg(p.col_rec + b_me * p.P + i) : make_int4(0, 0, 0, 0);
  }
  int incl = c_me;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += s_warp_sum[w];
  if (threadIdx.x == kThreads - 1) s_total = base + incl;
  const int first = base + incl - c_me;
  for (int i = 0; i < c_me; ++i) slots[first + i] = b_me * p.P + i;
  if (cl) {
    if (mine) {
      cl->req_first[b_me] = first;
      cl->req_cnt[b_me] = c_me;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < c_me) cl->recs[first + i] = r8[i];
    for (int i = 8; i < c_me; ++i) cl->recs[first + i] = __ldcg(p.col_rec + b_me * p.P + i);
  }
  __syncthreads();
  return s_total;
}

// [gh; p] = [W_hh; W1_S] x (+ [b_hh; 0]) for every active column, on CUDA
// cores in fp32 (the path for fp32 weights).
template <int WDT>
__device__ void gemm_phase(const ChainParams &p, unsigned char *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ds = p.d_s;
  const int R = 3 * ds + p.r;
  int *slots = reinterpret_cast<int *>(smem);  // [nb * P]
  const int total = compact_slots(p, slots);
  if (total == 0) return;
  float *stage = reinterpret_cast<float *>(smem + ((p.nb * p.P * 4 + 15) & ~15));  // [8][KC]
  const int nct = (total + kGemmCols - 1) / kGemmCols;
  int rparts = max(1, static_cast<int>(gridDim.x) / nct);
  const int rgroups = (R + 3) / 4;
  rparts = min(rparts, rgroups);
  const int groups_per_part = (rgroups + rparts - 1) / rparts;
  const int units = nct * rparts;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int ct = u % nct, rp = u / nct;
    const int c0 = ct * kGemmCols;
    const int ncol = min(kGemmCols, total - c0);
    const int g0 = rp * groups_per_part, g1 = min(rgroups, g0 + groups_per_part);
    for (int kc0 = 0; kc0 < ds; kc0 += kGemmKC) {
      const int kc1 = min(ds, kc0 + kGemmKC);
      const int kw = kc1 - kc0;
      // groups are processed per K chunk; accumulators live only within a group
      // when ds <= KC (the common case); for larger ds partial sums go to the
      // outputs through a second pass below.
      __syncthreads();
      for (int i = threadIdx.x; i < kGemmCols * (kw / 4); i += kThreads) {
        const int c = i / (kw / 4), q = i % (kw / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < ncol) {
          const int slot = slots[c0 + c];
          v = __ldcg(reinterpret_cast<const float4 *>(p.gin + static_cast<size_t>(slot) * ds +
                                                      kc0) + q);
        }
        reinterpret_cast<float4 *>(stage + c * kGemmKC)[q] = v;
      }
      __syncthreads();
      for (int g = g0 + warp; g < g1; g += kWarps) {
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        const void *wrow[4];
        bool rok[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) {
          const int row = g * 4 + ri;
          rok[ri] = row < R;
          if (row < 3 * ds) {
            wrow[ri] = static_cast<const char *>(p.W_hh) +
                       static_cast<size_t>(row) * ds * (WDT ? 2 : 4);
          } else {
            const int t = rok[ri] ? row - 3 * ds : 0;
            wrow[ri] = static_cast<const char *>(p.W1) +
                       (static_cast<size_t>(t) * (p.d + ds) + p.d) * (WDT ? 2 : 4);
          }
        }
        for (int k = lane * 8; k < kw; k += 256) {
          float wf[4][8];
#pragma unroll
          for (int ri = 0; ri < 4; ++ri) {
            if (rok[ri]) {
              load8<WDT>(wrow[ri], kc0 + k, wf[ri]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) wf[ri][e] = 0.f;
            }
          }
#pragma unroll
          for (int c = 0; c < kGemmCols; ++c) {
            const float4 x0 = *reinterpret_cast<const float4 *>(stage + c * kGemmKC + k);
            const float4 x1 = *reinterpret_cast<const float4 *>(stage + c * kGemmKC + k + 4);
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) {
              float a = acc[ri * 8 + c];
              a = fmaf(wf[ri][0], x0.x, a); a = fmaf(wf[ri][1], x0.y, a);
              a = fmaf(wf[ri][2], x0.z, a); a = fmaf(wf[ri][3], x0.w, a);
              a = fmaf(wf[ri][4], x1.x, a); a = fmaf(wf[ri][5], x1.y, a);
              a = fmaf(wf[ri][6], x1.z, a); a = fmaf(wf[ri][7], x1.w, a);
              acc[ri * 8 + c] = a;
            }
          }
        }
        const float sum = reduce_scatter32(acc, lane);
        const int ri = lane >> 3, c = lane & 7;
        const int row = g * 4 + ri;
        if (row < R && c < ncol) {
          const int slot = slots[c0 + c];
          const int b = slot / p.P;
          const int e = __ldcg(p.col_rec + slot).x;
          if (row < 3 * ds) {
            const int e_slot = (e == kState0) ? p.e_cap : e;
            float *dst = p.gh_store + (static_cast<size_t>(b) * (p.e_cap + 1) + e_slot) * 3 * ds + row;
            const float prev = (kc0 == 0) ? (p.b_hh ? p.b_hh[row] : 0.f) : __ldcg(dst);
            *dst = prev + sum;
          } else {
            float *dst = p.pbuf + static_cast<size_t>(slot) * p.r + (row - 3 * ds);
            const float prev = (kc0 == 0) ? 0.f : __ldcg(dst);
            *dst = prev + sum;
          }
        }
      }
    }
  }
}

// ------------------------------------------------- tensor-core GEMM phase

constexpr uint32_t kTmemCols = 256;   // fp32 accumulator columns per block

// (M tile, K chunk) of GEMM block g: consecutive blocks share the M tile.
__device__ __forceinline__ void gemm_tile(const ChainParams &p, int g, int &mt, int &kz) {
  mt = g / p.ks;
  kz = g % p.ks;
}

// Rows [mt*128, mt*128+128) of [W_hh; W1_S] and K columns [kz*kc, kz*kc+kc) as
// bf16 into the A tile (zero beyond R rows or d_s columns). Once per launch.
__device__ void load_a_tile(const ChainParams &p, unsigned char *sA) {
  int mt, kz;
  gemm_tile(p, blockIdx.x, mt, kz);
  const int R = 3 * p.d_s + p.r, k0 = kz * p.kc;
  const int kg = p.kc / 8;
  for (int i = threadIdx.x; i < 128 * kg; i += kThreads) {
    const int r = i / kg, q = i % kg;
    const int row = mt * 128 + r, k = k0 + q * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < R && k < p.d_s) {
      const uint16_t *src =
          (row < 3 * p.d_s)
              ? static_cast<const uint16_t *>(p.W_hh) + static_cast<size_t>(row) * p.d_s + k
              : static_cast<const uint16_t *>(p.W1) +
                    static_cast<size_t>(row - 3 * p.d_s) * (p.d + p.d_s) + p.d + k;
      v = __ldg(reinterpret_cast<const uint4 *>(src));
    }
    *reinterpret_cast<uint4 *>(sA + umma_offset(r, q * 8, p.kc)) = v;
  }
}

// B operand in global memory, already in the tensor cores' tile layout. Node
// column `slot` lives in pass slot / 256 at column c = slot % 256; K index k in
// chunk kz = k / kc at slice (k % kc) / 16. For each (pass, chunk, slice) the
// three bf16 terms follow one another, each a K-major no-swizzle tile of 256
// columns x 16 K (8 KB), so that one slice of a term is a single contiguous
// block whose first 32 * n bytes hold columns [0, n).
constexpr int kTermBytes = 256 * 16 * 2;
constexpr int kSliceBytes = 3 * kTermBytes;
constexpr int kMaxBufs = 4;                    // B slice buffers at most (p.nbufs: 2..4)

__device__ __forceinline__ size_t bcol_index(const ChainParams &p, int slot, int k) {
  const int kz = k / p.kc, kk = k - kz * p.kc;
  const int c = slot & 255;
  const size_t blk = (static_cast<size_t>((slot >> 8) * p.ks + kz) * (p.kc >> 4) + (kk >> 4)) * 3;
  return blk * (kTermBytes / 2) +
         static_cast<size_t>(((c >> 3) * 256 + ((kk >> 3) & 1) * 128 + (c & 7) * 16) / 2 + (kk & 7));
}

struct UmmaState {
  uint32_t tmem;      // TMEM base column address
  uint32_t next;      // global index of the next B slice (buffer = next % p.nbufs)
};

// Partial products of this block's (M tile, K chunk) for every active column,
// written to p.partial[kz][slot][row]. Every block also lists the active
// columns and their records (slots, cl): the request phase reassigns the
// columns' records while their gh sums and scores are still being made. D (TMEM, 128 rows x up to 256 node
// columns) = A B^T, A = 128 weight rows (K-major, resident), B = the node
// columns as hi / mid / lo bf16 terms; one MMA per (K step, term) covers a
// whole pass of 256 columns, since an MMA costs about the same for any N up to
// 256. Thread 0 issues the bulk copies into p.nbufs slice buffers, thread 32 the
// MMAs and commits; all warps read the accumulators back. Every block lists
// the active columns (slots, count in total_out) for the request phase.
__device__ bool gemm_phase_umma(const ChainParams &p, unsigned char *smem, int *slots,
                                const ColList &cl, UmmaState &u, int &total_out) {
  __shared__ int s_hi[16];           // per pass: last active column + 1
  __shared__ uint32_t s_mask[16][8]; // per pass: active columns
  __shared__ int s_fail;              // a bounded wait of an issuing thread ran out
  if (threadIdx.x == 0) s_fail = 0;
  const int total = compact_slots(p, slots, &cl);   // (synchronises the block)
  total_out = total;
  if (total == 0 || blockIdx.x >= p.n_mt * p.ks) return true;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int mt, kz;
  gemm_tile(p, blockIdx.x, mt, kz);
  const int R = 3 * p.d_s + p.r;
  const int n_pass = (p.cols_cap + 255) >> 8;
  if (threadIdx.x < 16 * 9) {
    if (threadIdx.x < 16) s_hi[threadIdx.x] = 0;
    else (&s_mask[0][0])[threadIdx.x - 16] = 0u;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const int slot = slots[i], c = slot & 255;
    atomicMax(&s_hi[slot >> 8], c + 1);
    atomicOr(&s_mask[slot >> 8][c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  unsigned char *sA = smem + p.sm_A;
  unsigned char *sB = smem + p.sm_B;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.sm_mbar);
  const uint32_t nbufs = static_cast<uint32_t>(p.nbufs);
  uint64_t *empty = full + kMaxBufs;
  const int nkb = p.kc >> 4;
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  for (int pass = 0; pass < n_pass; ++pass) {
    const int hi = s_hi[pass];
    if (hi == 0) continue;
    const uint64_t t0 = clock_me ? global_ns() : 0;
    const int npad = (hi + 15) & ~15;
    const uint32_t g0 = u.next;
    if (threadIdx.x == 0) {
      // producer: one bulk copy per K slice (the three term tiles are adjacent
      // in global memory; the last is needed up to npad columns only)
      const uint32_t bytes = 2 * kTermBytes + static_cast<uint32_t>(npad) * 32;
      const unsigned char *src = reinterpret_cast<const unsigned char *>(p.gin16) +
                                 static_cast<size_t>(pass * p.ks + kz) * nkb * kSliceBytes;
      fence_async_global();   // columns written before the grid barrier -> bulk reads
      fence_async_smem();     // earlier generic use of the buffers -> bulk writes
      long long c_empty = 0, c_copy = 0;
      for (int s = 0; s < nkb; ++s) {
        const uint32_t g = g0 + s, buf = g % nbufs;
        // the buffer's previous slice must be consumed by its MMAs
        const long long c0 = clock64();
        if (g >= nbufs && !mbar_wait(&empty[buf], ((g / nbufs) - 1) & 1u, p.limit_ns)) {
          s_fail = 1;
          break;
        }
        const long long c1 = clock64();
        mbar_expect_tx(&full[buf], bytes);
        bulk_g2s(sB + buf * kSliceBytes, src + static_cast<size_t>(s) * kSliceBytes, bytes,
                 &full[buf]);
        c_empty += c1 - c0;
        c_copy += clock64() - c1;
      }
      if (clock_me) {
        p.ctrl->t_ns[24] += c_empty;
        p.ctrl->t_ns[26] += c_copy;
      }
    } else if (threadIdx.x == 32) {
      // MMA issuer: three MMAs (hi, mid, lo terms) per K slice into one TMEM
      // accumulator, each slice's buffer released by a commit
      const uint32_t idesc = umma_idesc_bf16(128, npad);
      const uint32_t a0 = smem_u32(sA), b_base = smem_u32(sB);
      long long c_full = 0, c_mma = 0;
      int s = 0;
      for (; s < nkb; ++s) {
        const uint32_t g = g0 + s, buf = g % nbufs;
        const long long cf = clock64();
        if (!mbar_wait(&full[buf], (g / nbufs) & 1u, p.limit_ns)) {
          s_fail = 1;
          break;
        }
        const long long cm = clock64();
        tmem_fence_after();
        const uint64_t ad = umma_desc(a0 + s * 256, 128, 16u * p.kc);
        const uint32_t b0 = b_base + buf * kSliceBytes;
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
          umma_bf16(u.tmem, ad, umma_desc(b0 + sp * kTermBytes, 128, 256), idesc, s > 0 || sp > 0);
        umma_commit(&empty[buf]);
        c_full += cm - cf;
        c_mma += clock64() - cm;
      }
      const uint64_t tm = global_ns();
      if (s > 0) {   // commits complete in order: the last one covers every MMA
        const uint32_t last = g0 + s - 1;
        if (!mbar_wait(&empty[last % nbufs], (last / nbufs) & 1u, p.limit_ns)) s_fail = 1;
      }
      if (blockIdx.x == 0) {
        p.ctrl->t_ns[12] += global_ns() - tm;
        p.ctrl->t_ns[25] += c_full;
        p.ctrl->t_ns[27] += c_mma;
      }
    }
    u.next = g0 + nkb;
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint64_t t1 = clock_me ? global_ns() : 0;
    if (clock_me) p.ctrl->t_ns[9] += t1 - t0;
    // epilogue: TMEM lane = row of the tile; warps w and w+4 share a lane quarter
    const int quarter = warp & 3;
    const int row = mt * 128 + quarter * 32 + lane;
    for (int grp = warp >> 2; grp * 32 < hi; grp += 2) {
      const uint32_t m = s_mask[pass][grp];
      if (m == 0u) continue;
      float v[32];
      tmem_ld32(u.tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grp * 32, v);
      tmem_wait_ld();
      if (row < R) {
        float *dst = p.partial +
                     (static_cast<size_t>(kz) * p.cols_cap + pass * 256 + grp * 32) * R + row;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((m >> j) & 1u) dst[static_cast<size_t>(j) * R] = v[j];
      }
    }
    tmem_fence_before();
    __syncthreads();
    if (clock_me) p.ctrl->t_ns[10] += global_ns() - t1;
  }
  __syncthreads();
  return s_fail == 0;
}

// ------------------------------------------------------------ gh sums

__device__ __forceinline__ unsigned *gh_mark_of(const ChainParams &p, int b, int e) {
  return p.gh_mark + static_cast<size_t>(b) * (p.e_cap + 1) + (e < 0 ? p.e_cap : e);
}

// Sum of the K-chunk partials (fixed order) + b_hh of the column in `slot`
// (record rec) into the per-node store; then the expansion's gh mark
// (release, gpu scope), read by the blocks that run the GRU of its children.
__device__ void gh_column(const ChainParams &p, int slot, const int4 &rec) {
  const int ds = p.d_s, R = 3 * ds + p.r, n4 = 3 * ds / 4;
  const size_t plane = static_cast<size_t>(p.cols_cap) * R;
  const int b = slot / p.P, e = rec.x == kState0 ? -1 : rec.x;
  float *dst = p.gh_store +
               (static_cast<size_t>(b) * (p.e_cap + 1) + (e < 0 ? p.e_cap : e)) * 3 * ds;
  const float *src = p.partial + static_cast<size_t>(slot) * R;
  constexpr int IT = 3;
  for (int i0 = threadIdx.x; i0 < n4; i0 += IT * kThreads) {
    float4 acc[IT];
#pragma unroll
    for (int q = 0; q < IT; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int z0 = 0; z0 < p.ks; z0 += 4) {
      float4 v[4][IT];
#pragma unroll
      for (int z = 0; z < 4; ++z)
#pragma unroll
        for (int q = 0; q < IT; ++q) {
          const int i = i0 + q * kThreads;
          v[z][q] = (z0 + z < p.ks && i < n4)
                        ? __ldcg(reinterpret_cast<const float4 *>(src + (z0 + z) * plane) + i)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int z = 0; z < 4; ++z)
#pragma unroll
        for (int q = 0; q < IT; ++q) {
          acc[q].x += v[z][q].x; acc[q].y += v[z][q].y;
          acc[q].z += v[z][q].z; acc[q].w += v[z][q].w;
        }
    }
#pragma unroll
    for (int q = 0; q < IT; ++q) {
      const int i = i0 + q * kThreads;
      if (i >= n4) continue;
      float4 a = acc[q];
      if (p.b_hh) {   // 4-byte aligned only
        a.x += p.b_hh[4 * i]; a.y += p.b_hh[4 * i + 1];
        a.z += p.b_hh[4 * i + 2]; a.w += p.b_hh[4 * i + 3];
      }
      reinterpret_cast<float4 *>(dst)[i] = a;
    }
  }
  // the block barrier orders every thread's stores before thread 0's release
  __syncthreads();
  if (threadIdx.x == 0) st_release_u32(gh_mark_of(p, b, e), 1u);
}

// One grab from the step's column counter: the index of a column to sum, or
// a value >= total when none is left. Block-wide.
__device__ __forceinline__ int gh_grab(unsigned *counter) {
  __shared__ int s_idx;
  if (threadIdx.x == 0) s_idx = static_cast<int>(atomicAdd(counter, 1u));
  __syncthreads();
  const int col = s_idx;
  __syncthreads();
  return col;
}

// The step's gh sums, handed out one column at a time.
struct GhWork {
  const int *slots;
  const int4 *recs;
  int total;
  unsigned *counter;
};

// Sums this step's columns until the counter runs out.
__device__ void gh_help(const ChainParams &p, const GhWork &w) {
  while (true) {
    const int col = gh_grab(w.counter);
    if (col >= w.total) break;
    gh_column(p, w.slots[col], w.recs[col]);
  }
}

// Bounded wait, block-wide, until ready() (evaluated by thread 0, with
// acquire loads) holds. With `help` the block sums gh columns while it waits,
// so a wait on gh marks ends even when no other block is free to sum. False
// when the limit passes or another block aborted.
template <typename Ready>
__device__ bool wait_for(const ChainParams &p, const GhWork *help, Ready ready) {
  __shared__ int s_state;   // 0: wait, 1: ready, 2: give up
  uint64_t t0 = 0;
  bool idle = help == nullptr;
  for (uint32_t it = 0;; ++it) {
    if (threadIdx.x == 0) {
      int st = ready() ? 1 : 0;
      if (st == 0 && idle && (it & 15u) == 0u) {
        const uint64_t now = global_ns();
        if (t0 == 0) t0 = now;
        else if (now - t0 > p.limit_ns || ld_acquire_s32(&p.ctrl->abort)) st = 2;
      }
      s_state = st;
    }
    __syncthreads();
    const int st = s_state;
    __syncthreads();
    if (st) return st == 1;
    if (help) {
      const int col = gh_grab(help->counter);
      idle = col >= help->total;
      if (!idle) gh_column(p, help->slots[col], help->recs[col]);
    }
  }
}

// ---------------------------------------------------------------- request tables

struct Tables {
  float *child_score;    // [e_cap][k]
  int32_t *child_tok;    // [e_cap][k]
  int16_t *child_exp;    // [e_cap][k]
  int8_t *exp_depth;     // [e_cap]
  int16_t *exp_parent;   // [e_cap]
  float *exp_score;      // [e_cap]
  int32_t *exp_tok;      // [e_cap]
  int16_t *run_e;        // [N+1]
  uint8_t *run_head;     // [N+1]
  int16_t *run_pos;      // [N+1]
  uint8_t *vhead;        // [N+1]
  float *run_hs;         // [N+1] score of each run's head (NaN: exhausted)
  float *vhs;            // [N+1] the same for the virtual walk
  int16_t *par;          // [N+1] parents of the output rows
  float *scratch;
};

__device__ Tables tables(const ChainParams &p, unsigned char *smem) {
  Tables t;
  t.child_score = reinterpret_cast<float *>(smem + p.sm_child_score);
  t.child_tok = reinterpret_cast<int32_t *>(smem + p.sm_child_tok);
  t.child_exp = reinterpret_cast<int16_t *>(smem + p.sm_child_exp);
  t.exp_depth = reinterpret_cast<int8_t *>(smem + p.sm_exp_depth);
  t.exp_parent = reinterpret_cast<int16_t *>(smem + p.sm_exp_parent);
  t.exp_score = reinterpret_cast<float *>(smem + p.sm_exp_score);
  t.exp_tok = reinterpret_cast<int32_t *>(smem + p.sm_exp_tok);
  t.run_e = reinterpret_cast<int16_t *>(smem + p.sm_run_e);
  t.run_head = reinterpret_cast<uint8_t *>(smem + p.sm_run_head);
  t.run_pos = reinterpret_cast<int16_t *>(smem + p.sm_run_pos);
  t.vhead = reinterpret_cast<uint8_t *>(smem + p.sm_vhead);
  t.run_hs = reinterpret_cast<float *>(smem + p.sm_run_hs);
  t.vhs = reinterpret_cast<float *>(smem + p.sm_vhs);
  t.par = reinterpret_cast<int16_t *>(smem + p.sm_par);
  t.scratch = reinterpret_cast<float *>(smem + p.sm_scratch);
  return t;
}

// Frontier argmax, warp-level. Run r belongs to lane r % 32; every lane keeps,
// in registers, the best of its own runs as (key, run) with key = order image
// of the head score (0: exhausted). The warp's best run under (score desc, run
// index asc) is then one max-reduction, one vote and one min-reduction.
struct LaneBest {
  uint32_t key;
  int run;
};

__device__ __forceinline__ uint32_t hs_key(float s) { return s == s ? float_order_bits(s) : 0u; }

// this lane's best among runs lane, lane + 32, ... < n_runs (ascending, so ties keep the lowest)
__device__ __forceinline__ LaneBest lane_scan(const float *hs, int n_runs, int lane) {
  LaneBest lb{0u, -1};
  for (int r = lane; r < n_runs; r += 32) {
    const uint32_t k = hs_key(hs[r]);
    if (k > lb.key) { lb.key = k; lb.run = r; }
  }
  return lb;
}

// the warp's best run, or -1 when every run is exhausted
__device__ __forceinline__ int warp_best(const LaneBest &lb) {
  const uint32_t kmax = __reduce_max_sync(kFull, lb.key);
  if (kmax == 0u) return -1;
  const uint32_t r = (lb.key == kmax) ? static_cast<uint32_t>(lb.run) : 0xffffffffu;
  return static_cast<int>(__reduce_min_sync(kFull, r));
}

// score of entry h of run r's children, NaN past the last child
__device__ __forceinline__ float head_score(const ChainParams &p, const Tables &t, int er, int h) {
  return (h < p.k) ? t.child_score[er * p.k + h] : __int_as_float(0x7fc00000);
}

// The GEMM input column of a state: fp32 (CUDA-core path) or three bf16 terms
// hi + mid + lo that reproduce the fp32 value to about 24 bits (tensor-core
// path; the products with the exact bf16 weights then keep fp32 accuracy).
__device__ __forceinline__ void write_column(const ChainParams &p, int slot, int u, float s) {
  if (p.umma) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(s);
    const float r1 = s - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    uint16_t *c = p.gin16 + bcol_index(p, slot, u);
    c[0] = __bfloat16_as_ushort(hi);
    c[kTermBytes / 2] = __bfloat16_as_ushort(mid);
    c[kTermBytes] = __bfloat16_as_ushort(lo);
  } else {
    p.gin[static_cast<size_t>(slot) * p.d_s + u] = s;
  }
}

__device__ __forceinline__ void write_column4(const ChainParams &p, int slot, int u, float4 s) {
  if (p.umma) {
    const float v[4] = {s.x, s.y, s.z, s.w};
    uint32_t hb[4], mb[4], lb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v[i]);
      const float r1 = v[i] - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
      hb[i] = __bfloat16_as_ushort(hi);
      mb[i] = __bfloat16_as_ushort(mid);
      lb[i] = __bfloat16_as_ushort(lo);
    }
    uint16_t *c = p.gin16 + bcol_index(p, slot, u);
    *reinterpret_cast<uint2 *>(c) = make_uint2(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16));
    *reinterpret_cast<uint2 *>(c + kTermBytes / 2) =
        make_uint2(mb[0] | (mb[1] << 16), mb[2] | (mb[3] << 16));
    *reinterpret_cast<uint2 *>(c + kTermBytes) =
        make_uint2(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16));
  } else {
    *reinterpret_cast<float4 *>(p.gin + static_cast<size_t>(slot) * p.d_s + u) = s;
  }
}

// ------------------------------------------------------------ request phase

// The warp sums of G values at once (G a power of two, at most 32): at each
// halving exchange a lane keeps the half of its values selected by one lane
// bit and adds its partner's copy of that half, so after log2(G) exchanges a
// lane holds one value summed over 2^log2(G) lanes, then a plain butterfly
// finishes it; G - 1 + 5 - log2(G) shuffles instead of 5 G. Returns to lane q
// (q < G) the warp sum of a[q] (a fixed order of additions, deterministic).
template <int G>
__device__ __forceinline__ float warp_sum_many(float (&a)[G], int lane) {
  static_assert(G >= 1 && G <= 32 && (G & (G - 1)) == 0, "power of two");
  int lg = 0;
#pragma unroll
  for (int n = G; n > 1; n >>= 1) ++lg;
#pragma unroll
  for (int n = G, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? a[i] : a[i + n / 2];
      const float keep = upper ? a[i + n / 2] : a[i];
      a[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
#pragma unroll
  for (int o = 16 >> lg; o >= 1; o >>= 1) a[0] += __shfl_xor_sync(kFull, a[0], o);
  // value q sits at the lanes whose bits 4 .. 5 - lg spell q
  return __shfl_sync(kFull, a[0], (lane << (5 - lg)) & 31);
}

// Children of the nodes the last GEMM expanded for request b: the columns
// c = g, g + G, ... of the request (member g of its group of G blocks), one
// warp per node. A warp forms h = SiLU(U_j + p) (p summed over the K-chunk
// partials in fixed order) and the corrected logits L_c = (L_base^j[c] +
// W2[c,:] h) / T of the M candidates, then the log-sum-exp over them and the k
// best (L desc, id asc) as the node's children, with scores score(node) + L_c
// - lse: into the request's shared tables when this block is the group's
// leader (t != nullptr), else to global memory as self-validating words. The
// prepared rows of the four best children (the likeliest next expansions) are
// fetched into L2.
template <int WDT, int SLOTS, bool SMALL_R>
__device__ void score_cols(const ChainParams &p, const Tables *t, int b, int g, const ColList &cl,
                           const int *slots, float T, float *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nq = p.r / 8;
  const int R = 3 * p.d_s + p.r;
  const size_t plane = static_cast<size_t>(p.cols_cap) * R;
  const float ninf = -__int_as_float(0x7f800000);
  constexpr int G = WDT == 1 ? 16 : 8;   // candidate rows in flight
  const int first = cl.req_first[b], cnt = cl.req_cnt[b];
  const int nmine = cnt > g ? (cnt - g + p.grp - 1) / p.grp : 0;
  if (nmine == 0) return;
  // wpn warps share a node (a power of two): every node's candidates take one
  // round of row loads when the member has few nodes
  int wpn = kWarps;
  while (wpn > 1 && wpn * nmine > kWarps) wpn >>= 1;
  const int npr = kWarps / wpn;               // nodes per round
  const int wq = warp % wpn, slot_in_round = warp / wpn;
  const int mq = (p.M + wpn - 1) / wpn;       // candidates per warp
  float *Lw = sm + slot_in_round * p.M;
  float *hbuf = sm + kWarps * p.M + warp * p.r;   // used only when r > 256
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  for (int r0 = 0; r0 < nmine; r0 += npr) {
    const int i = r0 + slot_in_round;
    const int c = g + i * p.grp;
    const int4 rec = i < nmine ? cl.recs[first + c] : make_int4(kState0, 0, 0, 0);
    const bool live = rec.x != kState0;   // (the state0 column of the first step is not scored)
    const int e = rec.x;
    const int slot = live ? slots[first + c] : 0;
    const int j = live ? static_cast<int>(static_cast<unsigned>(rec.y) >> 16) : 1;
    const float base_score = __int_as_float(rec.w);
    const size_t row = static_cast<size_t>(p.b0 + b) * p.D + (j - 1);
    const int32_t *cid = p.cand_id + row * p.M;
    const float *cval = p.cand_val + row * p.M;
    const float *U = p.U + row * p.r;
    uint64_t t_in = clock_me ? global_ns() : 0;
    // the candidate ids of the finishing pass, loaded early
    int fid[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int ci = s * 32 + lane;
      fid[s] = (live && wq == 0 && ci < p.M) ? __ldg(cid + ci) : -1;
    }
    if (live) {
      const int c_beg = wq * mq, c_end = min(p.M, c_beg + mq);
      // the first group's ids and base values, in the same round trip as the
      // p partials and U below
      const bool mine0 = lane < G && c_beg + lane < c_end;
      const int id0 = mine0 ? __ldg(cid + c_beg + lane) : -1;
      const float base0 = mine0 ? __ldg(cval + c_beg + lane) : 0.f;
      float h[8];
      if (SMALL_R) {
        float pa[8], uu[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pa[q] = 0.f;
          uu[q] = lane < nq ? __ldg(U + 8 * lane + q) : 0.f;
        }
        if (lane < nq) {
          if (p.umma) {
            const float *src = p.partial + static_cast<size_t>(slot) * R + 3 * p.d_s + 8 * lane;
            for (int z0 = 0; z0 < p.ks; z0 += 4) {
              float4 v[4][2];
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                const bool ok = z0 + z < p.ks;
                const float4 *q = reinterpret_cast<const float4 *>(src + (z0 + z) * plane);
                v[z][0] = ok ? __ldcg(q) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[z][1] = ok ? __ldcg(q + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                pa[0] += v[z][0].x; pa[1] += v[z][0].y; pa[2] += v[z][0].z; pa[3] += v[z][0].w;
                pa[4] += v[z][1].x; pa[5] += v[z][1].y; pa[6] += v[z][1].z; pa[7] += v[z][1].w;
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              pa[q] = ldcg(p.pbuf + static_cast<size_t>(slot) * p.r + 8 * lane + q);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) h[q] = (lane < nq) ? siluf_(uu[q] + pa[q]) : 0.f;
      } else {
        // h in shared memory (r > 256): p summed over the chunks here
        for (int q = lane; q < p.r; q += 32) {
          float a = 0.f;
          if (p.umma) {
            for (int z = 0; z < p.ks; ++z)
              a += ldcg(p.partial + z * plane + static_cast<size_t>(slot) * R + 3 * p.d_s + q);
          } else {
            a = ldcg(p.pbuf + static_cast<size_t>(slot) * p.r + q);
          }
          hbuf[q] = siluf_(__ldg(U + q) + a);
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) h[q] = 0.f;
      }
      if (clock_me) {
        const uint64_t now = global_ns();
        p.ctrl->t_ns[13] += now - t_in;
        t_in = now;
      }
      for (int c0 = c_beg; c0 < c_end; c0 += G) {
        const int my_c = c0 + lane;
        const bool mine = lane < G && my_c < c_end;
        const int my_id = c0 == c_beg ? id0 : (mine ? __ldg(cid + my_c) : -1);
        const float my_base = c0 == c_beg ? base0 : (mine ? __ldg(cval + my_c) : 0.f);
        float acc[G];
        int ids[G];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          ids[q] = __shfl_sync(kFull, my_id, q);
          acc[q] = 0.f;
        }
        if (SMALL_R && WDT == 1) {
          uint4 raw[G];                      // eight bf16 weights per row and lane
#pragma unroll
          for (int q = 0; q < G; ++q)
            raw[q] = (ids[q] >= 0 && lane < nq)
                         ? __ldg(reinterpret_cast<const uint4 *>(
                               static_cast<const uint16_t *>(p.W2) +
                               static_cast<size_t>(ids[q]) * p.r + 8 * lane))
                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const uint32_t w4[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              acc[q] = fmaf(__uint_as_float(w4[x] << 16), h[2 * x], acc[q]);
              acc[q] = fmaf(__uint_as_float(w4[x] & 0xffff0000u), h[2 * x + 1], acc[q]);
            }
          }
        } else if (SMALL_R) {
          float wf[G][8];
#pragma unroll
          for (int q = 0; q < G; ++q) {
            if (ids[q] >= 0 && lane < nq) {
              load8<WDT>(p.W2, static_cast<size_t>(ids[q]) * p.r + 8 * lane, wf[q]);
            } else {
#pragma unroll
              for (int x = 0; x < 8; ++x) wf[q][x] = 0.f;
            }
          }
#pragma unroll
          for (int q = 0; q < G; ++q)
#pragma unroll
            for (int x = 0; x < 8; ++x) acc[q] = fmaf(wf[q][x], h[x], acc[q]);
        } else {
#pragma unroll 1
          for (int q = lane; q - lane < nq; q += 32) {
            if (q < nq) {
              float hq[8];
#pragma unroll
              for (int x = 0; x < 8; ++x) hq[x] = hbuf[8 * q + x];
#pragma unroll
              for (int y = 0; y < G; ++y) {
                if (ids[y] >= 0) {
                  float wf[8];
                  load8<WDT>(p.W2, static_cast<size_t>(ids[y]) * p.r + 8 * q, wf);
#pragma unroll
                  for (int x = 0; x < 8; ++x) acc[y] = fmaf(wf[x], hq[x], acc[y]);
                }
              }
            }
          }
        }
        const float my_dl = warp_sum_many<G>(acc, lane);   // lane q < G: candidate c0 + q
        if (mine) Lw[my_c] = my_id >= 0 ? __fdiv_rn(my_base + my_dl, T) : ninf;
      }
    }
    __syncthreads();
    if (clock_me) {
      const uint64_t now = global_ns();
      p.ctrl->t_ns[14] += now - t_in;
      t_in = now;
    }
    if (live && wq == 0) {
      uint64_t key[SLOTS];
      float Lv[SLOTS];
      float mx = ninf;
#pragma unroll
      for (int s2 = 0; s2 < SLOTS; ++s2) {
        const int ci = s2 * 32 + lane;
        key[s2] = 0ull;
        Lv[s2] = ninf;
        if (ci < p.M && fid[s2] >= 0) {
          Lv[s2] = Lw[ci];
          key[s2] = make_key(Lv[s2], static_cast<uint32_t>(fid[s2]));
        }
        mx = fmaxf(mx, Lv[s2]);
      }
      mx = warp_max(mx);
      float sum = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < SLOTS; ++s2)
        if (s2 * 32 + lane < p.M) sum += expf(Lv[s2] - mx);
      sum = warp_sum(sum);
      const float lse = (mx == ninf) ? ninf : mx + logf(sum);
      warp_sort_desc<SLOTS>(key, lane);
#pragma unroll
      for (int s2 = 0; s2 < SLOTS; ++s2) {
        const int x = s2 * 32 + lane;
        if (x < p.k) {
          const float L = key_value(key[s2]);
          const float lp = (lse == ninf) ? ninf : L - lse;
          const int tok = static_cast<int32_t>(key_id(key[s2]));
          if (t) {
            t->child_score[e * p.k + x] = base_score + lp;
            t->child_tok[e * p.k + x] = tok;
            t->child_exp[e * p.k + x] = -1;
          } else {
            // one 64-bit store per child: the leader sees it whole or not at all
            const unsigned long long w =
                (static_cast<unsigned long long>(static_cast<uint32_t>(tok)) << 32) |
                __float_as_uint(base_score + lp);
            st_relaxed_u64(p.kids + static_cast<size_t>(slot) * p.k + x, w);
          }
          // (a bulk prefetch of a bad address is a fault: the token is checked)
          if (x < 4 && j < p.D && tok >= 0 && tok < p.V)
            prefetch_l2(p.G + static_cast<size_t>(tok) * 3 * p.d_s,
                        static_cast<uint32_t>(12u * p.d_s));
        }
      }
      if (clock_me) p.ctrl->t_ns[15] += global_ns() - t_in;
    }
    __syncthreads();
  }
}

// GRU cells of member g's share of the request's chosen nodes (columns c = g,
// g + G, ... of its new selection): S_e = GRU(S_parent, x = E[tok]) with the
// input half the prepared row G[tok] (= W_ih E[tok] + b_ih) and the recurrent
// half gh_parent (= W_hh S_parent + b_hh) from the GEMM that expanded the
// parent (the root: state0 and the gh of the state0 column), once its gh mark
// is set. The new state goes to the node store and, as the next GEMM's input,
// to column b * P + c. Two items per thread in flight. False when a bounded
// wait ran out.
__device__ __forceinline__ float gru_unit(float gir, float giz, float gin, float ghr, float ghz,
                                          float ghn, float sp) {
  const float r = sigmoidf_(gir + ghr);
  const float z = sigmoidf_(giz + ghz);
  const float n = tanhf(gin + r * ghn);
  return (1.f - z) * n + z * sp;
}

__device__ bool gru_cols(const ChainParams &p, int b, int g, const GhWork &help,
                         const Tables *t, const TailState *ts) {
  __shared__ int4 s_rec[DT_MAX_SPEC];
  __shared__ int s_n;
  if (threadIdx.x == 0) {
    int m = 0;
    if (t) {   // the leader: its own tables (ts->n_sel is 0 once it is done)
      const int n = ts->done ? 0 : ts->n_sel;
      for (int c = g; c < n; c += p.grp) {
        const int e = ts->sel_e[c];
        s_rec[m++] = col_record(e, t->exp_parent[e], 0, t->exp_tok[e], 0.0f);
      }
    } else {
      const int n = __ldcg(p.col_count + b);
      for (int c = g; c < n; c += p.grp) s_rec[m++] = __ldcg(p.col_rec + b * p.P + c);
    }
    s_n = m;
  }
  __syncthreads();
  const int mine = s_n;
  if (mine == 0) return true;
  if (threadIdx.x < mine) {   // the rows that do not wait for a gh sum, on their way to L2
    const int4 rec = s_rec[threadIdx.x];
    const int pe = (rec.y & 0xffff) - 1;
    if (rec.z >= 0 && rec.z < p.V)
      prefetch_l2(p.G + static_cast<size_t>(rec.z) * 3 * p.d_s,
                  static_cast<uint32_t>(12u * p.d_s));
    if (pe >= 0)
      prefetch_l2(p.S_store + (static_cast<size_t>(b) * (p.e_cap + 1) + pe) * p.d_s,
                  static_cast<uint32_t>(4u * p.d_s));
  }
  // the parents' gh must be summed (tensor-core path: from this or an earlier step)
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  const uint64_t tw = clock_me ? global_ns() : 0;
  if (p.umma &&
      !wait_for(p, &help, [&] {
        for (int i = 0; i < mine; ++i) {
          const int r = s_rec[i].y & 0xffff;   // parent + 1
          if (ld_acquire_u32(gh_mark_of(p, b, r - 1)) == 0u) return false;
        }
        return true;
      }))
    return false;
  if (clock_me) p.ctrl->t_ns[8] += global_ns() - tw;
  const int ds = p.d_s, q4 = ds / 4;
  const int items = mine * q4;
  const size_t ebase = static_cast<size_t>(b) * (p.e_cap + 1);
  constexpr int IT = 2;
  for (int i0 = threadIdx.x; i0 < items; i0 += IT * kThreads) {
    float4 gi[IT][3], gh[IT][3], sp[IT];
    int col[IT], u[IT];
    size_t so[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      const int i = i0 + k * kThreads;
      col[k] = -1;
      if (i < items) {
        const int m = i / q4;
        u[k] = (i - m * q4) * 4;
        col[k] = g + m * p.grp;
        const int4 rec = s_rec[m];
        const int e = rec.x, pe = (rec.y & 0xffff) - 1, tok = rec.z;
        const float *gp = p.G + static_cast<size_t>(tok) * 3 * ds + u[k];
        const float *ghp = p.gh_store + (ebase + (pe < 0 ? p.e_cap : pe)) * 3 * ds + u[k];
        const float *spp = pe < 0 ? p.state0 + static_cast<size_t>(p.b0 + b) * ds + u[k]
                                  : p.S_store + (ebase + pe) * ds + u[k];
        so[k] = (ebase + e) * ds + u[k];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          gi[k][q] = __ldg(reinterpret_cast<const float4 *>(gp + q * ds));
          gh[k][q] = __ldcg(reinterpret_cast<const float4 *>(ghp + q * ds));
        }
        sp[k] = __ldcg(reinterpret_cast<const float4 *>(spp));
      }
    }
#pragma unroll
    for (int k = 0; k < IT; ++k) {
      if (col[k] < 0) continue;
      float4 v;
      v.x = gru_unit(gi[k][0].x, gi[k][1].x, gi[k][2].x, gh[k][0].x, gh[k][1].x, gh[k][2].x, sp[k].x);
      v.y = gru_unit(gi[k][0].y, gi[k][1].y, gi[k][2].y, gh[k][0].y, gh[k][1].y, gh[k][2].y, sp[k].y);
      v.z = gru_unit(gi[k][0].z, gi[k][1].z, gi[k][2].z, gh[k][0].z, gh[k][1].z, gh[k][2].z, sp[k].z);
      v.w = gru_unit(gi[k][0].w, gi[k][1].w, gi[k][2].w, gh[k][0].w, gh[k][1].w, gh[k][2].w, sp[k].w);
      *reinterpret_cast<float4 *>(p.S_store + so[k]) = v;
      write_column4(p, b * p.P + col[k], u[k], v);
    }
  }
  if (p.umma) fence_async_global();   // the columns are read by bulk copies next
  __syncthreads();
  return true;
}

__device__ void write_row(const ChainParams &p, int b, int pos, int tok, int par, int dep,
                          float sc) {
  const size_t o = static_cast<size_t>(p.b0 + b) * (p.N + 1) + pos;
  p.tokens[o] = tok;
  p.parents[o] = par;
  p.depths[o] = dep;
  p.scores[o] = sc;
}

// Rows after the last pop, the ancestor mask, the status; then leave the search.
__device__ void finalize(const ChainParams &p, const Tables &t, TailState &ts, int b,
                         bool counted) {
  __syncthreads();
  const int count = ts.count;
  const int first_empty = ts.status ? 0 : count + 1;
  for (int i = first_empty + threadIdx.x; i <= p.N; i += kThreads)
    write_row(p, b, i, -1, -1, -1, -__int_as_float(0x7f800000));
  if (p.mask) {
    const size_t n1 = static_cast<size_t>(p.N) + 1;
    uint8_t *mb = p.mask + static_cast<size_t>(p.b0 + b) * n1 * n1;
    for (size_t i = threadIdx.x; i < n1 * n1; i += kThreads) mb[i] = 0;
    __syncthreads();
    if (!ts.status) {
      for (int i = threadIdx.x; i <= count; i += kThreads)
        for (int a = i; a >= 0; a = t.par[a]) mb[static_cast<size_t>(i) * n1 + a] = 1;
    }
  }
  if (threadIdx.x == 0) {
    p.status[p.b0 + b] = ts.status;
    ts.done = 1;
    if (counted) atomicSub(&p.ctrl->active, 1);
  }
  __syncthreads();
}

// Pop in canonical order until done or until a popped node needs children that
// are not known yet; then choose the next nodes to expand. Warp 0 only. Shared
// tables are read by every lane (broadcast); a run's entries are written by the
// lane that owns it.
__device__ void replay_and_select(const ChainParams &p, const Tables &t, TailState &ts, int b,
                                  int lane) {
  int count = ts.count, n_runs = ts.n_runs;
  const bool clock_me = blockIdx.x == 0 && lane == 0;
  long long c_start = clock64();
  int it_pop = 0;
  LaneBest lb = lane_scan(t.run_hs, n_runs, lane);
  bool done = false;
  while (true) {
    ++it_pop;
    if (count >= p.N) { done = true; break; }
    const int r = warp_best(lb);
    if (r < 0) { done = true; break; }
    const int h = t.run_head[r], er = t.run_e[r];
    const int dep = t.exp_depth[er] + 1, pos = count + 1;
    const int ce = t.child_exp[er * p.k + h];
    const bool need = dep < p.D && pos < p.N;
    if (need && ce < 0) break;  // stall: this node's children are not known yet
    const int rpos = t.run_pos[r];
    if (lane == 0) {
      write_row(p, b, pos, t.child_tok[er * p.k + h], rpos, dep, t.child_score[er * p.k + h]);
      t.par[pos] = static_cast<int16_t>(rpos);
    }
    if (lane == (r & 31)) {
      t.run_head[r] = static_cast<uint8_t>(h + 1);
      t.run_hs[r] = head_score(p, t, er, h + 1);
      lb = lane_scan(t.run_hs, n_runs, lane);
    }
    if (need && lane == (n_runs & 31)) {
      const float hs0 = head_score(p, t, ce, 0);
      t.run_e[n_runs] = static_cast<int16_t>(ce);
      t.run_head[n_runs] = 0;
      t.run_hs[n_runs] = hs0;
      t.run_pos[n_runs] = static_cast<int16_t>(pos);
      const uint32_t k0 = hs_key(hs0);
      if (k0 > lb.key) { lb.key = k0; lb.run = n_runs; }
    }
    n_runs += need ? 1 : 0;
    count = pos;
    __syncwarp();
  }
  if (clock_me) {
    const long long c = clock64();
    p.ctrl->t_ns[28] += it_pop;
    p.ctrl->t_ns[29] += c - c_start;
    c_start = c;
  }
  if (done) {
    if (lane == 0) {
      ts.count = count; ts.n_runs = n_runs; ts.n_sel = 0; ts.done = 2;
      p.col_count[b] = 0;
    }
    __syncwarp();
    return;
  }
  // choose the stalled node plus up to P-1 of the next frontier nodes in order,
  // walking a copy of the run heads (vhead / vhs)
  const int spec_left = p.e_cap - p.N - ts.spec_used;
  for (int r = lane; r < n_runs; r += 32) {
    t.vhead[r] = t.run_head[r];
    t.vhs[r] = t.run_hs[r];
  }
  __syncwarp();
  int nsel = 0, nspec = 0, i = 0;
  const int e_count = ts.e_count;
  int it_sel = 0;
  while (nsel < p.P) {
    ++it_sel;
    const int r = warp_best(lb);
    if (r < 0) break;
    ++i;
    if (count + i >= p.N) break;
    const int h = t.vhead[r], er = t.run_e[r];
    const int dep = t.exp_depth[er] + 1;
    const int slot_c = er * p.k + h;
    const bool fresh = dep < p.D && t.child_exp[slot_c] < 0;
    const bool take = fresh && (nsel == 0 || nspec < spec_left);
    if (take && lane == 0) {
      const int e = e_count + nsel;
      t.child_exp[slot_c] = static_cast<int16_t>(e);
      t.exp_depth[e] = static_cast<int8_t>(dep);
      t.exp_parent[e] = static_cast<int16_t>(er);
      t.exp_score[e] = t.child_score[slot_c];
      t.exp_tok[e] = t.child_tok[slot_c];
      ts.sel_e[nsel] = e;
      p.col_rec[b * p.P + nsel] =
          col_record(e, er, dep + 1, t.child_tok[slot_c], t.child_score[slot_c]);
    }
    if (lane == (r & 31)) {
      t.vhead[r] = static_cast<uint8_t>(h + 1);
      t.vhs[r] = head_score(p, t, er, h + 1);
      lb = lane_scan(t.vhs, n_runs, lane);
    }
    if (take) {
      nspec += (nsel > 0) ? 1 : 0;
      ++nsel;
    }
    __syncwarp();
  }
  if (clock_me) {
    p.ctrl->t_ns[30] += it_sel;
    p.ctrl->t_ns[31] += clock64() - c_start;
  }
  if (lane == 0) {
    ts.count = count;
    ts.n_runs = n_runs;
    ts.e_count = e_count + nsel;
    ts.n_sel = nsel;
    ts.spec_used += nspec;
    p.col_count[b] = nsel;
    atomicAdd(&p.ctrl->expansions, static_cast<unsigned>(nsel));
  }
  __syncwarp();
}


// The same replay and selection with the run state in registers: run r lives
// in slot r / 32 of lane r % 32 as two packed words and its head score:
//   w1 = head h (6 bits) | expansion er (12 bits) << 6 | output row of its parent (11 bits) << 18
//   w2 = depth of its entries (8 bits) | (expansion of the head + 1) << 8
// so a pop needs two shuffles from the owning lane and no shared-memory lookup,
// and only the owner of the popped run (and of a new run) reads the next head's
// score and expansion. The output rows and the chosen expansions are logged in
// registers (pop i and choice i by lane i % 32) and written after the loops.
// Used while the runs fit (N + 1 <= 32 RS); the run state is loaded from and
// stored back to the shared tables.
template <int RS>
__device__ __forceinline__ uint32_t pick_slot(const uint32_t (&v)[RS], int s) {
  uint32_t x = v[0];
#pragma unroll
  for (int i = 1; i < RS; ++i) x = (s == i) ? v[i] : x;
  return x;
}

template <int RS>
__device__ __forceinline__ LaneBest lane_best_reg(const float (&hs)[RS], int n_runs, int lane) {
  LaneBest lb{0u, -1};
#pragma unroll
  for (int s = 0; s < RS; ++s) {
    const int r = s * 32 + lane;
    if (r < n_runs) {
      const uint32_t k = hs_key(hs[s]);
      if (k > lb.key) { lb.key = k; lb.run = r; }
    }
  }
  return lb;
}

__device__ __forceinline__ uint32_t run_w1(int h, int er, int pos) {
  return static_cast<uint32_t>(h) | (static_cast<uint32_t>(er) << 6) |
         (static_cast<uint32_t>(pos) << 18);
}
__device__ __forceinline__ uint32_t run_w2(int dep, int ce) {
  return static_cast<uint32_t>(dep) | (static_cast<uint32_t>(ce + 1) << 8);
}
// expansion of entry h of expansion er's children (-1: not expanded; -2: past the end)
__device__ __forceinline__ int head_exp(const ChainParams &p, const Tables &t, int er, int h) {
  return h < p.k ? t.child_exp[er * p.k + h] : -2;
}

// Per-run state of the register replay, slot s of lane l holding run
// r = 32 s + l: the head (w1, w2, score rh), the next head (its score nrh and
// w2 nw2) and, when the head is expanded, its first child (score fh, and fce
// the first child's expansion, -2 when there is none). With the next values at
// hand a pop needs one round of shared-memory loads, all issued together and
// off the path to the next pop's argmax.
template <int RS>
struct RunRegs {
  uint32_t w1[RS], w2[RS], nw2[RS];
  float rh[RS], nrh[RS], fh[RS];
  int fce[RS];
};

template <int RS>
__device__ __forceinline__ float pick_f(const float (&v)[RS], int s) {
  float x = v[0];
#pragma unroll
  for (int i = 1; i < RS; ++i) x = (s == i) ? v[i] : x;
  return x;
}
template <int RS>
__device__ __forceinline__ int pick_i(const int (&v)[RS], int s) {
  int x = v[0];
#pragma unroll
  for (int i = 1; i < RS; ++i) x = (s == i) ? v[i] : x;
  return x;
}

// the expansion field of a w2 word: run_w2 stores ce + 1 >= -1 in the upper 24
// bits, so an arithmetic shift gives back -2 (past the last child) as well
__device__ __forceinline__ int w2_exp(uint32_t w2) { return (static_cast<int>(w2) >> 8) - 1; }

template <int RS>
__device__ void replay_and_select_reg(const ChainParams &p, const Tables &t, TailState &ts, int b,
                                      int lane) {
  const float nan = __int_as_float(0x7fc00000);
  int count = ts.count, n_runs = ts.n_runs;
  const int count0 = count;
  const bool clock_me = blockIdx.x == 0 && lane == 0;
  long long c_start = clock64();
  int it_pop = 0;
  auto score_at = [&](int er, int h) { return h < p.k ? t.child_score[er * p.k + h] : nan; };
  auto exp_at = [&](int er, int h) { return h < p.k ? static_cast<int>(t.child_exp[er * p.k + h]) : -2; };
  RunRegs<RS> R;
  uint32_t plog[RS];
#pragma unroll
  for (int s = 0; s < RS; ++s) {
    const int r = s * 32 + lane;
    plog[s] = 0u;
    R.w1[s] = 0u; R.w2[s] = 0u; R.nw2[s] = 0u;
    R.rh[s] = nan; R.nrh[s] = nan; R.fh[s] = nan; R.fce[s] = -2;
    if (r < n_runs) {
      const int h = t.run_head[r], er = t.run_e[r];
      const int dep = t.exp_depth[er] + 1, ce = exp_at(er, h);
      R.w1[s] = run_w1(h, er, t.run_pos[r]);
      R.w2[s] = run_w2(dep, ce);
      R.rh[s] = t.run_hs[r];
      R.nrh[s] = score_at(er, h + 1);
      R.nw2[s] = run_w2(dep, exp_at(er, h + 1));
      if (ce >= 0) { R.fh[s] = score_at(ce, 0); R.fce[s] = exp_at(ce, 0); }
    }
  }
  LaneBest lb = lane_best_reg<RS>(R.rh, n_runs, lane);
  // one pop of run r (owner lane own, slot sl): its head advances to the next
  // entry; when `grow`, the popped node's children (expansion ce) become run
  // n_runs. Every lane evaluates the same loads (broadcast) and selects.
  auto advance = [&](int sl, int own, uint32_t a, int dep, uint32_t nw, float nr, bool grow,
                     int ce, float f, int fc, int pos) {
    const int h = a & 63, er = (a >> 6) & 4095;
    const int ce1 = w2_exp(nw);   // the new head's expansion
    const float s2 = score_at(er, h + 2);
    const int e2 = exp_at(er, h + 2);
    const float f1 = ce1 >= 0 ? score_at(ce1, 0) : nan;
    const int g1 = ce1 >= 0 ? exp_at(ce1, 0) : -2;
    float c1 = nan, fr = nan;
    int x1 = -2, xr = -2;
    if (grow) {
      c1 = score_at(ce, 1);
      x1 = exp_at(ce, 1);
      if (fc >= 0) { fr = score_at(fc, 0); xr = exp_at(fc, 0); }
    }
    const int ns = n_runs >> 5, nl = n_runs & 31;
#pragma unroll
    for (int s = 0; s < RS; ++s) {
      if (lane == own && s == sl) {
        R.w1[s] = a + 1u; R.w2[s] = nw; R.rh[s] = nr;
        R.nrh[s] = s2; R.nw2[s] = run_w2(dep, e2); R.fh[s] = f1; R.fce[s] = g1;
      }
      if (grow && lane == nl && s == ns) {
        R.w1[s] = run_w1(0, ce, pos); R.w2[s] = run_w2(dep + 1, fc); R.rh[s] = f;
        R.nrh[s] = c1; R.nw2[s] = run_w2(dep + 1, x1); R.fh[s] = fr; R.fce[s] = xr;
      }
    }
  };
  bool done = false;
  while (true) {
    ++it_pop;
    if (count >= p.N) { done = true; break; }
    const int r = warp_best(lb);
    if (r < 0) { done = true; break; }
    const int sl = r >> 5, own = r & 31;
    const uint32_t a = __shfl_sync(kFull, pick_slot<RS>(R.w1, sl), own);
    const uint32_t c = __shfl_sync(kFull, pick_slot<RS>(R.w2, sl), own);
    const uint32_t nw = __shfl_sync(kFull, pick_slot<RS>(R.nw2, sl), own);
    const float nr = __shfl_sync(kFull, pick_f<RS>(R.nrh, sl), own);
    const float f = __shfl_sync(kFull, pick_f<RS>(R.fh, sl), own);
    const int fc = __shfl_sync(kFull, pick_i<RS>(R.fce, sl), own);
    const int dep = c & 255, ce = w2_exp(c), pos = count + 1;
    const bool need = dep < p.D && pos < p.N;
    if (need && ce < 0) break;  // stall: this node's children are not known yet
    const int i = pos - count0 - 1;   // pop index within this step
    if (lane == (i & 31)) {
#pragma unroll
      for (int s = 0; s < RS; ++s)
        if (s == (i >> 5)) plog[s] = a;
    }
    advance(sl, own, a, dep, nw, nr, need, ce, f, fc, pos);
    n_runs += need ? 1 : 0;
    count = pos;
    lb = lane_best_reg<RS>(R.rh, n_runs, lane);
  }
  // the popped rows (pop i logged by lane i % 32), then the run state back to
  // the shared tables (it persists across steps)
  const int n_pop = count - count0;
#pragma unroll
  for (int s = 0; s < RS; ++s) {
    const int i = s * 32 + lane;
    if (i < n_pop) {
      const uint32_t a = plog[s];
      const int h = a & 63, er = (a >> 6) & 4095, rpos = static_cast<int>(a >> 18);
      const int pos = count0 + 1 + i;
      write_row(p, b, pos, t.child_tok[er * p.k + h], rpos, t.exp_depth[er] + 1,
                t.child_score[er * p.k + h]);
      t.par[pos] = static_cast<int16_t>(rpos);
    }
    const int r = s * 32 + lane;
    if (r < n_runs) {
      t.run_head[r] = static_cast<uint8_t>(R.w1[s] & 63);
      t.run_e[r] = static_cast<int16_t>((R.w1[s] >> 6) & 4095);
      t.run_pos[r] = static_cast<int16_t>(R.w1[s] >> 18);
      t.run_hs[r] = R.rh[s];
    }
  }
  __syncwarp();
  if (clock_me) {
    const long long cc = clock64();
    p.ctrl->t_ns[28] += it_pop;
    p.ctrl->t_ns[29] += cc - c_start;
    c_start = cc;
  }
  if (done) {
    if (lane == 0) {
      ts.count = count; ts.n_runs = n_runs; ts.n_sel = 0; ts.done = 2;
      p.col_count[b] = 0;
    }
    __syncwarp();
    return;
  }
  // choose the stalled node plus up to P-1 of the next frontier nodes in order,
  // walking the register copy of the run heads (the real state is stored)
  const int spec_left = p.e_cap - p.N - ts.spec_used;
  int nsel = 0, nspec = 0, vi = 0;
  const int e_count = ts.e_count;
  int it_sel = 0;
  uint32_t my_pick = 0xffffffffu;   // choice `lane`: entry (er, h), depth
  while (nsel < p.P) {
    ++it_sel;
    const int r = warp_best(lb);
    if (r < 0) break;
    ++vi;
    if (count + vi >= p.N) break;
    const int sl = r >> 5, own = r & 31;
    const uint32_t a = __shfl_sync(kFull, pick_slot<RS>(R.w1, sl), own);
    const uint32_t c = __shfl_sync(kFull, pick_slot<RS>(R.w2, sl), own);
    const uint32_t nw = __shfl_sync(kFull, pick_slot<RS>(R.nw2, sl), own);
    const float nr = __shfl_sync(kFull, pick_f<RS>(R.nrh, sl), own);
    const int dep = c & 255, ce = w2_exp(c);
    const bool fresh = dep < p.D && ce == -1;
    const bool take = fresh && (nsel == 0 || nspec < spec_left);
    if (take && lane == nsel) my_pick = (a & 0x3ffffu) | (static_cast<uint32_t>(dep) << 18);
    advance(sl, own, a, dep, nw, nr, false, -1, nan, -2, 0);
    lb = lane_best_reg<RS>(R.rh, n_runs, lane);
    if (take) {
      nspec += (nsel > 0) ? 1 : 0;
      ++nsel;
    }
  }
  // the chosen expansions (choice i by lane i)
  if (lane < nsel) {
    const int h = my_pick & 63, er = (my_pick >> 6) & 4095, dep = my_pick >> 18;
    const int slot_c = er * p.k + h;
    const int e = e_count + lane;
    const float sc = t.child_score[slot_c];
    const int tok = t.child_tok[slot_c];
    t.child_exp[slot_c] = static_cast<int16_t>(e);
    t.exp_depth[e] = static_cast<int8_t>(dep);
    t.exp_parent[e] = static_cast<int16_t>(er);
    t.exp_score[e] = sc;
    t.exp_tok[e] = tok;
    ts.sel_e[lane] = e;
    p.col_rec[b * p.P + lane] = col_record(e, er, dep + 1, tok, sc);
  }
  __syncwarp();
  if (clock_me) {
    p.ctrl->t_ns[30] += it_sel;
    p.ctrl->t_ns[31] += clock64() - c_start;
  }
  if (lane == 0) {
    ts.count = count;
    ts.n_runs = n_runs;
    ts.e_count = e_count + nsel;
    ts.n_sel = nsel;
    ts.spec_used += nspec;
    p.col_count[b] = nsel;
    atomicAdd(&p.ctrl->expansions, static_cast<unsigned>(nsel));
  }
  __syncwarp();
}

__device__ void tail_init(const ChainParams &p, const Tables &t, TailState &ts, int b) {
  if (threadIdx.x == 0) {
    ts.count = 0; ts.n_runs = 0; ts.e_count = 0; ts.done = 0; ts.n_sel = 0; ts.spec_used = 0;
    ts.status = DT_OK;
    float T = p.temperature ? p.temperature[p.b0 + b] : 1.0f;
    if (p.req_flags[p.b0 + b] & kReqFlagNonfinite) ts.status = DT_ERR_NONFINITE;
    else if (!(T >= 0.0f) || T == __int_as_float(0x7f800000)) ts.status = DT_ERR_BAD_TEMPERATURE;
    ts.T = (T == 0.0f) ? 1.0f : T;  // T = 0: greedy ordering, read as T = 1
    t.par[0] = -1;
    p.col_count[b] = 0;
  }
  __syncthreads();
  if (ts.status != DT_OK) { finalize(p, t, ts, b, false); return; }
  const int anchor = p.anchor[p.b0 + b];
  if (threadIdx.x == 0) write_row(p, b, 0, anchor, -1, 0, 0.0f);
  if (p.N == 0) { finalize(p, t, ts, b, false); return; }
  // first GEMM column: the initial state, for W_hh state0 + b_hh
  const float *s0 = p.state0 + static_cast<size_t>(p.b0 + b) * p.d_s;
  for (int u = threadIdx.x; u < p.d_s; u += kThreads) write_column(p, b * p.P, u, s0[u]);
  if (p.umma) fence_async_global();
  if (threadIdx.x == 0) {
    p.col_rec[b * p.P] = col_record(kState0, -1, 0, 0, 0.0f);
    p.col_count[b] = 1;
    atomicAdd(&p.ctrl->active, 1);
  }
  // warm L2 with the W2 rows of every candidate of this request (scored by the
  // expansions to come) when the whole wave's rows fit comfortably in L2
  const size_t row_bytes = static_cast<size_t>(p.r) * (p.umma ? 2 : 4);
  if (static_cast<size_t>(p.nb) * p.D * p.M * row_bytes <= (48u << 20)) {
    const int32_t *cid = p.cand_id + static_cast<size_t>(p.b0 + b) * p.D * p.M;
    for (int i = threadIdx.x; i < p.D * p.M; i += kThreads) {
      const int id = cid[i];
      if (id >= 0)
        prefetch_l2(static_cast<const char *>(p.W2) + static_cast<size_t>(id) * row_bytes,
                    static_cast<uint32_t>(row_bytes));
    }
  }
  __syncthreads();
}

// The leader's gather of the other members' children (columns c of request b
// with c % grp != 0): every thread polls its share of the child words until
// each is written, copies them into the tables and empties them again. The
// words were emptied at launch and after the previous step's gather, and the
// grid barrier orders both before this step's writes. False when the limit
// passes or another block aborted.
__device__ bool gather_kids(const ChainParams &p, const Tables &t, int b, const ColList &cl,
                            const int *slots) {
  __shared__ int s_give_up;
  const int first = cl.req_first[b], cnt = cl.req_cnt[b];
  const int nent = cnt * p.k;
  uint64_t t0 = 0;
  if (threadIdx.x == 0) s_give_up = 0;
  for (uint32_t it = 0;; ++it) {
    bool ok = true;
    for (int i = threadIdx.x; i < nent; i += kThreads) {
      const int c = i / p.k, rank = i - c * p.k;
      if (c % p.grp == 0) continue;
      const int e = cl.recs[first + c].x;
      if (e == kState0) continue;
      const unsigned long long w =
          ld_relaxed_u64(p.kids + static_cast<size_t>(slots[first + c]) * p.k + rank);
      if (w == kEmptyKid) {
        ok = false;
      } else {
        t.child_score[e * p.k + rank] = __uint_as_float(static_cast<uint32_t>(w));
        t.child_tok[e * p.k + rank] = static_cast<int32_t>(w >> 32);
        t.child_exp[e * p.k + rank] = -1;
      }
    }
    if (__syncthreads_and(ok)) break;
    if (threadIdx.x == 0 && (it & 15u) == 0u) {
      const uint64_t now = global_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > p.limit_ns || ld_acquire_s32(&p.ctrl->abort)) s_give_up = 1;
    }
    __syncthreads();
    if (s_give_up) return false;
  }
  for (int i = threadIdx.x; i < nent; i += kThreads) {
    const int c = i / p.k, rank = i - c * p.k;
    if (c % p.grp != 0 && cl.recs[first + c].x != kState0)
      p.kids[static_cast<size_t>(slots[first + c]) * p.k + rank] = kEmptyKid;
  }
  __syncthreads();
  return true;
}

// The request phase of one step, member g of request b's group (the leader,
// g = 0, holds the request's tables): score the member's share of the last
// GEMM's nodes; the leader gathers the members' children (waiting for their
// marks), pops, chooses the next nodes and publishes them (the request's
// mark); then every member runs the GRU of its share of them. False when a
// bounded wait ran out.
template <int WDT, int SLOTS>
__device__ bool group_step(const ChainParams &p, const Tables &t, TailState &ts, int b, int g,
                           float *sm, const int *slots, const ColList &cl, const GhWork &help,
                           unsigned mark) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int first = cl.req_first[b], cnt = cl.req_cnt[b];
  if (cnt == 0) return true;   // the request is done (or never started)
  const bool leader = g == 0;
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  uint64_t t0 = clock_me ? global_ns() : 0;
  auto lap = [&](int k) {
    if (clock_me) {
      const uint64_t now = global_ns();
      p.ctrl->t_ns[k] += now - t0;
      t0 = now;
    }
  };
  if (leader && ts.e_count == 0) {
    // the root: expansion 0, S_0 = GRU(state0, E[anchor]); its recurrent half
    // comes from the state0 column of this step
    const int anchor = p.anchor[p.b0 + b];
    if (threadIdx.x == 0) {
      t.exp_depth[0] = 0; t.exp_parent[0] = -1; t.exp_score[0] = 0.0f; t.exp_tok[0] = anchor;
      ts.e_count = 1;
      ts.n_sel = 1;
      ts.sel_e[0] = 0;
      atomicAdd(&p.ctrl->expansions, 1u);
      p.col_rec[b * p.P] = col_record(0, -1, 1, anchor, 0.0f);
      p.col_count[b] = 1;
    }
  } else {
    // 1. children of this member's nodes
    float T = p.temperature ? p.temperature[p.b0 + b] : 1.0f;
    T = (T == 0.0f) ? 1.0f : T;
    if (p.r <= 256) score_cols<WDT, SLOTS, true>(p, leader ? &t : nullptr, b, g, cl, slots, T, sm);
    else score_cols<WDT, SLOTS, false>(p, leader ? &t : nullptr, b, g, cl, slots, T, sm);
    lap(2);
    if (leader) {
      // 2. the other members' children: their words, polled until every one is
      //    written, then emptied again for the next step
      if (p.grp > 1 && cnt > 1 && !gather_kids(p, t, b, cl, slots)) return false;
      if (threadIdx.x == 0 && ts.n_runs == 0) {  // the root's children form the first run
        t.run_e[0] = 0; t.run_head[0] = 0; t.run_pos[0] = 0;
        t.run_hs[0] = head_score(p, t, 0, 0);
        ts.n_runs = 1;
      }
      __syncthreads();
      lap(3);
      // 3. canonical pops, then the next expansions
      if (warp == 0) {
        // runs are at most N + 1: the register replay while they fit 4 x 32
        if (p.N + 1 <= 64) replay_and_select_reg<2>(p, t, ts, b, lane);
        else if (p.N + 1 <= 96) replay_and_select_reg<3>(p, t, ts, b, lane);
        else if (p.N + 1 <= 128) replay_and_select_reg<4>(p, t, ts, b, lane);
        else replay_and_select(p, t, ts, b, lane);
      }
      __syncthreads();
      lap(4);
      if (ts.done == 2) finalize(p, t, ts, b, true);   // (col_count[b] is 0)
    }
  }
  // 4. the selection out (leader) or in (members), then the GRU cells
  if (leader) {
    __syncthreads();
    if (threadIdx.x == 0) st_release_u32(p.sel_mark + b, mark);
  } else if (!wait_for(p, &help, [&] { return ld_acquire_u32(p.sel_mark + b) == mark; })) {
    return false;
  }
  const bool ok = gru_cols(p, b, g, help, leader ? &t : nullptr, leader ? &ts : nullptr);
  lap(5);
  return ok;
}

template <int WDT, int SLOTS>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(ChainParams p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ TailState ts;
  __shared__ int s_active;
  const Tables t = tables(p, smem);
  // request groups: blocks [b G, b G + G) serve request b; member 0 leads
  const int b = blockIdx.x / p.grp, g = blockIdx.x % p.grp;
  const bool grouped = b < p.nb;
  const bool tail = grouped && g == 0;
  // tensor-core blocks: stationary A tile, the slice mbarriers, 256 TMEM columns
  const bool mma_block = p.umma && blockIdx.x < p.n_mt * p.ks;
  UmmaState u;
  u.tmem = 0;
  u.next = 0;
  if (mma_block) {
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + p.sm_mbar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + p.sm_tmem);
    if (threadIdx.x == 0)
      for (int i = 0; i < 2 * kMaxBufs; ++i) mbar_init(&mbar[i], 1);   // full, empty
    load_a_tile(p, smem + p.sm_A);
    fence_async_smem();   // generic stores of the A tile -> tensor-core reads
    if ((threadIdx.x >> 5) == 0) tmem_alloc(tslot, kTmemCols);
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    u.tmem = *tslot;
  }
  if (p.umma && p.ks * p.kc > p.d_s) {
    // K padding of every B column: zero once (A is zero there too, and 0 * NaN
    // from stale bytes must not reach an accumulator)
    const int pad = p.ks * p.kc - p.d_s;
    const int ncol = ((p.cols_cap + 255) >> 8) << 8;
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < ncol * pad; i += gridDim.x * kThreads) {
      uint16_t *c = p.gin16 + bcol_index(p, i / pad, p.d_s + i % pad);
      c[0] = 0; c[kTermBytes / 2] = 0; c[kTermBytes] = 0;
    }
    fence_async_global();
  }
  // marks and child words of an earlier launch must not read as this launch's
  {
    const int wave = p.cols_cap / p.P;
    const int nm = wave + wave * (p.e_cap + 1);
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < nm; i += gridDim.x * kThreads)
      p.sel_mark[i] = 0u;   // sel_mark and gh_mark are consecutive
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < p.cols_cap * p.k;
         i += gridDim.x * kThreads)
      p.kids[i] = kEmptyKid;
  }
  if (tail) tail_init(p, t, ts, b);
  unsigned bar_target = 0;
  bool ok = grid_barrier(&p.ctrl->bar_count, &p.ctrl->abort, gridDim.x, p.limit_ns, bar_target,
                         false, p.test_skip && blockIdx.x == gridDim.x - 1);
  // block 0 accounts its time per phase (for profiling; a few timer reads a step)
  const bool clock_me = blockIdx.x == 0 && threadIdx.x == 0;
  uint64_t t_prev = clock_me ? global_ns() : 0;
  auto lap = [&](int k) {
    if (clock_me) {
      const uint64_t now = global_ns();
      p.ctrl->t_ns[k] += now - t_prev;
      t_prev = now;
    }
  };
  int *slots = reinterpret_cast<int *>(smem + p.sm_slots);
  ColList cl;
  cl.recs = reinterpret_cast<int4 *>(smem + p.sm_recs);
  cl.req_first = slots + p.cols_cap;
  cl.req_cnt = cl.req_first + p.nb;
  float *scratch = reinterpret_cast<float *>(smem + p.sm_scratch);
  for (int step = 0; ok && step < p.N + 3; ++step) {
    if (clock_me) p.ctrl->steps = static_cast<unsigned>(step + 1);
    bool gemm_ok = true;
    int total = 0;
    if (p.umma) {
      gemm_ok = gemm_phase_umma(p, smem, slots, cl, u, total);
    } else {
      gemm_phase<WDT>(p, smem + p.sm_scratch);
      total = compact_slots(p, slots, &cl);
    }
    lap(0);
    ok = grid_barrier(&p.ctrl->bar_count, &p.ctrl->abort, gridDim.x, p.limit_ns, bar_target,
                      !gemm_ok);
    lap(1);
    if (!ok) break;
    // the column counter of the next step starts from zero (this one's was
    // last used before the previous barrier)
    unsigned *counter = (step & 1) ? &p.ctrl->red_next_odd : &p.ctrl->red_next;
    if (blockIdx.x == 0 && threadIdx.x == 0)
      *((step & 1) ? &p.ctrl->red_next : &p.ctrl->red_next_odd) = 0u;
    const unsigned mark = static_cast<unsigned>(step + 1);
    GhWork help;
    help.slots = slots;
    help.recs = cl.recs;
    help.total = p.umma ? total : 0;   // (the CUDA-core GEMM writes gh itself)
    help.counter = counter;
    bool req_ok = true;
    if (grouped) {
      req_ok = group_step<WDT, SLOTS>(p, t, ts, b, g, scratch, slots, cl, help, mark);
      if (clock_me) t_prev = global_ns();
    }
    if (!req_ok && threadIdx.x == 0) atomicExch(&p.ctrl->abort, 1);
    if (p.umma) gh_help(p, help);
    lap(6);
    ok = grid_barrier(&p.ctrl->bar_count, &p.ctrl->abort, gridDim.x, p.limit_ns, bar_target,
                      !req_ok);
    lap(7);
    if (!ok) break;
    if (threadIdx.x == 0) s_active = ld_acquire_s32(&p.ctrl->active);
    __syncthreads();
    if (s_active == 0) break;
  }
  if (tail && !ts.done) {
    if (threadIdx.x == 0) ts.status = DT_ERR_TIMEOUT;
    finalize(p, t, ts, b, true);
  }
  if (mma_block) {  // every MMA of this block has completed (waited in its phase)
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(u.tmem, kTmemCols);
  }
}

}  // namespace

// Shared-memory carve-up of the search kernel for e_cap expansion slots.
static int chain_smem_layout(const Plan &pl, int e_cap, int wave, ChainParams *cp) {
  const dt_dims &d = pl.dims;
  auto al = [](int x, int a) { return (x + a - 1) / a * a; };
  int off = 0;
  const int k = d.k, n1 = d.N + 1;
  cp->sm_child_score = off; off = al(off + e_cap * k * 4, 16);
  cp->sm_child_tok = off;   off = al(off + e_cap * k * 4, 16);
  cp->sm_child_exp = off;   off = al(off + e_cap * k * 2, 16);
  cp->sm_exp_depth = off;   off = al(off + e_cap, 16);
  cp->sm_exp_parent = off;  off = al(off + e_cap * 2, 16);
  cp->sm_exp_score = off;   off = al(off + e_cap * 4, 16);
  cp->sm_exp_tok = off;     off = al(off + e_cap * 4, 16);
  cp->sm_run_e = off;       off = al(off + n1 * 2, 16);
  cp->sm_run_head = off;    off = al(off + n1, 16);
  cp->sm_run_pos = off;     off = al(off + n1 * 2, 16);
  cp->sm_vhead = off;       off = al(off + n1, 16);
  cp->sm_par = off;         off = al(off + n1 * 2, 16);
  cp->sm_run_hs = off;      off = al(off + n1 * 4, 16);
  cp->sm_vhs = off;         off = al(off + n1 * 4, 16);
  cp->sm_A = cp->sm_B = cp->sm_mbar = cp->sm_tmem = 0;
  if (pl.umma) {
    cp->sm_A = off = al(off, 128);    off += 128 * pl.kc * 2;
    cp->sm_B = off = al(off, 128);    off += pl.nbufs * kSliceBytes;
    cp->sm_mbar = off = al(off, 16);  off += 16 * kMaxBufs;
    cp->sm_tmem = off;                off += 16;
  }
  cp->sm_slots = off = al(off, 16);   off += (wave * pl.spec + 2 * wave) * 4;   // slots, per request
  cp->sm_recs = off = al(off, 16);    off += wave * pl.spec * 16;
  cp->sm_scratch = off = al(off, 16);
  const int gemm_scratch = al(wave * pl.spec * 4, 16) + (pl.umma ? 0 : kGemmCols * kGemmKC * 4);
  const int score_scratch = kWarps * d.M * 4 + (d.r > 256 ? kWarps * d.r * 4 : 0);
  off += gemm_scratch > score_scratch ? gemm_scratch : score_scratch;
  cp->sm_total = off;
  return off;
}

int chain_smem_bytes(const Plan &pl, int e_cap, int wave) {
  ChainParams cp;
  return chain_smem_layout(pl, e_cap, wave, &cp);
}

template <int WDT, int SLOTS>
static const void *chain_fn() {
  return reinterpret_cast<const void *>(&chain_kernel<WDT, SLOTS>);
}

const void *chain_kernel_ptr(int wdtype, int M) {
  const int mp = M <= 32 ? 1 : M <= 64 ? 2 : M <= 128 ? 4 : 8;
  if (wdtype == DT_BF16) {
    switch (mp) {
      case 1: return chain_fn<1, 1>();
      case 2: return chain_fn<1, 2>();
      case 4: return chain_fn<1, 4>();
      default: return chain_fn<1, 8>();
    }
  }
  switch (mp) {
    case 1: return chain_fn<0, 1>();
    case 2: return chain_fn<0, 2>();
    case 4: return chain_fn<0, 4>();
    default: return chain_fn<0, 8>();
  }
}

cudaError_t launch_chain(const Plan &pl, const ChainArgs &a, void *ws, cudaStream_t st) {
  const dt_dims &d = pl.dims;
  char *w = static_cast<char *>(ws);
  ChainParams cp;
  chain_smem_layout(pl, pl.e_cap, pl.wave, &cp);
  cp.V = d.V; cp.d = d.d; cp.d_s = d.d_s; cp.r = d.r; cp.D = d.D; cp.M = d.M; cp.k = d.k;
  cp.N = d.N;
  cp.nb = a.nb; cp.b0 = a.b0; cp.P = pl.spec; cp.e_cap = pl.e_cap;
  cp.W_hh = a.w->W_hh; cp.W1 = a.w->W1; cp.W2 = a.w->W2; cp.b_hh = a.w->b_hh;
  cp.G = a.G;
  cp.state0 = a.state0; cp.anchor = a.anchor; cp.temperature = a.temperature;
  cp.cand_id = reinterpret_cast<const int32_t *>(w + pl.off_cand_id);
  cp.cand_val = reinterpret_cast<const float *>(w + pl.off_cand_val);
  cp.U = reinterpret_cast<const float *>(w + pl.off_U);
  cp.S_store = reinterpret_cast<float *>(w + pl.off_S);
  cp.gh_store = reinterpret_cast<float *>(w + pl.off_gh);
  cp.gin = reinterpret_cast<float *>(w + pl.off_gin);
  cp.pbuf = reinterpret_cast<float *>(w + pl.off_p);
  cp.col_rec = reinterpret_cast<int4 *>(w + pl.off_colinfo);
  cp.kids = reinterpret_cast<unsigned long long *>(w + pl.off_kids);
  cp.sel_mark = reinterpret_cast<unsigned *>(w + pl.off_ghflag);
  cp.gh_mark = cp.sel_mark + pl.wave;
  {
    const int gsz = pl.chain_grid / a.nb;
    cp.grp = gsz < 1 ? 1 : (gsz > pl.spec ? pl.spec : gsz);
  }
  cp.umma = pl.umma; cp.n_mt = pl.n_mt; cp.ks = pl.ks; cp.kc = pl.kc; cp.nbufs = pl.nbufs;
  cp.cols_cap = pl.wave * pl.spec;
  cp.partial = pl.umma ? reinterpret_cast<float *>(w + pl.off_partial) : nullptr;
  cp.gin16 = pl.umma ? reinterpret_cast<uint16_t *>(w + pl.off_gin16) : nullptr;
  cp.col_count = reinterpret_cast<int *>(w + pl.off_colexp);
  cp.ctrl = reinterpret_cast<Ctrl *>(w + pl.off_ctrl);
  cp.req_flags = reinterpret_cast<const int *>(w + pl.off_ctrl + kCtrlHeader +
                                               sizeof(unsigned) * static_cast<size_t>(d.batch) * d.D);
  cp.tokens = a.out->tokens; cp.parents = a.out->parents; cp.depths = a.out->depths;
  cp.scores = a.out->scores; cp.mask = a.out->mask; cp.status = a.out->status;
  cp.limit_ns = pl.test_timeout ? 2000000ull : 2000000000ull;  // per bounded wait
  cp.test_skip = pl.test_timeout;
  const void *fn = chain_kernel_ptr(pl.wdtype, d.M);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(pl.chain_smem));
  if (e != cudaSuccess) return e;
  // the barrier counters of the control block are re-zeroed for every wave
  e = cudaMemsetAsync(cp.ctrl, 0, sizeof(Ctrl), st);
  if (e != cudaSuccess) return e;
  void *args[] = {&cp};
  return cudaLaunchCooperativeKernel(fn, dim3(pl.chain_grid), dim3(kThreads), args,
                                     pl.chain_smem, st);
}

}  // namespace dt
