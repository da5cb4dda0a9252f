// dt_api.cu -- the C ABI of libdt.so (declared in include/dt.h): argument
// validation, workspace carve-up and the launch sequence of one round.
//
// Round = top-M selection over the base logits ("Riassunto Tecnico: DominoTree",
// Componenti Core 2) -> per-depth projection U_j = W1_H H_j (Componenti Core 1,
// H_i shared) -> the conditional best-first search and tree emission
// (Componenti Core 1, 4, 5). Nothing here allocates device memory.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>  // driver types for cuPointerGetAttribute, resolved at run time
#include <cuda_runtime.h>

#include "dt_internal.h"

namespace dt {

int chain_smem_bytes(const Plan &pl, int e_cap, int wave);
const void *chain_kernel_ptr(int wdtype, int M);

namespace {

constexpr size_t kAlign = 256;
inline size_t al(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int device_sm_count(int *sms, int *smem_optin) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
    return DT_ERR_CUDA;
  if (major != 10 || minor != 3) return DT_ERR_UNSUPPORTED;  // built for sm_103a only
  return DT_OK;
}

}  // namespace

int validate_dims(const dt_dims *d) {
  if (!d) return DT_ERR_INVALID_ARG;
  if (d->V < 1 || d->batch < 1) return DT_ERR_INVALID_ARG;
  if (d->d < 8 || d->d % 8) return DT_ERR_INVALID_ARG;
  if (d->d_s < 8 || d->d_s % 8 || d->d_s > DT_MAX_DS) return DT_ERR_INVALID_ARG;
  if (d->r < 8 || d->r % 8 || d->r > DT_MAX_R) return DT_ERR_INVALID_ARG;
  if (d->D < 1 || d->D > DT_MAX_D) return DT_ERR_INVALID_ARG;
  if (d->M < 1 || d->M > DT_MAX_M || d->M > d->V) return DT_ERR_INVALID_ARG;
  if (d->k < 1 || d->k > DT_MAX_K || d->k > d->M) return DT_ERR_INVALID_ARG;
  if (d->N < 0 || d->N > DT_MAX_N) return DT_ERR_INVALID_ARG;
  return DT_OK;
}

int make_plan_uncached(const dt_dims *dims, int wdtype, const dt_options *opt, Plan *p) {
  int rc = validate_dims(dims);
  if (rc) return rc;
  if (wdtype != DT_F32 && wdtype != DT_BF16) return DT_ERR_INVALID_ARG;
  if (opt && (opt->spec_width < 0 || opt->spec_width > DT_MAX_SPEC)) return DT_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof *p);
  p->dims = *dims;
  p->wdtype = wdtype;
  int smem_optin = 0;
  rc = device_sm_count(&p->num_sms, &smem_optin);
  if (rc) return rc;
  const dt_dims &d = *dims;
  p->spec = (opt && opt->spec_width > 0) ? opt->spec_width : 8;
  p->test_timeout = (opt && (opt->flags & DT_OPT_TEST_BARRIER_TIMEOUT)) ? 1 : 0;
  p->marginal = (opt && (opt->flags & DT_OPT_MARGINAL)) ? 1 : 0;

  // top-M segments: at most 64K elements per block, enough blocks to fill the GPU
  const long long rows = static_cast<long long>(d.batch) * d.D;
  if (rows > 65535) return DT_ERR_UNSUPPORTED;  // one grid row of the top-M launch per (b, j)
  const long long by_size = (d.V + 65535) / 65536;
  const long long by_util = (4LL * p->num_sms + rows - 1) / rows;
  const long long by_min = (d.V + 4095) / 4096;
  long long ns = by_size;
  if (by_util > ns) ns = by_util < by_min ? by_util : (by_min > ns ? by_min : ns);
  p->nsplit = static_cast<int>(ns < 1 ? 1 : ns);
  // rows of a multiple of 4 floats: one wave of blocks (3 per SM) over the
  // concatenated rows, each streaming a contiguous range (at least 2048 float4)
  p->topm_blocks = 0;
  if (d.V % 4 == 0) {
    const long long units = rows * (d.V / 4);
    long long nb = 3LL * p->num_sms;
    if (nb > units / 2048) nb = units / 2048;
    if (nb >= 1) {
      p->topm_blocks = static_cast<int>(nb);
      p->nsplit = static_cast<int>((nb + rows - 1) / rows) + 2;   // pieces of one row, at most
    }
  }

  // search kernel: expansion slots, shared memory and co-resident grid (the
  // marginal mode has no search: its workspace ends after the candidates)
  if (!p->marginal) {
    const void *fn = chain_kernel_ptr(wdtype, d.M);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return DT_ERR_CUDA;
    // the opt-in limit covers static + dynamic shared memory of a block
    const int smem_max = smem_optin - static_cast<int>(fa.sharedSizeBytes);
    const int wave0 = d.batch < 256 ? (d.batch < p->num_sms ? d.batch : p->num_sms) : 256;
    // e_cap (expansion slots), B slice buffers and shared memory for the GEMM
    // choice in *p: the full speculation budget with 4, 3 or 2 buffers, else
    // a halved budget with 2; false when even the smallest e_cap does not fit
    auto fit_smem = [&](Plan *q, int wave) {
      int e_cap = d.N + 1 + (q->spec > 1 ? d.N + 1 : 0);
      q->nbufs = 4;
      int smem = chain_smem_bytes(*q, e_cap, wave);
      while (smem > smem_max && q->umma && q->nbufs > 2) {
        --q->nbufs;
        smem = chain_smem_bytes(*q, e_cap, wave);
      }
      while (smem > smem_max && e_cap > d.N + 1) {
        e_cap = d.N + 1 + (e_cap - d.N - 1) / 2;
        smem = chain_smem_bytes(*q, e_cap, wave);
      }
      if (smem > smem_max) return false;
      q->e_cap = e_cap;
      q->chain_smem = static_cast<size_t>(smem);
      return true;
    };
    p->umma = 0;
    if (wdtype == DT_BF16) {
      // search GEMM on the tensor cores: 128-row tiles of [W_hh; W1_S] times K
      // chunks, one (tile, chunk) per block, at most 512 K columns per chunk;
      // the K-chunk partials are summed through global memory
      const int R = 3 * d.d_s + d.r;
      const int n_mt = (R + 127) / 128;
      int ks = p->num_sms / n_mt;
      if (ks >= 1) {
        int kc = ((d.d_s + ks - 1) / ks + 15) / 16 * 16;
        ks = (d.d_s + kc - 1) / kc;
        if (kc <= 512 && n_mt * ks <= p->num_sms) {
          p->umma = 1;
          p->n_mt = n_mt;
          p->ks = ks;
          p->kc = kc;
        }
      }
    }
    int wave = wave0;
    if (!fit_smem(p, wave)) return DT_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(p->chain_smem)) != cudaSuccess)
      return DT_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256,
                                                      static_cast<int>(p->chain_smem)) !=
        cudaSuccess)
      return DT_ERR_CUDA;
    if (per_sm < 1) return DT_ERR_UNSUPPORTED;
    p->chain_grid = per_sm * p->num_sms;
    if (wave > p->chain_grid) wave = p->chain_grid;
    p->wave = wave;
  }
  const int wave = p->wave;
  const int e_cap = p->e_cap;

  // projection U = W1[:, :d] H: on the tensor cores for bf16 weights (about
  // one block per SM), else the CUDA-core split-K GEMM, its K split so that
  // the tiles x chunks fill every SM once
  p->proj_umma = (!p->marginal && proj_umma_supported(d, wdtype)) ? 1 : 0;
  p->proj_ksplit = 1;
  if (p->proj_umma) {
    p->proj_ksplit = proj_umma_split(static_cast<int>(rows), d.r, d.d, p->num_sms);
  } else if (!p->marginal) {
    const int tiles = gemm_tiles(static_cast<int>(rows), d.r);
    int ks = p->num_sms / tiles;
    const int kmax = (d.d + 15) / 16;
    p->proj_ksplit = ks < 1 ? 1 : (ks > 32 ? 32 : (ks > kmax ? kmax : ks));
  }
  // workspace carve-up
  size_t off = 0;
  p->off_ctrl = off;
  p->off_gemm_tickets = kCtrlHeader + sizeof(unsigned) * rows + sizeof(int) * d.batch;
  off = al(off + p->off_gemm_tickets +
           sizeof(unsigned) * gemm_tiles(static_cast<int>(rows), d.r));
  p->off_part = off;
  off = al(off + (p->nsplit > 1 ? sizeof(uint64_t) * rows * p->nsplit * d.M : 0));
  p->off_cand_id = off;   off = al(off + sizeof(int32_t) * rows * d.M);
  p->off_cand_val = off;  off = al(off + sizeof(float) * rows * d.M);
  if (p->marginal) {
    p->off_U = p->off_S = p->off_gh = p->off_gin = p->off_p = p->off_colexp = p->off_colinfo =
        p->off_kids = p->off_ghflag = p->off_upart = p->off_partial = p->off_gin16 = p->off_end =
            off;
    return DT_OK;
  }
  p->off_U = off;         off = al(off + sizeof(float) * rows * d.r);
  const size_t slots_e = static_cast<size_t>(wave) * (e_cap + 1);
  p->off_S = off;         off = al(off + sizeof(float) * slots_e * d.d_s);
  p->off_gh = off;        off = al(off + sizeof(float) * slots_e * 3 * d.d_s);
  const size_t cols = static_cast<size_t>(wave) * p->spec;
  p->off_gin = off;       off = al(off + sizeof(float) * cols * d.d_s);
  p->off_p = off;         off = al(off + sizeof(float) * cols * d.r);
  p->off_colexp = off;    off = al(off + sizeof(int) * (cols + wave));
  p->off_colinfo = off;   off = al(off + (3 * sizeof(int) + sizeof(float)) * cols);
  p->off_kids = off;      off = al(off + sizeof(unsigned long long) * cols * d.k);
  // marks: per request, per (request, expansion slot)
  p->off_ghflag = off;
  off = al(off + sizeof(unsigned) * (wave + slots_e));
  p->off_upart = off;
  off = al(off + (p->proj_ksplit > 1 ? sizeof(float) * p->proj_ksplit * rows * d.r : 0));
  p->off_partial = off;
  off = al(off + (p->umma ? sizeof(float) * p->ks * cols * (3 * d.d_s + d.r) : 0));
  p->off_gin16 = off;
  // B operand of the tensor-core GEMM: passes of 256 columns, K padded to ks * kc
  const size_t cols256 = (cols + 255) / 256 * 256;
  off = al(off + (p->umma ? sizeof(uint16_t) * cols256 * 3 * p->ks * p->kc : 0));
  p->off_end = off;
  return DT_OK;
}

// Plans are pure functions of (device, dims, weight type, options) and cost
// several occupancy and attribute queries; the last few are kept so that a
// serving loop calling with the same shape pays for them once.
int make_plan(const dt_dims *dims, int wdtype, const dt_options *opt, Plan *p) {
  struct Entry {
    bool used;
    int device, wdtype, spec, flags;
    dt_dims dims;
    Plan plan;
  };
  static std::mutex mu;
  static Entry cache[8];
  static int next = 0;
  const int vrc = validate_dims(dims);   // before any device query
  if (vrc) return vrc;
  if (wdtype != DT_F32 && wdtype != DT_BF16) return DT_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  const int spec = opt ? opt->spec_width : 0, flags = opt ? opt->flags : 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
      if (e.used && e.device == dev && e.wdtype == wdtype && e.spec == spec && e.flags == flags &&
          std::memcmp(&e.dims, dims, sizeof(dt_dims)) == 0) {
        *p = e.plan;
        return DT_OK;
      }
  }
  const int rc = make_plan_uncached(dims, wdtype, opt, p);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(mu);
  Entry &e = cache[next];
  next = (next + 1) % 8;
  e.used = true;
  e.device = dev;
  e.wdtype = wdtype;
  e.spec = spec;
  e.flags = flags;
  e.dims = *dims;
  e.plan = *p;
  return DT_OK;
}

}  // namespace dt

using dt::Plan;

namespace {

bool is_marginal(const dt_options *opt) { return opt && (opt->flags & DT_OPT_MARGINAL); }

int check_weights(const dt_weights *w) {
  if (!w || !w->E || !w->W_ih || !w->W_hh || !w->W1 || !w->W2) return DT_ERR_INVALID_ARG;
  if (!dt::aligned16(w->E) || !dt::aligned16(w->W_ih) || !dt::aligned16(w->W_hh) ||
      !dt::aligned16(w->W1) || !dt::aligned16(w->W2))
    return DT_ERR_INVALID_ARG;
  if ((w->b_ih && !dt::aligned4(w->b_ih)) || (w->b_hh && !dt::aligned4(w->b_hh)))
    return DT_ERR_INVALID_ARG;
  if (w->wdtype != DT_F32 && w->wdtype != DT_BF16) return DT_ERR_INVALID_ARG;
  return DT_OK;
}

int check_out(const dt_tree_out *o) {
  if (!o || !o->tokens || !o->parents || !o->depths || !o->scores || !o->status)
    return DT_ERR_INVALID_ARG;
  if (!dt::aligned4(o->tokens) || !dt::aligned4(o->parents) || !dt::aligned4(o->depths) ||
      !dt::aligned4(o->scores) || !dt::aligned4(o->status) || (o->topm && !dt::aligned4(o->topm)))
    return DT_ERR_INVALID_ARG;
  return DT_OK;
}

int record(const dt_options *opt, int i, cudaStream_t st) {
  if (!opt || !opt->phase_events || !opt->phase_events[i]) return DT_OK;
  return cudaEventRecord(static_cast<cudaEvent_t>(opt->phase_events[i]), st) == cudaSuccess
             ? DT_OK
             : DT_ERR_CUDA;
}

// Range [start, start + size) of the registration that holds the device
// address `dp`, from the driver's pointer attributes (resolved through the
// runtime's entry-point query, so the library does not link the driver).
bool registration_range(const void *dp, uintptr_t *start, size_t *size) {
  using GetAttr = CUresult (*)(void *, CUpointer_attribute, CUdeviceptr);
  static GetAttr fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<GetAttr>(f);
  }();
  if (!fn) return false;
  CUdeviceptr st = 0;
  size_t sz = 0;
  const CUdeviceptr p = reinterpret_cast<CUdeviceptr>(dp);
  if (fn(&st, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, p) != CUDA_SUCCESS ||
      fn(&sz, CU_POINTER_ATTRIBUTE_RANGE_SIZE, p) != CUDA_SUCCESS || !sz)
    return false;
  *start = static_cast<uintptr_t>(st);
  *size = sz;
  return true;
}

// One library-owned non-blocking stream per device for the work that runs
// beside the caller's stream; created on first use, kept for the process.
cudaStream_t side_stream() {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

// Fork/join events of the side stream, created once per (device, caller
// stream) and kept for the process. Two calls on the same stream may record
// them in turn: a wait then covers a later record of the same stream, which
// orders no less work than the call needs.
struct Events {
  cudaEvent_t fork = nullptr, join = nullptr;
};

bool stream_events(cudaStream_t st, Events *ev) {
  struct Entry {
    int dev;
    cudaStream_t st;
    Events ev;
  };
  static std::mutex mu;
  static Entry table[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].dev == dev && table[i].st == st) {
      *ev = table[i].ev;
      return true;
    }
  Events e;
  if (cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(e.fork);
    return false;
  }
  if (used < 64) {
    table[used++] = Entry{dev, st, e};
  } else {
    // a full table drops its oldest entry; its events are not destroyed, since
    // work already queued may still wait on them
    for (int i = 1; i < 64; ++i) table[i - 1] = table[i];
    table[63] = Entry{dev, st, e};
  }
  *ev = e;
  return true;
}

int run_round(const Plan &pl, const dt_weights *w, const void *prepared, const float *base_logits,
              const float *H, const float *state0, const int32_t *anchor_tok,
              const float *temperature, void *ws, const dt_tree_out *out, const dt_options *opt,
              cudaStream_t st) {
  const dt_dims &d = pl.dims;
  int rc = record(opt, 0, st);
  if (rc) return rc;
  char *wsb = static_cast<char *>(ws);
  if (cudaMemsetAsync(wsb + pl.off_ctrl, 0, pl.off_part - pl.off_ctrl, st) != cudaSuccess)
    return DT_ERR_CUDA;
  if (pl.marginal) {
    if (dt::launch_topm(pl, base_logits, ws, out->topm, st) != cudaSuccess) return DT_ERR_CUDA;
    rc = record(opt, 1, st);
    if (!rc) rc = record(opt, 2, st);
    if (rc) return rc;
    const unsigned *ticket = reinterpret_cast<const unsigned *>(wsb + pl.off_ctrl + dt::kCtrlHeader);
    const int *req_flags = reinterpret_cast<const int *>(ticket + static_cast<size_t>(d.batch) * d.D);
    if (dt::launch_marginal(d, reinterpret_cast<const int32_t *>(wsb + pl.off_cand_id),
                            reinterpret_cast<const float *>(wsb + pl.off_cand_val), req_flags,
                            anchor_tok, temperature, out, st) != cudaSuccess)
      return DT_ERR_CUDA;
    return record(opt, 3, st);
  }
  // the projection runs on a side stream beside the top-M selection on the
  // main stream; the two touch disjoint workspace regions. On device-resident
  // logits the top-M blocks fill every SM first and the projection mostly runs
  // in the slots they free at the end; where the top-M is bound by the host
  // link (logits read in place from mapped memory) it is hidden entirely.
  cudaStream_t side = side_stream();
  if (!side) return DT_ERR_CUDA;
  Events ev;
  if (!stream_events(st, &ev)) return DT_ERR_CUDA;
  if (cudaEventRecord(ev.fork, st) != cudaSuccess || cudaStreamWaitEvent(side, ev.fork, 0) != cudaSuccess)
    return DT_ERR_CUDA;
  float *U = reinterpret_cast<float *>(wsb + pl.off_U);
  float *upart = reinterpret_cast<float *>(wsb + pl.off_upart);
  if (pl.proj_umma) {
    // a bounded wait of the projection that runs out aborts the search
    int *fail = reinterpret_cast<int *>(wsb + pl.off_ctrl + offsetof(dt::Ctrl, abort));
    if (dt::launch_proj_umma(d.batch * d.D, d.r, d.d, H, d.d, w->W1, d.d + d.d_s, U,
                             pl.proj_ksplit, upart, fail, side) != cudaSuccess)
      return DT_ERR_CUDA;
  } else if (dt::launch_gemm_nt(d.batch * d.D, d.r, d.d, H, DT_F32, d.d, w->W1, w->wdtype,
                                static_cast<size_t>(d.d) + d.d_s, nullptr, U, d.r,
                                pl.proj_ksplit, upart, side) != cudaSuccess) {
    return DT_ERR_CUDA;
  }
  if (cudaEventRecord(ev.join, side) != cudaSuccess) return DT_ERR_CUDA;
  if (dt::launch_topm(pl, base_logits, ws, out->topm, st) != cudaSuccess) return DT_ERR_CUDA;
  rc = record(opt, 1, st);
  if (rc) return rc;
  if (cudaStreamWaitEvent(st, ev.join, 0) != cudaSuccess) return DT_ERR_CUDA;
  rc = record(opt, 2, st);
  if (rc) return rc;
  dt::ChainArgs a;
  a.w = w;
  a.G = static_cast<const float *>(prepared);
  a.state0 = state0;
  a.anchor = anchor_tok;
  a.temperature = temperature;
  a.out = out;
  for (int b0 = 0; b0 < d.batch; b0 += pl.wave) {
    a.b0 = b0;
    a.nb = (d.batch - b0) < pl.wave ? (d.batch - b0) : pl.wave;
    if (dt::launch_chain(pl, a, ws, st) != cudaSuccess) return DT_ERR_CUDA;
  }
  return record(opt, 3, st);
}

// Chain-decoding plan: kernel shapes plus the workspace carve-up.
int decode_plan_for(const dt_dims *dims, dt::DecodePlan *pl) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  int sms = 0, smem = 0;
  rc = dt::device_sm_count(&sms, &smem);
  if (rc) return rc;
  rc = dt::decode_plan(*dims, sms, smem, pl);
  if (rc) return rc;
  const dt_dims &d = *dims;
  const size_t wave = static_cast<size_t>(pl->wave);
  const long long rows = static_cast<long long>(d.batch) * d.D;
  // the projection runs alone before the decoding kernel: on the tensor cores
  // with about one block per SM, else the CUDA-core GEMM filling every SM once
  pl->proj_umma = dt::proj_umma_supported(d, DT_BF16) ? 1 : 0;
  if (pl->proj_umma) {
    pl->proj_ksplit = dt::proj_umma_split(static_cast<int>(rows), d.r, d.d, sms);
  } else {
    const int tiles = dt::gemm_tiles(static_cast<int>(rows), d.r);
    const int ks = sms / tiles, kmax = (d.d + 15) / 16;
    pl->proj_ksplit = ks < 1 ? 1 : (ks > 32 ? 32 : (ks > kmax ? kmax : ks));
  }
  const size_t gn = static_cast<size_t>(pl->n_tV) * 4;
  size_t off = 0;
  pl->off_ctrl = off;  off = dt::al(off + sizeof(dt::Ctrl));
  pl->off_U = off;     off = dt::al(off + sizeof(float) * rows * d.r);
  pl->off_upart = off;
  off = dt::al(off + (pl->proj_ksplit > 1 ? sizeof(float) * pl->proj_ksplit * rows * d.r : 0));
  pl->off_ypart = off; off = dt::al(off + sizeof(float) * pl->n_kz * wave * pl->R);
  pl->off_S = off;     off = dt::al(off + sizeof(float) * wave * d.d_s);
  pl->off_stm = off;   off = dt::al(off + sizeof(float) * wave * gn);
  pl->off_sts = off;   off = dt::al(off + sizeof(float) * wave * gn);
  pl->off_sta = off;   off = dt::al(off + sizeof(int32_t) * wave * gn);
  pl->off_flags = off; off = dt::al(off + sizeof(int) * wave);
  pl->off_end = off;
  return DT_OK;
}

struct HostStaging {
  size_t base, H, state0, anchor, temp, tokens, parents, depths, scores, mask, topm, status, end;
};

HostStaging host_staging(const dt_dims &d, size_t start) {
  HostStaging s;
  const size_t n1 = static_cast<size_t>(d.N) + 1;
  size_t off = start;
  s.base = off;    off = dt::al(off + sizeof(float) * d.batch * d.D * static_cast<size_t>(d.V));
  s.H = off;       off = dt::al(off + sizeof(float) * d.batch * d.D * static_cast<size_t>(d.d));
  s.state0 = off;  off = dt::al(off + sizeof(float) * d.batch * static_cast<size_t>(d.d_s));
  s.anchor = off;  off = dt::al(off + sizeof(int32_t) * d.batch);
  s.temp = off;    off = dt::al(off + sizeof(float) * d.batch);
  s.tokens = off;  off = dt::al(off + sizeof(int32_t) * d.batch * n1);
  s.parents = off; off = dt::al(off + sizeof(int32_t) * d.batch * n1);
  s.depths = off;  off = dt::al(off + sizeof(int32_t) * d.batch * n1);
  s.scores = off;  off = dt::al(off + sizeof(float) * d.batch * n1);
  s.mask = off;    off = dt::al(off + d.batch * n1 * n1);
  s.topm = off;    off = dt::al(off + sizeof(int32_t) * d.batch * d.D * static_cast<size_t>(d.M));
  s.status = off;  off = dt::al(off + sizeof(int32_t) * d.batch);
  s.end = off;
  return s;
}

}  // namespace

extern "C" {

int dt_abi_version(void) { return DT_ABI_VERSION; }

const char *dt_status_string(int code) {
  switch (code) {
    case DT_OK: return "ok";
    case DT_ERR_INVALID_ARG: return "invalid argument (size, null pointer, alignment or limit)";
    case DT_ERR_UNSUPPORTED: return "unsupported device or shape";
    case DT_ERR_CUDA: return "CUDA runtime or launch error";
    case DT_ERR_NONFINITE: return "a base logit of the request is NaN or +inf";
    case DT_ERR_TIMEOUT: return "bounded inter-block wait expired; request output invalid";
    case DT_ERR_BAD_TEMPERATURE: return "temperature is negative or not finite";
    default: return "unknown status code";
  }
}

size_t dt_prepared_bytes(const dt_dims *dims) {
  if (dt::validate_dims(dims)) return 0;
  return sizeof(float) * static_cast<size_t>(dims->V) * 3 * dims->d_s;
}

int dt_prepare_weights(const dt_dims *dims, const dt_weights *w, void *prepared,
                       size_t prepared_bytes, void *stream) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  rc = check_weights(w);
  if (rc) return rc;
  if (!prepared || (reinterpret_cast<uintptr_t>(prepared) & 255u) ||
      prepared_bytes < dt_prepared_bytes(dims))
    return DT_ERR_INVALID_ARG;
  int sms = 0, smem = 0;
  rc = dt::device_sm_count(&sms, &smem);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dt::launch_gemm_nt(dims->V, 3 * dims->d_s, dims->d, w->E, w->wdtype, dims->d, w->W_ih,
                         w->wdtype, dims->d, w->b_ih, static_cast<float *>(prepared),
                         3 * static_cast<size_t>(dims->d_s), 1, nullptr, st) != cudaSuccess)
    return DT_ERR_CUDA;
  return DT_OK;
}

size_t dt_workspace_bytes(const dt_dims *dims, const dt_options *opt) {
  Plan pl;
  if (!dims) return 0;
  if (dt::make_plan(dims, DT_BF16, opt, &pl)) return 0;
  Plan pf;
  if (dt::make_plan(dims, DT_F32, opt, &pf)) return 0;
  return pl.off_end > pf.off_end ? pl.off_end : pf.off_end;
}

int dt_kernel_launches(const dt_dims *dims, int wdtype, const dt_options *opt) {
  Plan pl;
  if (!dims || (wdtype != DT_F32 && wdtype != DT_BF16)) return 0;
  if (dt::make_plan(dims, wdtype, opt, &pl)) return 0;
  if (pl.marginal) return 2;
  const int waves = (dims->batch + pl.wave - 1) / pl.wave;
  return 2 + (pl.proj_ksplit > 1 ? 1 : 0) + waves;
}

int dt_build_trees(const dt_dims *dims, const dt_weights *w, const void *prepared,
                   const float *base_logits, const float *H, const float *state0,
                   const int32_t *anchor_tok, const float *temperature, void *workspace,
                   size_t workspace_bytes, const dt_tree_out *out, const dt_options *opt,
                   void *stream) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  const bool marginal = is_marginal(opt);
  if (!marginal) {
    rc = check_weights(w);
    if (rc) return rc;
    if (!prepared || !H || !state0 || !dt::aligned16(prepared) || !dt::aligned16(H) ||
        !dt::aligned16(state0))
      return DT_ERR_INVALID_ARG;
  }
  rc = check_out(out);
  if (rc) return rc;
  if (!base_logits || !anchor_tok || !workspace) return DT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !dt::aligned4(base_logits) ||
      !dt::aligned4(anchor_tok) || (temperature && !dt::aligned4(temperature)))
    return DT_ERR_INVALID_ARG;
  if (dims->V % 4 == 0 && !dt::aligned16(base_logits)) return DT_ERR_INVALID_ARG;
  Plan pl;
  rc = dt::make_plan(dims, marginal ? DT_F32 : w->wdtype, opt, &pl);
  if (rc) return rc;
  if (workspace_bytes < pl.off_end) return DT_ERR_INVALID_ARG;
  return run_round(pl, w, prepared, base_logits, H, state0, anchor_tok, temperature, workspace,
                   out, opt, static_cast<cudaStream_t>(stream));
}

const void *dt_mapped_host_pointer(const void *host, size_t bytes) {
  if (!host || !bytes) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  // memory registered for one device only is not mapped for the others
  if (a.device != dev) {
    unsigned flags = 0;
    if (cudaHostGetFlags(&flags, const_cast<void *>(host)) != cudaSuccess ||
        !(flags & cudaHostAllocPortable)) {
      cudaGetLastError();
      return nullptr;
    }
  }
  uintptr_t start = 0;
  size_t size = 0;
  const uintptr_t dp = reinterpret_cast<uintptr_t>(a.devicePointer);
  if (!registration_range(a.devicePointer, &start, &size)) return nullptr;
  if (dp < start || dp - start > size || size - (dp - start) < bytes) return nullptr;
  return a.devicePointer;
}

size_t dt_host_workspace_bytes(const dt_dims *dims, const dt_options *opt) {
  size_t ws = dt_workspace_bytes(dims, opt);
  if (!ws) return 0;
  return host_staging(*dims, dt::al(ws)).end;
}

int dt_build_trees_host(const dt_dims *dims, const dt_weights *w, const void *prepared,
                        const float *base_logits, const float *H, const float *state0,
                        const int32_t *anchor_tok, const float *temperature, void *workspace,
                        size_t workspace_bytes, const dt_tree_out *host_out,
                        const dt_options *opt, void *stream) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  const bool marginal = is_marginal(opt);
  if (!marginal) {
    rc = check_weights(w);
    if (rc) return rc;
    if (!prepared || !H || !state0) return DT_ERR_INVALID_ARG;
  }
  if (!host_out || !host_out->tokens || !host_out->parents || !host_out->depths ||
      !host_out->scores || !host_out->status || !base_logits || !anchor_tok || !workspace ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return DT_ERR_INVALID_ARG;
  Plan pl;
  rc = dt::make_plan(dims, marginal ? DT_F32 : w->wdtype, opt, &pl);
  if (rc) return rc;
  const size_t ws_dev = dt_workspace_bytes(dims, opt);
  const HostStaging s = host_staging(*dims, dt::al(ws_dev));
  if (workspace_bytes < s.end) return DT_ERR_INVALID_ARG;
  const dt_dims &d = *dims;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *wsb = static_cast<char *>(workspace);
  const size_t n1 = static_cast<size_t>(d.N) + 1;
  auto h2d = [&](size_t off, const void *src, size_t bytes) {
    return cudaMemcpyAsync(wsb + off, src, bytes, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  auto d2h = [&](void *dst, size_t off, size_t bytes) {
    return cudaMemcpyAsync(dst, wsb + off, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  const size_t nb = static_cast<size_t>(d.batch);
  // mapped page-locked logits are read in place by the top-M scan (the only
  // reader of the full rows) instead of being copied first
  const size_t base_bytes = sizeof(float) * nb * d.D * d.V;
  const float *base_dev = nullptr;
  if (!(opt && (opt->flags & DT_OPT_STAGE_HOST_LOGITS))) {
    base_dev = static_cast<const float *>(dt_mapped_host_pointer(base_logits, base_bytes));
    if (base_dev && (!dt::aligned4(base_dev) || (d.V % 4 == 0 && !dt::aligned16(base_dev))))
      base_dev = nullptr;
  }
  if ((!base_dev && !h2d(s.base, base_logits, base_bytes)) ||
      (!marginal && !h2d(s.H, H, sizeof(float) * nb * d.D * d.d)) ||
      (!marginal && !h2d(s.state0, state0, sizeof(float) * nb * d.d_s)) ||
      !h2d(s.anchor, anchor_tok, sizeof(int32_t) * nb) ||
      (temperature && !h2d(s.temp, temperature, sizeof(float) * nb)))
    return DT_ERR_CUDA;
  dt_tree_out dev;
  dev.tokens = reinterpret_cast<int32_t *>(wsb + s.tokens);
  dev.parents = reinterpret_cast<int32_t *>(wsb + s.parents);
  dev.depths = reinterpret_cast<int32_t *>(wsb + s.depths);
  dev.scores = reinterpret_cast<float *>(wsb + s.scores);
  dev.mask = host_out->mask ? reinterpret_cast<uint8_t *>(wsb + s.mask) : nullptr;
  dev.topm = host_out->topm ? reinterpret_cast<int32_t *>(wsb + s.topm) : nullptr;
  dev.status = reinterpret_cast<int32_t *>(wsb + s.status);
  rc = run_round(pl, w, prepared,
                 base_dev ? base_dev : reinterpret_cast<const float *>(wsb + s.base),
                 reinterpret_cast<const float *>(wsb + s.H),
                 reinterpret_cast<const float *>(wsb + s.state0),
                 reinterpret_cast<const int32_t *>(wsb + s.anchor),
                 temperature ? reinterpret_cast<const float *>(wsb + s.temp) : nullptr, workspace,
                 &dev, opt, st);
  if (rc) return rc;
  if (!d2h(host_out->tokens, s.tokens, sizeof(int32_t) * nb * n1) ||
      !d2h(host_out->parents, s.parents, sizeof(int32_t) * nb * n1) ||
      !d2h(host_out->depths, s.depths, sizeof(int32_t) * nb * n1) ||
      !d2h(host_out->scores, s.scores, sizeof(float) * nb * n1) ||
      !d2h(host_out->status, s.status, sizeof(int32_t) * nb) ||
      (host_out->mask && !d2h(host_out->mask, s.mask, nb * n1 * n1)) ||
      (host_out->topm && !d2h(host_out->topm, s.topm, sizeof(int32_t) * nb * d.D * d.M)))
    return DT_ERR_CUDA;
  return DT_OK;
}

/* ------------------------------------------------- Domino chain decoding */

size_t dt_chain_prepared_bytes(const dt_dims *dims) {
  if (dt::validate_dims(dims)) return 0;
  return dt::decode_prepared_bytes(*dims);
}

int dt_prepare_chain(const dt_dims *dims, const dt_weights *w, void *chain_prepared,
                     size_t chain_prepared_bytes, void *stream) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  rc = check_weights(w);
  if (rc) return rc;
  if (w->wdtype != DT_BF16) return DT_ERR_UNSUPPORTED;
  if (!chain_prepared || (reinterpret_cast<uintptr_t>(chain_prepared) & 255u) ||
      chain_prepared_bytes < dt_chain_prepared_bytes(dims))
    return DT_ERR_INVALID_ARG;
  int sms = 0, smem = 0;
  rc = dt::device_sm_count(&sms, &smem);
  if (rc) return rc;
  if (dt::launch_decode_prepare(*dims, w, chain_prepared, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DT_ERR_CUDA;
  return DT_OK;
}

size_t dt_chain_workspace_bytes(const dt_dims *dims) {
  dt::DecodePlan pl;
  if (decode_plan_for(dims, &pl)) return 0;
  return pl.off_end;
}

int dt_chain_kernel_launches(const dt_dims *dims) {
  dt::DecodePlan pl;
  if (decode_plan_for(dims, &pl)) return 0;
  return 1 + (pl.proj_ksplit > 1 ? 1 : 0) + (dims->batch + pl.wave - 1) / pl.wave;
}

int dt_decode_chains(const dt_dims *dims, const dt_weights *w, const void *prepared,
                     const void *chain_prepared, const float *base_logits, const float *H,
                     const float *state0, const int32_t *anchor_tok, const float *temperature,
                     const float *uniforms, void *workspace, size_t workspace_bytes,
                     int32_t *tokens, float *logprobs, int32_t *status, void *stream) {
  int rc = dt::validate_dims(dims);
  if (rc) return rc;
  rc = check_weights(w);
  if (rc) return rc;
  if (w->wdtype != DT_BF16) return DT_ERR_UNSUPPORTED;
  if (!prepared || !chain_prepared || !base_logits || !H || !state0 || !anchor_tok ||
      !workspace || !tokens || !logprobs || !status)
    return DT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || !dt::aligned16(prepared) ||
      !dt::aligned16(chain_prepared) || !dt::aligned16(H) || !dt::aligned16(state0) ||
      !dt::aligned4(base_logits) || !dt::aligned4(anchor_tok) ||
      (temperature && !dt::aligned4(temperature)) || (uniforms && !dt::aligned4(uniforms)) ||
      !dt::aligned4(tokens) || !dt::aligned4(logprobs) || !dt::aligned4(status))
    return DT_ERR_INVALID_ARG;
  dt::DecodePlan pl;
  rc = decode_plan_for(dims, &pl);
  if (rc) return rc;
  if (workspace_bytes < pl.off_end) return DT_ERR_INVALID_ARG;
  const dt_dims &d = *dims;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *wsb = static_cast<char *>(workspace);
  float *U = reinterpret_cast<float *>(wsb + pl.off_U);
  float *upart = reinterpret_cast<float *>(wsb + pl.off_upart);
  // the control block starts at zero; a bounded wait of the projection that
  // runs out sets its abort flag, which every decoding wave then reports
  if (cudaMemsetAsync(wsb + pl.off_ctrl, 0, sizeof(dt::Ctrl), st) != cudaSuccess)
    return DT_ERR_CUDA;
  // U_i = W1[:, :d] H_i for every request and position (path independent)
  if (pl.proj_umma) {
    int *fail = reinterpret_cast<int *>(wsb + pl.off_ctrl + offsetof(dt::Ctrl, abort));
    if (dt::launch_proj_umma(d.batch * d.D, d.r, d.d, H, d.d, w->W1, d.d + d.d_s, U,
                             pl.proj_ksplit, upart, fail, st) != cudaSuccess)
      return DT_ERR_CUDA;
  } else if (dt::launch_gemm_nt(d.batch * d.D, d.r, d.d, H, DT_F32, d.d, w->W1, w->wdtype,
                                static_cast<size_t>(d.d) + d.d_s, nullptr, U, d.r,
                                pl.proj_ksplit, upart, st) != cudaSuccess) {
    return DT_ERR_CUDA;
  }
  dt::DecodeArgs a;
  a.chain_prepared = chain_prepared;
  a.G = static_cast<const float *>(prepared);
  a.b_hh = w->b_hh;
  a.U = U;
  a.base = base_logits;
  a.state0 = state0;
  a.temperature = temperature;
  a.uniforms = uniforms;
  a.anchor = anchor_tok;
  a.ypart = reinterpret_cast<float *>(wsb + pl.off_ypart);
  a.S = reinterpret_cast<float *>(wsb + pl.off_S);
  a.W2 = static_cast<const uint16_t *>(w->W2);
  a.st_m = reinterpret_cast<float *>(wsb + pl.off_stm);
  a.st_s = reinterpret_cast<float *>(wsb + pl.off_sts);
  a.st_a = reinterpret_cast<int32_t *>(wsb + pl.off_sta);
  a.flags = reinterpret_cast<int *>(wsb + pl.off_flags);
  a.ctrl = reinterpret_cast<dt::Ctrl *>(wsb + pl.off_ctrl);
  a.tokens = tokens;
  a.logprobs = logprobs;
  a.status = status;
  for (int b0 = 0; b0 < d.batch; b0 += pl.wave) {
    a.b0 = b0;
    a.nb = (d.batch - b0) < pl.wave ? (d.batch - b0) : pl.wave;
    if (b0 > 0) {   // a later wave: everything but the abort flag starts at zero again
      const size_t ab = offsetof(dt::Ctrl, abort), ae = ab + sizeof(int);
      if (cudaMemsetAsync(wsb + pl.off_ctrl, 0, ab, st) != cudaSuccess ||
          cudaMemsetAsync(wsb + pl.off_ctrl + ae, 0, sizeof(dt::Ctrl) - ae, st) != cudaSuccess)
        return DT_ERR_CUDA;
    }
    if (dt::launch_decode(pl, a, st) != cudaSuccess) return DT_ERR_CUDA;
  }
  return DT_OK;
}

}  // extern "C"
