// dt_noalloc.cu -- dt_select_topm_noalloc: the per-depth top-M selection for
// callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: a serving runtime that has
// reserved all device memory up front for its own pool (a new allocation would
// fail or fragment it), a latency-critical loop where cudaMalloc's implicit
// device synchronisation is unacceptable, or a plug-in that runs inside a host
// framework that owns every device allocation. They still pass inputs and
// outputs; the kernel's scratch (per-segment partial lists, per-row tickets,
// per-request flags, candidate values) lives in the file-scope device array
// below instead of a caller workspace.
//
// The array occupies DT_NOALLOC_SCRATCH_BYTES on every device that loads the
// library, until the process exits. Every call shares it and it keeps the last
// call's contents, so each call first clears the part that must start at zero
// (tickets and flags). Calls that overlap on the GPU -- on different streams, or
// on different host threads on the same device -- race on the array and must
// be serialised by the caller. The first call on a device resolves the array's
// device address with cudaGetSymbolAddress (with that device current); make
// that first call before any stream capture. The address is kept per device
// number, which is right for the primary context the runtime uses; it does not
// follow a cudaDeviceReset or another driver-API context on the same device.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dt_internal.h"

namespace dt {
cudaError_t launch_topm_raw(const float *base_logits, int batch, int D, int V, int M, int nsplit,
                            int nblk, uint64_t *partial, unsigned *ticket, int *req_flags,
                            int32_t *cand_id, float *cand_val, int32_t *topm_out, cudaStream_t st);
}

namespace {

static __device__ __align__(256) unsigned char g_topm_scratch[DT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char *g_scratch_addr[kMaxDevices];  // per device, resolved once

// Device address of g_topm_scratch on the current device (set-up on first use).
int scratch_address(unsigned char **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topm_scratch) != cudaSuccess || !p) return DT_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_scratch_addr[dev];
  return DT_OK;
}

__global__ void flags_to_status(const int *flags, int32_t *status, int batch) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) status[b] = (flags[b] & dt::kReqFlagNonfinite) ? DT_ERR_NONFINITE : DT_OK;
}

inline size_t al(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int dt_select_topm_noalloc(const float *base_logits, int batch, int D, int V, int M,
                                      int32_t *topm, int32_t *status, void *stream) {
  if (!base_logits || !topm || !status || batch < 1 || D < 1 || D > DT_MAX_D || V < 1 ||
      M < 1 || M > DT_MAX_M || M > V)
    return DT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(base_logits) & 3u) || (reinterpret_cast<uintptr_t>(topm) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u) ||
      (V % 4 == 0 && (reinterpret_cast<uintptr_t>(base_logits) & 15u)))
    return DT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(batch) * D;
  if (rows > 65535) return DT_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DT_ERR_CUDA;
  // segment count as in dt_build_trees, reduced until the scratch fits
  const long long by_size = (V + 65535) / 65536;
  const long long by_util = (4LL * sms + rows - 1) / rows;
  const long long by_min = (V + 4095) / 4096;
  long long ns = by_size;
  if (by_util > ns) ns = by_util < by_min ? by_util : (by_min > ns ? by_min : ns);
  auto need = [&](long long n) {
    const size_t part = n > 1 ? sizeof(uint64_t) * rows * n * M : 0;
    return al(sizeof(unsigned) * rows) + al(sizeof(int) * batch) + al(sizeof(float) * rows * M) +
           al(part);
  };
  // rows of a multiple of 4 floats: the contiguous-range launch of
  // dt_build_trees (one wave of blocks; at most ns pieces of a row)
  long long nblk = 0;
  if (V % 4 == 0) {
    const long long units = rows * (V / 4);
    nblk = 3LL * sms;
    if (nblk > units / 2048) nblk = units / 2048;
    if (nblk >= 1) ns = (nblk + rows - 1) / rows + 2;
    if (nblk >= 1 && need(ns) > DT_NOALLOC_SCRATCH_BYTES) nblk = 0;
    if (nblk < 1) nblk = 0;
  }
  while (nblk == 0 && ns > 1 && need(ns) > DT_NOALLOC_SCRATCH_BYTES) --ns;
  if (need(ns) > DT_NOALLOC_SCRATCH_BYTES) return DT_ERR_INVALID_ARG;  // beyond the static scratch
  unsigned char *base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  unsigned *ticket = reinterpret_cast<unsigned *>(base);
  int *flags = reinterpret_cast<int *>(base + al(sizeof(unsigned) * rows));
  float *cand_val = reinterpret_cast<float *>(base + al(sizeof(unsigned) * rows) +
                                              al(sizeof(int) * batch));
  uint64_t *partial = reinterpret_cast<uint64_t *>(
      reinterpret_cast<unsigned char *>(cand_val) + al(sizeof(float) * rows * M));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // tickets and flags must start at zero; the array keeps the previous call's values
  if (cudaMemsetAsync(base, 0, al(sizeof(unsigned) * rows) + al(sizeof(int) * batch), st) !=
      cudaSuccess)
    return DT_ERR_CUDA;
  if (dt::launch_topm_raw(base_logits, batch, D, V, M, static_cast<int>(ns),
                          static_cast<int>(nblk), partial, ticket,
                          flags, topm, cand_val, nullptr, st) != cudaSuccess)
    return DT_ERR_CUDA;
  flags_to_status<<<(batch + 255) / 256, 256, 0, st>>>(flags, status, batch);
  return cudaGetLastError() == cudaSuccess ? DT_OK : DT_ERR_CUDA;
}
