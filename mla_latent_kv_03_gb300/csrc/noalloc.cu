// mla_decode_paged_noalloc: the paged decode (plan, split-KV attention and
// the merge of the splits) for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they decode: code
// that runs inside a host framework's per-step callback with a fixed device
// memory budget, a real-time serving loop where an allocation would
// synchronise the device or fail under fragmentation, or a plugin whose
// contract forbids allocating. They still own and pass every input and the
// output; only the scratch the decode needs (the split plan, the per-split
// partial outputs and the device status word) comes from a fixed array built
// into this library.
//
// The array is file-scope device memory of kScratchBytes. Every GPU that
// loads the library holds it until the process exits. All calls on a device
// share it: calls whose GPU work overlaps (two streams, or two host threads)
// race on it and must not be issued. Each call clears the part that has to
// start at zero (the status word and plan header) and rebuilds the rest.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

// The host-side name g_scratch is only a stand-in for the device array; the
// kernels get its device address, resolved once per device. The address is
// kept for the life of the process: after cudaDeviceReset the module may be
// loaded again elsewhere, so the library must not be called on that device
// again in this process.
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

mla_status mla_decode_paged_noalloc(const mla_config* cfg, const void* q_abs, const void* cache,
                                    int64_t num_blocks, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t batch, int64_t num_q,
                                    float* o_lat, uint32_t* dev_status, void* stream) {
  // every argument check of mla_decode_paged first, so that a refused call
  // has touched nothing, the scratch included
  mla_status s = mla::decode_paged_checks(cfg, q_abs, cache, num_blocks, block_table,
                                          max_blocks_per_seq, seq_lens, query_start_loc, batch,
                                          num_q);
  if (s != MLA_OK) return s;
  if (num_q == 0) return MLA_OK;
  if (!o_lat || (reinterpret_cast<uintptr_t>(o_lat) & 15) != 0) return MLA_ERR_INVALID_ARGUMENT;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3) != 0)
    return MLA_ERR_INVALID_ARGUMENT;
  // the scratch must hold this launch's workspace; with the arguments valid,
  // a zero size means the device query failed
  const size_t need = mla_decode_workspace_size(cfg, num_q, batch);
  if (need == 0) return MLA_ERR_CUDA;
  mla_config fit = *cfg;
  if (need > kScratchBytes) {
    if (cfg->num_ctas > 0) return MLA_ERR_WORKSPACE_TOO_SMALL;
    // default CTA count: take the largest count below it whose workspace fits
    // (the size does not decrease with the count, so bisect)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
    int lo = 0, hi = sms;  // size(lo) fits (lo > 0) or lo == 0; size(hi) does not
    while (hi - lo > 1) {
      const int mid = lo + (hi - lo) / 2;
      fit.num_ctas = mid;
      if (mla_decode_workspace_size(&fit, num_q, batch) <= kScratchBytes) lo = mid; else hi = mid;
    }
    if (lo == 0) return MLA_ERR_WORKSPACE_TOO_SMALL;
    fit.num_ctas = lo;
  }
  void* ws = nullptr;
  if (scratch_for_current_device(&ws) != cudaSuccess) return MLA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // status word and plan header start at zero on every call
  if (cudaMemsetAsync(ws, 0, sizeof(mla::WsHeader), st) != cudaSuccess) return MLA_ERR_CUDA;
  s = mla_decode_paged(&fit, q_abs, cache, num_blocks, block_table, max_blocks_per_seq, seq_lens,
                       query_start_loc, batch, num_q, ws, kScratchBytes, stream);
  if (s != MLA_OK) return s;
  s = mla_combine(&fit, ws, kScratchBytes, batch, num_q, o_lat, stream);
  if (s != MLA_OK) return s;
  if (dev_status &&
      cudaMemcpyAsync(dev_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // extern "C"
