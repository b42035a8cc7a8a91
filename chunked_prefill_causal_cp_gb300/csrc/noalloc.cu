// noalloc.cu -- cp_mixed_step_noalloc: the mixed token-budget step for callers
// that cannot allocate device memory.
//
// cp_mixed_step needs a caller-provided workspace for the decode rows' split-KV
// partial results.  Some callers have no way to provide one: code that runs
// inside an engine whose device memory is fully reserved up front (a serving
// process with a fixed memory budget that forbids allocation on the request
// path), plugins that are handed only input and output tensors by a host
// framework that owns every allocation, and code running where the CUDA
// runtime does not allow cudaMalloc at all (for example from a stream
// callback).  This entry point gives them the same step with its scratch in a
// fixed array that is part of the library image itself.
//
// This translation unit is its own CUDA module.  Under the runtime's lazy
// module loading (the default) the module, and with it the array's 8 MiB of
// device memory, is loaded on a device by the first call that needs it: the
// address lookup in this entry point's first call on that device.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "cp_internal.h"

namespace {

// Split-KV scratch of the no-allocation entry point: 8 MiB on every GPU that
// loads this module, held until the process exits.  Enough for, e.g., 16
// sequences x 32 query heads x contexts up to 8192 keys at head_dim 128.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the symbol itself is only a host-side
// stand-in and must never be passed to a kernel.  The cached address belongs
// to the device's primary context: after cudaDeviceReset it is stale, so calls
// after a reset are not supported.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CP_OK;
}

}  // namespace

extern "C" {

size_t cp_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int cp_mixed_step_noalloc(const cp_layer_desc* desc, const void* q, const void* k_new, const void* v_new,
                          void* k_pages, void* v_pages, const int32_t* block_table, const int32_t* cu_rows,
                          int32_t* past_len, int32_t num_seqs, int32_t total_rows, int32_t max_ctx, void* out,
                          int32_t* dev_status, void* stream) {
  // The same checks as cp_mixed_step, in the same order and with the same
  // status codes, then the size check against the fixed scratch -- all before
  // any CUDA call.
  size_t need = 0;
  const int r0 = cp::mixed_step_check(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len,
                                      num_seqs, total_rows, max_ctx, out, &need);
  if (r0 != CP_OK) return r0;
  if (total_rows == 0) return CP_OK;
  if (need > kNoAllocScratchBytes) return CP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int r = scratch_for_current_device(&scratch);
  if (r != CP_OK) return r;
  // The split partials are written before they are read.
  return cp_mixed_step(desc, q, k_new, v_new, k_pages, v_pages, block_table, cu_rows, past_len, num_seqs,
                       total_rows, max_ctx, out, scratch, kNoAllocScratchBytes, dev_status, stream);
}

}  // extern "C"
