// Sparse MLA decode for callers that cannot allocate device memory.
//
// Some users of this library are not in a position to hand it a workspace:
// a serving runtime that reserves nearly all HBM up front for its KV pools
// (one more cudaMalloc may fail, or fragment the reservation), a plugin whose
// host framework owns every device allocation, or a latency-critical path on
// which a synchronizing cudaMalloc / cudaFree cannot be afforded.  For them
// dsa_sparse_mla_decode_noalloc keeps the split-K partials in one fixed
// device array that is part of the library's device image: every GPU that
// loads the library holds DSA_NOALLOC_SCRATCH_BYTES of it until the process
// exits, and this file never allocates or frees anything.
//
// The array is a file-scope __device__ symbol.  On the host its name is only a
// stand-in, not a device address, so the real address is looked up once per
// device (with that device current) through cudaGetSymbolAddress and cached;
// that lookup happens inside the first call made on each device.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_decode.h"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" int dsa_sparse_mla_decode_noalloc(const uint16_t* q, int32_t heads, float sm_scale,
                                             const dsa_paged_cache* kv, const dsa_rows* rows,
                                             const int32_t* idx, const int32_t* count, int32_t k,
                                             int32_t num_splits, float* out, float* out_lse,
                                             int32_t* d_err, void* stream) {
  if (rows == nullptr || rows->num_rows < 0) return DSA_ERR_INVALID_ARG;
  // the partials of this call must fit in the fixed array
  const size_t need = dsa_sparse_mla_decode_workspace_size(rows->num_rows, heads, k, num_splits);
  if (need > kScratchBytes) return DSA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (need > 0) {
    const int st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
  }
  // Nothing in the array has to start at zero: the split kernel writes every
  // partial LSE, and the merge reads a partial output only where its LSE is
  // finite, i.e. where this call wrote it.
  return dsa_sparse_mla_decode(q, heads, sm_scale, kv, rows, idx, count, k, num_splits, out,
                               out_lse, scratch, need > 0 ? kScratchBytes : 0, d_err, stream);
}
