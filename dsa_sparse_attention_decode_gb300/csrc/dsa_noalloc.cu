// Sparse MLA decode for callers that cannot allocate device memory.
//
// Some users of this library are not in a position to hand it a workspace:
// a serving runtime that reserves nearly all HBM up front for its KV pools
// (one more cudaMalloc may fail, or fragment the reservation), a plugin whose
// host framework owns every device allocation, or a latency-critical path on
// which a synchronizing cudaMalloc / cudaFree cannot be afforded.  For them
// dsa_sparse_mla_decode_noalloc keeps the split-K partials in one fixed
// device array that is part of the library's device image, and this file
// never allocates or frees anything itself.  The array (DSA_NOALLOC_SCRATCH_BYTES)
// is reserved on a device when the library's device code is loaded there:
// with CUDA's default lazy loading that is the first call of this entry point
// on the device, so such callers should make one call at start-up, before
// they reserve their KV pools.  It is then held until the process exits (or
// the context is reset).
//
// The array is a file-scope __device__ symbol.  On the host its name is only a
// stand-in, not a device address, so every call looks the real address up
// through cudaGetSymbolAddress with the call's device current.  The lookup is
// cheap and is not cached: after a cudaDeviceReset the module may be loaded
// again at another address, and a remembered address would then point at
// memory this library no longer owns.
#include <cuda_runtime.h>

#include "dsa_decode.h"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch on the current device.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
  *out = p;
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
