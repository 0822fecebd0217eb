// Self-test of the bounded on-chip wait every kernel of this library uses.
//
// "Harden DeepSeek V4 DSpark DP2 serving", fail-closed convention: a wait that
// cannot complete must end in a reported error, not a hang.  Each kernel waits
// on mbarriers through mbar_wait (dsa_common.cuh), which gives up after a time
// limit, sets the CTA's abort flag and lets the kernel record
// DSA_DEVERR_TIMEOUT and return.  This kernel runs that same wait on a phase
// that nothing completes (one CTA, one thread waiting, nothing in flight), so
// the give-up path can be exercised on a GPU without disturbing it.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

__global__ void bounded_wait_kernel(uint64_t limit_ns, int32_t* d_err, uint64_t* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival completes the phase; none comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(smem_u32(&bar), 0u, &abort_flag, limit_ns);
    *waited_ns = globaltimer_ns() - t0;
    if (!ok && abort_flag) raise_err(d_err, DSA_DEVERR_TIMEOUT);
    // complete the phase so that the barrier is not left mid-phase
    mbar_arrive(smem_u32(&bar));
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* d_err, uint64_t* waited_ns,
                                         cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, d_err, waited_ns);
  return cudaGetLastError();
}

}  // namespace dsa
