// Device helpers shared by the sm_103a kernels: mbarriers with bounded waits,
// TMA loads, tcgen05 (MMA, TMEM) wrappers, smem descriptors, error word.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_decode.h"

#define DSA_DEV __device__ __forceinline__

namespace dsa {

constexpr int kIdxHeads = DSA_INDEX_HEADS;
constexpr int kIdxDim = DSA_INDEX_DIM;
constexpr int kKvDim = DSA_KV_DIM;
constexpr int kVDim = DSA_V_DIM;
constexpr int kMaxShards = DSA_MAX_SHARDS;
constexpr int kRowsPerGroup = 8;  // indexer query rows one CTA holds at a time

// A bounded on-chip wait gives up after this long (ns of %globaltimer).  Every
// kernel here finishes in well under a millisecond, so reaching it means the
// pipeline is broken; the kernel then records DSA_DEVERR_TIMEOUT and exits.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

DSA_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DSA_DEV void raise_err(int32_t* d_err, int bits) {
  if (d_err != nullptr) atomicOr(d_err, bits);
}

// Programmatic dependent launch.  A kernel lets the next kernel of its stream
// start launching once every one of its CTAs has started (the next grid's CTAs
// then take SMs as this grid's CTAs leave), and waits for the previous grid
// to complete, memory included, before it reads what that grid wrote or
// writes anything itself.  Both are no-ops in a plain launch.
DSA_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DSA_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host: launch `kern`, as a programmatic dependent of the stream's previous
// kernel when `pdl` is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

DSA_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier

DSA_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

DSA_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

DSA_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

DSA_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

DSA_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}


// Wait for the phase with the given parity to complete.  Returns false when
// the CTA-wide abort flag is set or the wait runs past limit_ns (the kernels
// use kWaitTimeoutNs; it then sets the flag itself).  Never spins forever.
DSA_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                       uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}


// ----------------------------------------------------------------- TMA

DSA_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

DSA_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                         int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes global -> shared (both
// addresses 16-byte aligned, bytes a multiple of 16), completing on `bar`.
DSA_DEV void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}


DSA_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

DSA_DEV void named_bar_sync(int id, int nthreads) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}


// ----------------------------------------------------------------- clusters

DSA_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders shared-memory writes before
// the barrier with reads (also remote ones) after it
DSA_DEV void cluster_sync() {
  __syncwarp();  // the .aligned forms need a converged warp
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the shared-memory address `saddr` of this CTA, mapped into CTA `rank`
DSA_DEV uint32_t dsmem_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
DSA_DEV uint4 dsmem_ld_v4(uint32_t caddr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}
DSA_DEV uint32_t dsmem_ld(uint32_t caddr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
  return v;
}

// ----------------------------------------------------------------- tcgen05
//
// Every helper below whose instruction is warp-collective (.sync.aligned, like
// the bar.sync named barrier and the cluster barrier above) first reconverges
// the warp with __syncwarp(): those forms are undefined when the warp arrives
// diverged, and the compiler does not know that an inline-asm instruction
// needs it.

DSA_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
DSA_DEV void tmem_relinquish() {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DSA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
DSA_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
DSA_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 or f16 inputs, f32 accumulate)
DSA_DEV void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A . B^T with e4m3 operands (both the same type) and an fp32 accumulator
DSA_DEV void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive once on the mbarrier when all prior tcgen05 async ops of this thread end
DSA_DEV void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}

DSA_DEV void tmem_wait_ld() {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// cp.async 16 bytes global -> shared (L2 only)
DSA_DEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
DSA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DSA_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane
DSA_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes stacked along
// M/N (stride byte offset 1024); the atom must be 1024-byte aligned.
DSA_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, K-major operands;
// a_bf16/b_bf16 select bf16 (1) or f16 (0) inputs.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_bf16, int b_bf16) {
  return (1u << 4) | (static_cast<uint32_t>(a_bf16) << 7) |
         (static_cast<uint32_t>(b_bf16) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0 for
// both), f32 accumulator, K-major operands.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ----------------------------------------------------------------- misc

// Orderable key of an fp32 score: larger score <-> larger key; -0 == +0.
DSA_DEV uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
DSA_DEV float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

DSA_DEV int shard_valid_len(int pos, int W, int w) {
  return pos < w ? 0 : (pos - w) / W + 1;
}

}  // namespace dsa
