// Shared pieces of the exact selections (top-k of a score row, top-k of the
// union of shard candidate lists): a 1024-thread block finds the exact k-th
// largest order-preserving key with histograms over key bit ranges.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

constexpr int kSelThreads = 1024;

// inclusive suffix sum over the 1024 threads (sum of values of threads >= tid)
__device__ __forceinline__ uint32_t block_suffix_sum(uint32_t v, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t s = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, s, o);
    if (lane + o < 32) s += t;
  }
  if (lane == 0) scratch[warp] = s;
  __syncthreads();
  uint32_t add = 0;
  for (int w = warp + 1; w < (kSelThreads / 32); ++w) add += scratch[w];
  __syncthreads();
  return s + add;
}

// Find the bin holding the k_rem-th largest key: writes (bin, k_rem within the
// bin, bin count) to out[0..2].  Every thread calls it.
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, uint32_t k_rem,
                                         uint32_t* scratch, uint32_t* out) {
  const int per = nb / kSelThreads;  // bins per thread (0: nb < 1024, one bin)
  const int tid = threadIdx.x;
  uint32_t mine = 0;
  if (per >= 1) {
    for (int j = 0; j < per; ++j) mine += hist[tid * per + j];
  } else if (tid < nb) {
    mine = hist[tid];
  }
  const uint32_t incl = block_suffix_sum(mine, scratch);
  const uint32_t above = incl - mine;
  if (above < k_rem && incl >= k_rem) {
    const int p = per >= 1 ? per : 1;
    uint32_t acc = above;
    for (int j = p - 1; j >= 0; --j) {
      const uint32_t h = hist[tid * p + j];
      if (acc + h >= k_rem) {
        out[0] = static_cast<uint32_t>(tid * p + j);
        out[1] = k_rem - acc;
        out[2] = h;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

// Bins of a key range [rlo, rhi] (inclusive): bin(key) = (key - rlo) >>
// shift, with shift the bits of (rhi - rlo) beyond nbits, so that the range
// splits into at most 2^nbits bins of 2^shift keys.
DSA_DEV int range_shift(uint32_t rlo, uint32_t rhi, int nbits) {
  const uint32_t wdt = rhi - rlo;
  const int len = wdt == 0u ? 0 : 32 - __clz(wdt);
  return len > nbits ? len - nbits : 0;
}
// the keys of bin b of [rlo, rhi] (the last bin may be short)
DSA_DEV void bin_range(uint32_t rlo, uint32_t rhi, int shift, uint32_t b, uint32_t* blo,
                       uint32_t* bhi) {
  const uint64_t l = static_cast<uint64_t>(rlo) + (static_cast<uint64_t>(b) << shift);
  const uint64_t h = l + (1ull << shift) - 1ull;
  *blo = static_cast<uint32_t>(l);
  *bhi = h < rhi ? static_cast<uint32_t>(h) : rhi;
}

constexpr int kSelBins1 = 8192;  // histogram bins of one selection round

}  // namespace dsa
