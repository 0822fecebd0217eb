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

constexpr int kSelBins1 = 8192;  // key bits [31:19]
constexpr int kSelShift1 = 19;
constexpr int kSelShift2 = 9;    // key bits [18:9]
constexpr int kSelBins2 = 1024;
constexpr int kSelBins3 = 512;   // key bits [8:0]

// With `hist` holding the histogram of key >> kSelShift1 over the items that
// take part, find the exact k-th largest key T and how many of the keys equal
// to T belong to the top k (the rest of the top k is every key above T).
// key_of(i) gives item i's key and valid(i) whether it takes part; two more
// histograms touch only the items still in play.  `sh` holds 3 scratch words.
template <class KeyFn, class ValidFn>
__device__ __forceinline__ void refine_threshold(KeyFn key_of, ValidFn valid, int n, uint32_t k,
                                                 uint32_t* hist, uint32_t* scratch,
                                                 uint32_t* sh, uint32_t& T, uint32_t& k_rem) {
  const int tid = threadIdx.x;
  find_bin(hist, kSelBins1, k, scratch, sh);
  const uint32_t b1 = sh[0];
  k_rem = sh[1];
  for (int b = tid; b < kSelBins2; b += kSelThreads) hist[b] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kSelThreads) {
    if (!valid(i)) continue;
    const uint32_t key = key_of(i);
    if ((key >> kSelShift1) == b1)
      atomicAdd(hist + ((key >> kSelShift2) & (kSelBins2 - 1)), 1u);
  }
  __syncthreads();
  find_bin(hist, kSelBins2, k_rem, scratch, sh);
  const uint32_t pre2 = (b1 << (kSelShift1 - kSelShift2)) | sh[0];
  k_rem = sh[1];
  for (int b = tid; b < kSelBins3; b += kSelThreads) hist[b] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kSelThreads) {
    if (!valid(i)) continue;
    const uint32_t key = key_of(i);
    if ((key >> kSelShift2) == pre2) atomicAdd(hist + (key & (kSelBins3 - 1)), 1u);
  }
  __syncthreads();
  find_bin(hist, kSelBins3, k_rem, scratch, sh);
  T = (pre2 << kSelShift2) | sh[0];
  k_rem = sh[1];
  __syncthreads();
}

}  // namespace dsa
