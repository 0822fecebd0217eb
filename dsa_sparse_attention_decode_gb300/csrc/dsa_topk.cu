// Exact top-k of indexer score rows.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Motivation: DSA keeps the top 2048 tokens of the whole sequence; Modifications
// / Indexer decode: every shard first keeps a local top-k of its own tokens.
//
// One CTA of 1024 threads per score row:
//   1. scores become order-preserving uint32 keys (-0 == +0), cached in shared
//      memory when the row fits; the same pass builds a histogram of the top
//      13 key bits;
//   2. the bin holding the k-th largest key is refined with two more
//      histograms (10 and 9 bits) over only the keys still in play, giving the
//      exact threshold key T and how many keys equal to T are taken;
//   3. keys above T are appended; keys equal to T are appended when all of
//      them are taken, else the lowest positions are taken in position order;
//   4. the k survivors are bitonic-sorted on (key, ~position) so that the
//      output is ordered by score descending, then position ascending; the
//      strides below 64 run in registers with warp shuffles.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBins1 = 8192;  // key bits [31:19]
constexpr int kShift1 = 19;
constexpr int kShift2 = 9;    // key bits [18:9]
constexpr int kBins2 = 1024;
constexpr int kBins3 = 512;   // key bits [8:0]

struct TopkSmem {
  int cap;         // keys cached in smem
  int sort_n;      // power of two >= max(k, 64)
  int off_keys, off_cand, off_hist, off_misc, total;
};

__host__ inline TopkSmem topk_smem(int k) {
  TopkSmem s{};
  int p = 64;
  while (p < k) p <<= 1;
  s.sort_n = p;
  s.off_cand = 0;
  s.off_hist = s.sort_n * 8;
  s.off_misc = s.off_hist + kBins1 * 4;
  s.off_keys = s.off_misc + 1024;
  s.cap = ((kSmemLimit - s.off_keys) / 4) & ~1023;
  s.total = s.off_keys + s.cap * 4;
  return s;
}

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
  for (int w = warp + 1; w < kWarps; ++w) add += scratch[w];
  __syncthreads();
  return s + add;
}

// Find the bin holding the k_rem-th largest key: writes (bin, k_rem within the
// bin, bin count) to out[0..2].  Every thread calls it.
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, uint32_t k_rem,
                                         uint32_t* scratch, uint32_t* out) {
  const int per = nb / kThreads;  // >= 1 (nb is 8192, 1024 or 512 -> handle 512 below)
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

__device__ __forceinline__ uint64_t composite(uint32_t key, int i) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i);
}

// append the lanes' items with `pred` at buf[base + counter ...) (any order)
__device__ __forceinline__ void warp_append(bool pred, uint64_t item, uint32_t* counter,
                                            uint64_t* buf, uint32_t base) {
  const int lane = threadIdx.x & 31;
  const unsigned m = __ballot_sync(0xffffffffu, pred);
  if (m == 0u) return;
  const int leader = __ffs(m) - 1;
  uint32_t b0 = 0;
  if (lane == leader) b0 = atomicAdd(counter, static_cast<uint32_t>(__popc(m)));
  b0 = __shfl_sync(0xffffffffu, b0, leader);
  if (pred) buf[base + b0 + __popc(m & ((1u << lane) - 1u))] = item;
}

__device__ void bitonic_sort_desc(uint64_t* buf, int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int size = 2; size <= n; size <<= 1) {
    int stride = size >> 1;
    for (; stride >= 64; stride >>= 1) {
      for (int t = tid; t < (n >> 1); t += kThreads) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const uint64_t a = buf[i], b = buf[j];
        const bool desc = (i & size) == 0;
        if (desc ? (a < b) : (a > b)) {
          buf[i] = b;
          buf[j] = a;
        }
      }
      __syncthreads();
    }
    // strides < 64: chunks of 64 elements, two per lane, in registers
    for (int c = warp; c < (n >> 6); c += kWarps) {
      const int i0 = c * 64 + lane, i1 = i0 + 32;
      uint64_t v0 = buf[i0], v1 = buf[i1];
      for (int s = stride; s > 0; s >>= 1) {
        if (s == 32) {
          const bool desc = (i0 & size) == 0;
          if (desc ? (v0 < v1) : (v0 > v1)) {
            const uint64_t t = v0;
            v0 = v1;
            v1 = t;
          }
        } else {
          const uint64_t o0 = __shfl_xor_sync(0xffffffffu, v0, s);
          const uint64_t o1 = __shfl_xor_sync(0xffffffffu, v1, s);
          const bool lower = (lane & s) == 0;
          const bool d0 = (i0 & size) == 0, d1 = (i1 & size) == 0;
          v0 = (lower == d0) ? (v0 > o0 ? v0 : o0) : (v0 < o0 ? v0 : o0);
          v1 = (lower == d1) ? (v1 > o1 ? v1 : o1) : (v1 < o1 ? v1 : o1);
        }
      }
      buf[i0] = v0;
      buf[i1] = v1;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const TopkLaunch P, const TopkSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + S.off_cand);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);
  uint32_t* scratch = misc;       // 32 words
  uint32_t* sh = misc + 64;       // shared scalars

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int q = blockIdx.x;
  const int w = q / P.rows;
  const int r = q - w * P.rows;
  const int k = P.k;

  int n;
  if (P.valid_len) {
    n = P.valid_len[q];
  } else {
    n = shard_valid_len(P.row_pos[r], P.W, w + P.shard_offset);
  }
  if (n < 0 || n > P.ld) {
    if (tid == 0) raise_err(P.d_err, DSA_DEVERR_INDEX);
    n = n < 0 ? 0 : static_cast<int>(P.ld);
  }
  const float* src = P.scores + static_cast<long long>(w) * P.shard_stride +
                     static_cast<long long>(r) * P.ld;
  const bool in_smem = n <= S.cap;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int cnt = n < k ? n : k;
  int sort_n = 64;
  while (sort_n < cnt) sort_n <<= 1;

  for (int b = tid; b < kBins1; b += kThreads) hist[b] = 0;
  if (tid < 16) sh[tid] = 0;
  __syncthreads();

  // ---------------- pass 1: keys (+ smem copy) and the 13-bit histogram
  const bool need_select = n > k;
  bool nan_seen = false;
  {
    const int nv = vec ? (n >> 2) : 0;
    const float4* src4 = reinterpret_cast<const float4*>(src);
    for (int base = 0; base < nv; base += kThreads * 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kThreads + tid;
        v[u] = i < nv ? __ldg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < nv) {
          const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          uint4 kk;
          uint32_t* kp = reinterpret_cast<uint32_t*>(&kk);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            nan_seen |= (f[e] != f[e]);
            kp[e] = score_key(f[e]);
            if (need_select) atomicAdd(hist + (kp[e] >> kShift1), 1u);
          }
          if (in_smem) reinterpret_cast<uint4*>(keys)[i] = kk;
        }
      }
    }
    for (int i = nv * 4 + tid; i < n; i += kThreads) {
      const float f = __ldg(src + i);
      nan_seen |= (f != f);
      const uint32_t key = score_key(f);
      if (need_select) atomicAdd(hist + (key >> kShift1), 1u);
      if (in_smem) keys[i] = key;
    }
  }
  if (nan_seen) sh[0] = 1;
  __syncthreads();
  if (tid == 0 && sh[0]) raise_err(P.d_err, DSA_DEVERR_NAN);

  auto key_at = [&](int i) -> uint32_t {
    return in_smem ? keys[i] : score_key(__ldg(src + i));
  };

  if (!need_select) {
    for (int i = tid; i < sort_n; i += kThreads) cand[i] = i < n ? composite(key_at(i), i) : 0ull;
  } else {
    // ---------------- refine the threshold bin to the exact k-th key
    find_bin(hist, kBins1, static_cast<uint32_t>(k), scratch, sh + 4);
    const uint32_t b1 = sh[4];
    uint32_t k_rem = sh[5];
    for (int b = tid; b < kBins2; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key >> kShift1) == b1) atomicAdd(hist + ((key >> kShift2) & (kBins2 - 1)), 1u);
    }
    __syncthreads();
    find_bin(hist, kBins2, k_rem, scratch, sh + 4);
    const uint32_t pre2 = (b1 << (kShift1 - kShift2)) | sh[4];
    k_rem = sh[5];
    for (int b = tid; b < kBins3; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key >> kShift2) == pre2) atomicAdd(hist + (key & (kBins3 - 1)), 1u);
    }
    __syncthreads();
    find_bin(hist, kBins3, k_rem, scratch, sh + 4);
    const uint32_t T = (pre2 << kShift2) | sh[4];
    k_rem = sh[5];
    const uint32_t eq_count = sh[6];
    const uint32_t n_gt = static_cast<uint32_t>(k) - k_rem;
    const bool take_all_eq = eq_count == k_rem;
    __syncthreads();

    // ---------------- collect
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + tid;
      const uint32_t key = i < n ? key_at(i) : 0u;
      warp_append(i < n && key > T, composite(key, i), sh + 1, cand, 0u);
      if (take_all_eq) warp_append(i < n && key == T, composite(key, i), sh + 2, cand, n_gt);
    }
    if (!take_all_eq) {
      // ties at the threshold: the k_rem lowest positions, in position order
      uint32_t taken = 0;
      for (int base = 0; base < n && taken < k_rem; base += kThreads) {
        const int i = base + tid;
        const bool eq = i < n && key_at(i) == T;
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) scratch[tid >> 5] = static_cast<uint32_t>(__popc(m));
        __syncthreads();
        uint32_t off = 0, tot = 0;
        for (int wv = 0; wv < kWarps; ++wv) {
          const uint32_t c = scratch[wv];
          if (wv < (tid >> 5)) off += c;
          tot += c;
        }
        if (eq) {
          const uint32_t rank = taken + off + __popc(m & ((1u << lane) - 1u));
          if (rank < k_rem) cand[n_gt + rank] = composite(T, i);
        }
        taken += tot;
        __syncthreads();
      }
    }
    for (int i = cnt + tid; i < sort_n; i += kThreads) cand[i] = 0ull;
  }
  __syncthreads();

  bitonic_sort_desc(cand, sort_n);

  // ---------------- write
  const int off = P.index_offset + (P.offset_per_shard ? (w + P.shard_offset) : 0);
  int32_t* oi = P.out_idx + static_cast<long long>(q) * k;
  float* os = P.out_score ? P.out_score + static_cast<long long>(q) * k : nullptr;
  for (int i = tid; i < k; i += kThreads) {
    if (i < cnt) {
      const uint64_t c = cand[i];
      const int j = static_cast<int>(~static_cast<uint32_t>(c));
      oi[i] = j * P.index_stride + off;
      if (os) os[i] = key_score(static_cast<uint32_t>(c >> 32));
    } else {
      oi[i] = -1;
      if (os) os[i] = -__int_as_float(0x7f800000);
    }
  }
  if (tid == 0) P.out_count[q] = cnt;
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& p, cudaStream_t stream) {
  const TopkSmem S = topk_smem(p.k);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
  if (e != cudaSuccess) return e;
  const int grid = p.nshards * p.rows;
  if (grid == 0) return cudaSuccess;
  topk_kernel<<<grid, kThreads, S.total, stream>>>(p, S);
  return cudaGetLastError();
}

}  // namespace dsa
