// Exact top-k of indexer score rows.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Motivation: DSA keeps the top 2048 tokens of the whole sequence; Modifications
// / Indexer decode: every shard first keeps a local top-k of its own tokens.
//
// One CTA of 1024 threads per score row:
//   1. scores become order-preserving uint32 keys (-0 == +0), cached in shared
//      memory when the row fits;
//   2. radix select of the k-th largest key in three passes (11, 11, 10 bits)
//      with shared-memory histograms fed by warp-aggregated atomics
//      (__match_any_sync), which keeps the hot bins of similar scores cheap;
//   3. keys above the threshold are appended; keys equal to it are taken in
//      ascending position order (only the first ones needed);
//   4. the k survivors are bitonic-sorted on (key, ~position) so the output
//      order is score descending, then position ascending.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemLimit = 227 * 1024;

struct TopkSmem {
  int cap;         // keys cached in smem
  int sort_n;      // power of two >= k
  int off_keys, off_cand, off_hist, off_misc, total;
};

__host__ inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__host__ inline TopkSmem topk_smem(int k) {
  TopkSmem s{};
  s.sort_n = pow2_at_least(k);
  const int cand = s.sort_n * 8;
  const int hist = 2048 * 4;
  const int misc = 1024;
  s.off_cand = 0;
  s.off_hist = cand;
  s.off_misc = cand + hist;
  s.off_keys = cand + hist + misc;
  s.cap = ((kSmemLimit - s.off_keys) / 4) & ~1023;
  s.total = s.off_keys + s.cap * 4;
  return s;
}

__device__ __forceinline__ void agg_add(uint32_t* hist, bool active, uint32_t digit) {
  const unsigned m = __ballot_sync(0xffffffffu, active);
  if (active) {
    const unsigned peers = __match_any_sync(m, digit);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1))
      atomicAdd(hist + digit, static_cast<uint32_t>(__popc(peers)));
  }
}

// inclusive suffix sums over the 1024 threads' values (sum of values of
// threads >= tid); `scratch` holds 32 ints
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

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const TopkLaunch P, const TopkSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + S.off_cand);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);
  uint32_t* scratch = misc;            // 32 words
  uint32_t* sh = misc + 64;            // shared scalars

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

  if (tid == 0) {
    sh[0] = 0;  // NaN seen
    sh[1] = 0;  // append counter (above threshold)
    sh[2] = 0;  // append counter (equal to threshold)
  }
  // load keys (and check NaN)
  bool nan_seen = false;
  for (int i = tid; i < n; i += kThreads) {
    const float f = __ldg(src + i);
    nan_seen |= (f != f);
    if (in_smem) keys[i] = score_key(f);
  }
  if (nan_seen) sh[0] = 1;
  __syncthreads();
  if (tid == 0 && sh[0]) raise_err(P.d_err, DSA_DEVERR_NAN);

  auto key_at = [&](int i) -> uint32_t {
    return in_smem ? keys[i] : score_key(__ldg(src + i));
  };

  const int cnt = n < k ? n : k;
  int sort_n = 1;
  while (sort_n < cnt) sort_n <<= 1;

  if (n <= k) {
    for (int i = tid; i < sort_n; i += kThreads)
      cand[i] = i < n ? ((static_cast<uint64_t>(key_at(i)) << 32) | static_cast<uint32_t>(~i))
                      : 0ull;
  } else {
    // ---------------- radix select of the k-th largest key
    uint32_t prefix = 0, pmask = 0;
    uint32_t k_rem = static_cast<uint32_t>(k);
    uint32_t eq_count = 0;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = shifts[pass];
      const int nb = 1 << widths[pass];
      const uint32_t dmask = static_cast<uint32_t>(nb - 1);
      for (int b = tid; b < nb; b += kThreads) hist[b] = 0;
      __syncthreads();
      for (int base = 0; base < n; base += kThreads) {
        const int i = base + tid;
        uint32_t key = 0;
        bool act = false;
        if (i < n) {
          key = key_at(i);
          act = (key & pmask) == prefix;
        }
        agg_add(hist, act, (key >> shift) & dmask);
      }
      __syncthreads();
      // thread t owns bins [t*per, (t+1)*per); find the bin where the count
      // of keys >= bin reaches k_rem
      const int per = nb / kThreads;  // 2 or 1
      uint32_t mine = 0;
      for (int j = 0; j < per; ++j) mine += hist[tid * per + j];
      const uint32_t incl = block_suffix_sum(mine, scratch);
      const uint32_t above = incl - mine;  // keys in bins above my range
      if (above < k_rem && incl >= k_rem) {
        uint32_t acc = above;
        for (int j = per - 1; j >= 0; --j) {
          const uint32_t h = hist[tid * per + j];
          if (acc + h >= k_rem) {
            sh[4] = static_cast<uint32_t>(tid * per + j);
            sh[5] = k_rem - acc;
            sh[6] = h;
            break;
          }
          acc += h;
        }
      }
      __syncthreads();
      prefix |= sh[4] << shift;
      pmask |= dmask << shift;
      k_rem = sh[5];
      eq_count = sh[6];
      __syncthreads();
    }
    const uint32_t T = prefix;
    const uint32_t n_gt = static_cast<uint32_t>(k) - k_rem;
    const bool take_all_eq = eq_count == k_rem;
    // ---------------- collect: keys > T anywhere in [0, n_gt); keys == T
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + tid;
      uint32_t key = 0;
      if (i < n) key = key_at(i);
      const bool gt = i < n && key > T;
      const bool eq = i < n && key == T && take_all_eq;
      {
        const unsigned m = __ballot_sync(0xffffffffu, gt);
        if (m) {
          uint32_t b0 = 0;
          if (lane == __ffs(m) - 1) b0 = atomicAdd(sh + 1, static_cast<uint32_t>(__popc(m)));
          b0 = __shfl_sync(0xffffffffu, b0, __ffs(m) - 1);
          if (gt) {
            const uint32_t pos = b0 + __popc(m & ((1u << lane) - 1u));
            cand[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i);
          }
        }
      }
      {
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        if (m) {
          uint32_t b0 = 0;
          if (lane == __ffs(m) - 1) b0 = atomicAdd(sh + 2, static_cast<uint32_t>(__popc(m)));
          b0 = __shfl_sync(0xffffffffu, b0, __ffs(m) - 1);
          if (eq) {
            const uint32_t pos = n_gt + b0 + __popc(m & ((1u << lane) - 1u));
            cand[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i);
          }
        }
      }
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
          if (rank < k_rem)
            cand[n_gt + rank] = (static_cast<uint64_t>(T) << 32) | static_cast<uint32_t>(~i);
        }
        taken += tot;
        __syncthreads();
      }
    }
    for (int i = cnt + tid; i < sort_n; i += kThreads) cand[i] = 0ull;
  }
  __syncthreads();

  // ---------------- bitonic sort, descending
  for (int size = 2; size <= sort_n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < (sort_n >> 1); t += kThreads) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const uint64_t a = cand[i], b = cand[j];
        const bool desc = (i & size) == 0;
        if (desc ? (a < b) : (a > b)) {
          cand[i] = b;
          cand[j] = a;
        }
      }
      __syncthreads();
    }
  }

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
