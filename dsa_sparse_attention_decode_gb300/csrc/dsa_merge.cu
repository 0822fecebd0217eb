// The two merge steps of the sharded decode.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Modifications / Indexer decode: the shards' (score, global position)
// candidates are merged into the exact global top-k and the merge emits the
// rows every shard owns (no separate compaction pass); Modifications / Sparse
// decode: the shards' partial (O, LSE) results are merged by their LSE.  The
// same LSE merge also combines split-K partials.
#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_select.cuh"

namespace dsa {
namespace {

// ------------------------------------------------------------ top-k merge
//
// The global top-k is the top-k of the union of the shards' candidate lists
// (every token of the global top-k is in its own shard's local top-k).  One
// 1024-thread CTA per query row:
//   1. the exact threshold key T over the union: 8192-bin histogram rounds
//      over a key range that starts as the candidates' smallest to largest
//      key (candidates all come from the upper tail of their rows, so fixed
//      top key bits would put them into a few bins); ties at T go to the
//      lowest global positions;
//   2. a candidate's rank among the ties, and later its output slot, is the
//      number of tied (selected) candidates with a lower global position in
//      every list: per-list prefix counts + a binary search in each list,
//      whose positions ascend;
//   3. selected positions go to the global list in ascending order and, as
//      local positions (p / W), to their own shard's owned list.
constexpr int kMergeThreads = kSelThreads;

struct MergeSmem {
  int off_keys, off_pos, off_pre, off_hist, off_misc, total;
};

__host__ __device__ inline MergeSmem merge_smem(int W, int k) {
  MergeSmem m{};
  const int N = W * k;
  m.off_keys = 0;
  m.off_pos = N * 4;
  m.off_pre = 2 * N * 4;
  m.off_hist = 3 * N * 4;
  m.off_misc = m.off_hist + kSelBins1 * 4;
  m.total = m.off_misc + 1024;
  return m;
}

// exclusive prefix of flag(e) over list w's first cnt entries -> pre[w*k + i];
// returns the list total.  Called by one whole warp.
template <class FlagFn>
__device__ __forceinline__ uint32_t warp_list_prefix(FlagFn flag, int w, int k, int cnt,
                                                     uint32_t* pre) {
  const int lane = threadIdx.x & 31;
  uint32_t run = 0;
  for (int i0 = 0; i0 < cnt; i0 += 32) {
    const int i = i0 + lane;
    const bool f = i < cnt && flag(w * k + i);
    const unsigned m = __ballot_sync(0xffffffffu, f);
    if (i < cnt) pre[w * k + i] = run + __popc(m & ((1u << lane) - 1u));
    run += __popc(m);
  }
  return run;
}

// number of entries of ascending list [p0, p0 + n) below x
__device__ __forceinline__ int lower_bound(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kMergeThreads, 1) shard_topk_merge_kernel(const MergeTopkLaunch P) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = P.W, k = P.k, R = P.rows, N = W * k;
  const MergeSmem S = merge_smem(W, k);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);  // later: selected flags
  int* pos = reinterpret_cast<int*>(smem + S.off_pos);
  uint32_t* pre = reinterpret_cast<uint32_t*>(smem + S.off_pre);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* scratch = misc;                             // 32
  uint32_t* sh = misc + 32;                             // 8
  int* cnt = reinterpret_cast<int*>(misc + 64);         // [8]
  uint32_t* tot = misc + 80;                            // [8] per-list totals
  const int r = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // the candidate lists come from the previous grid

  if (tid < W) {
    int c = __ldcg(P.cand_count + tid * R + r);
    if (c < 0 || c > k) {
      raise_err(P.d_err, DSA_DEVERR_INDEX);
      c = c < 0 ? 0 : k;
    }
    cnt[tid] = c;
  }
  __syncthreads();
  int total = 0;
  for (int v = 0; v < W; ++v) total += cnt[v];
  const bool all = total <= k;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  {
    // the candidates, 8 loads in flight per thread
    constexpr int kU = 8;
    for (int e0 = 0; e0 < N; e0 += kMergeThreads * kU) {
      uint32_t key[kU];
      int pv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = e0 + u * kMergeThreads + tid;
        const int w = e / k, i = e - w * k;
        pv[u] = -2;
        if (e < N && i < cnt[w]) {
          const long long g = (static_cast<long long>(w) * R + r) * k + i;
          key[u] = score_key(__ldcg(P.cand_score + g));
          pv[u] = __ldcg(P.cand_pos + g);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = e0 + u * kMergeThreads + tid;
        if (pv[u] == -2) continue;
        const int w = e / k;
        if (pv[u] < 0 || pv[u] % W != w) raise_err(P.d_err, DSA_DEVERR_INDEX);
        keys[e] = key[u];
        pos[e] = pv[u];
        kmin = min(kmin, key[u]);
        kmax = max(kmax, key[u]);
      }
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((tid & 31) == 0) {
    scratch[warp] = kmin;
    hist[warp] = kmax;  // the histogram is not in use yet
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = __reduce_min_sync(0xffffffffu, scratch[tid]);
    const uint32_t b = __reduce_max_sync(0xffffffffu, hist[tid]);
    if (tid == 0) {
      sh[4] = a;
      sh[5] = b;
    }
  }
  __syncthreads();
  uint32_t T = 0, k_rem = static_cast<uint32_t>(k);
  if (!all) {
    // [rlo, rhi] holds T; k_rem is T's rank in it from the top
    uint32_t rlo = sh[4], rhi = sh[5];
    __syncthreads();  // sh is read before find_bin writes it
    auto valid = [&](int e) { return (e % k) < cnt[e / k]; };
    while (rlo < rhi) {
      const int shift = range_shift(rlo, rhi, 13);
      for (int b = tid; b < kSelBins1; b += kMergeThreads) hist[b] = 0;
      __syncthreads();
      for (int e = tid; e < N; e += kMergeThreads) {
        if (!valid(e)) continue;
        const uint32_t key = keys[e];
        if (key >= rlo && key <= rhi) atomicAdd(hist + ((key - rlo) >> shift), 1u);
      }
      __syncthreads();
      find_bin(hist, kSelBins1, k_rem, scratch, sh);  // ends with a barrier
      bin_range(rlo, rhi, shift, sh[0], &rlo, &rhi);
      k_rem = sh[1];
      __syncthreads();  // sh and hist are read before the next round writes them
    }
    T = rlo;
  }

  // ranks of the ties at T, by global position
  if (warp < W) {
    const uint32_t t =
        warp_list_prefix([&](int e) { return !all && keys[e] == T; }, warp, k, cnt[warp], pre);
    if ((tid & 31) == 0) tot[warp] = t;
  }
  __syncthreads();
  uint32_t selflag[(DSA_MAX_SHARDS * 4096 + kMergeThreads - 1) / kMergeThreads];
  for (int e = tid, it = 0; e < N; e += kMergeThreads, ++it) {
    const int w = e / k, i = e - w * k;
    bool sel = false;
    if (i < cnt[w]) {
      const uint32_t key = keys[e];
      if (all || key > T) {
        sel = true;
      } else if (key == T) {
        uint32_t rank = pre[e];
        for (int v = 0; v < W; ++v) {
          if (v == w) continue;
          const int j = lower_bound(pos + v * k, cnt[v], pos[e]);
          rank += j < cnt[v] ? pre[v * k + j] : tot[v];
        }
        sel = rank < k_rem;
      }
    }
    selflag[it] = sel ? 1u : 0u;
  }
  __syncthreads();
  for (int e = tid, it = 0; e < N; e += kMergeThreads, ++it) keys[e] = selflag[it];
  __syncthreads();
  // output slots: selected candidates with a lower global position
  if (warp < W) {
    const uint32_t t = warp_list_prefix([&](int e) { return keys[e] != 0u; }, warp, k, cnt[warp], pre);
    if ((tid & 31) == 0) tot[warp] = t;
  }
  __syncthreads();
  uint32_t out_cnt = 0;
  for (int v = 0; v < W; ++v) out_cnt += tot[v];
  int32_t* oidx = P.out_idx + static_cast<long long>(r) * k;
  for (int e = tid; e < N; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i >= cnt[w] || keys[e] == 0u) continue;
    const int p = pos[e];
    uint32_t slot = pre[e];
    for (int v = 0; v < W; ++v) {
      if (v == w) continue;
      const int j = lower_bound(pos + v * k, cnt[v], p);
      slot += j < cnt[v] ? pre[v * k + j] : tot[v];
    }
    oidx[slot] = p;
    P.owned_local[(static_cast<long long>(w) * R + r) * k + pre[e]] = p / W;
  }
  for (int j = static_cast<int>(out_cnt) + tid; j < k; j += kMergeThreads) oidx[j] = -1;
  for (int e = tid; e < N; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i >= static_cast<int>(tot[w])) P.owned_local[(static_cast<long long>(w) * R + r) * k + i] = -1;
  }
  if (tid < W) P.owned_count[tid * R + r] = static_cast<int>(tot[tid]);
  if (tid == 0) P.out_count[r] = static_cast<int>(out_cnt);
}

// ------------------------------------------------------------ top-k merge,
// bitmap form
//
// With every candidate position below a known bound: the same exact
// threshold T, then the selection is marked in two bitmaps over the row's
// global positions (above T; equal to T).  Walking the bitmap words in
// position order takes the ties lowest positions first and gives every
// selected position its slot in the global list; a shard's owned list is the
// same walk restricted to the bits p with p % W == w.  No search per
// candidate, and both lists come out in ascending order.
constexpr int kMaxBitmapWords = 8192;  // positions below 262144

struct MergeBmSmem {
  int nw, off_keys, off_pos, off_hist, off_gt, off_eq, off_misc, total;
};

__host__ __device__ inline MergeBmSmem merge_bm_smem(int W, int k, int pos_bound) {
  MergeBmSmem m{};
  const int N = W * k;
  m.nw = ((pos_bound + 31) / 32 + 3) / 4 * 4;
  m.off_keys = 0;
  m.off_pos = N * 4;
  m.off_hist = 2 * N * 4;
  m.off_gt = m.off_hist + kSelBins1 * 4;
  m.off_eq = m.off_gt + m.nw * 4;
  m.off_misc = m.off_eq + m.nw * 4;
  m.total = m.off_misc + 1024;
  return m;
}

// exclusive prefix sum of v over the 1024 threads; *total gets the sum
__device__ __forceinline__ uint32_t excl_scan1024(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();  // scratch is free
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  const uint32_t wt = scratch[lane];
  uint32_t winc = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, winc, o);
    if (lane >= o) winc += t;
  }
  *total = __shfl_sync(0xffffffffu, winc, 31);
  return __shfl_sync(0xffffffffu, winc - wt, warp) + incl - v;
}

__global__ void __launch_bounds__(kMergeThreads, 1)
    shard_merge_bitmap_kernel(const MergeTopkLaunch P, const MergeBmSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = P.W, k = P.k, R = P.rows, N = W * k;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);
  int* pos = reinterpret_cast<int*>(smem + S.off_pos);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* gtb = reinterpret_cast<uint32_t*>(smem + S.off_gt);
  uint32_t* eqb = reinterpret_cast<uint32_t*>(smem + S.off_eq);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* scratch = misc;                      // 32
  uint32_t* sh = misc + 32;                      // 8
  int* cnt = reinterpret_cast<int*>(misc + 64);  // [8]
  const int r = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int bound = P.pos_bound;
  pdl_trigger();
  pdl_wait();  // the candidate lists come from the previous grid

  if (tid < W) {
    int c = __ldcg(P.cand_count + tid * R + r);
    if (c < 0 || c > k) {
      raise_err(P.d_err, DSA_DEVERR_INDEX);
      c = c < 0 ? 0 : k;
    }
    cnt[tid] = c;
  }
  for (int j = tid; j < S.nw; j += kMergeThreads) {
    gtb[j] = 0u;
    eqb[j] = 0u;
  }
  __syncthreads();
  int total = 0;
  for (int v = 0; v < W; ++v) total += cnt[v];
  const bool all = total <= k;
  // a candidate slot holds a position (>= 0) or -1 (past its list, or left out)
  auto valid = [&](int e) { return pos[e] >= 0; };
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  {
    // two slots of every list per thread and round: up to 16 loads in flight
    constexpr int kU = 2;
    for (int i0 = 0; i0 < k; i0 += kMergeThreads * kU) {
      uint32_t key[kU][DSA_MAX_SHARDS];
      int pv[kU][DSA_MAX_SHARDS];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int w = 0; w < DSA_MAX_SHARDS; ++w) {
          const int i = i0 + u * kMergeThreads + tid;
          key[u][w] = 0u;
          pv[u][w] = -1;
          if (w < W && i < cnt[w]) {
            const long long g = (static_cast<long long>(w) * R + r) * k + i;
            key[u][w] = score_key(__ldcg(P.cand_score + g));
            pv[u][w] = __ldcg(P.cand_pos + g);
          }
        }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int w = 0; w < DSA_MAX_SHARDS; ++w) {
          const int i = i0 + u * kMergeThreads + tid;
          if (w >= W || i >= k) continue;
          int p = pv[u][w];
          if (i < cnt[w] && (p < 0 || p >= bound || p % W != w)) {
            raise_err(P.d_err, DSA_DEVERR_INDEX);
            p = -1;  // left out
          }
          keys[w * k + i] = key[u][w];
          pos[w * k + i] = p;
          if (p >= 0) {
            kmin = min(kmin, key[u][w]);
            kmax = max(kmax, key[u][w]);
          }
        }
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((tid & 31) == 0) {
    scratch[warp] = kmin;
    hist[warp] = kmax;  // the histogram is not in use yet
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = __reduce_min_sync(0xffffffffu, scratch[tid]);
    const uint32_t b = __reduce_max_sync(0xffffffffu, hist[tid]);
    if (tid == 0) {
      sh[4] = a;
      sh[5] = b;
    }
  }
  __syncthreads();
  uint32_t T = 0, k_rem = static_cast<uint32_t>(k);
  if (!all) {
    uint32_t rlo = sh[4], rhi = sh[5];
    __syncthreads();  // sh is read before find_bin writes it
    while (rlo < rhi) {
      const int shift = range_shift(rlo, rhi, 13);
      for (int b = tid; b < kSelBins1; b += kMergeThreads) hist[b] = 0;
      __syncthreads();
      for (int e = tid; e < N; e += kMergeThreads) {
        if (!valid(e)) continue;
        const uint32_t key = keys[e];
        if (key >= rlo && key <= rhi) atomicAdd(hist + ((key - rlo) >> shift), 1u);
      }
      __syncthreads();
      find_bin(hist, kSelBins1, k_rem, scratch, sh);  // ends with a barrier
      bin_range(rlo, rhi, shift, sh[0], &rlo, &rhi);
      k_rem = sh[1];
      __syncthreads();  // sh and hist are read before the next round writes them
    }
    T = rlo;
  }
  // the selection in the bitmaps: above T for sure; ties at T taken later
  for (int e = tid; e < N; e += kMergeThreads) {
    if (!valid(e)) continue;
    const uint32_t key = keys[e];
    const int p = pos[e];
    if (all || key > T) atomicOr(gtb + (p >> 5), 1u << (p & 31));
    else if (key == T) atomicOr(eqb + (p >> 5), 1u << (p & 31));
  }
  __syncthreads();
  // walk the words in position order: thread t a contiguous run of words
  const int nwu = (bound + 31) >> 5;
  const int per = (nwu + kMergeThreads - 1) / kMergeThreads;
  const int j0 = min(nwu, tid * per), j1 = min(nwu, j0 + per);
  uint32_t e_mine = 0;
  for (int j = j0; j < j1; ++j) e_mine += __popc(eqb[j]);
  uint32_t e_tot;
  uint32_t eq_before = excl_scan1024(e_mine, scratch, &e_tot);
  for (int j = j0; j < j1; ++j) {
    uint32_t ew = eqb[j];
    const uint32_t room = eq_before < k_rem ? k_rem - eq_before : 0u;
    const uint32_t pe = __popc(ew);
    if (pe > room) {  // keep the lowest `room` ties of the word
      uint32_t keep = 0u;
      for (uint32_t t = 0; t < room; ++t) {
        const uint32_t bit = ew & (0u - ew);
        keep |= bit;
        ew ^= bit;
      }
      ew = keep;
    }
    eq_before += pe;
    gtb[j] |= ew;  // the final selection (this thread's words only)
  }
  // global list
  uint32_t s_mine = 0;
  for (int j = j0; j < j1; ++j) s_mine += __popc(gtb[j]);
  uint32_t s_tot;
  uint32_t slot = excl_scan1024(s_mine, scratch, &s_tot);
  int32_t* oidx = P.out_idx + static_cast<long long>(r) * k;
  for (int j = j0; j < j1; ++j) {
    uint32_t sel = gtb[j];
    while (sel != 0u) {
      const int b = __ffs(sel) - 1;
      sel &= sel - 1u;
      if (slot < static_cast<uint32_t>(k)) oidx[slot] = j * 32 + b;
      ++slot;
    }
  }
  const uint32_t out_cnt = min(s_tot, static_cast<uint32_t>(k));
  for (int j = static_cast<int>(out_cnt) + tid; j < k; j += kMergeThreads) oidx[j] = -1;
  if (tid == 0) P.out_count[r] = static_cast<int>(out_cnt);
  // every shard's owned list: the bits p of word j with p % W == w
  for (int w = 0; w < W; ++w) {
    auto mask_of = [&](int j) {
      // bits b with (32 j + b) % W == w: the first is b0, then every W-th
      const int b0 = ((w - (32 * j) % W) % W + W) % W;
      uint32_t m = 0u;
      for (int b = b0; b < 32; b += W) m |= 1u << b;
      return m;
    };
    uint32_t o_mine = 0;
    for (int j = j0; j < j1; ++j) o_mine += __popc(gtb[j] & mask_of(j));
    uint32_t o_tot;
    uint32_t os = excl_scan1024(o_mine, scratch, &o_tot);
    int32_t* ol = P.owned_local + (static_cast<long long>(w) * R + r) * k;
    for (int j = j0; j < j1; ++j) {
      uint32_t sel = gtb[j] & mask_of(j);
      while (sel != 0u) {
        const int b = __ffs(sel) - 1;
        sel &= sel - 1u;
        if (os < static_cast<uint32_t>(k)) ol[os] = (j * 32 + b) / W;
        ++os;
      }
    }
    const uint32_t oc = min(o_tot, static_cast<uint32_t>(k));
    for (int j = static_cast<int>(oc) + tid; j < k; j += kMergeThreads) ol[j] = -1;
    if (tid == 0) P.owned_count[w * R + r] = static_cast<int>(oc);
  }
}

// ------------------------------------------------------------ LSE merge
//
// lse = ln sum_p exp(lse_p), out = sum_p exp(lse_p - lse) O_p; parts whose
// lse is -inf hold no tokens and are not read.  One CTA per (row, head), one
// float4 of the value vector per thread.
// One CTA per (row, head), one float4 of the value dims per thread.  Up to
// kFastParts partials, every load (LSEs and partial outputs alike) is issued
// before any is used, so the kernel waits for one round trip to L2; an
// empty partial (LSE -inf, output not written) is skipped by selection.
constexpr int kFastParts = 8;
// With more partials: every thread loads a share of the parts' LSEs, a
// block reduction gives their maximum, the live parts (LSE finite) are
// listed in part order by a block scan with their weights exp(lse_p - m),
// and the value dims accumulate the live partial outputs: kListGroups groups
// of threads take turns of kMergeUnroll consecutive live parts (that many
// loads in flight per thread), and group 0 adds the groups' sums in order.
// The order of every sum is fixed, so the result does not depend on
// scheduling.
constexpr int kMaxListParts = 1024;
constexpr int kMergeUnroll = 8;
constexpr int kListGroups = 4;          // thread groups of the live-list path
constexpr int kMaxGroupThreads = 768;   // (groups - 1) * padded dv / 4 it reduces over

// sum (kMax: maximum) of v over the CTA; every thread gets it.  red holds 33
// words.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float t = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, t) : v + t;
  }
  __syncthreads();  // red is free
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float x = lane < nw ? red[lane] : (kMax ? -__int_as_float(0x7f800000) : 0.0f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float t = __shfl_xor_sync(0xffffffffu, x, o);
      x = kMax ? fmaxf(x, t) : x + t;
    }
    if (lane == 0) red[32] = x;
  }
  __syncthreads();
  return red[32];
}

__global__ void lse_merge_kernel(const float* __restrict__ O_parts,
                                 const float* __restrict__ lse_parts, int parts, int rows,
                                 int heads, int dv, float* __restrict__ out,
                                 float* __restrict__ out_lse, const float* __restrict__ max_parts,
                                 float* __restrict__ out_max) {
  const int rh = blockIdx.x;  // r * heads + h
  pdl_trigger();
  pdl_wait();  // the partials come from the previous grid
  const long long stride_p = static_cast<long long>(rows) * heads;
  // groups of dpad threads, one float4 of the value dims per thread; more
  // than one group (the live-list path) splits the live partials between them
  const int dpad = ((dv / 4 + 31) / 32) * 32;
  const int d4 = threadIdx.x % dpad, grp = threadIdx.x / dpad, ngrp = blockDim.x / dpad;
  const bool has_d = d4 < dv / 4;
  const float kNegInf = -__int_as_float(0x7f800000);
  float m = kNegInf, den = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (parts <= kFastParts) {
    float l[kFastParts];
    float4 v[kFastParts];
#pragma unroll
    for (int p = 0; p < kFastParts; ++p) {
      l[p] = p < parts ? __ldcg(lse_parts + p * stride_p + rh) : kNegInf;
      v[p] = (p < parts && has_d)
                 ? __ldcg(reinterpret_cast<const float4*>(O_parts + (p * stride_p + rh) * dv) + d4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int p = 0; p < kFastParts; ++p) m = fmaxf(m, l[p]);
    if (m != kNegInf) {
#pragma unroll
      for (int p = 0; p < kFastParts; ++p) {
        const bool live = l[p] != kNegInf;
        const float e = live ? expf(l[p] - m) : 0.0f;
        den += e;
        acc.x = live ? fmaf(e, v[p].x, acc.x) : acc.x;
        acc.y = live ? fmaf(e, v[p].y, acc.y) : acc.y;
        acc.z = live ? fmaf(e, v[p].z, acc.z) : acc.z;
        acc.w = live ? fmaf(e, v[p].w, acc.w) : acc.w;
      }
    }
  } else if (parts <= kMaxListParts) {
    __shared__ float wgt[kMaxListParts];
    __shared__ int live[kMaxListParts];
    __shared__ float red[33];
    __shared__ int nlive_s;
    const int nt = blockDim.x;
    float lm = kNegInf;
    for (int p = threadIdx.x; p < parts; p += nt) {
      const float l = __ldcg(lse_parts + p * stride_p + rh);
      wgt[p] = l;
      lm = fmaxf(lm, l);
    }
    m = block_reduce<true>(lm, red);  // its barriers publish wgt
    if (m != kNegInf) {
      // live parts in part order: thread t takes a contiguous run of parts
      const int per = (parts + nt - 1) / nt;
      const int p0 = min(parts, static_cast<int>(threadIdx.x) * per), p1 = min(parts, p0 + per);
      int mine = 0;
      float dsum = 0.0f;
      for (int p = p0; p < p1; ++p) {
        const float l = wgt[p];
        if (l != kNegInf) {
          ++mine;
          dsum += expf(l - m);
        }
      }
      // exclusive scan of the live counts over the threads
      int incl = mine;
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      __shared__ int wsum[32];
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      int off = incl - mine;
      for (int w2 = 0; w2 < warp; ++w2) off += wsum[w2];
      if (threadIdx.x == nt - 1) nlive_s = off + mine;
      __syncthreads();  // every thread has read wsum and the raw LSEs of its run
      for (int p = p0; p < p1; ++p) {
        const float l = wgt[p];
        if (l != kNegInf) live[off++] = p;
      }
      den = block_reduce<false>(dsum, red);  // its barriers publish live
      const int nl = nlive_s;
      if (has_d) {
        for (int i0 = grp * kMergeUnroll; i0 < nl; i0 += ngrp * kMergeUnroll) {
          float4 v[kMergeUnroll];
          float e[kMergeUnroll];
#pragma unroll
          for (int u = 0; u < kMergeUnroll; ++u) {
            const int p = i0 + u < nl ? live[i0 + u] : -1;
            e[u] = p >= 0 ? expf(__ldcg(lse_parts + p * stride_p + rh) - m) : 0.0f;
            v[u] = p >= 0 ? __ldcg(reinterpret_cast<const float4*>(O_parts + (p * stride_p + rh) * dv) + d4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < kMergeUnroll; ++u) {
            acc.x = fmaf(e[u], v[u].x, acc.x);
            acc.y = fmaf(e[u], v[u].y, acc.y);
            acc.z = fmaf(e[u], v[u].z, acc.z);
            acc.w = fmaf(e[u], v[u].w, acc.w);
          }
        }
      }
    }
    if (ngrp > 1) {  // the groups' sums: group 0 adds the others
      __shared__ float4 gacc[kMaxGroupThreads];
      if (grp > 0 && has_d) gacc[threadIdx.x - dpad] = acc;
      __syncthreads();
      if (grp == 0 && has_d)
        for (int g2 = 1; g2 < ngrp; ++g2) {
          const float4 o = gacc[(g2 - 1) * dpad + d4];
          acc.x += o.x;
          acc.y += o.y;
          acc.z += o.z;
          acc.w += o.w;
        }
    }
  } else {
    for (int p = 0; p < parts; ++p) m = fmaxf(m, __ldcg(lse_parts + p * stride_p + rh));
    if (m != kNegInf) {
      for (int p = 0; p < parts; ++p) {
        const float l = __ldcg(lse_parts + p * stride_p + rh);
        if (l == kNegInf) continue;
        const float e = expf(l - m);
        den += e;
        if (has_d) {
          const float4 v =
              __ldcg(reinterpret_cast<const float4*>(O_parts + (p * stride_p + rh) * dv) + d4);
          acc.x = fmaf(e, v.x, acc.x);
          acc.y = fmaf(e, v.y, acc.y);
          acc.z = fmaf(e, v.z, acc.z);
          acc.w = fmaf(e, v.w, acc.w);
        }
      }
    }
  }
  const float inv = m == kNegInf ? 0.0f : 1.0f / den;
  if (has_d && grp == 0)
    reinterpret_cast<float4*>(out + static_cast<long long>(rh) * dv)[d4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (threadIdx.x == 0) out_lse[rh] = m == kNegInf ? m : m + logf(den);
  // the largest scaled logit over the parts (an empty part holds -inf)
  if (out_max != nullptr && threadIdx.x == 0) {
    float mx = kNegInf;
    for (int p = 0; p < parts; ++p) mx = fmaxf(mx, __ldcg(max_parts + p * stride_p + rh));
    out_max[rh] = mx;
  }
}

}  // namespace

int merge_smem_bytes(int W, int k) { return merge_smem(W, k).total; }

cudaError_t launch_shard_topk_merge(const MergeTopkLaunch& p, cudaStream_t stream, bool pdl) {
  if (p.rows == 0) return cudaSuccess;
  if (p.pos_bound > 0 && (p.pos_bound + 31) / 32 <= kMaxBitmapWords) {
    const MergeBmSmem S = merge_bm_smem(p.W, p.k, p.pos_bound);
    if (S.total <= 227 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(shard_merge_bitmap_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
      if (e != cudaSuccess) return e;
      return launch_ex(shard_merge_bitmap_kernel, dim3(p.rows), dim3(kMergeThreads), S.total,
                       stream, pdl, p, S);
    }
  }
  const int smem = merge_smem_bytes(p.W, p.k);
  cudaError_t e = cudaFuncSetAttribute(shard_topk_merge_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_ex(shard_topk_merge_kernel, dim3(p.rows), dim3(kMergeThreads), smem, stream, pdl,
                   p);
}

cudaError_t launch_lse_merge(const float* O_parts, const float* lse_parts, int parts, int rows,
                             int heads, int dv, float* out, float* out_lse, cudaStream_t stream,
                             bool pdl, const float* max_parts, float* out_max) {
  if (rows * heads == 0) return cudaSuccess;
  if (dv % 4 != 0 || dv / 4 > 1024) return cudaErrorInvalidValue;
  const int dpad = ((dv / 4 + 31) / 32) * 32;  // one float4 of the value dims per thread
  // the live-list path splits the partials between groups of dpad threads
  const int groups = (parts > kFastParts && parts <= kMaxListParts &&
                      (kListGroups - 1) * dpad <= kMaxGroupThreads)
                         ? kListGroups
                         : 1;
  const int threads = dpad * groups;
  if ((max_parts == nullptr) != (out_max == nullptr)) return cudaErrorInvalidValue;
  return launch_ex(lse_merge_kernel, dim3(rows * heads), dim3(threads), 0, stream, pdl, O_parts,
                   lse_parts, parts, rows, heads, dv, out, out_lse, max_parts, out_max);
}

}  // namespace dsa
