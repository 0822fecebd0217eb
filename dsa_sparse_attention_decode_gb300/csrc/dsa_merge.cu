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
//   1. the exact threshold key T over the union (histograms, as for one row),
//      ties at T going to the lowest global positions;
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
  for (int b = tid; b < kSelBins1; b += kMergeThreads) hist[b] = 0;
  __syncthreads();
  int total = 0;
  for (int v = 0; v < W; ++v) total += cnt[v];
  const bool all = total <= k;
  auto valid = [&](int e) { return (e % k) < cnt[e / k]; };
  for (int e = tid; e < N; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i < cnt[w]) {
      const long long g = (static_cast<long long>(w) * R + r) * k + i;
      const uint32_t key = score_key(__ldcg(P.cand_score + g));
      const int p = __ldcg(P.cand_pos + g);
      if (p < 0 || p % W != w) raise_err(P.d_err, DSA_DEVERR_INDEX);
      keys[e] = key;
      pos[e] = p;
      if (!all) atomicAdd(hist + (key >> kSelShift1), 1u);
    }
  }
  __syncthreads();
  uint32_t T = 0, k_rem = 0;
  if (!all)
    refine_threshold([&](int e) { return keys[e]; }, valid, N, static_cast<uint32_t>(k), hist,
                     scratch, sh, T, k_rem);

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

__global__ void lse_merge_kernel(const float* __restrict__ O_parts,
                                 const float* __restrict__ lse_parts, int parts, int rows,
                                 int heads, int dv, float* __restrict__ out,
                                 float* __restrict__ out_lse, const float* __restrict__ max_parts,
                                 float* __restrict__ out_max) {
  const int rh = blockIdx.x;  // r * heads + h
  pdl_trigger();
  pdl_wait();  // the partials come from the previous grid
  const long long stride_p = static_cast<long long>(rows) * heads;
  const int d4 = threadIdx.x;
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
  if (has_d)
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
  const int threads = ((dv / 4 + 31) / 32) * 32;  // one float4 of the value dims per thread
  if ((max_parts == nullptr) != (out_max == nullptr)) return cudaErrorInvalidValue;
  return launch_ex(lse_merge_kernel, dim3(rows * heads), dim3(threads), 0, stream, pdl, O_parts,
                   lse_parts, parts, rows, heads, dv, out, out_lse, max_parts, out_max);
}

}  // namespace dsa
