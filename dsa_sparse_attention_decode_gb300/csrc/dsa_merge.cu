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

namespace dsa {
namespace {

// ------------------------------------------------------------ top-k merge
//
// Every candidate's place in the merged order is its index in its own list
// plus, for every other list, the number of entries that precede it there
// (binary search: lists are sorted by score descending, position ascending;
// positions of different shards differ, so there are no exact ties).
constexpr int kMergeThreads = 1024;

__device__ __forceinline__ bool precedes(float as, int ap, float bs, int bp) {
  return as > bs || (as == bs && ap < bp);
}

__global__ void __launch_bounds__(kMergeThreads, 1) shard_topk_merge_kernel(const MergeTopkLaunch P) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = P.W, k = P.k, R = P.rows;
  float* cs = reinterpret_cast<float*>(smem);
  int* cp = reinterpret_cast<int*>(smem + static_cast<size_t>(W) * k * 4);
  int* cnt = reinterpret_cast<int*>(smem + static_cast<size_t>(W) * k * 8);
  int* owned = cnt + DSA_MAX_SHARDS;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;

  if (tid < W) {
    int c = P.cand_count[tid * R + r];
    if (c < 0 || c > k) {
      raise_err(P.d_err, DSA_DEVERR_INDEX);
      c = c < 0 ? 0 : k;
    }
    cnt[tid] = c;
    owned[tid] = 0;
  }
  __syncthreads();
  for (int e = tid; e < W * k; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i < cnt[w]) {
      cs[e] = P.cand_score[(static_cast<long long>(w) * R + r) * k + i];
      cp[e] = P.cand_pos[(static_cast<long long>(w) * R + r) * k + i];
    }
  }
  __syncthreads();
  int total = 0;
  for (int w = 0; w < W; ++w) total += cnt[w];
  const int out_cnt = total < k ? total : k;

  int32_t* oidx = P.out_idx + static_cast<long long>(r) * k;
  for (int e = tid; e < W * k; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i >= cnt[w]) continue;
    const float s = cs[e];
    const int p = cp[e];
    if (p < 0 || p % W != w) raise_err(P.d_err, DSA_DEVERR_INDEX);
    int rank = i;
    for (int v = 0; v < W; ++v) {
      if (v == w) continue;
      int lo = 0, hi = cnt[v];  // first entry of list v that does not precede (s, p)
      const float* vs = cs + v * k;
      const int* vp = cp + v * k;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (precedes(vs[mid], vp[mid], s, p)) lo = mid + 1;
        else hi = mid;
      }
      rank += lo;
    }
    if (rank < k) {
      oidx[rank] = p;
      P.owned_local[(static_cast<long long>(w) * R + r) * k + i] = p / W;
      atomicAdd(owned + w, 1);
    }
  }
  __syncthreads();
  for (int j = out_cnt + tid; j < k; j += kMergeThreads) oidx[j] = -1;
  for (int e = tid; e < W * k; e += kMergeThreads) {
    const int w = e / k, i = e - w * k;
    if (i >= owned[w]) P.owned_local[(static_cast<long long>(w) * R + r) * k + i] = -1;
  }
  if (tid < W) P.owned_count[tid * R + r] = owned[tid];
  if (tid == 0) P.out_count[r] = out_cnt;
}

// ------------------------------------------------------------ LSE merge
//
// lse = ln sum_p exp(lse_p), out = sum_p exp(lse_p - lse) O_p; parts whose
// lse is -inf hold no tokens and are not read.  One CTA per (row, head), one
// float4 of the value vector per thread.
__global__ void lse_merge_kernel(const float* __restrict__ O_parts,
                                 const float* __restrict__ lse_parts, int parts, int rows,
                                 int heads, int dv, float* __restrict__ out,
                                 float* __restrict__ out_lse) {
  const int rh = blockIdx.x;  // r * heads + h
  const long long stride_p = static_cast<long long>(rows) * heads;
  float m = -__int_as_float(0x7f800000);
  for (int p = 0; p < parts; ++p) m = fmaxf(m, __ldg(lse_parts + p * stride_p + rh));
  const bool empty = (m == -__int_as_float(0x7f800000));
  float den = 0.0f;
  if (!empty)
    for (int p = 0; p < parts; ++p) den += expf(__ldg(lse_parts + p * stride_p + rh) - m);
  const float inv = empty ? 0.0f : 1.0f / den;
  for (int d4 = threadIdx.x; d4 < dv / 4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
      for (int p = 0; p < parts; ++p) {
        const float l = __ldg(lse_parts + p * stride_p + rh);
        if (l == -__int_as_float(0x7f800000)) continue;
        const float wgt = expf(l - m) * inv;
        const float4 v = __ldg(reinterpret_cast<const float4*>(O_parts + (p * stride_p + rh) * dv) + d4);
        acc.x = fmaf(wgt, v.x, acc.x);
        acc.y = fmaf(wgt, v.y, acc.y);
        acc.z = fmaf(wgt, v.z, acc.z);
        acc.w = fmaf(wgt, v.w, acc.w);
      }
    }
    reinterpret_cast<float4*>(out + static_cast<long long>(rh) * dv)[d4] = acc;
  }
  if (threadIdx.x == 0) out_lse[rh] = empty ? m : m + logf(den);
}

}  // namespace

int merge_smem_bytes(int W, int k) { return W * k * 8 + 2 * DSA_MAX_SHARDS * 4; }

cudaError_t launch_shard_topk_merge(const MergeTopkLaunch& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int smem = merge_smem_bytes(p.W, p.k);
  cudaError_t e = cudaFuncSetAttribute(shard_topk_merge_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  shard_topk_merge_kernel<<<p.rows, kMergeThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float* O_parts, const float* lse_parts, int parts, int rows,
                             int heads, int dv, float* out, float* out_lse, cudaStream_t stream) {
  if (rows * heads == 0) return cudaSuccess;
  const int threads = dv / 4 >= 128 ? 128 : ((dv / 4 + 31) / 32) * 32;
  lse_merge_kernel<<<rows * heads, threads, 0, stream>>>(O_parts, lse_parts, parts, rows, heads,
                                                          dv, out, out_lse);
  return cudaGetLastError();
}

}  // namespace dsa
