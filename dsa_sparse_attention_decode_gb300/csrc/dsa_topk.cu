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
//      exact threshold key T and how many keys equal to T are taken (the
//      lowest positions win ties);
//   3. an order-preserving compaction writes the selected positions in
//      ascending order: every warp owns a contiguous segment of the row,
//      counts its keys above / equal to T, and after one exclusive scan over
//      the warps writes its selected positions at their final slots.
// No sort: the list comes out in position order.
#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_select.cuh"

namespace dsa {
namespace {

constexpr int kThreads = kSelThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBins1 = kSelBins1;
constexpr int kShift1 = kSelShift1;

struct TopkSmem {
  int cap;         // keys cached in smem
  int off_keys, off_hist, off_misc, total;
};

__host__ inline TopkSmem topk_smem() {
  TopkSmem s{};
  s.off_hist = 0;
  s.off_misc = s.off_hist + kBins1 * 4;
  s.off_keys = s.off_misc + 1024;
  s.cap = ((kSmemLimit - s.off_keys) / 4) & ~1023;
  s.total = s.off_keys + s.cap * 4;
  return s;
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const TopkLaunch P, const TopkSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
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

  const int off = P.index_offset + (P.offset_per_shard ? (w + P.shard_offset) : 0);
  int32_t* oi = P.out_idx + static_cast<long long>(q) * k;
  float* os = P.out_score ? P.out_score + static_cast<long long>(q) * k : nullptr;

  uint32_t T = 0, k_rem = 0;
  bool all = true;  // n <= k: every position is selected
  if (need_select) {
    all = false;
    // ---------------- refine the threshold bin to the exact k-th key
    refine_threshold(key_at, [](int) { return true; }, n, static_cast<uint32_t>(k), hist,
                     scratch, sh + 4, T, k_rem);
    // k_rem: keys equal to T that are taken (the lowest positions)
  }

  // ---------------- order-preserving compaction by warp segments
  const int warp = tid >> 5;
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  uint32_t* wgt = misc + 128;  // [32] keys above T per warp
  uint32_t* weq = misc + 160;  // [32] keys equal to T per warp
  {
    uint32_t cg = 0, ce = 0;
    if (!all) {
      for (int i0 = s0; i0 < s1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t key = i < s1 ? key_at(i) : 0u;
        cg += __popc(__ballot_sync(0xffffffffu, i < s1 && key > T));
        ce += __popc(__ballot_sync(0xffffffffu, i < s1 && key == T));
      }
    } else {
      cg = static_cast<uint32_t>(s1 - s0);
    }
    if (lane == 0) {
      wgt[warp] = cg;
      weq[warp] = ce;
    }
  }
  __syncthreads();
  uint32_t eq_before = 0, sel_before = 0;
  for (int v = 0; v < warp; ++v) {
    const uint32_t e = weq[v];
    const uint32_t take = eq_before >= k_rem ? 0u : min(e, k_rem - eq_before);
    sel_before += wgt[v] + take;
    eq_before += e;
  }
  for (int i0 = s0; i0 < s1; i0 += 32) {
    const int i = i0 + lane;
    const bool in = i < s1;
    const uint32_t key = (in && !all) ? key_at(i) : 0u;
    const bool gt = in && (all || key > T);
    const bool eq = in && !all && key == T;
    const unsigned me = __ballot_sync(0xffffffffu, eq);
    const uint32_t eq_rank = eq_before + __popc(me & ((1u << lane) - 1u));
    const bool sel = gt || (eq && eq_rank < k_rem);
    const unsigned ms = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const uint32_t slot = sel_before + __popc(ms & ((1u << lane) - 1u));
      oi[slot] = i * P.index_stride + off;
      if (os) os[slot] = all ? __ldg(src + i) : key_score(key);
    }
    eq_before += __popc(me);
    sel_before += __popc(ms);
  }
  for (int i = cnt + tid; i < k; i += kThreads) {
    oi[i] = -1;
    if (os) os[i] = -__int_as_float(0x7f800000);
  }
  if (tid == 0) P.out_count[q] = cnt;
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& p, cudaStream_t stream) {
  const TopkSmem S = topk_smem();
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
  if (e != cudaSuccess) return e;
  const int grid = p.nshards * p.rows;
  if (grid == 0) return cudaSuccess;
  topk_kernel<<<grid, kThreads, S.total, stream>>>(p, S);
  return cudaGetLastError();
}

}  // namespace dsa
