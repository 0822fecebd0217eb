// Exact top-k of indexer score rows.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Motivation: DSA keeps the top 2048 tokens of the whole sequence; Modifications
// / Indexer decode: every shard first keeps a local top-k of its own tokens.
//
// One cluster of kCluster CTAs (1024 threads each) per score row; CTA c owns
// the c-th contiguous segment of the row:
//   1. its scores become order-preserving uint32 keys (-0 == +0), cached in
//      shared memory when the segment fits; the same pass builds the segment's
//      histogram of the top 13 key bits;
//   2. every CTA sums the cluster's histograms through distributed shared
//      memory and finds the bin holding the k-th largest key; two more
//      histograms (10 and 9 bits) over only the keys still in play refine it
//      to the exact threshold key T and how many keys equal to T are taken
//      (the lowest positions win ties);
//   3. an order-preserving compaction writes the selected positions in
//      ascending order: each CTA learns from the others' counts where its
//      segment's selections start, then every warp owns a contiguous piece of
//      the segment and writes its selected positions at their final slots.
// No sort: the list comes out in position order.
#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_select.cuh"

namespace dsa {
namespace {

constexpr int kThreads = kSelThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 4;  // CTAs per score row
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBins1 = kSelBins1;
constexpr int kShift1 = kSelShift1;

struct TopkSmem {
  int cap;         // keys of the CTA's segment cached in smem
  int off_hist, off_red, off_misc, off_keys, total;
};

__host__ inline TopkSmem topk_smem() {
  TopkSmem s{};
  s.off_hist = 0;                       // this CTA's histogram (read by the cluster)
  s.off_red = s.off_hist + kBins1 * 4;  // the cluster's summed histogram
  s.off_misc = s.off_red + kBins1 * 4;
  s.off_keys = s.off_misc + 1024;
  s.cap = ((kSmemLimit - s.off_keys) / 4) & ~1023;
  s.total = s.off_keys + s.cap * 4;
  return s;
}

// red[b] = sum over the cluster's CTAs of hist[b], b < nb (nb a multiple of
// 4 * kThreads or smaller than it, and of 4)
__device__ __forceinline__ void cluster_sum_hist(const uint32_t* hist, uint32_t* red, int nb) {
  const uint32_t base = smem_u32(hist);
  for (int v = threadIdx.x; v < nb / 4; v += kThreads) {
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < kCluster; ++c) {
      const uint4 x = dsmem_ld_v4(dsmem_map(base + v * 16, c));
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    reinterpret_cast<uint4*>(red)[v] = acc;
  }
  __syncthreads();
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    topk_kernel(const TopkLaunch P, const TopkSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + S.off_red);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);
  uint32_t* scratch = misc;       // 32 words
  uint32_t* sh = misc + 64;       // shared scalars
  uint32_t* cnt = misc + 96;      // [2] this CTA's keys above / equal to T (read by the cluster)
  uint32_t* wgt = misc + 128;     // [32] keys above T per warp
  uint32_t* weq = misc + 160;     // [32] keys equal to T per warp

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t crank = cluster_ctarank();
  const int q = blockIdx.x / kCluster;
  const int w = q / P.rows;
  const int r = q - w * P.rows;
  const int k = P.k;

  // every CTA of the cluster derives the same n, so all take the same branches
  // and pass the same cluster barriers
  int n;
  if (P.valid_len) {
    n = P.valid_len[q];
  } else {
    n = shard_valid_len(P.row_pos[r], P.W, w + P.shard_offset);
  }
  if (n < 0 || n > P.ld) {
    if (tid == 0 && crank == 0) raise_err(P.d_err, DSA_DEVERR_INDEX);
    n = n < 0 ? 0 : static_cast<int>(P.ld);
  }
  const float* src = P.scores + static_cast<long long>(w) * P.shard_stride +
                     static_cast<long long>(r) * P.ld;
  // this CTA's segment [c0, c1) of the row, 32-aligned starts
  const int cseg = (((n + kCluster - 1) / kCluster) + 31) & ~31;
  const int c0 = min(n, static_cast<int>(crank) * cseg);
  const int c1 = min(n, c0 + cseg);
  const int m = c1 - c0;
  const bool in_smem = m <= S.cap;
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int cnt_all = n < k ? n : k;
  const bool need_select = n > k;

  for (int b = tid; b < kBins1; b += kThreads) hist[b] = 0;
  if (tid < 16) sh[tid] = 0;
  __syncthreads();

  // ---------------- pass 1: keys (+ smem copy) and the 13-bit histogram
  bool nan_seen = false;
  {
    const float* seg = src + c0;
    const int nv = vec ? (m >> 2) : 0;
    const float4* src4 = reinterpret_cast<const float4*>(seg);
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
    for (int i = nv * 4 + tid; i < m; i += kThreads) {
      const float f = __ldg(seg + i);
      nan_seen |= (f != f);
      const uint32_t key = score_key(f);
      if (need_select) atomicAdd(hist + (key >> kShift1), 1u);
      if (in_smem) keys[i] = key;
    }
  }
  if (nan_seen) sh[0] = 1;
  __syncthreads();
  if (tid == 0 && sh[0]) raise_err(P.d_err, DSA_DEVERR_NAN);

  // key of row position i of this CTA's segment
  auto key_at = [&](int i) -> uint32_t {
    return in_smem ? keys[i - c0] : score_key(__ldg(src + i));
  };

  uint32_t T = 0, k_rem = 0;
  if (need_select) {
    // ---------------- the exact k-th largest key over the cluster's histograms
    cluster_sync();                       // every CTA's 13-bit histogram is complete
    cluster_sum_hist(hist, red, kBins1);
    find_bin(red, kBins1, static_cast<uint32_t>(k), scratch, sh + 4);
    const uint32_t b1 = sh[4];
    k_rem = sh[5];
    cluster_sync();                       // every CTA has read the histograms
    for (int b = tid; b < kSelBins2; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = c0 + tid; i < c1; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key >> kShift1) == b1) atomicAdd(hist + ((key >> kSelShift2) & (kSelBins2 - 1)), 1u);
    }
    cluster_sync();
    cluster_sum_hist(hist, red, kSelBins2);
    find_bin(red, kSelBins2, k_rem, scratch, sh + 4);
    const uint32_t pre2 = (b1 << (kShift1 - kSelShift2)) | sh[4];
    k_rem = sh[5];
    cluster_sync();
    for (int b = tid; b < kSelBins3; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = c0 + tid; i < c1; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key >> kSelShift2) == pre2) atomicAdd(hist + (key & (kSelBins3 - 1)), 1u);
    }
    cluster_sync();
    cluster_sum_hist(hist, red, kSelBins3);
    find_bin(red, kSelBins3, k_rem, scratch, sh + 4);
    T = (pre2 << kSelShift2) | sh[4];
    k_rem = sh[5];  // keys equal to T that are taken (the lowest positions)
  }

  // ---------------- order-preserving compaction
  const int off = P.index_offset + (P.offset_per_shard ? (w + P.shard_offset) : 0);
  int32_t* oi = P.out_idx + static_cast<long long>(q) * k;
  float* os = P.out_score ? P.out_score + static_cast<long long>(q) * k : nullptr;
  const bool all = !need_select;  // n <= k: every position is selected
  const int wseg = ((m + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(c1, c0 + warp * wseg), s1 = min(c1, s0 + wseg);
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
  if (tid == 0) {
    uint32_t g = 0, e = 0;
    for (int v = 0; v < kWarps; ++v) {
      g += wgt[v];
      e += weq[v];
    }
    cnt[0] = g;
    cnt[1] = e;
  }
  cluster_sync();  // every CTA's counts are visible to the cluster
  // selections and ties of the segments before this one (lower positions)
  uint32_t eq_before = 0, sel_before = 0;
  for (uint32_t c = 0; c < crank; ++c) {
    const uint32_t g = dsmem_ld(dsmem_map(smem_u32(cnt), c));
    const uint32_t e = dsmem_ld(dsmem_map(smem_u32(cnt + 1), c));
    const uint32_t take = eq_before >= k_rem ? 0u : min(e, k_rem - eq_before);
    sel_before += g + take;
    eq_before += e;
  }
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
  if (crank == 0) {
    for (int i = cnt_all + tid; i < k; i += kThreads) {
      oi[i] = -1;
      if (os) os[i] = -__int_as_float(0x7f800000);
    }
    if (tid == 0) P.out_count[q] = cnt_all;
  }
  cluster_sync();  // no CTA leaves while another may still read its counts
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& p, cudaStream_t stream) {
  const TopkSmem S = topk_smem();
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
  if (e != cudaSuccess) return e;
  const int rows = p.nshards * p.rows;
  if (rows == 0) return cudaSuccess;
  topk_kernel<<<rows * kCluster, kThreads, S.total, stream>>>(p, S);
  return cudaGetLastError();
}

}  // namespace dsa
