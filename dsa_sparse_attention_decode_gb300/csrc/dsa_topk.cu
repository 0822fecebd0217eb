// Exact top-k of indexer score rows.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Motivation: DSA keeps the top 2048 tokens of the whole sequence; Modifications
// / Indexer decode: every shard first keeps a local top-k of its own tokens.
//
// A cluster of C CTAs (1024 threads each; C = 4, 2 or 1, the most that keeps
// every row's cluster resident at once) per score row; CTA c owns the c-th
// contiguous segment of the row:
//   1. the segment's scores become order-preserving uint32 keys (-0 == +0),
//      cached in shared memory as far as they fit; the row's smallest and
//      largest keys bound the bits in which keys differ;
//   2. one histogram of the top 11 of those bits (summed over the cluster
//      through distributed shared memory) gives the bin b1 holding the k-th
//      largest key.  Keys above b1 are selected for sure; one classifying pass
//      counts them per warp and lists the few keys inside b1 (the candidates,
//      with their positions) in shared memory;
//   3. every CTA reads the cluster's candidates and resolves the remaining
//      bits on them alone: the exact threshold key T and how many keys equal
//      to T are taken (the lowest positions win ties).  A degenerate row whose
//      b1 holds too many keys instead resolves them with more histogram
//      rounds over the whole row;
//   4. an order-preserving compaction writes the selected positions in
//      ascending order: from the per-warp counts every warp knows its first
//      output slot, and writes 128 keys' selections per step (4 per lane,
//      warp scans for the slots).
// No sort: the list comes out in position order.  This cluster form serves
// launches of few rows (at most half the SM count: every row then gets a
// cluster of 2 or 4 CTAs at once) and score rows too long for the position
// bitmaps of the segment form below.
#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "dsa_select.cuh"

namespace dsa {
namespace {

constexpr int kThreads = kSelThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kRoundBits = 11;          // key bits resolved per histogram round
constexpr int kBins = 1 << kRoundBits;
constexpr int kCand = 4096;             // candidates of a row (cluster-wide)
constexpr int kSmemLimit = 227 * 1024;

// misc words
constexpr int kSh = 32;        // [32] shared scalars
constexpr int kWgt = 64;       // [32] per warp: keys above T
constexpr int kWeq = 96;       // [32] per warp: keys equal to T
constexpr int kWdef = 128;     // [32] per warp: keys above the bin b1
constexpr int kPub = 160;      // [16] read by the cluster: min, max, candidates, keys above b1
constexpr int kTmp = 192;      // [64] reductions
constexpr int kCtaCnt = 256;   // [8] per CTA of the cluster: keys above T, keys equal to T
constexpr int kWtot = 320;     // [32] per warp: the bin search's suffix sums
constexpr int kMiscWords = 512;

struct TopkSmem {
  int cap;         // keys of the CTA's segment cached in smem
  int off_hist, off_misc, off_cand, off_all, off_keys, total;
};

__host__ inline TopkSmem topk_smem(int C) {
  TopkSmem s{};
  s.off_hist = 0;                                  // this CTA's histogram (read by the cluster)
  s.off_misc = s.off_hist + kBins * 4;
  s.off_cand = s.off_misc + kMiscWords * 4;        // this CTA's candidates (key, position)
  s.off_all = s.off_cand + kCand * 8;              // the cluster's candidates
  s.off_keys = s.off_all + (C > 1 ? kCand * 8 : 0);
  s.cap = ((kSmemLimit - s.off_keys) / 4) & ~127;
  s.total = s.off_keys + s.cap * 4;
  return s;
}

// inclusive prefix sum over the lanes of a warp
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// sum of v over the lanes at and above this one
__device__ __forceinline__ uint32_t warp_suffix_incl(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v += t;
  }
  return v;
}

// One warp: the bin of hist[0, nb) (nb a power of two up to 2048; a higher
// bin holds larger keys) that holds the k_rem-th largest key.  Lane 0 writes
// (bin, k_rem within the bin, the bin's count) to out[0..2].  Two levels:
// every lane sums a contiguous run of nb / 32 bins, a suffix scan finds the
// run, and the run's bins are spread over the lanes for a second scan.
__device__ void warp_find_bin(const uint32_t* hist, int nb, uint32_t k_rem, uint32_t* out,
                              int lane) {
  const int per = nb >= 32 ? nb / 32 : 1;
  const int base = lane * per;
  uint32_t mine = 0;
  if (base < nb) {
    if (per >= 4) {
      for (int j = 0; j < per; j += 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(hist + base + j);
        mine += x.x + x.y + x.z + x.w;
      }
    } else {
      for (int j = 0; j < per; ++j) mine += hist[base + j];
    }
  }
  const uint32_t incl = warp_suffix_incl(mine, lane);
  const uint32_t above = incl - mine;
  const unsigned hit = __ballot_sync(0xffffffffu, base < nb && above < k_rem && incl >= k_rem);
  const int fl = hit ? __ffs(hit) - 1 : 0;
  const uint32_t abv = __shfl_sync(0xffffffffu, above, fl);
  // the found run, per2 bins per lane
  const int per2 = per >= 32 ? per / 32 : 1;
  const int b0 = fl * per + lane * per2;
  const bool in2 = lane * per2 < per;
  uint32_t m2 = 0;
  if (in2)
    for (int j = 0; j < per2; ++j) m2 += hist[b0 + j];
  const uint32_t incl2 = warp_suffix_incl(m2, lane) + abv;
  const uint32_t above2 = incl2 - m2;
  const unsigned hit2 = __ballot_sync(0xffffffffu, in2 && above2 < k_rem && incl2 >= k_rem);
  const int fl2 = hit2 ? __ffs(hit2) - 1 : 0;
  if (lane == fl2) {
    uint32_t acc = above2;
    for (int j = per2 - 1; j >= 0; --j) {
      const uint32_t h = hist[b0 + j];
      if (acc + h >= k_rem || j == 0) {
        out[0] = static_cast<uint32_t>(b0 + j);
        out[1] = k_rem - acc;
        out[2] = h;
        break;
      }
      acc += h;
    }
  }
  __syncwarp();
}

__device__ __forceinline__ uint2 dsmem_ld_v2(uint32_t caddr) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(caddr)
               : "memory");
  return v;
}

// Every thread of the CTA: the bin of the cluster's histogram (the sum over
// the cluster's CTAs of hist[0, nb), nb a power of two up to kBins; a higher
// bin holds larger keys) that holds the k_rem-th largest key.  For C > 1 the
// caller has passed a cluster barrier after every CTA's histogram, and no CTA
// writes its histogram again before the next one.  Thread t sums its own
// nb / kThreads bins (at least one; threads past nb hold none) over the
// cluster, a suffix sum over the threads (per warp, then over the 32 warp
// totals in wtot) gives the keys above them, and the one thread whose bins
// hold the k_rem-th key writes (bin, k_rem within the bin, the bin's count)
// to out[0..2].  The caller's __syncthreads publishes them.
template <int C>
__device__ __forceinline__ void cta_find_bin(const uint32_t* hist, int nb, uint32_t k_rem,
                                             uint32_t* out, uint32_t* wtot, int tid) {
  static_assert(kWarps == 32 && kThreads * 2 >= kBins, "one warp total per lane, two bins per thread");
  const int lane = tid & 31, warp = tid >> 5;
  const bool two = nb > kThreads;  // two bins per thread
  const int b0 = two ? 2 * tid : tid;
  uint32_t h0 = 0, h1 = 0;
  if (b0 < nb) {
    if constexpr (C > 1) {
      const uint32_t a = smem_u32(hist + b0);
#pragma unroll
      for (int c = 0; c < C; ++c) {
        if (two) {
          const uint2 x = dsmem_ld_v2(dsmem_map(a, c));
          h0 += x.x;
          h1 += x.y;
        } else {
          h0 += dsmem_ld(dsmem_map(a, c));
        }
      }
    } else if (two) {
      const uint2 x = *reinterpret_cast<const uint2*>(hist + b0);
      h0 = x.x;
      h1 = x.y;
    } else {
      h0 = hist[b0];
    }
  }
  const uint32_t mine = h0 + h1;
  const uint32_t incl = warp_suffix_incl(mine, lane);
  if (lane == 0) wtot[warp] = incl;
  __syncthreads();
  const uint32_t wt = wtot[lane];
  const uint32_t wincl = warp_suffix_incl(wt, lane);
  const uint32_t total = __shfl_sync(0xffffffffu, wincl, 0);
  const uint32_t above = __shfl_sync(0xffffffffu, wincl - wt, warp) + (incl - mine);
  // thread 0 answers (with its lowest bin) if the histogram holds fewer keys
  if ((above < k_rem && above + mine >= k_rem) || (tid == 0 && total < k_rem)) {
    if (two && above + h1 >= k_rem) {
      out[0] = static_cast<uint32_t>(b0 + 1);
      out[1] = k_rem - above;
      out[2] = h1;
    } else {
      out[0] = static_cast<uint32_t>(b0);
      out[1] = k_rem - (above + h1);
      out[2] = h0;
    }
  }
}

template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(kThreads, 1)
    topk_kernel(const TopkLaunch P, const TopkSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint2* cand = reinterpret_cast<uint2*>(smem + S.off_cand);
  uint2* cand_all = C > 1 ? reinterpret_cast<uint2*>(smem + S.off_all) : cand;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + S.off_keys);
  uint32_t* sh = misc + kSh;
  uint32_t* wgt = misc + kWgt;
  uint32_t* weq = misc + kWeq;
  uint32_t* wdef = misc + kWdef;
  uint32_t* pub = misc + kPub;
  uint32_t* wtot = misc + kWtot;
  uint32_t* tmp = misc + kTmp;
  uint32_t* ctacnt = misc + kCtaCnt;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;  // the lanes below this one
  const uint32_t crank = C > 1 ? cluster_ctarank() : 0u;
  const int q = blockIdx.x / C;
  const int w = q / P.rows;
  const int r = q - w * P.rows;
  const int k = P.k;
  pdl_trigger();
  pdl_wait();  // the scores come from the previous grid

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
  // this CTA's segment [c0, c0 + m) of the row, 32-aligned starts
  const int cseg = C > 1 ? ((((n + C - 1) / C) + 31) & ~31) : n;
  const int c0 = min(n, static_cast<int>(crank) * cseg);
  const int m = min(n, c0 + cseg) - c0;
  const float* seg = src + c0;
  const bool vec = (reinterpret_cast<uintptr_t>(seg) & 15u) == 0;
  const int cached = min(m, S.cap);  // segment keys [0, cached) live in smem
  const int cnt_all = n < k ? n : k;
  const bool need_select = n > k;

  for (int i = tid; i < kMiscWords; i += kThreads) misc[i] = 0;
  __syncthreads();

  // ---------------- pass 1: keys (+ smem copy), smallest and largest key
  bool nan_seen = false;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  {
    const int nv = vec ? (m >> 2) : 0;
    const float4* src4 = reinterpret_cast<const float4*>(seg);
    for (int base = 0; base < nv; base += kThreads * 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = base + u * kThreads + tid;
        v[u] = i < nv ? __ldcg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
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
            kmin = min(kmin, kp[e]);
            kmax = max(kmax, kp[e]);
          }
          // cached is m or a multiple of 128: a vector lies wholly on one side
          if (4 * i < cached) reinterpret_cast<uint4*>(keys)[i] = kk;
        }
      }
    }
    for (int i = nv * 4 + tid; i < m; i += kThreads) {
      const float f = __ldcg(seg + i);
      nan_seen |= (f != f);
      const uint32_t key = score_key(f);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
      if (i < cached) keys[i] = key;
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  const bool nan_warp = __any_sync(0xffffffffu, nan_seen);
  if (lane == 0) {
    tmp[warp] = kmin;
    tmp[32 + warp] = kmax;
    if (nan_warp) sh[2] = 1;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = __reduce_min_sync(0xffffffffu, tmp[lane]);
    const uint32_t b = __reduce_max_sync(0xffffffffu, tmp[32 + lane]);
    if (lane == 0) {
      pub[0] = a;
      pub[1] = b;
    }
  }
  __syncthreads();
  if constexpr (C > 1) {
    cluster_sync();  // every CTA's min and max are visible to the cluster
    if (warp == 0) {
      uint32_t a = 0xFFFFFFFFu, b = 0u;
      if (lane < C) {
        a = dsmem_ld(dsmem_map(smem_u32(pub), lane));
        b = dsmem_ld(dsmem_map(smem_u32(pub + 1), lane));
      }
      a = __reduce_min_sync(0xffffffffu, a);
      b = __reduce_max_sync(0xffffffffu, b);
      if (lane == 0) {
        sh[0] = a;
        sh[1] = b;
      }
    }
  } else {
    if (tid == 0) {
      sh[0] = pub[0];
      sh[1] = pub[1];
    }
  }
  __syncthreads();
  kmin = sh[0];
  kmax = sh[1];
  if (tid == 0 && sh[2]) raise_err(P.d_err, DSA_DEVERR_NAN);

  // key of segment position j
  auto key_at = [&](int j) -> uint32_t {
    return j < cached ? keys[j] : score_key(__ldcg(seg + j));
  };
  // the keys of segment positions j0 .. j0 + 3 below lim (j0 a multiple of 4)
  auto load4 = [&](int j0, int lim, uint32_t* kv, bool* ok) {
    if (j0 + 3 < lim && j0 + 3 < cached) {
      const uint4 x = *reinterpret_cast<const uint4*>(keys + j0);
      kv[0] = x.x;
      kv[1] = x.y;
      kv[2] = x.z;
      kv[3] = x.w;
      ok[0] = ok[1] = ok[2] = ok[3] = true;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ok[e] = j0 + e < lim;
        kv[e] = ok[e] ? key_at(j0 + e) : 0u;
      }
    }
  };

  // warp pieces of the segment (segment positions), 32-aligned
  const int wseg = ((m + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(m, warp * wseg), s1 = min(m, s0 + wseg);

  // mode 0: n <= k, every position; 1: threshold from the candidates;
  // 2: threshold from rounds over the whole row (or a single key value)
  int mode = 0;
  uint32_t T = 0, k_rem = 0;
  uint64_t pre = 0;  // the threshold's bits above bit lo - 1
  int lo = 0;
  const uint32_t diff = kmin ^ kmax;
  if (need_select) {
    if (diff == 0) {
      mode = 2;
      T = kmax;  // one key value: the first k positions
      k_rem = static_cast<uint32_t>(k);
    } else {
      const int top = 31 - __clz(diff);  // highest bit in which keys differ
      const int nbits = min(kRoundBits, top + 1);
      lo = top + 1 - nbits;
      const int nb = 1 << nbits;
      for (int b = tid; b < nb; b += kThreads) hist[b] = 0;
      __syncthreads();
      const uint32_t bmask = static_cast<uint32_t>(nb - 1);
      for (int j4 = tid; j4 < (cached >> 2); j4 += kThreads) {
        const uint4 x = reinterpret_cast<const uint4*>(keys)[j4];
        atomicAdd(hist + ((x.x >> lo) & bmask), 1u);
        atomicAdd(hist + ((x.y >> lo) & bmask), 1u);
        atomicAdd(hist + ((x.z >> lo) & bmask), 1u);
        atomicAdd(hist + ((x.w >> lo) & bmask), 1u);
      }
      for (int j = (cached & ~3) + tid; j < m; j += kThreads)
        atomicAdd(hist + ((key_at(j) >> lo) & bmask), 1u);
      __syncthreads();
      if constexpr (C > 1) cluster_sync();  // every CTA's histogram is complete
      cta_find_bin<C>(hist, nb, static_cast<uint32_t>(k), sh + 4, wtot, tid);
      __syncthreads();
      pre = ((static_cast<uint64_t>(kmax) >> (top + 1)) << nbits) | sh[4];
      k_rem = sh[5];
      mode = sh[6] <= static_cast<uint32_t>(kCand) ? 1 : 2;
    }
  }

  if (mode == 1) {
    // ---------------- classify: keys above b1 per warp, candidates listed
    uint32_t ndef = 0;
    for (int s = s0; s < s1; s += 128) {
      const int j0 = s + 4 * lane;
      uint32_t kv[4];
      bool ok[4];
      load4(j0, s1, kv, ok);
      uint32_t c_lo = 0, tot = 0;  // candidates in lower lanes / in the warp
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint64_t hi = kv[e] >> lo;
        ndef += (ok[e] && hi > pre) ? 1u : 0u;
        const uint32_t b = __ballot_sync(0xffffffffu, ok[e] && hi == pre);
        c_lo += __popc(b & lt_mask);
        tot += __popc(b);
      }
      if (tot != 0) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(sh + 8, tot);
        base = __shfl_sync(0xffffffffu, base, 0);
        uint32_t slot = base + c_lo;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (ok[e] && (static_cast<uint64_t>(kv[e] >> lo) == pre)) {
            cand[slot] = make_uint2(kv[e], static_cast<uint32_t>(c0 + j0 + e));
            ++slot;
          }
        }
      }
    }
    ndef = __reduce_add_sync(0xffffffffu, ndef);
    if (lane == 0) wdef[warp] = ndef;
    __syncthreads();
    const uint32_t nloc = sh[8];
    uint32_t total = nloc;
    if constexpr (C > 1) {
      if (warp == 0) {
        const uint32_t d = __reduce_add_sync(0xffffffffu, wdef[lane]);
        if (lane == 0) {
          pub[2] = nloc;
          pub[3] = d;
        }
      }
      __syncthreads();
      // every CTA's candidates and counts are visible, and every CTA is done
      // reading the others' histograms
      cluster_sync();
      if (warp == 0) {
        uint32_t nc = 0, d = 0;
        if (lane < C) {
          nc = dsmem_ld(dsmem_map(smem_u32(pub + 2), lane));
          d = dsmem_ld(dsmem_map(smem_u32(pub + 3), lane));
        }
        const uint32_t incl = warp_incl_scan(nc, lane);
        if (lane < C) {
          tmp[lane] = incl - nc;
          tmp[8 + lane] = nc;
          tmp[16 + lane] = d;
        }
        if (lane == 31) sh[9] = incl;
      }
      __syncthreads();
      total = sh[9];
      for (int c = 0; c < C; ++c) {
        const uint32_t nc = tmp[8 + c], o = tmp[c];
        for (uint32_t e = tid; e < nc; e += kThreads) {
          const uint32_t ca = dsmem_map(smem_u32(cand + e), c);
          cand_all[o + e] = make_uint2(dsmem_ld(ca), dsmem_ld(ca + 4));
        }
      }
      __syncthreads();
    }
    // ---------------- the remaining bits of T, from the candidates alone
    if (total <= static_cast<uint32_t>(kThreads)) {
      // rank every candidate among them: T is the key with fewer than k_rem
      // candidates above it and at least k_rem at or above it
      if (static_cast<uint32_t>(tid) < total) {
        const uint32_t key = cand_all[tid].x;
        uint32_t gt = 0, eq = 0;
#pragma unroll 4
        for (uint32_t j = 0; j < total; ++j) {
          const uint32_t kj = cand_all[j].x;
          gt += kj > key ? 1u : 0u;
          eq += kj == key ? 1u : 0u;
        }
        if (gt < k_rem && k_rem <= gt + eq) {
          sh[12] = key;  // every writer writes the same two words
          sh[13] = k_rem - gt;
        }
      }
    } else if (warp == 0) {
      // histogram rounds (warp 0; the histogram is free: every CTA is past
      // its cluster sum)
      int t = lo - 1;
      while (t >= 0) {
        const int nbits = min(kRoundBits, t + 1);
        const int lo2 = t + 1 - nbits;
        const int nb = 1 << nbits;
        for (int b = lane; b < nb; b += 32) hist[b] = 0;
        __syncwarp();
        for (uint32_t e = lane; e < total; e += 32) {
          const uint32_t key = cand_all[e].x;
          if (static_cast<uint64_t>(key >> (t + 1)) == pre)
            atomicAdd(hist + ((key >> lo2) & static_cast<uint32_t>(nb - 1)), 1u);
        }
        __syncwarp();
        warp_find_bin(hist, nb, k_rem, sh + 4, lane);
        pre = (pre << nbits) | sh[4];
        k_rem = sh[5];
        __syncwarp();
        t = lo2 - 1;
      }
      if (lane == 0) {
        sh[12] = static_cast<uint32_t>(pre);
        sh[13] = k_rem;
      }
    }
    __syncthreads();
    T = sh[12];
    k_rem = sh[13];
    // candidates above / equal to T, per warp of this CTA and per CTA
    for (uint32_t e = tid; e < nloc; e += kThreads) {
      const uint2 c = cand[e];
      const int wj = (static_cast<int>(c.y) - c0) / wseg;
      if (c.x > T) atomicAdd(wgt + wj, 1u);
      else if (c.x == T) atomicAdd(weq + wj, 1u);
    }
    if constexpr (C > 1) {
      for (uint32_t e = tid; e < total; e += kThreads) {
        const uint2 c = cand_all[e];
        const int cc = static_cast<int>(c.y) / cseg;
        if (c.x > T) atomicAdd(ctacnt + 2 * cc, 1u);
        else if (c.x == T) atomicAdd(ctacnt + 2 * cc + 1, 1u);
      }
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t g = 0, eqb = 0;
      if constexpr (C > 1) {
        for (uint32_t c = 0; c < crank; ++c) {
          g += tmp[16 + c] + ctacnt[2 * c];
          eqb += ctacnt[2 * c + 1];
        }
      }
      sh[10] = g;
      sh[11] = eqb;
    }
  } else if (mode == 2) {
    // ---------------- degenerate rows: rounds over the whole row
    while (diff != 0 && lo > 0) {
      if constexpr (C > 1) cluster_sync();  // every CTA is done reading the histograms
      const int t = lo - 1;
      const int nbits = min(kRoundBits, t + 1);
      const int lo2 = t + 1 - nbits;
      const int nb = 1 << nbits;
      for (int b = tid; b < nb; b += kThreads) hist[b] = 0;
      __syncthreads();
      for (int j = tid; j < m; j += kThreads) {
        const uint32_t key = key_at(j);
        if (static_cast<uint64_t>(key >> (t + 1)) == pre)
          atomicAdd(hist + ((key >> lo2) & static_cast<uint32_t>(nb - 1)), 1u);
      }
      __syncthreads();
      if constexpr (C > 1) cluster_sync();
      cta_find_bin<C>(hist, nb, k_rem, sh + 4, wtot, tid);
      __syncthreads();
      pre = (pre << nbits) | sh[4];
      k_rem = sh[5];
      lo = lo2;
      __syncthreads();  // sh is read before the next round writes it
    }
    if (diff != 0) T = static_cast<uint32_t>(pre);
    // keys above / equal to T per warp
    uint32_t cg = 0, ce = 0;
    for (int s = s0; s < s1; s += 128) {
      uint32_t kv[4];
      bool ok[4];
      load4(s + 4 * lane, s1, kv, ok);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        cg += (ok[e] && kv[e] > T) ? 1u : 0u;
        ce += (ok[e] && kv[e] == T) ? 1u : 0u;
      }
    }
    cg = __reduce_add_sync(0xffffffffu, cg);
    ce = __reduce_add_sync(0xffffffffu, ce);
    if (lane == 0) {
      wgt[warp] = cg;
      weq[warp] = ce;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t g = 0, e = 0;
      for (int v = 0; v < kWarps; ++v) {
        g += wgt[v];
        e += weq[v];
      }
      pub[4] = g;
      pub[5] = e;
    }
    __syncthreads();
    if constexpr (C > 1) cluster_sync();  // every CTA's counts are visible
    if (warp == 0) {
      uint32_t g = 0, e = 0;
      if constexpr (C > 1) {
        if (static_cast<uint32_t>(lane) < crank) {
          g = dsmem_ld(dsmem_map(smem_u32(pub + 4), lane));
          e = dsmem_ld(dsmem_map(smem_u32(pub + 5), lane));
        }
      }
      g = __reduce_add_sync(0xffffffffu, g);
      e = __reduce_add_sync(0xffffffffu, e);
      if (lane == 0) {
        sh[10] = g;
        sh[11] = e;
      }
    }
  } else {
    if (tid == 0) {
      sh[10] = static_cast<uint32_t>(c0);  // every position before the segment
      sh[11] = 0;
    }
  }
  __syncthreads();
  // sh[10], sh[11]: keys above T and keys equal to T in the CTAs before this
  // one.  Ties are taken in position order, so the ties taken before any
  // point are min(ties before it, k_rem).

  // ---------------- order-preserving compaction
  const int off = P.index_offset + (P.offset_per_shard ? (w + P.shard_offset) : 0);
  int32_t* oi = P.out_idx + static_cast<long long>(q) * k;
  float* os = P.out_score ? P.out_score + static_cast<long long>(q) * k : nullptr;
  const bool all = mode == 0;
  uint32_t sel_before, eq_before;
  {
    const int v0 = min(m, lane * wseg);
    const uint32_t g = all ? static_cast<uint32_t>(min(m, v0 + wseg) - v0) : wdef[lane] + wgt[lane];
    const uint32_t e = weq[lane];
    const uint32_t gi = warp_incl_scan(g, lane), ei = warp_incl_scan(e, lane);
    // this warp's exclusive prefix over the warps before it
    const uint32_t gx = __shfl_sync(0xffffffffu, gi - g, warp);
    const uint32_t ex = __shfl_sync(0xffffffffu, ei - e, warp);
    eq_before = sh[11] + ex;
    sel_before = sh[10] + gx + min(eq_before, k_rem);
  }
  for (int s = s0; s < s1; s += 128) {
    const int j0 = s + 4 * lane;
    uint32_t kv[4];
    bool ok[4];
    if (all) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ok[e] = j0 + e < s1;
        kv[e] = 0u;
      }
    } else {
      load4(j0, s1, kv, ok);
    }
    // position order is lane-major (lane l holds positions j0 .. j0 + 3), so
    // the ties and selections before this lane's first are the lower lanes'
    // bits of one ballot per e
    bool eqf[4];
    uint32_t eq_lo = 0, eq_all = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      eqf[e] = ok[e] && !all && kv[e] == T;
      const uint32_t b = __ballot_sync(0xffffffffu, eqf[e]);
      eq_lo += __popc(b & lt_mask);
      eq_all += __popc(b);
    }
    uint32_t er = eq_before + eq_lo;  // rank of this lane's first tie
    bool self[4];
    uint32_t sel_lo = 0, sel_all = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (eqf[e]) {
        self[e] = er < k_rem;
        ++er;
      } else {
        self[e] = ok[e] && (all || kv[e] > T);
      }
      const uint32_t b = __ballot_sync(0xffffffffu, self[e]);
      sel_lo += __popc(b & lt_mask);
      sel_all += __popc(b);
    }
    uint32_t slot = sel_before + sel_lo;  // selections before this lane's first
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (self[e]) {
        const int pos = c0 + j0 + e;
        oi[slot] = pos * P.index_stride + off;
        if (os) os[slot] = all ? __ldcg(seg + j0 + e) : key_score(kv[e]);
        ++slot;
      }
    }
    eq_before += eq_all;
    sel_before += sel_all;
  }
  if (crank == 0) {
    for (int i = cnt_all + tid; i < k; i += kThreads) {
      oi[i] = -1;
      if (os) os[i] = -__int_as_float(0x7f800000);
    }
    if (tid == 0) P.out_count[q] = cnt_all;
  }
  if constexpr (C > 1) cluster_sync();  // no CTA leaves while another may still read its smem
}

// ======================================================================
// Segment-parallel selection with position bitmaps.
//
// Three kernels, so that every SM takes part in the passes over the scores
// whatever the number and the lengths of the rows:
//   K1 (one CTA per 16K-position segment of a row): a 1024-bin histogram of
//      the segment's keys over a key window drawn from a sample of the row
//      (keys below it count in bin 0, keys above it in the last bin), added
//      to the row's histogram in the workspace;
//   K2 (the same segments): the row's histogram gives the key range (bin)
//      holding the k-th largest key; the segment's keys above the range are
//      written as bits of the row's position bitmap (32 positions per word),
//      and the keys inside it are listed as candidates (key, position);
//   K3 (one 512-thread CTA per row): the threshold key T comes from 10-bit
//      histogram rounds over the candidates alone; candidates above T join
//      the bitmap and those equal to T go to a bitmap of ties; compaction
//      walks the bitmap words in position order, takes ties lowest positions
//      first (as many as the selection still needs), and prefix sums over
//      the threads give every selected position its output slot.  The list
//      comes out in ascending position order without a sort.
// A row whose threshold bin holds more keys than the candidate list takes
// (only rows with massive ties or a degenerate spread) is resolved by K3
// alone with further 4096-bin rounds over the row.  Without a workspace K3
// runs alone and makes its own histogram and bitmap pass.
// A window that follows the row's own spread keeps neighbouring keys in
// different bins: fixed top key bits would put a row of scores within one
// octave into a few bins, whose shared-memory atomics serialize.
constexpr int kRThreads = 512;      // K3
constexpr int kSThreads = 256;      // K1, K2
constexpr int kWBits = 10;          // first histogram: 1024 bins over the sampled window
constexpr int kWBins = 1 << kWBits;
constexpr int kRBits = 12;          // further rounds over a row: 4096 bins
constexpr int kRCand = 4096;        // candidate list capacity
constexpr int kCBits = 10;          // rounds over the candidates
constexpr int kSample = 512;        // sampled positions of a row
constexpr int kRMisc = 256;         // words: [0, 32) scalars, [32, 128) scratch
constexpr int kU = 6;               // quads in flight per thread and step

struct RowsSmem {
  int nw;  // bitmap words (covers ld positions, a multiple of 4)
  int off_hist, off_cand, off_eq, off_gt, off_chist, off_misc, total;
};

__host__ inline RowsSmem rows_smem(int64_t ld) {
  RowsSmem s{};
  s.nw = static_cast<int>(((ld + 31) / 32 + 3) / 4 * 4);
  const int a_hist = (1 << kRBits) * 4;
  const int a_cand = kRCand * 8 + s.nw * 4;  // the candidates and the tie bitmap
  // the histogram is dead before the candidate list and the tie bitmap are written
  const int a = a_hist > a_cand ? a_hist : a_cand;
  s.off_hist = 0;
  s.off_cand = 0;
  s.off_eq = kRCand * 8;
  s.off_gt = a;
  s.off_chist = s.off_gt + s.nw * 4;
  s.off_misc = s.off_chist + (1 << kCBits) * 4;
  s.total = s.off_misc + kRMisc * 4;
  return s;
}

// Exclusive prefix sum of v over the CTA's NT threads; *total gets the sum.
// Uses scratch[0, NT / 32); every thread calls it.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch,
                                                    uint32_t* total) {
  constexpr int kW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v, lane);
  __syncthreads();  // scratch is free (an earlier call may still be reading it)
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  const uint32_t wt = lane < kW ? scratch[lane] : 0u;
  const uint32_t winc = warp_incl_scan(wt, lane);
  const uint32_t wex = __shfl_sync(0xffffffffu, winc - wt, warp);
  *total = __shfl_sync(0xffffffffu, winc, kW - 1);
  return wex + incl - v;
}

// The bin of hist[0, nb) (nb a power of two, 2 .. 4096; a higher bin holds
// larger keys) that holds the k_rem-th largest key: (bin, k_rem within the
// bin, the bin's count) to out[0..2].  Every thread calls it; the caller's
// __syncthreads publishes the answer.
template <int NT>
__device__ void block_find_bin(const uint32_t* hist, int nb, uint32_t k_rem, uint32_t* out,
                               uint32_t* scratch) {
  const int tid = threadIdx.x;
  const int per = nb >= NT ? nb / NT : 1;
  const int b0 = tid * per;
  uint32_t mine = 0;
  if (b0 < nb) {
    if (per >= 4) {
      for (int j = 0; j < per; j += 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(hist + b0 + j);
        mine += x.x + x.y + x.z + x.w;
      }
    } else {
      for (int j = 0; j < per; ++j) mine += hist[b0 + j];
    }
  }
  // keys in the bins of the threads above this one = total - inclusive prefix
  uint32_t total;
  const uint32_t ex = block_excl_scan<NT>(mine, scratch, &total);
  const uint32_t above = total - ex - mine;
  if (b0 < nb && above < k_rem && above + mine >= k_rem) {
    uint32_t acc = above;
    for (int j = per - 1; j >= 0; --j) {
      const uint32_t h = hist[b0 + j];
      if (acc + h >= k_rem) {
        out[0] = static_cast<uint32_t>(b0 + j);
        out[1] = k_rem - acc;
        out[2] = h;
        break;
      }
      acc += h;
    }
  }
}

// A score row: its valid count and where it lives.
struct RowRef {
  const float* src;
  int n;
  int nq;    // quads of positions, (n + 3) / 4
  bool vec;  // float4 loads: 16-byte aligned row start and stride a multiple of 4
};

__device__ __forceinline__ RowRef row_ref(const TopkLaunch& P, int q) {
  const int w = q / P.rows;
  const int r = q - w * P.rows;
  RowRef R;
  int n = P.valid_len ? P.valid_len[q] : shard_valid_len(P.row_pos[r], P.W, w + P.shard_offset);
  n = n < 0 ? 0 : (n > P.ld ? static_cast<int>(P.ld) : n);
  R.n = n;
  R.nq = (n + 3) >> 2;
  R.src = P.scores + static_cast<long long>(w) * P.shard_stride + static_cast<long long>(r) * P.ld;
  R.vec = (reinterpret_cast<uintptr_t>(R.src) & 15u) == 0 && (P.ld & 3) == 0;
  return R;
}

// The keys of quad qd (positions 4qd .. 4qd + 3); returns the valid mask.
// With float4 loads every quad with 4qd < n lies inside the row's storage.
__device__ __forceinline__ uint32_t load_quad(const RowRef& R, int qd, uint32_t* kv) {
  if (qd >= R.nq) return 0u;
  const int p = qd * 4;
  float f[4];
  if (R.vec) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(R.src + p));
    f[0] = x.x;
    f[1] = x.y;
    f[2] = x.z;
    f[3] = x.w;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = p + e < R.n ? __ldcg(R.src + p + e) : 0.0f;
  }
  uint32_t ok = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    kv[e] = score_key(f[e]);
    ok |= (p + e < R.n ? 1u : 0u) << e;
  }
  return ok;
}

// The row's key window: the smallest and the largest key of kSample evenly
// spread positions (the same positions in every kernel) -> win[0], win[1].
// Every thread calls it (n >= 1).
template <int NT>
__device__ void sample_window(const RowRef& R, uint32_t* scratch, uint32_t* win) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int i = threadIdx.x; i < kSample; i += NT) {
    const int p = static_cast<int>((static_cast<long long>(i) * R.n) / kSample);
    const uint32_t key = score_key(__ldcg(R.src + p));
    mn = min(mn, key);
    mx = max(mx, key);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  __syncthreads();  // scratch is free
  if (lane == 0) {
    scratch[warp] = mn;
    scratch[32 + warp] = mx;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = __reduce_min_sync(0xffffffffu, lane < NT / 32 ? scratch[lane] : 0xFFFFFFFFu);
    const uint32_t b = __reduce_max_sync(0xffffffffu, lane < NT / 32 ? scratch[32 + lane] : 0u);
    if (lane == 0) {
      win[0] = a;
      win[1] = b;
    }
  }
  __syncthreads();
}

// bin of a key in the first histogram (window [wlo, ...] split 2^wshift wide)
__device__ __forceinline__ uint32_t window_bin(uint32_t key, uint32_t wlo, int wshift) {
  return key < wlo ? 0u : min(static_cast<uint32_t>(kWBins - 1), (key - wlo) >> wshift);
}
// the keys of first-histogram bin b (bin 0 reaches down to 0, the last bin up to ~0)
__device__ __forceinline__ void window_range(uint32_t wlo, int wshift, uint32_t b, uint32_t* rlo,
                                             uint32_t* rhi) {
  bin_range(wlo, 0xFFFFFFFFu, wshift, b, rlo, rhi);
  if (b == 0u) *rlo = 0u;
  if (b == static_cast<uint32_t>(kWBins - 1)) *rhi = 0xFFFFFFFFu;
}

// One step of the first histogram: this thread's kU quads (loaded by
// hist_load); returns whether a NaN was seen.
template <int NT>
__device__ __forceinline__ void hist_load(const RowRef& R, int base, int q1, uint32_t (*kv)[4],
                                          uint32_t* ok) {
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int qd = base + u * NT + static_cast<int>(threadIdx.x);
    ok[u] = qd < q1 ? load_quad(R, qd, kv[u]) : 0u;
  }
}
__device__ __forceinline__ bool hist_step(const uint32_t (*kv)[4], const uint32_t* ok,
                                          uint32_t wlo, int wshift, uint32_t* hist) {
  bool nan_seen = false;
#pragma unroll
  for (int u = 0; u < kU; ++u)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((ok[u] >> e) & 1u) {
        const uint32_t key = kv[u][e];
        // NaN keys: above 0xFF800000 (+inf) or below 0x007FFFFF (-inf)
        nan_seen |= key > 0xFF800000u || key < 0x007FFFFFu;
        atomicAdd(hist + window_bin(key, wlo, wshift), 1u);
      }
  return nan_seen;
}

// First histogram over quads [q0, q1) of the row; returns whether a NaN was seen.
template <int NT>
__device__ bool window_hist_pass(const RowRef& R, int q0, int q1, uint32_t wlo, int wshift,
                                 uint32_t* hist) {
  bool nan_seen = false;
  for (int base = q0; base < q1; base += NT * kU) {
    uint32_t kv[kU][4], ok[kU];
    hist_load<NT>(R, base, q1, kv, ok);
    nan_seen |= hist_step(kv, ok, wlo, wshift, hist);
  }
  return nan_seen;
}

// One step of the marking pass: this warp's kU runs starting at run s0
// (loaded by mark_load).
__device__ __forceinline__ void mark_load(const RowRef& R, int s0, int r1, uint32_t (*kv)[4],
                                          uint32_t* ok) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kU; ++u) ok[u] = s0 + u < r1 ? load_quad(R, (s0 + u) * 32 + lane, kv[u]) : 0u;
}
__device__ __forceinline__ void mark_step(const RowRef& R, const uint32_t (*kv)[4],
                                          const uint32_t* ok, int s0, int r1, uint32_t rlo,
                                          uint32_t rhi, bool exact, uint32_t* gt_out,
                                          uint32_t* eq_out, uint32_t* cand_cnt, uint2* cand_out) {
  const int lane = threadIdx.x & 31;
  const int nwu = (R.n + 31) >> 5;
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (s0 + u >= r1) break;  // warp-uniform
    uint32_t gn = 0u, en = 0u;  // 4-bit masks: above / inside the range
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool v = (ok[u] >> e) & 1u;
      const uint32_t key = kv[u][e];
      gn |= (v && key > rhi ? 1u : 0u) << e;
      en |= (v && key >= rlo && key <= rhi ? 1u : 0u) << e;
    }
    const int sh4 = 4 * (lane & 7);
    uint32_t gw = gn << sh4, ew = en << sh4;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      gw |= __shfl_xor_sync(0xffffffffu, gw, o);
      ew |= __shfl_xor_sync(0xffffffffu, ew, o);
    }
    const int word = (s0 + u) * 4 + (lane >> 3);
    if ((lane & 7) == 0 && word < nwu) {
      gt_out[word] = gw;
      if (exact) eq_out[word] = ew;
    }
    if (!exact && __any_sync(0xffffffffu, en != 0u)) {
      const uint32_t c = __popc(en);
      const uint32_t incl = warp_incl_scan(c, lane);
      uint32_t slot = 0;
      if (lane == 31) slot = atomicAdd(cand_cnt, incl);
      slot = __shfl_sync(0xffffffffu, slot, 31) + incl - c;
      const int p0 = ((s0 + u) * 32 + lane) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((en >> e) & 1u) {
          if (slot < static_cast<uint32_t>(kRCand))
            cand_out[slot] = make_uint2(kv[u][e], static_cast<uint32_t>(p0 + e));
          ++slot;
        }
    }
  }
}

// Marking pass over the runs [r0, r1) of 32 quads (128 positions) of the
// row: keys above rhi become bits of gt_out (word = position / 32); keys in
// [rlo, rhi] become bits of eq_out when `exact`, else candidates appended at
// cand_out[atomicAdd(cand_cnt)] (at most kRCand kept).  Lane l holds
// positions 4l .. 4l + 3 of a run, so the word of positions 32j .. 32j + 31
// is the OR of the 4-bit masks of lanes 8j .. 8j + 7.
template <int NT>
__device__ void mark_pass(const RowRef& R, int r0, int r1, uint32_t rlo, uint32_t rhi, bool exact,
                          uint32_t* gt_out, uint32_t* eq_out, uint32_t* cand_cnt, uint2* cand_out) {
  const int warp = threadIdx.x >> 5;
  for (int s0 = r0 + warp * kU; s0 < r1; s0 += (NT / 32) * kU) {
    uint32_t kv[kU][4], ok[kU];
    mark_load(R, s0, r1, kv, ok);
    mark_step(R, kv, ok, s0, r1, rlo, rhi, exact, gt_out, eq_out, cand_cnt, cand_out);
  }
}

// ---------------------------------------------------------------- K1
__global__ void __launch_bounds__(kSThreads) topk_hist_kernel(const TopkLaunch P) {
  __shared__ __align__(16) uint32_t hist[kWBins];
  __shared__ uint32_t misc[128];
  const int q = blockIdx.y;
  pdl_trigger();
  pdl_wait();  // the scores come from the previous grid
  const RowRef R = row_ref(P, q);
  const int q0 = blockIdx.x * P.seg_quads;
  if (R.n <= P.k || q0 >= R.nq) return;
  const int q1 = min(R.nq, q0 + P.seg_quads);
  // the first step's keys in flight while the window is sampled
  uint32_t kv0[kU][4], ok0[kU];
  hist_load<kSThreads>(R, q0, q1, kv0, ok0);
  for (int i = threadIdx.x; i < kWBins; i += kSThreads) hist[i] = 0u;
  sample_window<kSThreads>(R, misc + 32, misc);  // its barriers also publish the zeroed bins
  const uint32_t wlo = misc[0];
  const int wshift = range_shift(wlo, misc[1], kWBits);
  bool nan_seen = hist_step(kv0, ok0, wlo, wshift, hist);
  nan_seen |= window_hist_pass<kSThreads>(R, q0 + kSThreads * kU, q1, wlo, wshift, hist);
  if (__any_sync(0xffffffffu, nan_seen) && (threadIdx.x & 31) == 0) raise_err(P.d_err, DSA_DEVERR_NAN);
  __syncthreads();
  uint32_t* g = P.ghist + static_cast<long long>(q) * kWBins;
  for (int i = threadIdx.x; i < kWBins; i += kSThreads)
    if (hist[i] != 0u) atomicAdd(g + i, hist[i]);
}

// ---------------------------------------------------------------- K2
// at most 64 registers, so that four CTAs fit on an SM (the pass is latency-
// bound: at 73 registers three fit, and it ran 2-6 % slower)
__global__ void __launch_bounds__(kSThreads, 4) topk_mark_kernel(const TopkLaunch P) {
  __shared__ __align__(16) uint32_t hist[kWBins];
  __shared__ uint32_t misc[128];
  const int q = blockIdx.y;
  pdl_trigger();
  pdl_wait();  // the row histograms come from the previous grid
  const RowRef R = row_ref(P, q);
  const int q0 = blockIdx.x * P.seg_quads;
  if (R.n <= P.k || q0 >= R.nq) return;
  const int q1 = min(R.nq, q0 + P.seg_quads);
  const int r0 = q0 / 32, r1 = (q1 + 31) / 32;
  // the first step's keys in flight while the window and the bin are found
  uint32_t kv0[kU][4], ok0[kU];
  const int s0 = r0 + (static_cast<int>(threadIdx.x) >> 5) * kU;
  mark_load(R, s0, r1, kv0, ok0);
  const uint32_t* g = P.ghist + static_cast<long long>(q) * kWBins;
  for (int i = threadIdx.x; i < kWBins; i += kSThreads) hist[i] = __ldcg(g + i);
  sample_window<kSThreads>(R, misc + 32, misc);
  const uint32_t wlo = misc[0];
  const int wshift = range_shift(wlo, misc[1], kWBits);
  block_find_bin<kSThreads>(hist, kWBins, static_cast<uint32_t>(P.k), misc + 4, misc + 32);
  __syncthreads();
  if (misc[6] > static_cast<uint32_t>(kRCand)) return;  // crowded: K3 resolves the row alone
  uint32_t rlo, rhi;
  window_range(wlo, wshift, misc[4], &rlo, &rhi);
  uint32_t* gt_out = P.gbits + static_cast<long long>(q) * P.nw;
  uint2* cand_out = P.gcand + static_cast<long long>(q) * kRCand;
  mark_step(R, kv0, ok0, s0, r1, rlo, rhi, false, gt_out, nullptr, P.gcnt + q, cand_out);
  mark_pass<kSThreads>(R, r0 + (kSThreads / 32) * kU, r1, rlo, rhi, false, gt_out, nullptr,
                       P.gcnt + q, cand_out);
}

// ---------------------------------------------------------------- K3
__global__ void __launch_bounds__(kRThreads, 2) topk_rows_kernel(const TopkLaunch P,
                                                              const RowsSmem S) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + S.off_hist);
  uint2* cand = reinterpret_cast<uint2*>(smem + S.off_cand);
  uint32_t* eqb = reinterpret_cast<uint32_t*>(smem + S.off_eq);
  uint32_t* gtb = reinterpret_cast<uint32_t*>(smem + S.off_gt);
  uint32_t* chist = reinterpret_cast<uint32_t*>(smem + S.off_chist);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S.off_misc);
  uint32_t* sh = misc;            // [0] NaN seen, [1] candidates, [4..6] bin search, [8..9] window
  uint32_t* scratch = misc + 32;  // [96] scan and reduction scratch

  const int tid = threadIdx.x, lane = tid & 31;
  const int q = blockIdx.x;
  const int w = q / P.rows;
  const int r = q - w * P.rows;
  const int k = P.k;
  pdl_trigger();
  pdl_wait();  // the scores (or the marks of K2) come from the previous grid

  {
    const int nraw = P.valid_len ? P.valid_len[q]
                                 : shard_valid_len(P.row_pos[r], P.W, w + P.shard_offset);
    if ((nraw < 0 || nraw > P.ld) && tid == 0) raise_err(P.d_err, DSA_DEVERR_INDEX);
  }
  const RowRef R = row_ref(P, q);
  const int n = R.n;
  const int off = P.index_offset + (P.offset_per_shard ? (w + P.shard_offset) : 0);
  int32_t* oi = P.out_idx + static_cast<long long>(q) * k;
  float* os = P.out_score ? P.out_score + static_cast<long long>(q) * k : nullptr;
  const int cnt_all = n < k ? n : k;
  if (tid < 32) sh[tid] = 0;

  if (n <= k) {
    // every valid position, in order
    bool nan_seen = false;
    for (int i = tid; i < n; i += kRThreads) {
      const float f = __ldcg(R.src + i);
      nan_seen |= (f != f);
      oi[i] = i * P.index_stride + off;
      if (os) os[i] = f;
    }
    for (int i = n + tid; i < k; i += kRThreads) {
      oi[i] = -1;
      if (os) os[i] = -__int_as_float(0x7f800000);
    }
    if (tid == 0) P.out_count[q] = cnt_all;
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_err(P.d_err, DSA_DEVERR_NAN);
    return;
  }

  // ---------------- the first histogram: K1's, or made here
  if (P.ghist != nullptr) {
    const uint32_t* g = P.ghist + static_cast<long long>(q) * kWBins;
    for (int i = tid; i < kWBins; i += kRThreads) hist[i] = __ldcg(g + i);
  } else {
    for (int i = tid; i < kWBins; i += kRThreads) hist[i] = 0u;
  }
  sample_window<kRThreads>(R, scratch, sh + 8);  // its barriers publish the bins and sh
  const uint32_t wlo = sh[8];
  const int wshift = range_shift(wlo, sh[9], kWBits);
  if (P.ghist == nullptr) {
    const bool nan_seen = window_hist_pass<kRThreads>(R, 0, R.nq, wlo, wshift, hist);
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_err(P.d_err, DSA_DEVERR_NAN);
    __syncthreads();
  }
  block_find_bin<kRThreads>(hist, kWBins, static_cast<uint32_t>(k), sh + 4, scratch);
  __syncthreads();
  // [rlo, rhi]: the keys of the bin holding T; k_rem: T's rank in it from the
  // top; cnt: the row's keys in it
  uint32_t rlo, rhi, k_rem = sh[5], cnt = sh[6];
  window_range(wlo, wshift, sh[4], &rlo, &rhi);
  const int nwu = (n + 31) >> 5;  // bitmap words in use
  bool exact = false;
  uint32_t nc;
  if (P.ghist != nullptr && cnt <= static_cast<uint32_t>(kRCand)) {
    // ---------------- K2's bitmap and candidates
    __syncthreads();  // the histogram is dead: its memory holds the candidates next
    const uint32_t* gb = P.gbits + static_cast<long long>(q) * P.nw;
    for (int j = tid; j < S.nw; j += kRThreads) {
      gtb[j] = j < nwu ? __ldcg(gb + j) : 0u;
      eqb[j] = 0u;
    }
    nc = min(__ldcg(P.gcnt + q), static_cast<uint32_t>(kRCand));
    const uint2* gc = P.gcand + static_cast<long long>(q) * kRCand;
    for (uint32_t e = tid; e < nc; e += kRThreads) cand[e] = __ldcg(gc + e);
    __syncthreads();
  } else {
    // ---------------- further rounds while the bin is crowded
    while (cnt > static_cast<uint32_t>(kRCand) && rlo < rhi) {
      const int shift = range_shift(rlo, rhi, kRBits);
      __syncthreads();  // every thread has read sh and the previous histogram
      for (int i = tid; i < (1 << kRBits); i += kRThreads) hist[i] = 0u;
      __syncthreads();
      for (int base = 0; base < R.nq; base += kRThreads * kU) {
        uint32_t kv[kU][4], ok[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) ok[u] = load_quad(R, base + u * kRThreads + tid, kv[u]);
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t key = kv[u][e];
            if (((ok[u] >> e) & 1u) && key >= rlo && key <= rhi)
              atomicAdd(hist + ((key - rlo) >> shift), 1u);
          }
      }
      __syncthreads();
      block_find_bin<kRThreads>(hist, 1 << kRBits, k_rem, sh + 4, scratch);
      __syncthreads();
      bin_range(rlo, rhi, shift, sh[4], &rlo, &rhi);
      k_rem = sh[5];
      cnt = sh[6];
    }
    exact = rlo == rhi;  // T is known: every key in the range equals it
    __syncthreads();     // the histogram is dead: its memory holds the candidates next
    for (int j = tid; j < S.nw; j += kRThreads) {
      gtb[j] = 0u;
      eqb[j] = 0u;
    }
    __syncthreads();
    mark_pass<kRThreads>(R, 0, (R.nq + 31) / 32, rlo, rhi, exact, gtb, eqb, sh + 1, cand);
    __syncthreads();
    nc = min(sh[1], static_cast<uint32_t>(kRCand));
  }

  // ---------------- T from the candidates alone (10-bit rounds over the range)
  if (!exact) {
    while (rlo < rhi) {
      const int shift = range_shift(rlo, rhi, kCBits);
      for (int i = tid; i < (1 << kCBits); i += kRThreads) chist[i] = 0u;
      __syncthreads();
      for (uint32_t e = tid; e < nc; e += kRThreads) {
        const uint32_t key = cand[e].x;
        if (key >= rlo && key <= rhi) atomicAdd(chist + ((key - rlo) >> shift), 1u);
      }
      __syncthreads();
      block_find_bin<kRThreads>(chist, 1 << kCBits, k_rem, sh + 4, scratch);
      __syncthreads();
      bin_range(rlo, rhi, shift, sh[4], &rlo, &rhi);
      k_rem = sh[5];
      __syncthreads();  // sh and chist are read before the next round writes them
    }
    // candidates above T are selected; those equal to T are ties
    for (uint32_t e = tid; e < nc; e += kRThreads) {
      const uint2 c = cand[e];
      if (c.x > rlo) atomicOr(gtb + (c.y >> 5), 1u << (c.y & 31u));
      else if (c.x == rlo) atomicOr(eqb + (c.y >> 5), 1u << (c.y & 31u));
    }
    __syncthreads();
  }
  // k_rem: ties (keys equal to T) to take, lowest positions first

  // ---------------- compaction in position order
  const int per = (nwu + kRThreads - 1) / kRThreads;
  const int j0 = tid * per, j1 = min(nwu, j0 + per);
  uint32_t e_mine = 0;
  for (int j = j0; j < j1; ++j) e_mine += __popc(eqb[j]);
  uint32_t e_tot;
  uint32_t eq_before = block_excl_scan<kRThreads>(e_mine, scratch, &e_tot);
  uint32_t s_mine = 0;
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
    eqb[j] = ew;  // this thread's words only
    s_mine += __popc(gtb[j] | ew);
  }
  uint32_t s_tot;
  uint32_t slot = block_excl_scan<kRThreads>(s_mine, scratch, &s_tot);
  for (int j = j0; j < j1 && slot < static_cast<uint32_t>(k); ++j) {
    uint32_t sel = gtb[j] | eqb[j];
    while (sel != 0u && slot < static_cast<uint32_t>(k)) {
      const int b = __ffs(sel) - 1;
      sel &= sel - 1u;
      const int pos = j * 32 + b;
      oi[slot] = pos * P.index_stride + off;
      if (os) os[slot] = key_score(score_key(__ldcg(R.src + pos)));  // -0 listed as +0
      ++slot;
    }
  }
  for (int i = cnt_all + tid; i < k; i += kRThreads) {
    oi[i] = -1;
    if (os) os[i] = -__int_as_float(0x7f800000);
  }
  if (tid == 0) P.out_count[q] = cnt_all;
}

template <int C>
cudaError_t launch_c(const TopkLaunch& p, int rows, cudaStream_t stream, bool pdl) {
  const TopkSmem S = topk_smem(C);
  cudaError_t e =
      cudaFuncSetAttribute(topk_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
  if (e != cudaSuccess) return e;
  return launch_ex(topk_kernel<C>, dim3(rows * C), dim3(kThreads), S.total, stream, pdl, p, S);
}

}  // namespace

size_t topk_workspace_bytes(int rows, int64_t ld) {
  if (rows <= 0) return 0;
  const int64_t nw = ((ld + 31) / 32 + 3) / 4 * 4;
  const int64_t R = rows;
  const int64_t hist = R * kWBins * 4 + (R * 4 + 255) / 256 * 256;  // histograms, counts
  return static_cast<size_t>(hist + R * kRCand * 8 + R * nw * 4);
}

void topk_set_workspace(TopkLaunch& p, void* ws) {
  const int64_t R = static_cast<int64_t>(p.nshards) * p.rows;
  p.nw = static_cast<int32_t>(((p.ld + 31) / 32 + 3) / 4 * 4);
  if (ws == nullptr || R == 0) {
    p.ghist = p.gcnt = p.gbits = nullptr;
    p.gcand = nullptr;
    return;
  }
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.ghist = reinterpret_cast<uint32_t*>(b);
  p.gcnt = reinterpret_cast<uint32_t*>(b + R * kWBins * 4);
  b += R * kWBins * 4 + (R * 4 + 255) / 256 * 256;
  p.gcand = reinterpret_cast<uint2*>(b);
  b += R * kRCand * 8;
  p.gbits = reinterpret_cast<uint32_t*>(b);
}

size_t topk_workspace_clear_bytes(int rows) {
  const int64_t R = rows;
  return static_cast<size_t>(R * kWBins * 4 + R * 4);
}

bool topk_uses_workspace(int rows, int64_t ld) {
  const int sms = num_sms() > 0 ? num_sms() : 148;
  return rows > 0 && rows <= 65535 && rows * 2 > sms && rows_smem(ld).total <= kSmemLimit;
}

cudaError_t launch_topk(const TopkLaunch& p0, cudaStream_t stream, bool pdl) {
  const int rows = p0.nshards * p0.rows;
  if (rows == 0) return cudaSuccess;
  TopkLaunch p = p0;
  const RowsSmem RS = rows_smem(p.ld);
  const int sms = num_sms() > 0 ? num_sms() : 148;
  // Few rows (every row gets a cluster of 2 or 4 CTAs at once) or rows too
  // long for the bitmaps: the cluster form, the widest cluster that still
  // runs every row at once (one CTA per SM).  Measured on one GB300: 32 rows
  // of 32768 scores in 18.4 us, against 33 us in the segment form.
  if (!topk_uses_workspace(rows, p.ld) && (RS.total > kSmemLimit || rows * 2 <= sms)) {
    if (rows * 4 <= sms) return launch_c<4>(p, rows, stream, pdl);
    if (rows * 2 <= sms) return launch_c<2>(p, rows, stream, pdl);
    return launch_c<1>(p, rows, stream, pdl);
  }
  cudaError_t e;
  if (!topk_uses_workspace(rows, p.ld)) topk_set_workspace(p, nullptr);
  if (p.ghist != nullptr) {
    // segments: 16K positions, fewer when that leaves most SMs idle
    const int sms = num_sms() > 0 ? num_sms() : 148;
    p.seg_quads = 4096;
    while (p.seg_quads > 1024 &&
           static_cast<long long>(rows) * ((p.ld + 4LL * p.seg_quads - 1) / (4LL * p.seg_quads)) <
               2LL * sms)
      p.seg_quads /= 2;
    const dim3 grid(static_cast<unsigned>((p.ld + 4LL * p.seg_quads - 1) / (4LL * p.seg_quads)),
                    static_cast<unsigned>(rows));
    e = launch_ex(topk_hist_kernel, grid, dim3(kSThreads), 0, stream, pdl, p);
    if (e != cudaSuccess) return e;
    e = launch_ex(topk_mark_kernel, grid, dim3(kSThreads), 0, stream, true, p);
    if (e != cudaSuccess) return e;
    pdl = true;
  }
  e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RS.total);
  if (e != cudaSuccess) return e;
  return launch_ex(topk_rows_kernel, dim3(rows), dim3(kRThreads), RS.total, stream, pdl, p, RS);
}

}  // namespace dsa
