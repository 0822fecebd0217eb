// DSA indexer scoring on the sm_103a tensor cores.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Motivation and Modifications / Indexer decode: every cached token (of a
// shard) gets an indexer score before the top-2048 selection.  Score of token
// t for query row r: sum_h w[r][h] * relu(q[r][h] . k[t]) over 64 heads x 128.
//
// Design (one persistent CTA per SM, 8 or 12 warps):
//   warp 0      TMA producer: 128-token tiles of the paged index-K cache,
//               two 64-token page halves per tile, into a ring of stages.
//   warp 1      tcgen05 issuer: D[128 tokens x 64*rows] = K_tile . Q^T with
//               the accumulator in TMEM (two slots, so the epilogue of one
//               tile overlaps the MMA of the next).
//   warps 2-3   Q staging.  bf16 keys: the query as is (kind::f16).  fp8
//               keys: the MMA runs kind::f8f6f4 on the e4m3 tile as it lands,
//               and each head's query, scaled by 2^e so that its largest |q|
//               sits in [224, 448], is split into two e4m3 terms hi + lo (lo
//               holds the rounding remainder of hi; together they keep every
//               bf16 digit down to 2^-9 at that scale) that accumulate into
//               the same TMEM columns; 2^-e goes into the head weight.
//   warps 4-7   epilogue (and warps 8-11, a second set, for fp8 keys or
//               several rows per request: then each set takes one of the two
//               accumulator slots): one thread per token row of the tile reads its
//               TMEM lane, applies relu, the head weights (and the fp8
//               per-token scale, read from the key stage, which is released
//               only once the MMA and both epilogue sets are done with it)
//               and stores the fp32 score.
// Work units are (shard, request, tile); the flattened unit list is split
// evenly over the CTAs.  All rows of a request share one key stream.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kBlockT = 128;  // tokens of one M-block (the M of one tcgen05 MMA)
// 4 warps (producer, issuer, Q staging) + 4 epilogue warps per epilogue set
__host__ __device__ constexpr int threads_of(int sets) { return 128 + 128 * sets; }
constexpr int kOpBytes = kBlockT * kIdxDim * 2;     // 32 KB bf16 key tile
constexpr int kRawFp8Block = kBlockT * kIdxDim;     // 16 KB e4m3 keys of one M-block
// an fp8 stage: the e4m3 tile (one or two M-blocks), then the (page, slot)
// of its 64-token boxes for the epilogue's scale loads, padded to the
// 1024-byte alignment of the 128B-swizzled operand
__host__ __device__ constexpr int fp8_stage_bytes(int blocks) { return blocks * kRawFp8Block + 1024; }
constexpr int kHalfBf16Box = 64 * 64 * 2;          // one TMA box: 64 tokens x 64 dims
constexpr int kSmemLimit = 227 * 1024;

struct PairMeta {           // per (shard, request) pair, written by the aux warps
  float w[kRowsPerGroup][kIdxHeads];
  int valid[kRowsPerGroup];
  int row[kRowsPerGroup];
};

struct Layout {
  int stages;      // TMA ring depth
  int stage_bytes;
  int q_rows;      // max_rows * 64
  int q_kb_stride; // bytes between the two 64-dim halves of Q
  int off_ring, off_q, off_meta, off_rows, off_bar, total;
  int rows_smem;   // row_start and row_pos copied to shared memory (they fit)
  int slot_cols, tmem_cols, rows_per_chunk;
  int blocks;      // M-blocks of 128 tokens per tile (2: one-row fp8 requests)
};

__host__ __device__ inline int rows_per_chunk_of(int nr) {
  int nch = (nr + 3) / 4;
  return (nr + nch - 1) / nch;
}

// row_ints: num_reqs + 1 + num_rows, the row metadata a CTA copies to
// shared memory for its schedule when it fits in kRowsSmemCap bytes.
constexpr int kRowsSmemCap = 8192;

__host__ inline Layout make_layout(int fp8, int max_rows, int row_ints, int blocks) {
  Layout L{};
  L.blocks = blocks;
  L.rows_smem = row_ints * 4 <= kRowsSmemCap;
  const int rows_bytes = L.rows_smem ? (row_ints * 4 + 15) / 16 * 16 : 0;
  L.q_rows = max_rows * kIdxHeads;
  L.q_kb_stride = L.q_rows * 128;
  L.rows_per_chunk = rows_per_chunk_of(max_rows);
  L.slot_cols = blocks * L.rows_per_chunk * kIdxHeads;
  int cols = 32;
  while (cols < 2 * L.slot_cols) cols *= 2;
  L.tmem_cols = cols;
  const int q_bytes = 2 * L.q_kb_stride;
  const int meta_bytes = 2 * static_cast<int>(sizeof(PairMeta));
  const int bar_bytes = 512;
  const int fixed = 1024 /*align*/ + q_bytes + meta_bytes + rows_bytes + bar_bytes;
  L.stage_bytes = fp8 ? fp8_stage_bytes(blocks) : kOpBytes;
  L.stages = (kSmemLimit - fixed) / L.stage_bytes;
  if (L.stages > 8) L.stages = 8;
  int off = 0;
  L.off_ring = off;
  off += L.stages * L.stage_bytes;
  L.off_q = off;
  off += q_bytes;
  L.off_meta = off;
  off += meta_bytes;
  L.off_rows = off;
  off += rows_bytes;
  L.off_bar = off;
  off += bar_bytes;
  L.total = off + 1024;
  return L;
}

struct PairInfo {
  int row0, nr, len, ntiles;
};

// A work pair is (shard cache, request, row group): the rows of a request
// form groups of at most max_rows consecutive rows (the query rows one CTA
// holds in shared memory), and every group streams the request's keys.
__device__ __forceinline__ int pair_shard(const IndexerLaunch& P, int pair) {
  return pair / (P.num_reqs * P.groups);
}
__device__ __forceinline__ int pair_req(const IndexerLaunch& P, int pair) {
  return (pair / P.groups) % P.num_reqs;
}

// The request's row range and the rows' positions, from the shared-memory
// copy when the layout holds one.
struct RowMeta {
  const int* rs;  // row_start copy, or nullptr: read the global arrays
  const int* rp;
  __device__ int start(const IndexerLaunch& P, int b) const {
    return rs ? rs[b] : __ldg(P.row_start + b);
  }
  __device__ int pos(const IndexerLaunch& P, int r) const {
    return rs ? rp[r] : __ldg(P.row_pos + r);
  }
};

__device__ PairInfo pair_info(const IndexerLaunch& P, const RowMeta& M, int pair, bool report,
                              int tile_t) {
  const int sl = pair_shard(P, pair);
  const int b = pair_req(P, pair);
  const int g = pair % P.groups;
  const int shard = P.shard_base + sl;
  PairInfo pi{0, 0, 0, 0};
  const int q0 = M.start(P, b);
  const int q1 = M.start(P, b + 1);
  if (q0 < 0 || q1 < q0 || q1 > P.num_rows) {
    if (report) raise_err(P.d_err, DSA_DEVERR_ROWS);
    return pi;
  }
  if (q1 - q0 > P.max_rows * P.groups) {
    if (report && g == 0) raise_err(P.d_err, DSA_DEVERR_GROUP);
    return pi;
  }
  const int r0 = q0 + g * P.max_rows;
  const int r1 = min(q1, r0 + P.max_rows);
  if (r0 >= r1) return pi;  // the request has fewer groups
  int len = 0;
  for (int r = r0; r < r1; ++r) {
    const int pos = M.pos(P, r);
    if (pos < 0) {
      if (report) raise_err(P.d_err, DSA_DEVERR_POS);
      return pi;
    }
    len = max(len, shard_valid_len(pos, P.W, shard));
  }
  if (static_cast<long long>(len) >
          static_cast<long long>(P.max_blocks[sl]) * P.page_size ||
      len > P.ld) {
    if (report) raise_err(P.d_err, DSA_DEVERR_POS);
    return pi;
  }
  pi.row0 = r0;
  pi.nr = r1 - r0;
  pi.len = len;
  pi.ntiles = (len + tile_t - 1) / tile_t;
  return pi;
}

// Walks this CTA's units in order: (pair, tile).  The pair's shard and
// request are kept, so that a tile needs no division.
struct Walker {
  int pair, tile, npairs, tile_t, sl, b;
  PairInfo pi;
  RowMeta M;
  __device__ void start(const IndexerLaunch& P, const RowMeta& m, int p, int t, int tt) {
    M = m;
    pair = p;
    tile = t;
    tile_t = tt;
    npairs = P.nshards * P.num_reqs * P.groups;
    set_pair(P);
    skip(P);
  }
  __device__ void set_pair(const IndexerLaunch& P) {
    pi = pair_info(P, M, pair, false, tile_t);
    sl = pair_shard(P, pair);
    b = pair_req(P, pair);
  }
  __device__ void skip(const IndexerLaunch& P) {
    while (tile >= pi.ntiles && pair + 1 < npairs) {
      ++pair;
      tile = 0;
      set_pair(P);
    }
  }
  __device__ void next(const IndexerLaunch& P) {
    ++tile;
    skip(P);
  }
};

__device__ __forceinline__ int page_of(const IndexerLaunch& P, int sl, int b, int lp) {
  const int32_t* bt = P.block_table[sl];
  return bt ? __ldg(bt + static_cast<long long>(b) * P.max_blocks[sl] + lp)
            : b * P.max_blocks[sl] + lp;
}

// logical page of token t (a shift when the page size is a power of two)
__device__ __forceinline__ int page_of_token(const IndexerLaunch& P, int t) {
  return P.page_shift >= 0 ? (t >> P.page_shift) : t / P.page_size;
}

// Two e4m3 terms of a float pair (a, b): hi = e4m3(x), lo = e4m3(x - hi),
// each packed as two bytes with a in the low byte.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_fp8x2_storage_t h =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_fp8x2_storage_t l =
      __nv_cvt_float2_to_fp8x2(make_float2(a - back.x, b - back.y), __NV_SATFINITE, __NV_E4M3);
  hi = static_cast<uint32_t>(h);
  lo = static_cast<uint32_t>(l);
}

template <bool kFp8, int kSets, int kBlocks>
__global__ void __launch_bounds__(threads_of(kSets), 1)
    indexer_kernel(const __grid_constant__ IndexerLaunch P, const Layout L) {
  constexpr int kThreads = threads_of(kSets);
  constexpr int kTileT = kBlockT * kBlocks;  // tokens per tile
  constexpr int kBoxes = kTileT / 64;        // 64-token TMA boxes per tile
  static_assert(kBlocks == 1 || (kFp8 && kSets == 2), "two-block tiles: fp8 keys, two sets");
  // with two-block tiles each epilogue set takes one block of every chunk
  constexpr bool kSetPerBlock = kBlocks == 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw_base);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  pdl_trigger();

  uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + L.off_bar);
  // barrier indices
  const int B_KFULL = 0, B_KEMPTY = 8, B_QFULL = 20, B_QEMPTY = 21, B_ACCFULL = 22,
            B_ACCEMPTY = 24, B_PFULL = 26, B_PEMPTY = 28, B_DRAIN = 30;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 32);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 33);
  int* s_start = reinterpret_cast<int*>(bars + 34);   // [pair, tile, nunits]
  int* s_scan = reinterpret_cast<int*>(bars + 36);    // 12 warp sums
  PairMeta* meta = reinterpret_cast<PairMeta*>(sbase + L.off_meta);

  if (tid == 0) {
    for (int s = 0; s < L.stages; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      // released by lane 0 of each epilogue warp, once each set
      // has seen the accumulators of its chunks of the tile land (the MMAs,
      // which read the stage, are then done)
      // released when the tile's MMAs complete (a commit of the issuing
      // thread) and, for fp8 keys, once every epilogue warp has read the
      // tile's page and slot words from the stage
      mbar_init(bar(B_KEMPTY + s), 1 + (kFp8 ? 4 * kSets : 0));
    }
    for (int o = 0; o < 2; ++o) {
      mbar_init(bar(B_ACCFULL + o), 1);
      mbar_init(bar(B_ACCEMPTY + o), kSetPerBlock ? 128 * kSets : 128);
      mbar_init(bar(B_PFULL + o), 1);
      mbar_init(bar(B_PEMPTY + o), 128 * kSets);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < P.nshards; ++i) tma_prefetch_desc(&P.kmap[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(L.tmem_cols));
    tmem_relinquish();
  }

  pdl_wait();  // inputs may come from the previous grid

  // L2 prefetch of the block tables and the queries of this launch (each
  // thread of the grid takes every n-th 128-byte line), so that the first
  // tile's page lookups and the query staging find them in L2
  {
    const long long nthreads = static_cast<long long>(gridDim.x) * kThreads;
    const long long first = static_cast<long long>(blockIdx.x) * kThreads + tid;
    auto prefetch = [&](const void* base, long long bytes) {
      for (long long off = first * 128; off < bytes; off += nthreads * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(base) + off));
    };
    for (int i = 0; i < P.nshards; ++i)
      if (P.block_table[i] != nullptr)
        prefetch(P.block_table[i], static_cast<long long>(P.num_reqs) * P.max_blocks[i] * 4);
    prefetch(P.q_idx, static_cast<long long>(P.num_rows) * kIdxHeads * kIdxDim * 2);
    prefetch(P.w_idx, static_cast<long long>(P.num_rows) * kIdxHeads * 4);
  }
  // every request's row range and every row's position, in one round of
  // loads (the schedule below would otherwise wait for two dependent ones)
  RowMeta rm{nullptr, nullptr};
  if (L.rows_smem) {
    int* rs = reinterpret_cast<int*>(sbase + L.off_rows);
    int* rp = rs + P.num_reqs + 1;
    for (int i = tid; i <= P.num_reqs; i += kThreads) rs[i] = __ldg(P.row_start + i);
    for (int i = tid; i < P.num_rows; i += kThreads) rp[i] = __ldg(P.row_pos + i);
    __syncthreads();
    rm = RowMeta{rs, rp};
  }

  // ---- schedule: count units of every (shard, request) pair, split evenly
  const int npairs = P.nshards * P.num_reqs * P.groups;
  {
    const int chunk = (npairs + kThreads - 1) / kThreads;
    const int p0 = min(npairs, tid * chunk);
    const int p1 = min(npairs, p0 + chunk);
    int mine = 0;
    for (int p = p0; p < p1; ++p) mine += pair_info(P, rm, p, blockIdx.x == 0, kTileT).ntiles;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    int woff = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) woff += s_scan[w];
      total += s_scan[w];
    }
    const int excl = woff + incl - mine;
    const long long u0 = static_cast<long long>(blockIdx.x) * total / gridDim.x;
    const long long u1 = static_cast<long long>(blockIdx.x + 1) * total / gridDim.x;
    if (tid == 0) s_start[2] = static_cast<int>(u1 - u0);
    if (u0 < u1 && excl <= u0 && u0 < excl + mine) {
      int acc = excl;
      for (int p = p0; p < p1; ++p) {
        const int n = pair_info(P, rm, p, false, kTileT).ntiles;
        if (u0 < acc + n) {
          s_start[0] = p;
          s_start[1] = static_cast<int>(u0 - acc);
          break;
        }
        acc += n;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nunits = s_start[2];
  const uint32_t tmem_base = *tmem_slot;

  if (nunits > 0) {
    const int start_pair = s_start[0];
    const int start_tile = s_start[1];
    const uint32_t ring = base + L.off_ring;
    const uint32_t qbase = base + L.off_q;

    if (warp == 0) {
      // ------------------------------------------------ TMA producer
      // The whole warp walks the units and lane 0 issues the copies.  The
      // block-table entries are read 32 at a time (one coalesced load holds
      // the pages of 16 tiles) and handed to lane 0 by a shuffle, so that a
      // tile waits for no global load of its own.
      Walker wk;
      wk.start(P, rm, start_pair, start_tile, kTileT);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int pc_pair = -1, pc_base = 0, pc_val = -1;  // this lane holds entry pc_base + lane
      for (int u = 0; u < nunits; ++u) {
        const bool got = __shfl_sync(
            0xffffffffu,
            lane == 0 ? mbar_wait(bar(B_KEMPTY + stage), phase ^ 1u, abort_flag) : true, 0);
        if (!got) break;
        ++issued;
        const int sl = wk.sl;
        const int b = wk.b;
        const int32_t* bt = P.block_table[sl];
        const int t0 = wk.tile * kTileT;
        const int lpa = page_of_token(P, t0);                // the tile's first page
        const int lpz = page_of_token(P, t0 + kTileT - 1);   // and its last
        if (bt != nullptr && (wk.pair != pc_pair || lpa < pc_base || lpz >= pc_base + 32)) {
          pc_pair = wk.pair;
          pc_base = lpa;
          const int e = pc_base + lane;
          pc_val = e < P.max_blocks[sl]
                       ? __ldg(bt + static_cast<long long>(b) * P.max_blocks[sl] + e)
                       : -1;
        }
        int pages[kBoxes], slots[kBoxes];
        uint32_t bytes = 0;
#pragma unroll
        for (int h = 0; h < kBoxes; ++h) {
          pages[h] = -1;
          slots[h] = 0;
          const int th = t0 + h * 64;
          const int lp = page_of_token(P, th);
          const int cached = __shfl_sync(0xffffffffu, pc_val, (lp - pc_base) & 31);
          if (th >= wk.pi.len) continue;
          const int pg = bt != nullptr ? cached : b * P.max_blocks[sl] + lp;
          if (pg < 0 || pg >= P.num_pages[sl]) {
            if (lane == 0) raise_err(P.d_err, DSA_DEVERR_PAGE);
            continue;
          }
          pages[h] = pg;
          slots[h] = th - lp * P.page_size;
          bytes += kFp8 ? 64u * 128u : 2u * kHalfBf16Box;
        }
        if (lane == 0) {
          const uint32_t fb = bar(B_KFULL + stage);
          const uint32_t dst = ring + stage * L.stage_bytes;
          if (kFp8) {
            // where the epilogue finds the tile's token scales (it loads its
            // token's scale itself): the boxes' pages, then their first
            // slots; released to it by the arrival below
            int* where = reinterpret_cast<int*>(sbase + L.off_ring + stage * L.stage_bytes +
                                                kBlocks * kRawFp8Block);
#pragma unroll
            for (int h = 0; h < kBoxes; ++h) {
              where[h] = pages[h];
              where[kBoxes + h] = slots[h];
            }
          }
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int h = 0; h < kBoxes; ++h) {
            if (pages[h] < 0) continue;
            if (kFp8) {
              tma_load_3d(dst + h * 8192, &P.kmap[sl], fb, 0, slots[h], pages[h]);
            } else {
              tma_load_3d(dst + h * 8192, &P.kmap[sl], fb, 0, slots[h], pages[h]);
              tma_load_3d(dst + 16384 + h * 8192, &P.kmap[sl], fb, 64, slots[h], pages[h]);
            }
          }
        }
        if (++stage == L.stages) {
          stage = 0;
          phase ^= 1u;
        }
        wk.next(P);
      }
      if (lane == 0) {
        // every stage's last release before the CTA exits (the epilogue is
        // behind this thread), so that no barrier is left mid-phase
        if (!*abort_flag) {
          for (int s = 0; s < L.stages && s < issued; ++s) {
            const int last = s + ((issued - 1 - s) / L.stages) * L.stages;
            mbar_wait(bar(B_KEMPTY + s), static_cast<uint32_t>(last / L.stages) & 1u, abort_flag);
          }
        }
        // every issued load must land before the CTA exits (only pending
        // after an abort; otherwise the consumers already waited for them)
        if (*abort_flag) {
          volatile int no_abort = 0;
          for (int s = 0; s < L.stages; ++s) {
            const int last = issued - 1 - ((issued - 1 - s) % L.stages + L.stages) % L.stages;
            if (last < 0 || (last % L.stages) != s) continue;
            mbar_wait(bar(B_KFULL + s), static_cast<uint32_t>(last / L.stages) & 1u, &no_abort);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        Walker wk;
        wk.start(P, rm, start_pair, start_tile, kTileT);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_iter = 0;
        int pair_j = -1, last_pair = -1;
        for (int u = 0; u < nunits; ++u) {
          if (wk.pair != last_pair) {
            if (pair_j >= 0) tc_commit(bar(B_QEMPTY));
            ++pair_j;
            last_pair = wk.pair;
            if (!mbar_wait(bar(B_QFULL), static_cast<uint32_t>(pair_j) & 1u, abort_flag)) break;
            tc_fence_after();
          }
          if (!mbar_wait(bar(B_KFULL + stage), phase, abort_flag)) break;
          const uint32_t a_base = ring + stage * L.stage_bytes;
          tc_fence_after();
          const int nr = wk.pi.nr;
          const int rpc = L.rows_per_chunk;
          bool ok = true;
          for (int c0 = 0; c0 < nr; c0 += rpc) {
            const int rows_c = min(rpc, nr - c0);
            const int slot = static_cast<int>(acc_iter & 1u);
            const uint32_t aph = (acc_iter >> 1) & 1u;
            if (!mbar_wait(bar(B_ACCEMPTY + slot), aph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t idesc = kFp8 ? idesc_e4m3(128, rows_c * kIdxHeads)
                                        : idesc_f16(128, rows_c * kIdxHeads, 1, 1);
            // descriptors: the start address field (bits 0..13, in 16-byte
            // units) of the block's first K-step, stepped by adding offsets
            const uint64_t bd0 =
                smem_desc_sw128(qbase + static_cast<uint32_t>(c0 * kIdxHeads * 128));
#pragma unroll
            for (int blk = 0; blk < kBlocks; ++blk) {
              // block blk: tokens blk * 128 .. + 127 of the tile, its own
              // accumulator columns in the slot
              const uint32_t d = tmem_base + static_cast<uint32_t>(
                                                 slot * L.slot_cols + blk * rpc * kIdxHeads);
              const uint64_t ad0 = smem_desc_sw128(a_base + blk * kRawFp8Block);
              // bf16: kb walks the two 64-dim halves of keys and query.
              // fp8: the 128-dim e4m3 block is one 128-byte row per token, met
              // once by the hi terms of the query (kb 0) and once by the lo
              // terms (kb 1), both into the same accumulator.
#pragma unroll
              for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = ad0 + static_cast<uint64_t>(((kFp8 ? 0 : kb * 16384) + k * 32) >> 4);
                  const uint64_t bd = bd0 + static_cast<uint64_t>((kb * L.q_kb_stride + k * 32) >> 4);
                  if (kFp8)
                    tc_mma_f8(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                  else
                    tc_mma_f16(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                }
              }
            }
            tc_commit(bar(B_ACCFULL + slot));
            ++acc_iter;
          }
          if (!ok) break;
          // the stage is free for the next fill once these MMAs are done
          tc_commit(bar(B_KEMPTY + stage));
          if (++stage == L.stages) {
            stage = 0;
            phase ^= 1u;
          }
          wk.next(P);
        }
        // all MMAs issued by this thread must finish before TMEM is freed
        volatile int no_abort = 0;
        tc_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0u, &no_abort);
      }
    } else if (warp == 2 || warp == 3) {
      // ------------------------------------------------ Q staging
      const int at = tid - 64;  // 0..63
      Walker wk;
      wk.start(P, rm, start_pair, start_tile, kTileT);
      int pair_j = -1, last_pair = -1;
      // A failed (timed-out) wait stops the work of this thread but it keeps
      // passing the same named barriers as its partner warp.
      bool ok = true;
      for (int u = 0; u < nunits; ++u) {
        if (wk.pair != last_pair) {
          ++pair_j;
          last_pair = wk.pair;
          const int mslot = pair_j & 1;
          if (ok && pair_j >= 2)
            ok = mbar_wait(bar(B_PEMPTY + mslot), static_cast<uint32_t>((pair_j >> 1) - 1) & 1u,
                           abort_flag);
          if (ok && pair_j >= 1)
            ok = mbar_wait(bar(B_QEMPTY), static_cast<uint32_t>(pair_j - 1) & 1u, abort_flag);
          const int sl = pair_shard(P, wk.pair);
          const int shard = P.shard_base + sl;
          const int nr = wk.pi.nr;
          const int row0 = wk.pi.row0;
          PairMeta& m = meta[mslot];
          // one query head-row (128 dims) per thread and step
          for (int n = at; ok && n < nr * kIdxHeads; n += 64) {
            const int g = n / kIdxHeads;
            const int h = n - g * kIdxHeads;
            const uint4* src = reinterpret_cast<const uint4*>(
                P.q_idx + (static_cast<long long>(row0 + g) * kIdxHeads + h) * kIdxDim);
            uint4 v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = __ldg(src + c);
            float wv = __ldg(P.w_idx + static_cast<long long>(row0 + g) * kIdxHeads + h);
            const uint32_t qrow = static_cast<uint32_t>(L.off_q + n * 128);
            if (kFp8) {
              // scale the head's query by 2^e so that its largest |q| lands in
              // [224, 448] (the top of the e4m3 range), then split every value
              // x into hi = e4m3(x) and lo = e4m3(x - hi)
              uint32_t mx = 0;
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const uint32_t* wds = reinterpret_cast<const uint32_t*>(&v[c]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  mx = max(mx, wds[j] & 0x7FFFu);
                  mx = max(mx, (wds[j] >> 16) & 0x7FFFu);
                }
              }
              // mx is the bf16 pattern of the largest |q|: biased exponent in
              // bits 7..14, mantissa in bits 0..6 (0x60 = 1.75, i.e. 448 / 256)
              const int ebits = static_cast<int>(mx >> 7);
              const int e = (ebits == 0)
                                ? 0
                                : max(-100, min(100, ((mx & 0x7Fu) <= 0x60u ? 135 : 134) - ebits));
              const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
              wv = wv * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
              for (int ch = 0; ch < 8; ++ch) {
                // 16 dims: the 8 bf16 pairs of v[2ch] and v[2ch + 1]
                const uint32_t* wds = reinterpret_cast<const uint32_t*>(&v[2 * ch]);
                uint32_t ho[4], lo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint32_t h0, l0, h1, l1;
                  const uint32_t wa = wds[2 * q], wb = wds[2 * q + 1];
                  split_e4m3x2(__uint_as_float(wa << 16) * sc, __uint_as_float(wa & 0xFFFF0000u) * sc,
                               h0, l0);
                  split_e4m3x2(__uint_as_float(wb << 16) * sc, __uint_as_float(wb & 0xFFFF0000u) * sc,
                               h1, l1);
                  ho[q] = h0 | (h1 << 16);
                  lo[q] = l0 | (l1 << 16);
                }
                const uint32_t off = qrow + static_cast<uint32_t>((ch ^ (n & 7)) << 4);
                *reinterpret_cast<uint4*>(sbase + off) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
                *reinterpret_cast<uint4*>(sbase + off + L.q_kb_stride) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
              }
            } else {
              // the K-major 128B-swizzled operand layout, 64 dims per half
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int kb = c >> 3;
                const int ch = c & 7;
                const uint32_t off = qrow + static_cast<uint32_t>(kb * L.q_kb_stride + ((ch ^ (n & 7)) << 4));
                *reinterpret_cast<uint4*>(sbase + off) = v[c];
              }
            }
            m.w[g][h] = wv;
          }
          if (ok && at < nr) {
            const int r = row0 + at;
            m.row[at] = r;
            m.valid[at] = shard_valid_len(__ldg(P.row_pos + r), P.W, shard);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 64);
          if (ok && at == 0) {
            mbar_arrive(bar(B_QFULL));
            mbar_arrive(bar(B_PFULL + mslot));
          }
        }
        wk.next(P);
      }
    } else {
      // ------------------------------------------------ epilogue (warps 4..)
      // With two sets of four warps and one-block tiles each set takes one
      // accumulator slot: set 0 (warps 4..7) the chunks that land in slot 0,
      // set 1 (warps 8..11) those in slot 1, so two chunks are summed at
      // once.  With two-block tiles set e takes block e of every chunk.
      const int eset = (warp - 4) >> 2;    // this warp's set
      const int eblk = kSetPerBlock ? eset : 0;  // the block of the tile it reads
      const int et = (tid - 128) & 127;    // token row of the block / TMEM lane
      const int q4 = warp & 3;             // TMEM lane quarter of this warp
      Walker wk;
      wk.start(P, rm, start_pair, start_tile, kTileT);
      uint32_t acc_iter = 0;
      int stage = 0;
      uint32_t phase = 0;
      int pair_j = -1, last_pair = -1;
      for (int u = 0; u < nunits; ++u) {
        if (wk.pair != last_pair) {
          if (pair_j >= 0) mbar_arrive(bar(B_PEMPTY + (pair_j & 1)));
          ++pair_j;
          last_pair = wk.pair;
          const bool got = mbar_wait(bar(B_PFULL + (pair_j & 1)),
                                     static_cast<uint32_t>(pair_j >> 1) & 1u, abort_flag);
          if (!__all_sync(0xffffffffu, got)) break;
        }
        const PairMeta& m = meta[pair_j & 1];
        const int sl = wk.sl;
        const int tt = eblk * kBlockT + et;  // token of the tile
        const int t = wk.tile * kTileT + tt;
        float kscale = 1.0f;
        if (kFp8) {
          // the token's scale, from the (page, slot) the producer left behind
          // the keys; loaded now, used after the accumulator wait.  Every set
          // reads its words once the tile has landed (also the set without a
          // chunk in it: its arrival must not run ahead of the fill, where it
          // would count towards the stage's previous use) and then lets the
          // stage go.
          const bool got = mbar_wait(bar(B_KFULL + stage), phase, abort_flag);
          if (!__all_sync(0xffffffffu, got)) break;
          const int* where = reinterpret_cast<const int*>(
              sbase + L.off_ring + stage * L.stage_bytes + kBlocks * kRawFp8Block);
          const int h = tt >> 6;
          const int pg = where[h];
          const int slot0 = where[kBoxes + h];
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_KEMPTY + stage));
          kscale = pg >= 0 ? __ldg(P.kscale[sl] + static_cast<long long>(pg) * P.page_size +
                                   slot0 + (tt & 63))
                           : 0.0f;
        }
        float* out_base = P.scores + static_cast<long long>(sl) * P.shard_stride;
        const int nr = wk.pi.nr;
        const int rpc = L.rows_per_chunk;
        bool ok = true;
        for (int c0 = 0; c0 < nr; c0 += rpc) {
          const int rows_c = min(rpc, nr - c0);
          const int slot = static_cast<int>(acc_iter & 1u);
          const uint32_t aph = (acc_iter >> 1) & 1u;
          if (kSets == 2 && !kSetPerBlock && slot != eset) {  // the other set's chunk
            ++acc_iter;
            continue;
          }
          if (!mbar_wait(bar(B_ACCFULL + slot), aph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int gi = 0; gi < rows_c; ++gi) {
            const int g = c0 + gi;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) +
                static_cast<uint32_t>(slot * L.slot_cols + (eblk * rpc + gi) * kIdxHeads);
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(taddr, v0);
            tmem_ld_32x32b_x32(taddr + 32, v1);
            tmem_wait_ld();
            // eight independent partial sums: one warp per scheduler has no
            // other work to hide a 64-long dependent chain behind
            float ps[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) ps[j] = 0.0f;
#pragma unroll
            for (int h = 0; h < 32; ++h)
              ps[h & 7] = fmaf(m.w[g][h], fmaxf(__uint_as_float(v0[h]), 0.0f), ps[h & 7]);
#pragma unroll
            for (int h = 0; h < 32; ++h)
              ps[h & 7] = fmaf(m.w[g][32 + h], fmaxf(__uint_as_float(v1[h]), 0.0f), ps[h & 7]);
            const float s = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            if (t < m.valid[g]) {
              out_base[static_cast<long long>(m.row[g]) * P.ld + t] = s * kscale;
            }
          }
          tc_fence_before();
          mbar_arrive(bar(B_ACCEMPTY + slot));
          ++acc_iter;
        }
        if (!ok) break;
        if (++stage == L.stages) {
          stage = 0;
          phase ^= 1u;
        }
        wk.next(P);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) raise_err(P.d_err, DSA_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(L.tmem_cols));
  }
}


template <bool kFp8, int kSets, int kBlocks>
cudaError_t launch_one(const IndexerLaunch& p, const Layout& L, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<kFp8, kSets, kBlocks>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (e != cudaSuccess) return e;
  indexer_kernel<kFp8, kSets, kBlocks><<<grid, threads_of(kSets), L.total, stream>>>(p, L);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer(const IndexerLaunch& p0, cudaStream_t stream) {
  IndexerLaunch p = p0;
  p.page_shift = -1;
  for (int s = 6; s < 31; ++s)
    if (p.page_size == (1 << s)) p.page_shift = s;
  // one-row fp8 requests: 256-token tiles (two M-blocks), so that a tile
  // carries as many key bytes as a bf16 tile and the per-tile work of every
  // role is paid per 32 KB
  const int blocks = (p.fp8 && p.max_rows == 1) ? 2 : 1;
  const Layout L = make_layout(p.fp8, p.max_rows, p.num_reqs + 1 + p.num_rows, blocks);
  if (L.stages < 2) return cudaErrorInvalidValue;
  int grid = num_sms();
  if (grid <= 0) return cudaErrorInvalidDevice;
  // A second epilogue set pays off where the epilogue carries weight: fp8
  // keys (a scale load per token, half the key bytes per tile) or several
  // rows per request; for one bf16 row the MMA issue is the bound and the
  // extra warps only crowd the issuing thread's sub-partition.
  if (p.fp8)
    return blocks == 2 ? launch_one<true, 2, 2>(p, L, grid, stream)
                       : launch_one<true, 2, 1>(p, L, grid, stream);
  if (p.max_rows > 1) return launch_one<false, 2, 1>(p, L, grid, stream);
  return launch_one<false, 1, 1>(p, L, grid, stream);
}

}  // namespace dsa
