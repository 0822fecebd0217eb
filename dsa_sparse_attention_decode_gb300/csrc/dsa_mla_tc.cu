// Absorbed-MLA sparse decode over an fp8 (e4m3) latent cache on the sm_103a
// tensor cores, split-K with LSE.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Modifications / Sparse decode: every (shard of a) query row attends only its
// selected latent rows with a split-K kernel that also returns the natural-log
// LSE; with a single split the partial is the final result.
//
// One CTA per (work row, split), 32 heads, 128-token tiles, 13 warps:
//   warps 0-3   gather: every tile is 32 groups of 4 selected tokens; lanes
//               0..7 of warp w take groups w, w + 4, ...  A lane resolves its
//               group (selection -> block table -> cache row) two tiles
//               ahead, its loads in flight while it issues, and issues the TMA
//               tile::gather4 copies of the 4 rows: five 128-byte column boxes
//               (dims 0..639; 576..639 lie past the row and are filled with
//               zeros) into a 128B-swizzled tile [column box b][token][128 B].
//               Two tile buffers.
//   warp 12     MMA issuer (one thread), kind::f8f6f4 with fp32 accumulators
//               in TMEM, issuing whichever of the next S^T and the next value
//               product is ready:
//                 S^T[tokens x heads] = KV[tokens x 576] . Q^T (the tile as a
//                 K-major operand; the query's hi and lo e4m3 terms are the
//                 two halves of one N = 64 operand, summed when read);
//                 O^T[dims x heads] += V^T[dims x tokens] . P^T (the same tile
//                 read as an MN-major operand, dims 0..511 in four 128-dim
//                 blocks; P's hi and lo terms again as one N = 64 operand).
//   warps 4-11  softmax: two threads per token lane of S^T (warps 4-7 heads
//               0..15, warps 8-11 heads 16..31).  The scaled logit
//               of token t and head h is z = sm_scale * scale_t * (q_h . code_t)
//               in base 2; the value product carries the token scale, so
//               P is taken of a = z + log2(scale_t) against the running max M
//               of a, which is raised lazily (only by more than 2): then O^T
//               (in TMEM) and the denominators are rescaled.  P * 64 is
//               split into e4m3 hi + lo terms; the denominator sums
//               exp2(z - M) per thread and is reduced over the tokens at the
//               end.  They also stage the query (per-head power of two into
//               [224, 448], hi + lo e4m3 terms), load their tokens' scales
//               and write the output.
// The query's hi and lo terms keep every bf16 digit of q down to 2^-9 of the
// head's largest |q|; P's two terms keep about 8 significant bits.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kH = 32;                   // heads
constexpr int kT = 128;                  // tokens per tile (the M of S^T)
constexpr int kThreads = 448;   // warps 0-3 gather, 4-11 softmax, 12 MMA, 13 scales
constexpr int kMmaWarp = 12;
constexpr int kScaleWarp = 13;
constexpr int kSmx = 256;       // softmax threads
constexpr int kHH = kH / 2;     // heads of one softmax thread
constexpr int kBoxes = 5;                // 128-byte column boxes of a latent row
constexpr int kBoxBytes = kT * 128;      // one column box of a tile: 16 KB
constexpr int kTileBytes = kBoxes * kBoxBytes;
constexpr int kQBytes = kBoxes * kH * 128;  // one e4m3 term of the query: 20 KB
constexpr int kPBytes = kH * kT;            // one e4m3 term of P^T: 4 KB
constexpr float kPScale = 64.0f;            // P is stored times 64
constexpr float kLazy = 2.0f;               // raise the running max only past +2
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// shared memory (offsets from a 1024-aligned base)
constexpr int kOffKV = 0;                              // 2 tiles
constexpr int kOffQ = kOffKV + 2 * kTileBytes;         // hi, lo
constexpr int kOffP = kOffQ + 2 * kQBytes;             // [slot][hi, lo]
constexpr int kOffKs = kOffP + 4 * kPBytes;            // [buf][128] token scales (-1: no token)
constexpr int kOffRows = kOffKs + 2 * kT * 4;          // [buf][128] cache rows (-1: no token)
constexpr int kOffRed = kOffRows + 2 * kT * 4;         // [4 lane quarters][32] reductions
constexpr int kOffMisc = kOffRed + 4 * kH * 4;         // [32] per-head factors, flags
constexpr int kOffBar = kOffMisc + 4 * kH * 4 + 64;
constexpr int kSmemBytes = kOffBar + 256 + 1024;       // + alignment slack

static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// TMEM columns: S^T slots at 0 and 64 (hi terms, then lo terms), O^T blocks
// at 128 + 64 m (hi, then lo)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 128;

DSA_DEV void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int col, int r0,
                         int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(col), "r"(r0), "r"(r1), "r"(r2),
      "r"(r3)
      : "memory");
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 128-byte rows of 128 consecutive M elements (e4m3), one row per K index,
// 8-row atoms of 1024 bytes stacked along K.  An MMA reads M = 128 (one atom
// wide), so both the leading and the stride offsets are the atom stride.
DSA_DEV uint64_t smem_desc_sw128_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1024u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

DSA_DEV void tmem_wait_st() {
  __syncwarp();
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// e4m3 code of x (round to nearest even, saturating), and the remainder
DSA_DEV uint32_t e4m3_of(float x) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
DSA_DEV float e4m3_val(uint32_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

// Warp transpose-reduction of 16 per-lane values v[0..15] (one per head):
// afterwards lanes l and l ^ 16 hold the reduction over the 32 lanes of
// value l & 15.
template <bool kMax>
DSA_DEV float warp_transpose_reduce16(float* v, int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  const float o = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], o) : v[0] + o;
}

// named barrier `id` of `n` threads that also ORs a predicate over them
DSA_DEV bool named_bar_or(int id, int n, int pred) {
  uint32_t r;
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(id), "r"(n), "r"(pred)
      : "memory");
  return r != 0;
}

DSA_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t* r) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
DSA_DEV void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
  __syncwarp();  // the .aligned form needs a converged warp
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

struct MlaTcLaunch {
  MlaLaunch p;
  CUtensorMap kvmap[DSA_MAX_SHARDS];
  int32_t page_shift;  // log2(page_size) when a power of two, else -1
};

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ MlaTcLaunch T) {
  const MlaLaunch& P = T.p;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* sb = smem_raw + (base - raw_base);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int qrow = blockIdx.y;  // w * R + r
  const int w = qrow / P.rows;
  const int r = qrow - w * P.rows;
  const int part = w * P.num_splits + split;
  const bool direct = (P.nshards * P.num_splits == 1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kOffBar);
  // barriers: KV_FULL[2], KV_EMPTY[2], S_FULL[2], S_EMPTY[2], P_FULL[2], O_FULL
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int B_KVF = 0, B_KVE = 2, B_SF = 4, B_SE = 6, B_PF = 8, B_OF = 10, B_DRAIN = 11,
            B_ROWS = 12;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 14);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  int* misc_i = reinterpret_cast<int*>(bars + 16);  // [0] request index
  float* qexp = reinterpret_cast<float*>(sb + kOffMisc);  // [32] logit factor per head
  float* lsum = qexp + kH;                                // [32] denominators
  float* Ms = lsum + kH;                                  // [32] running maxima of a
  float* Mn = Ms + kH;                                    // [32] their candidates for a tile
  float* red = reinterpret_cast<float*>(sb + kOffRed);    // [4][32]
  float* ks_s = reinterpret_cast<float*>(sb + kOffKs);    // [2][128] token scales
  int* rows_s = reinterpret_cast<int*>(sb + kOffRows);    // [2][128] cache rows

  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_KVF + i), 64);   // every gather lane (its copies), every scale lane
      mbar_init(bar(B_ROWS + i), 32);  // every gather lane wrote its rows
      mbar_init(bar(B_KVE + i), 1);    // MMA commit after the tile's value product
      mbar_init(bar(B_SF + i), 1);     // MMA commit after S^T
      mbar_init(bar(B_SE + i), kSmx);  // softmax threads read S^T
      mbar_init(bar(B_PF + i), kSmx);  // softmax threads wrote P^T
    }
    mbar_init(bar(B_OF), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    misc_i[0] = -1;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&T.kvmap[w]);
  __syncthreads();
  // request of this row (row_start is an input the previous grid does not write)
  for (int i = tid; i < P.num_reqs; i += kThreads)
    if (__ldg(P.row_start + i) <= r && r < __ldg(P.row_start + i + 1)) misc_i[0] = i;

  // ---- the query: per-head power of two, hi + lo e4m3 terms, K-major SW128
  // [box b][term][head][128 B] (each box's hi and lo rows form one N = 64
  // operand); dims 576..639 of box 4 stay unread
  if (warp >= 4 && warp < 8) {
    const int st = tid - 128;           // 0..127
    const int h = st >> 2, qp = st & 3;  // head, quarter of its 576 dims (144 each)
    const uint16_t* qs = P.q + (static_cast<long long>(r) * kH + h) * kKvDim + qp * 144;
    uint32_t mx = 0;
    for (int i = 0; i < 144; i += 2) {
      const uint32_t two = __ldg(reinterpret_cast<const uint32_t*>(qs + i));
      mx = max(mx, max(two & 0x7FFFu, (two >> 16) & 0x7FFFu));
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // mx: bf16 pattern of the head's largest |q| (exponent bits 7..14)
    const int ebits = static_cast<int>(mx >> 7);
    const int e = (ebits == 0) ? 0 : max(-100, min(100, ((mx & 0x7Fu) <= 0x60u ? 135 : 134) - ebits));
    const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    for (int c = 0; c < 9; ++c) {  // 16 dims per chunk
      const int d0 = qp * 144 + c * 16;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float x = __bfloat162float(__ushort_as_bfloat16(__ldg(qs + c * 16 + 4 * j + b))) * sc;
          const uint32_t ch = e4m3_of(x);
          const uint32_t cl = e4m3_of(x - e4m3_val(ch));
          hw |= ch << (8 * b);
          lw |= cl << (8 * b);
        }
        hi[j] = hw;
        lo[j] = lw;
      }
      const int bx = d0 >> 7, cc = (d0 & 127) >> 4;
      const uint32_t off = static_cast<uint32_t>(bx * 2 * kH * 128 + h * 128 + ((cc ^ (h & 7)) << 4));
      *reinterpret_cast<uint4*>(sb + kOffQ + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sb + kOffQ + kH * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (qp == 0) qexp[h] = P.sm_scale * kLog2e * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    fence_proxy_async_smem();  // the query is read by the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int b = misc_i[0];

  pdl_wait();  // the selections come from the previous grid
  int cnt = __ldcg(P.count + qrow);
  if (cnt < 0 || cnt > P.k) {
    if (tid == 0) raise_err(P.d_err, DSA_DEVERR_INDEX);
    cnt = cnt < 0 ? 0 : P.k;
  }
  const int begin = split * P.chunk;
  const int ntok = max(0, min(cnt, begin + P.chunk) - begin);
  const int ntiles = (ntok + kT - 1) / kT;

  float* out_o = direct ? P.out + static_cast<long long>(r) * kH * kVDim
                        : P.part_out + (static_cast<long long>(part) * P.rows + r) * kH * kVDim;
  float* out_l = direct ? P.out_lse + static_cast<long long>(r) * kH
                        : P.part_lse + (static_cast<long long>(part) * P.rows + r) * kH;

  if (ntiles > 0) {
    if (tid == 0 && b < 0) raise_err(P.d_err, DSA_DEVERR_ROWS);
    if (warp < 4) {
      // ================================================= gather (warps 0..3)
      const int32_t* ilist = P.idx + static_cast<long long>(qrow) * P.k + begin;
      const int32_t* bt = P.block_table[w];
      const int psz = P.page_size;
      const long long span = static_cast<long long>(P.max_blocks[w]) * psz;
      const int oob = P.num_pages[w] * psz;  // a row past the cache: zero-filled
      const bool vec_idx = (reinterpret_cast<uintptr_t>(ilist) & 15u) == 0;
      // lanes 0..7 each own one group per tile: group g = warp + 4 * lane
      const bool active = lane < 8;
      const int g = warp + 4 * lane;
      // selections of the group in tile `tile` (-1: none)
      auto load_idx = [&](int tile, int* t4) {
        const int i0 = tile * kT + 4 * g;
        if (!active || tile >= ntiles) {
          t4[0] = t4[1] = t4[2] = t4[3] = -1;
        } else if (vec_idx && i0 + 3 < ntok) {
          const int4 v = __ldcg(reinterpret_cast<const int4*>(ilist + i0));
          t4[0] = v.x;
          t4[1] = v.y;
          t4[2] = v.z;
          t4[3] = v.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) t4[q] = i0 + q < ntok ? __ldcg(ilist + i0 + q) : -1;
        }
      };
      // page ids of the selections (loads left in flight); -2: bad position
      auto load_pages = [&](const int* t4, int* pg4, int* sl4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int t = t4[q];
          pg4[q] = -1;
          sl4[q] = 0;
          if (t < 0) continue;
          if (b < 0 || static_cast<long long>(t) >= span) {
            pg4[q] = -2;
            continue;
          }
          const int lp = T.page_shift >= 0 ? (t >> T.page_shift) : t / psz;
          sl4[q] = t - lp * psz;
          pg4[q] = bt ? __ldg(bt + static_cast<long long>(b) * P.max_blocks[w] + lp)
                      : b * P.max_blocks[w] + lp;
        }
      };
      int tA[4], tB[4], pgA[4], slA[4];
      load_idx(0, tA);
      load_pages(tA, pgA, slA);
      load_idx(1, tB);
      int issued = 0;
      for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1, use = tile >> 1;
        const bool ok = lane == 0 && use >= 1
                            ? mbar_wait(bar(B_KVE + buf), static_cast<uint32_t>(use - 1) & 1u, abort_flag)
                            : true;
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        if (active) {
          // the rows of this tile (the page loads were issued a tile ago)
          int rows[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int pg = pgA[q];
            rows[q] = oob;
            if (pg == -2 || (tA[q] >= 0 && pg < 0 && pg != -2) || pg >= P.num_pages[w]) {
              raise_err(P.d_err, pg == -2 ? DSA_DEVERR_INDEX : DSA_DEVERR_PAGE);
            } else if (pg >= 0) {
              rows[q] = pg * psz + slA[q];
            }
          }
          const uint32_t full = bar(B_KVF + buf);
          // the rows go to the scale warp, which loads the token scales
          *reinterpret_cast<int4*>(rows_s + buf * kT + 4 * g) =
              make_int4(rows[0] == oob ? -1 : rows[0], rows[1] == oob ? -1 : rows[1],
                        rows[2] == oob ? -1 : rows[2], rows[3] == oob ? -1 : rows[3]);
          mbar_arrive(bar(B_ROWS + buf));
          mbar_arrive_expect_tx(full, kBoxes * 512u);
          const uint32_t dst = base + kOffKV + buf * kTileBytes + g * 512;
#pragma unroll
          for (int bx = 0; bx < kBoxes; ++bx)
            tma_gather4(dst + bx * kBoxBytes, &T.kvmap[w], full, bx * 128, rows[0], rows[1],
                        rows[2], rows[3]);
        }
        ++issued;
        // two tiles ahead: the next tile's page loads, the selections after it
        load_pages(tB, pgA, slA);
#pragma unroll
        for (int q = 0; q < 4; ++q) tA[q] = tB[q];
        load_idx(tile + 2, tB);
      }
      // every issued tile must land before the CTA exits (after an abort the
      // consumers stop waiting for them)
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int tile = max(0, issued - 2); tile < issued; ++tile)
          mbar_wait(bar(B_KVF + (tile & 1)), static_cast<uint32_t>(tile >> 1) & 1u, &no_abort);
      }
    } else if (warp == kScaleWarp) {
      // ================================================= token scales
      // For every tile, once its rows are known: 4 tokens' scales per lane,
      // released to the softmax by the arrival on the tile's full barrier.
      for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        if (!mbar_wait(bar(B_ROWS + buf), static_cast<uint32_t>(tile >> 1) & 1u, abort_flag)) break;
        const int4 rw = *reinterpret_cast<const int4*>(rows_s + buf * kT + 4 * lane);
        const int r4[4] = {rw.x, rw.y, rw.z, rw.w};
        float ks[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) ks[q] = r4[q] >= 0 ? __ldg(P.kscale[w] + r4[q]) : -1.0f;
        *reinterpret_cast<float4*>(ks_s + buf * kT + 4 * lane) = make_float4(ks[0], ks[1], ks[2], ks[3]);
        mbar_arrive(bar(B_KVF + buf));
      }
    } else if (warp == kMmaWarp) {
      // ================================================= MMA issuer
      if (lane == 0) {
        const uint32_t idesc_s = idesc_e4m3(kT, 2 * kH);
        const uint32_t idesc_o = idesc_e4m3(kT, 2 * kH) | (1u << 15);  // A (V^T) MN-major
        const uint64_t q0 = smem_desc_sw128(base + kOffQ);
        auto issue_s = [&](int i) {  // S^T of tile i: 18 K-steps (boxes 0..3: 4, box 4: 2)
          const int buf = i & 1;
          const uint32_t kv = base + kOffKV + buf * kTileBytes;
          const uint32_t d = tmem + 64u * buf;
          int step = 0;
#pragma unroll
          for (int bx = 0; bx < kBoxes; ++bx) {
            const uint64_t a0 = smem_desc_sw128(kv + bx * kBoxBytes);
#pragma unroll
            for (int s = 0; s < (bx < 4 ? 4 : 2); ++s) {
              tc_mma_f8(d, a0 + static_cast<uint64_t>((s * 32) >> 4),
                        q0 + static_cast<uint64_t>((bx * 2 * kH * 128 + s * 32) >> 4), idesc_s,
                        step == 0 ? 0u : 1u);
              ++step;
            }
          }
          tc_commit(bar(B_SF + buf));
        };
        auto issue_pv = [&](int j) {  // O^T += V^T . P^T of tile j
          const int buf = j & 1;
          const uint32_t kv = base + kOffKV + buf * kTileBytes;
          const uint64_t p0 = smem_desc_sw128(base + kOffP + buf * 2 * kPBytes);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint64_t a0 = smem_desc_sw128_mn(kv + m * kBoxBytes);
            const uint32_t d = tmem + kOCol + 64u * m;
#pragma unroll
            for (int s = 0; s < kT / 32; ++s)
              tc_mma_f8(d, a0 + static_cast<uint64_t>((s * 32 * 128) >> 4),
                        p0 + static_cast<uint64_t>((s * 32) >> 4), idesc_o,
                        (j == 0 && s == 0) ? 0u : 1u);
          }
          tc_commit(bar(B_KVE + buf));  // the tile buffer and the P slot are free
        };
        // whichever is ready first: the next S^T (its tile landed, its S slot
        // read) or the next value product (its P written)
        int sn = 0, pn = 0;
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (pn < ntiles) {
          bool did = false;
          if (sn < ntiles) {
            const int buf = sn & 1;
            if (mbar_try_wait(bar(B_KVF + buf), static_cast<uint32_t>(sn >> 1) & 1u) &&
                (sn < 2 || mbar_try_wait(bar(B_SE + buf), static_cast<uint32_t>((sn >> 1) - 1) & 1u))) {
              tc_fence_after();
              issue_s(sn++);
              did = true;
            }
          }
          if (pn < sn && mbar_try_wait(bar(B_PF + (pn & 1)), static_cast<uint32_t>(pn >> 1) & 1u)) {
            tc_fence_after();
            issue_pv(pn++);
            did = true;
          }
          if (did) {
            spins = 0;
            continue;
          }
          if (spins++ == 0) t0 = globaltimer_ns();
          if ((spins & 15u) == 0u) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
              *abort_flag = 1;
              break;
            }
          }
        }
        if (pn == ntiles) tc_commit(bar(B_OF));
        // all MMAs of this thread finish before TMEM is freed
        volatile int no_abort = 0;
        tc_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0u, &no_abort);
      }
    } else {
      // ================================================= softmax (warps 4..11)
      const int st = 32 * (warp & 3) + lane;  // token lane of S^T, TMEM lane of O^T
      const int wq = warp & 3;                // lane quarter
      const int hh = (warp - 4) >> 2;         // head half: heads 16 hh .. 16 hh + 15
      const int sid = tid - 128;              // 0 .. 255
      const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
      // running maxima of a per head in shared memory (the same for every
      // thread); lanes l and l ^ 16 hold the partial denominator of head
      // 16 hh + (l & 15) over the warp's tokens
      if (sid < kH) Ms[sid] = -__int_as_float(0x7f800000);
      float lacc = 0.0f;
      named_bar_sync(1, kSmx);
      // A wait that gives up (the abort flag is set; every later wait then
      // returns at once) does not leave the loop: the eight warps keep passing
      // the same named barriers, compute on whatever is there, and the error
      // word reports it.
      bool ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int buf = i & 1;
        ok &= mbar_wait(bar(B_SF + buf), static_cast<uint32_t>(i >> 1) & 1u, abort_flag);
        // the token's scale (the MMA issuer saw the tile land before S^T)
        ok &= mbar_wait(bar(B_KVF + buf), static_cast<uint32_t>(i >> 1) & 1u, abort_flag);
        const float ks = ks_s[buf * kT + st];
        const bool valid = i * kT + st < ntok && ks >= 0.0f;
        tc_fence_after();
        // a = z + log2(scale), z = sm_scale * scale * (q . code) in base 2
        float a[kHH];
        const float lks = log2f(fmaxf(ks, 7.888609052210118e-31f));  // scale >= 2^-100
        {
          uint32_t vh[kHH], vl[kHH];
          tmem_ld_32x32b_x16(tmem + lane_addr + 64u * buf + kHH * hh, vh);
          tmem_ld_32x32b_x16(tmem + lane_addr + 64u * buf + kH + kHH * hh, vl);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(B_SE + buf));
#pragma unroll
          for (int h = 0; h < kHH; ++h)
            a[h] = valid ? fmaf(__uint_as_float(vh[h]) + __uint_as_float(vl[h]),
                                ks * qexp[kHH * hh + h], lks)
                         : -__int_as_float(0x7f800000);
        }
        // tile maxima of a per head: transpose-reduce in the warp, then over
        // the four lane quarters
        {
          float t[kHH];
#pragma unroll
          for (int h = 0; h < kHH; ++h) t[h] = a[h];
          const float m = warp_transpose_reduce16<true>(t, lane);  // head 16 hh + (lane & 15)
          if (lane < kHH) red[wq * kH + kHH * hh + lane] = m;
        }
        named_bar_sync(1, kSmx);
        // thread h < 32: head h's candidate maximum; whether any head moves
        // past the lazy margin goes to every thread with the barrier
        int up = 0;
        if (sid < kH) {
          const float nm = fmaxf(Ms[sid], fmaxf(fmaxf(red[sid], red[kH + sid]),
                                                fmaxf(red[2 * kH + sid], red[3 * kH + sid])));
          Mn[sid] = nm;
          up = nm > Ms[sid] + kLazy;
        }
        const bool raise = named_bar_or(1, kSmx, up);
        auto new_max = [&](int h) { return Mn[h]; };
        if (raise) {
          // rescale O^T (after the previous tile's value product) and the
          // denominators to the new maxima: this thread's lane, its 16 heads
          if (i >= 1) {
            ok &= mbar_wait(bar(B_KVE + ((i - 1) & 1)), static_cast<uint32_t>((i - 1) >> 1) & 1u,
                            abort_flag);
            tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 8; ++m) {  // block m / 2, hi (even) or lo (odd) terms
              const uint32_t col = kOCol + 64u * (m >> 1) + kH * (m & 1) + kHH * hh;
              uint32_t v[kHH];
              tmem_ld_32x32b_x16(tmem + lane_addr + col, v);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kHH; ++h) {
                const int hg = kHH * hh + h;
                v[h] = __float_as_uint(__uint_as_float(v[h]) * exp2f(Ms[hg] - new_max(hg)));
              }
              tmem_st_32x32b_x16(tmem + lane_addr + col, v);
            }
            tmem_wait_st();
            const int hl = kHH * hh + (lane & 15);
            lacc *= exp2f(Ms[hl] - new_max(hl));
          }
          named_bar_sync(1, kSmx);  // every thread has read the old maxima
          if (sid < kH) Ms[sid] = new_max(sid);
        }
        named_bar_sync(1, kSmx);  // red is read, Ms is final for this tile
        // P^T slot buf is free once the value product of tile i - 2 is done
        if (i >= 2)
          ok &= mbar_wait(bar(B_KVE + buf), static_cast<uint32_t>((i >> 1) - 1) & 1u, abort_flag);
        // P (times 64) as e4m3 hi + lo terms: the K-major SW128 P^T operand,
        // rows 0..31 the hi terms of heads 0..31, rows 32..63 the lo terms;
        // row j holds tokens 0..127, token st at chunk (st / 16) ^ (j & 7)
        uint8_t* p0 = sb + kOffP + buf * 2 * kPBytes;
        const int cst = st >> 4, bst = st & 15;
        {
          float t[kHH];
#pragma unroll
          for (int h = 0; h < kHH; h += 2) {
            const int hg = kHH * hh + h;
            const float pa = exp2f(a[h] - Ms[hg]) * kPScale;
            const float pb = exp2f(a[h + 1] - Ms[hg + 1]) * kPScale;
            t[h] = exp2f(a[h] - lks - Ms[hg]);  // exp2(z - M): the denominator's term
            t[h + 1] = exp2f(a[h + 1] - lks - Ms[hg + 1]);
            const __nv_fp8x2_storage_t c2 =
                __nv_cvt_float2_to_fp8x2(make_float2(pa, pb), __NV_SATFINITE, __NV_E4M3);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c2, __NV_E4M3);
            const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(
                make_float2(pa - back.x, pb - back.y), __NV_SATFINITE, __NV_E4M3);
            const int offa = ((cst ^ (hg & 7)) << 4) + bst;
            const int offb = ((cst ^ ((hg + 1) & 7)) << 4) + bst;
            p0[hg * 128 + offa] = static_cast<uint8_t>(c2 & 0xFFu);
            p0[(hg + 1) * 128 + offb] = static_cast<uint8_t>(c2 >> 8);
            p0[(kH + hg) * 128 + offa] = static_cast<uint8_t>(l2 & 0xFFu);
            p0[(kH + hg + 1) * 128 + offb] = static_cast<uint8_t>(l2 >> 8);
          }
          lacc += warp_transpose_reduce16<false>(t, lane);
        }
        fence_proxy_async_smem();  // P^T is read by the tensor core
        tc_fence_before();
        mbar_arrive(bar(B_PF + buf));
      }
      // ---- denominators: sum the lane quarters' partials
      if (lane < kHH) red[wq * kH + kHH * hh + lane] = lacc;
      named_bar_sync(1, kSmx);
      if (sid < kH) lsum[sid] = (red[sid] + red[kH + sid]) + (red[2 * kH + sid] + red[3 * kH + sid]);
      named_bar_sync(1, kSmx);
      // ---- O = (O^T hi + lo) / 64 / l, LSE = (M + log2 l) ln 2
      const bool got = __all_sync(0xffffffffu, ok) && mbar_wait(bar(B_OF), 0u, abort_flag);
      if (__all_sync(0xffffffffu, got)) {
        tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          uint32_t vh[kHH], vl[kHH];
          tmem_ld_32x32b_x16(tmem + lane_addr + kOCol + 64u * m + kHH * hh, vh);
          tmem_ld_32x32b_x16(tmem + lane_addr + kOCol + 64u * m + kH + kHH * hh, vl);
          tmem_wait_ld();
          const int dim = 128 * m + st;
#pragma unroll
          for (int h = 0; h < kHH; ++h) {
            const int hg = kHH * hh + h;
            const float l = lsum[hg];
            out_o[hg * kVDim + dim] =
                l > 0.0f ? (__uint_as_float(vh[h]) + __uint_as_float(vl[h])) * (1.0f / kPScale) / l : 0.0f;
          }
        }
      }
      if (sid < kH) {
        const float l = lsum[sid];
        out_l[sid] = l > 0.0f ? (Ms[sid] + log2f(l)) * kLn2 : -__int_as_float(0x7f800000);
      }
    }
  } else {
    // an empty split: LSE -inf (and O = 0 when it is the final output)
    for (int h = tid; h < kH; h += kThreads) out_l[h] = -__int_as_float(0x7f800000);
    if (direct)
      for (int i = tid; i < kH * kVDim; i += kThreads) out_o[i] = 0.0f;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) raise_err(P.d_err, DSA_DEVERR_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool sparse_mla_tc_supported(const MlaLaunch& p) {
  return p.fp8 && p.heads == kH && p.out_max == nullptr;
}

cudaError_t launch_sparse_mla_tc(const MlaLaunch& p, cudaStream_t stream, bool pdl) {
  if (p.nshards * p.rows == 0 || p.num_splits == 0) return cudaSuccess;
  MlaTcLaunch T{};
  T.p = p;
  T.page_shift = -1;
  for (int s = 0; s < 31; ++s)
    if (p.page_size == (1 << s)) T.page_shift = s;
  for (int i = 0; i < p.nshards; ++i) {
    cudaError_t e = make_kv_fp8_tmap(&T.kvmap[i], p.kv[i], p.num_pages[i], p.page_size);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.nshards * p.rows);
  return launch_ex(sparse_mla_tc_kernel, grid, dim3(kThreads), kSmemBytes, stream, pdl, T);
}

}  // namespace dsa
