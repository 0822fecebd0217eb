// Absorbed-MLA sparse decode, split-K with LSE.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Modifications / Sparse decode: every (shard of a) query row attends only
// its selected latent rows with a split-K kernel that also returns the
// natural-log LSE; the commit "store a lone split's output and LSE in place":
// with a single split the partial is the final result and goes straight to
// the caller's output.
//
// One CTA per (work row, split), 10 warps.  Warps 8-9 gather 64-token tiles
// of 576-wide latent rows into a double buffer, one bulk copy per selected row
// (selection -> block table -> row, resolved one tile ahead), each landing on
// the tile's mbarrier, so the gather runs while warps 0-7 compute on the
// previous tile; fp8 rows land raw and are widened to f16 by the compute warps
// (e4m3 values are f16 values).  Every head of the row shares each gathered
// tile:
//   S = q . kv^T (all 576 dims), online softmax in fp32 (base 2), P split into
//   two bf16 parts (f16 for fp8 rows), O += P . v (first 512 dims).
// With bf16 rows and 32 heads the compute warps form two groups of 16 heads
// that take turns on S, so that one group's S (shared-memory reads) overlaps
// the other's P . v (tensor pipe).
// The fp8 path multiplies each logit by the token's scale and folds the scale
// into P for the value product; its query is converted to f16 with a per-head
// power-of-two factor that the logit scale undoes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kCompute = 256;                 // warps 0..7: tensor-core math
constexpr int kGather = 64;                   // warps 8..9: the row gather
constexpr int kThreads = kCompute + kGather;
constexpr int kTile = 64;                 // tokens per tile
constexpr int kRowB = kKvDim * 2 + 16;    // padded smem row of 576 16-bit values
constexpr int kPRowB = kTile * 2 + 16;    // padded smem row of P
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MlaSmem {
  int off_q, off_kv, off_raw, off_p, off_red, off_kscale, off_misc, off_bt, off_bar, total;
  int kv_bufs;
};

// bt_ints: entries of a request's block-table row kept in shared memory (0:
// the gather reads the global table)
__host__ __device__ inline MlaSmem mla_smem(int heads, int fp8, int chunk, int bt_ints = 0) {
  MlaSmem s{};
  int off = 0;
  s.off_q = off;
  off += heads * kRowB;
  s.kv_bufs = fp8 ? 1 : 2;
  s.off_kv = off;
  off += s.kv_bufs * kTile * kRowB;
  s.off_raw = off;
  off += fp8 ? 2 * kTile * kKvDim : 0;
  s.off_p = off;
  off += (fp8 ? 1 : 2) * heads * kPRowB;  // bf16 path: P = hi + lo
  s.off_red = off;
  off += 2 * 8 * heads * 4;
  s.off_kscale = off;
  off += fp8 ? chunk * 4 : 0;
  s.off_misc = off;
  off += 64 * 4 + heads * 4;
  s.off_bt = off;
  off += bt_ints * 4;
  off = (off + 15) & ~15;
  s.off_bar = off;  // mbarriers: full[2], empty[2], abort flag
  off += 64;
  s.total = off;
  return s;
}


DSA_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
DSA_DEV void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
DSA_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// arrive on named barrier `id` (of `nthreads` threads) without waiting
DSA_DEV void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <bool kF16>
DSA_DEV void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                      uint32_t b1) {
  if (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <bool kF16>
DSA_DEV uint32_t pack2(float lo, float hi) {
  if (kF16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// H heads (16 or 32); kFp8: e4m3 cache, f16 MMAs; else bf16 cache and MMAs.
template <int H, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const MlaLaunch P) {
  // The compute warps form kGroups groups, each owning H / kGroups heads with
  // its own online softmax and O.  Two groups (bf16, 32 heads) take turns on
  // S = q.kv^T, which is bound by shared-memory reads, so that one group's S
  // runs while the other's O += P.v keeps the tensor pipe busy.  The fp8 path
  // (one widened tile buffer) and 16 heads (one m16 tile) use one group.
  constexpr int kGroups = (!kFp8 && H == 32) ? 2 : 1;
  constexpr int kGW = (kCompute / 32) / kGroups;  // warps per group
  constexpr int MT = H / kGroups / 16;   // m16 tiles of the group's heads
  constexpr int TGS = kGW / MT;          // token groups of S
  constexpr int NTW = 8 / TGS;           // n8 token tiles per warp in S
  constexpr int DW = kVDim / kGW;        // value dims per warp in O += P.v
  extern __shared__ __align__(16) uint8_t smem[];
  const MlaSmem S = mla_smem(H, kFp8, P.chunk, P.bt_smem);
  uint8_t* q_s = smem + S.off_q;
  int* bt_s = reinterpret_cast<int*>(smem + S.off_bt);
  uint8_t* kv_s = smem + S.off_kv;
  uint8_t* raw_s = smem + S.off_raw;
  uint8_t* p_s = smem + S.off_p;
  float* red = reinterpret_cast<float*>(smem + S.off_red);      // [2][TGS][H]
  float* kscale_s = reinterpret_cast<float*>(smem + S.off_kscale);
  int* misc = reinterpret_cast<int*>(smem + S.off_misc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S.off_bar);  // full[2], empty[2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4);
  float* qexp = reinterpret_cast<float*>(smem + S.off_misc + 64 * 4);  // [H] logit scales

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int split = blockIdx.x;
  const int qrow = blockIdx.y;                 // w * R + r
  const int w = qrow / P.rows;
  const int r = qrow - w * P.rows;
  const int part = w * P.num_splits + split;
  const bool direct = (P.nshards * P.num_splits == 1);

  pdl_trigger();
  // The query and the row's request are inputs that the previous grid (when
  // this grid is its programmatic dependent) does not write: they are fetched
  // while it finishes.  The bf16 query copy stays in flight meanwhile.
  const uint16_t* qsrc = P.q + static_cast<long long>(r) * H * kKvDim;
  if (!kFp8 && tid < kCompute) {
    for (int c = tid; c < H * 72; c += kCompute) {
      const int h = c / 72, cc = c - h * 72;
      cp_async16(smem_u32(q_s + h * kRowB + cc * 16), qsrc + h * kKvDim + cc * 8);
    }
    cp_async_commit();
  }

  // request of this row: the one i with row_start[i] <= r < row_start[i + 1]
  // (row_start is non-decreasing, so at most one non-empty request matches)
  if (tid == 0) misc[0] = -1;
  __syncthreads();
  for (int i = tid; i < P.num_reqs; i += kThreads) {
    if (__ldg(P.row_start + i) <= r && r < __ldg(P.row_start + i + 1)) misc[0] = i;
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(bars + i), kGather);   // tile landed: every gather thread's copies
      mbar_init(smem_u32(bars + 2 + i), kGroups);  // buffer free: one thread per group
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();  // the request index and the barriers
  const int b = misc[0];
  // the request's block-table row (an input the previous grid does not write)
  const bool bt_smem = P.bt_smem > 0 && b >= 0 && P.block_table[w] != nullptr;
  if (bt_smem) {
    const int32_t* row = P.block_table[w] + static_cast<long long>(b) * P.max_blocks[w];
    for (int j = tid; j < P.max_blocks[w]; j += kThreads) bt_s[j] = __ldg(row + j);
  }
  __syncthreads();
  pdl_wait();  // the selections come from the previous grid

  // a gather thread's first selection is loaded together with the count
  const int gt0 = tid - kCompute;
  const int t_first = (warp >= kCompute / 32 && split * P.chunk + gt0 < P.k)
                          ? __ldcg(P.idx + static_cast<long long>(qrow) * P.k + split * P.chunk + gt0)
                          : -1;
  int cnt = __ldcg(P.count + qrow);
  if (cnt < 0 || cnt > P.k) {
    if (tid == 0) raise_err(P.d_err, DSA_DEVERR_INDEX);
    cnt = cnt < 0 ? 0 : P.k;
  }
  const int begin = split * P.chunk;
  const int ntok = max(0, min(cnt, begin + P.chunk) - begin);

  float* out_o = direct ? P.out + static_cast<long long>(r) * H * kVDim
                        : P.part_out + (static_cast<long long>(part) * P.rows + r) * H * kVDim;
  float* out_l = direct ? P.out_lse + static_cast<long long>(r) * H
                        : P.part_lse + (static_cast<long long>(part) * P.rows + r) * H;
  // the largest scaled logit, when the caller asks for it
  float* out_m = P.out_max == nullptr ? nullptr
                 : direct ? P.out_max + static_cast<long long>(r) * H
                          : P.part_max + (static_cast<long long>(part) * P.rows + r) * H;
  if (ntok == 0) {
    for (int h = tid; h < H; h += kThreads) {
      out_l[h] = -__int_as_float(0x7f800000);
      if (out_m) out_m[h] = -__int_as_float(0x7f800000);
    }
    if (direct)
      for (int i = tid; i < H * kVDim; i += kThreads) out_o[i] = 0.0f;
    if (!kFp8 && tid < kCompute) cp_async_wait<0>();  // no copy may land after the CTA leaves
    return;
  }

  if (tid == 0 && b < 0) raise_err(P.d_err, DSA_DEVERR_ROWS);
  const uint8_t* kvbase = static_cast<const uint8_t*>(P.kv[w]);
  const int ntiles = (ntok + kTile - 1) / kTile;

  if (warp >= kCompute / 32) {
    // ================================================= row gather (warps 8, 9)
    // Tile i goes to buffer i & 1 once the compute warps have released it.
    // Each of the 64 threads moves one selected latent row with one bulk copy
    // (the copy engine takes whole rows; scattered 16-byte copies were bound
    // by their issue rate) and arrives on the tile's barrier with the bytes it
    // expects; a row past the split is zero-filled before the arrival.
    // Every thread resolves its own row of the next tile (selection ->
    // block table -> element offset, and the fp8 token scale) right after it
    // issues the current tile's copy, while the compute warps work.
    const int gt = tid - kCompute;  // the tile row this thread moves
    constexpr uint32_t kRowBytes = kFp8 ? kKvDim : kKvDim * 2;
    const int32_t* ilist = P.idx + static_cast<long long>(qrow) * P.k + begin;
    const int32_t* bt = P.block_table[w];
    const int psz = P.page_size;
    const long long span = static_cast<long long>(P.max_blocks[w]) * psz;
    auto resolve = [&](int tile, long long& off, float& ks) {
      off = -1;
      ks = 0.0f;
      const int i = tile * kTile + gt;
      if (tile >= ntiles || i >= ntok) return;  // no row: zero-filled
      const int t = tile == 0 ? t_first : __ldcg(ilist + i);
      if (b < 0 || t < 0 || static_cast<long long>(t) >= span) {
        raise_err(P.d_err, DSA_DEVERR_INDEX);
        return;
      }
      const int lp = t / psz;
      const int pg = bt_smem ? bt_s[lp]
                     : bt ? __ldg(bt + static_cast<long long>(b) * P.max_blocks[w] + lp)
                          : b * P.max_blocks[w] + lp;
      if (pg < 0 || pg >= P.num_pages[w]) {
        raise_err(P.d_err, DSA_DEVERR_PAGE);
        return;
      }
      off = static_cast<long long>(pg) * psz + (t - lp * psz);
      if (kFp8) ks = __ldg(P.kscale[w] + off);
    };
    long long off_next;
    float ks_next;
    resolve(0, off_next, ks_next);
    int issued = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int buf = tile & 1, use = tile >> 1;
      if (use >= 1 &&
          !mbar_wait(smem_u32(bars + 2 + buf), static_cast<uint32_t>(use - 1) & 1u, abort_flag))
        break;
      const int t0 = tile * kTile;
      const uint32_t full = smem_u32(bars + buf);
      const long long off = off_next;
      if (kFp8 && t0 + gt < ntok) kscale_s[t0 + gt] = ks_next;  // read after the tile's barrier
      uint8_t* dst = kFp8 ? raw_s + buf * kTile * kKvDim + gt * kKvDim
                          : kv_s + buf * kTile * kRowB + gt * kRowB;
      if (off >= 0) {
        mbar_arrive_expect_tx(full, kRowBytes);
        bulk_copy_g2s(smem_u32(dst), kvbase + off * kRowBytes, kRowBytes, full);
      } else {
        for (uint32_t c = 0; c < kRowBytes; c += 16)
          *reinterpret_cast<uint4*>(dst + c) = make_uint4(0u, 0u, 0u, 0u);
        mbar_arrive(full);
      }
      ++issued;
      resolve(tile + 1, off_next, ks_next);
    }
    // after an abort the compute warps stop waiting: every copy still in
    // flight must land before the CTA exits
    if (*abort_flag) {
      volatile int no_abort = 0;
      for (int tile = max(0, issued - 2); tile < issued; ++tile)
        mbar_wait(smem_u32(bars + (tile & 1)), static_cast<uint32_t>(tile >> 1) & 1u, &no_abort);
    }
  } else {
    // ================================================= compute (warps 0..7)
    // bf16: wait for the query copy.  fp8: the query as f16 with a per-head
    // power of two; every warp loads all of its heads before converting any
    if (!kFp8) {
      cp_async_wait<0>();
      if (tid < H) qexp[tid] = P.sm_scale * kLog2e;
    } else {
      constexpr int kHpw = H / (kCompute / 32);  // heads per warp
      uint32_t qv[kHpw][kKvDim / 64];
#pragma unroll
      for (int x = 0; x < kHpw; ++x) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(qsrc + (warp + x * 8) * kKvDim);
#pragma unroll
        for (int j = 0; j < kKvDim / 64; ++j) qv[x][j] = __ldg(src + lane + 32 * j);
      }
#pragma unroll
      for (int x = 0; x < kHpw; ++x) {
        const int h = warp + x * 8;
        uint32_t mx = 0;
#pragma unroll
        for (int j = 0; j < kKvDim / 64; ++j)
          mx = max(mx, max(qv[x][j] & 0x7FFFu, (qv[x][j] >> 16) & 0x7FFFu));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int ebits = static_cast<int>(mx >> 7);
        const int e = (ebits == 0) ? 0 : max(-100, min(100, 141 - ebits));
        const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
        for (int j = 0; j < kKvDim / 64; ++j) {
          const uint32_t two = qv[x][j];
          const float lo = __uint_as_float(two << 16) * sc;
          const float hi = __uint_as_float(two & 0xFFFF0000u) * sc;
          *reinterpret_cast<uint32_t*>(q_s + h * kRowB + (lane + 32 * j) * 4) = pack2<true>(lo, hi);
        }
        if (lane == 0)
          qexp[h] = P.sm_scale * kLog2e * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      }
    }
    named_bar_sync(1, kCompute);  // the query is in shared memory
    const int grp = warp / kGW, wg = warp - grp * kGW;  // group, warp within it
    const int mt0 = grp * MT;                           // the group's first head tile
    // the group's barrier (id 1 when a single group spans all compute warps)
    const int gbar = kGroups == 1 ? 1 : 2 + grp;
    // per-thread state: O accumulators for dims [DW*wg, DW*wg+DW) of the group's heads
    float o[MT][DW / 8][4];
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
      for (int j = 0; j < DW / 8; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[a][j][c] = 0.0f;
    float m_run[MT][2];
#pragma unroll
    for (int a = 0; a < MT; ++a) m_run[a][0] = m_run[a][1] = -__int_as_float(0x7f800000);
    float l_part[2] = {0.0f, 0.0f};  // row sums of this thread's S rows

    const int ml_s = wg % MT;            // S role: head tile within the group
    const int mt_s = mt0 + ml_s;         // S role: head tile
    const int tg = wg / MT;              // S role: token group
    const int n_s0 = tg * (8 * NTW);     // first token of the group in the tile
    const float qsc0 = qexp[mt_s * 16 + g];
    const float qsc1 = qexp[mt_s * 16 + g + 8];
    // S turns: group 0 computes S of tile i once group 1 is done with S of
    // tile i - 1 (barrier 4), group 1 once group 0 is done with S of tile i
    // (barrier 5); group 1's first arrival opens group 0's first turn
    if (kGroups == 2 && grp == 1) named_bar_arrive(4, kCompute);

    for (int tile = 0; tile < ntiles; ++tile) {
      const int fb = tile & 1;  // the gathered tile's buffer (raw rows for fp8)
      // a timed-out wait (abort flag set) computes on whatever is there; the
      // error word reports it and every barrier below is still passed
      mbar_wait(smem_u32(bars + fb), static_cast<uint32_t>(tile >> 1) & 1u, abort_flag);
      const int buf = kFp8 ? 0 : fb;
      uint8_t* kv = kv_s + buf * kTile * kRowB;
      if (kFp8) {
        const uint8_t* rawp = raw_s + fb * kTile * kKvDim;
        for (int c = tid; c < kTile * 72; c += kCompute) {
          const int row = c / 72, cc = c - row * 72;
          const uint2 v = *reinterpret_cast<const uint2*>(rawp + row * kKvDim + cc * 8);
          uint4 out;
          __half2_raw h;
          h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v.x & 0xFFFFu), __NV_E4M3);
          out.x = h.x | (static_cast<uint32_t>(h.y) << 16);
          h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v.x >> 16), __NV_E4M3);
          out.y = h.x | (static_cast<uint32_t>(h.y) << 16);
          h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v.y & 0xFFFFu), __NV_E4M3);
          out.z = h.x | (static_cast<uint32_t>(h.y) << 16);
          h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v.y >> 16), __NV_E4M3);
          out.w = h.x | (static_cast<uint32_t>(h.y) << 16);
          *reinterpret_cast<uint4*>(kv + row * kRowB + cc * 16) = out;
        }
        named_bar_sync(1, kCompute);
        if (tid == 0) mbar_arrive(smem_u32(bars + 2 + fb));  // the raw buffer is free
      }
      const int t0 = tile * kTile;
      const uint32_t kv_a = smem_u32(kv);
      const uint32_t q_a = smem_u32(q_s);
      if (kGroups == 2) named_bar_sync(4 + grp, kCompute);  // this group's S turn

      // ---- S = q . kv^T for head tile mt_s, tokens n_s0 .. n_s0 + 8*NTW
      // Software-pipelined: the fragments of step kk + 1 are requested before
      // the MMAs of step kk issue (the asm statements keep program order), and
      // even and odd steps accumulate into separate registers so that no MMA
      // waits for the one just before it.
      float sacc[NTW][4];
      {
        float sacc2[2][NTW][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int j = 0; j < NTW; ++j)
            sacc2[h2][j][0] = sacc2[h2][j][1] = sacc2[h2][j][2] = sacc2[h2][j][3] = 0.0f;
        const uint32_t a_addr = q_a + (mt_s * 16 + (lane & 15)) * kRowB + (lane >> 4) * 16;
        const uint32_t b_addr =
            NTW == 2 ? kv_a + (n_s0 + (lane & 7) + ((lane >> 4) << 3)) * kRowB + ((lane >> 3) & 1) * 16
                     : kv_a + (n_s0 + (lane & 7)) * kRowB + ((lane >> 3) & 1) * 16;
        uint32_t fa[2][4], fb[2][4];
        auto load_step = [&](int kk, int sl) {
          ldsm_x4(a_addr + kk * 32, fa[sl][0], fa[sl][1], fa[sl][2], fa[sl][3]);
          if (NTW == 2)
            ldsm_x4(b_addr + kk * 32, fb[sl][0], fb[sl][1], fb[sl][2], fb[sl][3]);
          else
            ldsm_x2(b_addr + kk * 32, fb[sl][0], fb[sl][1]);
        };
        load_step(0, 0);
#pragma unroll
        for (int kk = 0; kk < kKvDim / 16; ++kk) {
          const int sl = kk & 1;
          if (kk + 1 < kKvDim / 16) load_step(kk + 1, sl ^ 1);
          mma16816<kFp8>(sacc2[sl][0], fa[sl][0], fa[sl][1], fa[sl][2], fa[sl][3], fb[sl][0], fb[sl][1]);
          if (NTW == 2)
            mma16816<kFp8>(sacc2[sl][NTW - 1], fa[sl][0], fa[sl][1], fa[sl][2], fa[sl][3], fb[sl][2],
                           fb[sl][3]);
        }
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c) sacc[j][c] = sacc2[0][j][c] + sacc2[1][j][c];
      }
      // the other group's S turn (group 1 opens no turn after its last tile)
      if (kGroups == 2 && !(grp == 1 && tile + 1 == ntiles)) named_bar_arrive(5 - grp, kCompute);
      // logits in base 2, masked past the split's end
      float mx0 = -__int_as_float(0x7f800000), mx1 = mx0;
#pragma unroll
      for (int j = 0; j < NTW; ++j) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tok = n_s0 + 8 * j + 2 * t4 + c;
          const bool ok = t0 + tok < ntok;
          float ks = 1.0f;
          if (kFp8) ks = ok ? kscale_s[t0 + tok] : 0.0f;
          const float z0 = ok ? sacc[j][c] * qsc0 * ks : -__int_as_float(0x7f800000);
          const float z1 = ok ? sacc[j][2 + c] * qsc1 * ks : -__int_as_float(0x7f800000);
          sacc[j][c] = z0;
          sacc[j][2 + c] = z1;
          mx0 = fmaxf(mx0, z0);
          mx1 = fmaxf(mx1, z1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      if (t4 == 0) {
        red[tg * H + mt_s * 16 + g] = mx0;
        red[tg * H + mt_s * 16 + g + 8] = mx1;
      }
      named_bar_sync(gbar, kGW * 32);
      // new running max for every head row this thread touches
      float alpha[MT][2];
#pragma unroll
      for (int a = 0; a < MT; ++a) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = (mt0 + a) * 16 + g + hh * 8;
          float tm = red[h];
#pragma unroll
          for (int x = 1; x < TGS; ++x) tm = fmaxf(tm, red[x * H + h]);
          const float mn = fmaxf(m_run[a][hh], tm);
          const float msafe = (mn == -__int_as_float(0x7f800000)) ? 0.0f : mn;
          alpha[a][hh] = exp2f(m_run[a][hh] - msafe);
          m_run[a][hh] = mn;
        }
      }
      // P for the S rows of this warp
      {
        const float mA = (m_run[ml_s][0] == -__int_as_float(0x7f800000)) ? 0.0f : m_run[ml_s][0];
        const float mB = (m_run[ml_s][1] == -__int_as_float(0x7f800000)) ? 0.0f : m_run[ml_s][1];
        float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
        for (int j = 0; j < NTW; ++j) {
          const int tok = n_s0 + 8 * j + 2 * t4;
          const float p00 = exp2f(sacc[j][0] - mA), p01 = exp2f(sacc[j][1] - mA);
          const float p10 = exp2f(sacc[j][2] - mB), p11 = exp2f(sacc[j][3] - mB);
          ls0 += p00 + p01;
          ls1 += p10 + p11;
          float v00 = p00, v01 = p01, v10 = p10, v11 = p11;
          if (kFp8) {
            const float k0 = (t0 + tok < ntok) ? kscale_s[t0 + tok] : 0.0f;
            const float k1 = (t0 + tok + 1 < ntok) ? kscale_s[t0 + tok + 1] : 0.0f;
            v00 *= k0;
            v01 *= k1;
            v10 *= k0;
            v11 *= k1;
          }
          const uint32_t h0 = pack2<kFp8>(v00, v01), h1 = pack2<kFp8>(v10, v11);
          *reinterpret_cast<uint32_t*>(p_s + (mt_s * 16 + g) * kPRowB + tok * 2) = h0;
          *reinterpret_cast<uint32_t*>(p_s + (mt_s * 16 + g + 8) * kPRowB + tok * 2) = h1;
          if (!kFp8) {
            // bf16 keeps 8 significant bits: carry the rounding remainder of P
            // in a second bf16 operand so that P . v is exact to ~2^-17
            *reinterpret_cast<uint32_t*>(p_s + (H + mt_s * 16 + g) * kPRowB + tok * 2) =
                pack2<false>(v00 - __uint_as_float(h0 << 16), v01 - __uint_as_float(h0 & 0xFFFF0000u));
            *reinterpret_cast<uint32_t*>(p_s + (H + mt_s * 16 + g + 8) * kPRowB + tok * 2) =
                pack2<false>(v10 - __uint_as_float(h1 << 16), v11 - __uint_as_float(h1 & 0xFFFF0000u));
          }
        }
        l_part[0] = l_part[0] * alpha[ml_s][0] + ls0;
        l_part[1] = l_part[1] * alpha[ml_s][1] + ls1;
      }
      named_bar_sync(gbar, kGW * 32);

      // ---- O += P . v for value dims [DW*wg, DW*wg + DW) of the group's heads
#pragma unroll
      for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int j = 0; j < DW / 8; ++j) {
          o[a][j][0] *= alpha[a][0];
          o[a][j][1] *= alpha[a][0];
          o[a][j][2] *= alpha[a][1];
          o[a][j][3] *= alpha[a][1];
        }
      {
        // 4 token slices x DW / 16 pairs of 8-dim column tiles, each step's
        // fragments requested one step ahead; the hi terms of P issue before
        // the lo terms so that no MMA waits for its accumulator
        constexpr int kJP = DW / 16;  // column-tile pairs per token slice
        const uint32_t p_a = smem_u32(p_s) + (mt0 * 16 + (lane & 15)) * kPRowB + (lane >> 4) * 16;
        const uint32_t v_a =
            kv_a + ((lane & 7) + ((lane >> 3) & 1) * 8) * kRowB + (wg * DW + (lane >> 4) * 8) * 2;
        uint32_t af[2][MT][4], al[2][MT][4], bv[2][4];
        auto load_p = [&](int kk, int sl) {
#pragma unroll
          for (int a = 0; a < MT; ++a) {
            ldsm_x4(p_a + a * 16 * kPRowB + kk * 32, af[sl][a][0], af[sl][a][1], af[sl][a][2],
                    af[sl][a][3]);
            if (!kFp8)
              ldsm_x4(p_a + (H + a * 16) * kPRowB + kk * 32, al[sl][a][0], al[sl][a][1],
                      al[sl][a][2], al[sl][a][3]);
          }
        };
        auto load_v = [&](int st, int sl) {
          const int kk = st / kJP, jp = st % kJP;
          ldsm_x4_t(v_a + kk * 16 * kRowB + jp * 32, bv[sl][0], bv[sl][1], bv[sl][2], bv[sl][3]);
        };
        load_p(0, 0);
        load_v(0, 0);
#pragma unroll
        for (int st = 0; st < (kTile / 16) * kJP; ++st) {
          const int kk = st / kJP, j = (st % kJP) * 2, sv = st & 1, sp = kk & 1;
          if (st + 1 < (kTile / 16) * kJP) {
            if ((st + 1) % kJP == 0) load_p(kk + 1, sp ^ 1);
            load_v(st + 1, sv ^ 1);
          }
#pragma unroll
          for (int a = 0; a < MT; ++a) {
            mma16816<kFp8>(o[a][j], af[sp][a][0], af[sp][a][1], af[sp][a][2], af[sp][a][3],
                           bv[sv][0], bv[sv][1]);
            mma16816<kFp8>(o[a][j + 1], af[sp][a][0], af[sp][a][1], af[sp][a][2], af[sp][a][3],
                           bv[sv][2], bv[sv][3]);
          }
          if (!kFp8) {
#pragma unroll
            for (int a = 0; a < MT; ++a) {
              mma16816<false>(o[a][j], al[sp][a][0], al[sp][a][1], al[sp][a][2], al[sp][a][3],
                              bv[sv][0], bv[sv][1]);
              mma16816<false>(o[a][j + 1], al[sp][a][0], al[sp][a][1], al[sp][a][2],
                              al[sp][a][3], bv[sv][2], bv[sv][3]);
            }
          }
        }
      }
      named_bar_sync(gbar, kGW * 32);
      // the tile's buffer is free once every group is past it
      if (!kFp8 && wg == 0 && lane == 0) mbar_arrive(smem_u32(bars + 2 + fb));
    }

    // ---- softmax denominators: sum the row partials over t4 and token groups
    float l0 = l_part[0], l1 = l_part[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    float* red2 = red + TGS * H;
    if (t4 == 0) {
      red2[tg * H + mt_s * 16 + g] = l0;
      red2[tg * H + mt_s * 16 + g + 8] = l1;
    }
    named_bar_sync(gbar, kGW * 32);
    const int d0 = wg * DW;
#pragma unroll
    for (int a = 0; a < MT; ++a) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = (mt0 + a) * 16 + g + hh * 8;
        float l = 0.0f;
#pragma unroll
        for (int x = 0; x < TGS; ++x) l += red2[x * H + h];
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
        for (int j = 0; j < DW / 8; ++j) {
          float2 v = make_float2(o[a][j][2 * hh] * inv, o[a][j][2 * hh + 1] * inv);
          *reinterpret_cast<float2*>(out_o + h * kVDim + d0 + 8 * j + 2 * t4) = v;
        }
        if (wg == 0 && t4 == 0) {
          out_l[h] = l > 0.0f ? (m_run[a][hh] + log2f(l)) * kLn2 : -__int_as_float(0x7f800000);
          // m_run is the largest logit in base 2 (tau * q.kv * log2 e)
          if (out_m) out_m[h] = l > 0.0f ? m_run[a][hh] * kLn2 : -__int_as_float(0x7f800000);
        }
      }
    }
  }

  __syncthreads();
  if (tid == 0 && *abort_flag) raise_err(P.d_err, DSA_DEVERR_TIMEOUT);
}

template <int H, bool F>
cudaError_t launch_one(const MlaLaunch& p, cudaStream_t stream, bool pdl) {
  const MlaSmem S = mla_smem(H, F, p.chunk, p.bt_smem);
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel<H, F>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, S.total);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.nshards * p.rows);
  return launch_ex(sparse_mla_kernel<H, F>, grid, dim3(kThreads), S.total, stream, pdl, p);
}

}  // namespace

int mla_smem_bytes(int heads, int fp8, int chunk) { return mla_smem(heads, fp8, chunk).total; }

int auto_mla_splits(int work_rows, int k, int expected_count) {
  // aim for about one CTA per SM; splits are whole 64-token tiles
  const int sms = num_sms() > 0 ? num_sms() : 148;
  int target = sms / (work_rows > 0 ? work_rows : 1);
  if (target < 1) target = 1;
  int per = (expected_count + target - 1) / target;
  per = ((per + kTile - 1) / kTile) * kTile;
  if (per < kTile) per = kTile;
  int s = (k + per - 1) / per;
  if (s < 1) s = 1;
  return s;
}

cudaError_t launch_sparse_mla(const MlaLaunch& p0, cudaStream_t stream, bool pdl) {
  if (p0.nshards * p0.rows == 0 || p0.num_splits == 0) return cudaSuccess;
  if (sparse_mla_tc_supported(p0)) return launch_sparse_mla_tc(p0, stream, pdl);
  // keep a request's block-table row in shared memory when it is short
  // enough and fits beside the tiles
  MlaLaunch p = p0;
  int maxb = 0;
  for (int i = 0; i < p.nshards; ++i)
    if (p.block_table[i] != nullptr && p.max_blocks[i] > maxb) maxb = p.max_blocks[i];
  constexpr int kBtSmemCap = 4096;
  p.bt_smem = (maxb > 0 && maxb <= kBtSmemCap &&
               mla_smem(p.heads, p.fp8, p.chunk, maxb).total <= 227 * 1024)
                  ? maxb
                  : 0;
  if (p.heads == 16)
    return p.fp8 ? launch_one<16, true>(p, stream, pdl) : launch_one<16, false>(p, stream, pdl);
  if (p.heads == 32)
    return p.fp8 ? launch_one<32, true>(p, stream, pdl) : launch_one<32, false>(p, stream, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
