// One decode step's cache write: RoPE on the new tokens' rows, fp8
// quantization for fp8 caches, and the owner-rule placement into the shard
// caches, in one launch.
//
// "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2",
// Modifications / Writes: MLA KV and indexer K land only on the owner rank
// (slot % W == rank); the page lists a fused RoPE + KV-cache write kernel,
// and its decode-gap analysis traces hundreds of small kernels per step to
// computing the owner-rule write location outside the write kernels.  Here
// the location is derived in the kernel from (request, position, W).
//
// Two warps per token, four tokens per CTA: the even warp writes the
// 576-wide latent row, the odd one the 128-wide index-K row.  Lane l holds
// the bf16 pairs l, l + 32, ...; its last pair is RoPE pair l (the rope dims
// are the last 64 of each row).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTokPerCta = 4;
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;

// Shard cache `w` of a launch: where token (req, pos) lives, or -1 (and an
// error bit) when the request, position or page is out of range.
__device__ long long owner_row(const CacheWriteSide& c, int w, int req, int p,
                               int page_size, int32_t* d_err) {
  const int lp = p / page_size;
  if (lp >= c.max_blocks[w]) {
    raise_err(d_err, DSA_DEVERR_POS);
    return -1;
  }
  const long long bi = static_cast<long long>(req) * c.max_blocks[w] + lp;
  const int pg = c.block_table[w] ? __ldg(c.block_table[w] + bi) : static_cast<int>(bi);
  if (pg < 0 || pg >= c.num_pages[w]) {
    raise_err(d_err, DSA_DEVERR_PAGE);
    return -1;
  }
  return static_cast<long long>(pg) * page_size + (p - lp * page_size);
}

// RoPE, rounding / quantization and the store of one D-wide row by one warp.
template <int D>
__device__ void write_row(const uint16_t* in, int pos, double theta, int fp8, void* data,
                          float* scale, long long row, int lane) {
  constexpr int kPer = D / 64;          // bf16 pairs per lane
  constexpr int kRope0 = (D - 64) / 2;  // first rope pair
  float2 v[kPer];
  const uint32_t* src = reinterpret_cast<const uint32_t*>(in);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const uint32_t wd = __ldg(src + lane + 32 * j);
    v[j] = make_float2(__uint_as_float(wd << 16), __uint_as_float(wd & 0xFFFF0000u));
  }
  {
    // the lane's rope pair i = lane: angle pos * base^(-i/32), formed and
    // reduced by 2 pi in double (a few double operations) so that long
    // positions keep their phase
    const double a0 = static_cast<double>(pos) * theta;
    const double a = fma(-floor(a0 * kInvTwoPi), kTwoPi, a0);
    float sn, cs;
    sincosf(static_cast<float>(a), &sn, &cs);
    const float2 x = v[kPer - 1];
    v[kPer - 1] = make_float2(x.x * cs - x.y * sn, x.x * sn + x.y * cs);
  }
  static_assert(kRope0 == 32 * (kPer - 1), "the last pair of every lane is a rope pair");
  if (!fp8) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(data) + row * D);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[j].x, v[j].y);
      dst[lane + 32 * j] = *reinterpret_cast<const uint32_t*>(&b);
    }
  } else {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) amax = fmaxf(amax, fmaxf(fabsf(v[j].x), fabsf(v[j].y)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    uint16_t* dst = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(data) + row * D);
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      dst[lane + 32 * j] = static_cast<uint16_t>(
          __nv_cvt_float2_to_fp8x2(make_float2(v[j].x / s, v[j].y / s), __NV_SATFINITE, __NV_E4M3));
    if (lane == 0) scale[row] = s;
  }
}

__global__ void __launch_bounds__(64 * kTokPerCta) cache_write_kernel(const CacheWriteLaunch P) {
  const int lane = threadIdx.x & 31;
  const int warp = (threadIdx.x >> 5) & 1;  // 0: latent row, 1: index-K row
  const int j = blockIdx.x * kTokPerCta + (threadIdx.x >> 6);
  if (j >= P.num_tokens || (warp == 1 && P.idx_in == nullptr)) return;
  const int req = __ldg(P.tok_req + j);
  const int pos = __ldg(P.tok_pos + j);
  if (req < 0 || req >= P.num_reqs) {
    if (lane == 0) raise_err(P.d_err, DSA_DEVERR_ROWS);
    return;
  }
  if (pos < 0) {
    if (lane == 0) raise_err(P.d_err, DSA_DEVERR_POS);
    return;
  }
  const int w = pos % P.W;  // the owner shard and the local position there
  const int p = pos / P.W;
  const CacheWriteSide& c = warp == 0 ? P.kv : P.idx;
  long long row = -1;
  if (lane == 0) row = owner_row(c, w, req, p, P.page_size, P.d_err);
  row = __shfl_sync(0xffffffffu, row, 0);
  if (row < 0) return;
  if (warp == 0)
    write_row<kKvDim>(P.kv_in + static_cast<long long>(j) * kKvDim, pos, P.theta[lane], c.fp8,
                      c.data[w], c.scale[w], row, lane);
  else
    write_row<kIdxDim>(P.idx_in + static_cast<long long>(j) * kIdxDim, pos, P.theta[lane], c.fp8,
                       c.data[w], c.scale[w], row, lane);
}

}  // namespace

cudaError_t launch_cache_write(const CacheWriteLaunch& p, cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  cache_write_kernel<<<(p.num_tokens + kTokPerCta - 1) / kTokPerCta, 64 * kTokPerCta, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
