// Launchers of the kernels behind the C ABI (host side).  Every launcher only
// enqueues work on `stream`; argument validation happens in dsa_abi.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_decode.h"

namespace dsa {

// ------------------------------------------------------------- indexer

// One launch scores the rows against `num_shards_in_launch` shard caches
// (shard ids shard_base .. shard_base + n - 1 of a group of W shards).
struct IndexerLaunch {
  CUtensorMap kmap[DSA_MAX_SHARDS];       // index-K tensor maps (TMA)
  const int32_t* block_table[DSA_MAX_SHARDS];
  const float* kscale[DSA_MAX_SHARDS];    // fp8 per-token scales
  int32_t num_pages[DSA_MAX_SHARDS];
  int32_t max_blocks[DSA_MAX_SHARDS];
  int32_t page_size;
  int32_t page_shift;   // log2(page_size) when a power of two, else -1 (set by the launcher)
  int32_t fp8;
  int32_t W;            // shards of the group
  int32_t shard_base;   // id of kmap[0]
  int32_t nshards;      // caches in this launch
  const uint16_t* q_idx;
  const float* w_idx;
  const int32_t* row_start;
  const int32_t* row_pos;
  int32_t num_rows;
  int32_t num_reqs;
  int32_t max_rows;     // rows per group (1..8): query rows one CTA holds at a time
  int32_t groups;       // row groups per request (rows per request <= max_rows * groups)
  float* scores;        // cache i writes rows at scores + i * shard_stride
  int64_t ld;
  int64_t shard_stride;
  int32_t* d_err;
};

// Host: fill kmap[i] for a cache; returns cudaSuccess or an error.
cudaError_t make_index_k_tmap(CUtensorMap* map, const dsa_paged_cache& c);
cudaError_t launch_indexer(const IndexerLaunch& p, cudaStream_t stream);

// ------------------------------------------------------------- top-k

struct TopkLaunch {
  const float* scores;
  int64_t ld;
  int64_t shard_stride;       // scores of row q = w * R + r at scores + w*stride + r*ld
  const int32_t* valid_len;   // explicit per-row valid counts, or NULL:
  const int32_t* row_pos;     //   valid = shard_valid_len(row_pos[r], W, w)
  int32_t W;
  int32_t shard_offset;       // shard id of w = 0 (single-shard calls)
  int32_t rows;               // R (rows per shard)
  int32_t nshards;            // shards in this launch (grid = nshards * R)
  int32_t k;
  int32_t index_stride;       // out index = j * stride + (w + shard_offset) * per_shard_offset
  int32_t index_offset;
  int32_t offset_per_shard;   // 1: add the shard id to index_offset
  int32_t* out_idx;           // row q at out_idx + q * k
  float* out_score;           // or NULL
  int32_t* out_count;
  int32_t* d_err;
  // workspace of the segment-parallel form (all NULL: one CTA per row does
  // every pass); set by topk_set_workspace
  uint32_t* ghist;            // [rows][1024] first histograms (zeroed before the launch)
  uint32_t* gcnt;             // [rows] candidates listed (zeroed before the launch)
  uint2* gcand;               // [rows][4096] candidates (key, position)
  uint32_t* gbits;            // [rows][nw] position bitmaps of the keys above the range
  int32_t nw;                 // bitmap words per row
  int32_t seg_quads;          // positions / 4 per segment CTA (set by the launcher)
};
// pdl: launch as a programmatic dependent of the stream's previous kernel (only
// after kernels of this library whose outputs the kernel waits for).  With a
// workspace, its first topk_workspace_clear_bytes() bytes must be zero when
// the launch starts (the caller clears them on the stream beforehand).
cudaError_t launch_topk(const TopkLaunch& p, cudaStream_t stream, bool pdl = false);
// workspace bytes of the segment-parallel form for `rows` score rows of stride ld
size_t topk_workspace_bytes(int rows, int64_t ld);
size_t topk_workspace_clear_bytes(int rows);
// whether launch_topk uses a workspace for these sizes (else it ignores it)
bool topk_uses_workspace(int rows, int64_t ld);
// point p's workspace fields into ws (NULL: the one-CTA-per-row form); needs
// p.nshards, p.rows and p.ld
void topk_set_workspace(TopkLaunch& p, void* ws);

// ------------------------------------------------------------- shard merge

struct MergeTopkLaunch {
  const float* cand_score;
  const int32_t* cand_pos;
  const int32_t* cand_count;
  int32_t W, rows, k;
  int32_t* out_idx;
  int32_t* out_count;
  int32_t* owned_local;
  int32_t* owned_count;
  int32_t* d_err;
  int32_t pos_bound;  // every candidate position is below it (0: unknown)
};
// With a position bound whose bitmaps fit in shared memory the merge marks the
// selection in a bitmap of global positions; otherwise it ranks candidates by
// binary searches in the other lists.
cudaError_t launch_shard_topk_merge(const MergeTopkLaunch& p, cudaStream_t stream,
                                   bool pdl = false);

// ------------------------------------------------------------- sparse MLA

struct MlaLaunch {
  const void* kv[DSA_MAX_SHARDS];
  const float* kscale[DSA_MAX_SHARDS];
  const int32_t* block_table[DSA_MAX_SHARDS];
  int32_t num_pages[DSA_MAX_SHARDS];
  int32_t max_blocks[DSA_MAX_SHARDS];
  int32_t page_size;
  int32_t fp8;
  int32_t nshards;         // caches in this launch; work row q = w * R + r
  const uint16_t* q;       // [R][H][576]
  int32_t heads;
  float sm_scale;
  const int32_t* row_start;
  int32_t num_reqs;
  int32_t rows;            // R
  const int32_t* idx;      // row q's list at idx + q * k
  const int32_t* count;    // [nshards * R]
  int32_t k;
  int32_t num_splits;      // S
  int32_t chunk;           // tokens per split (multiple of 64)
  int32_t bt_smem;         // block-table entries cached in shared memory (set by the launcher)
  float* out;              // when parts == 1: [R][H][512]
  float* out_lse;
  float* part_out;         // else: part p = w * S + s at part_out + p*R*H*512
  float* part_lse;
  float* out_max;          // optional max scaled logit [R][H] (nullptr: not written)
  float* part_max;         // with it and parts > 1: part p at part_max + p*R*H
  int32_t* d_err;
};
// pdl: the kernel reads the query, row_start and block tables before it waits
// for the previous grid, which therefore must not write them
cudaError_t launch_sparse_mla(const MlaLaunch& p, cudaStream_t stream, bool pdl = false);
int auto_mla_splits(int work_rows, int k, int expected_count);
// the tensor-core form for fp8 caches with 32 heads (tiles of 128 tokens):
// launch_sparse_mla takes it when sparse_mla_tc_supported(p)
bool sparse_mla_tc_supported(const MlaLaunch& p);
cudaError_t launch_sparse_mla_tc(const MlaLaunch& p, cudaStream_t stream, bool pdl);
// Host: the TMA map of an fp8 latent cache as [num_pages * page_size][576]
// rows with 128-byte column boxes of one row (for tile::gather4 loads)
cudaError_t make_kv_fp8_tmap(CUtensorMap* map, const void* data, int num_pages, int page_size);

// ------------------------------------------------------------- cache write

struct CacheWriteSide {    // the shard caches of one kind (latent or index-K)
  void* data[DSA_MAX_SHARDS];
  float* scale[DSA_MAX_SHARDS];
  const int32_t* block_table[DSA_MAX_SHARDS];
  int32_t num_pages[DSA_MAX_SHARDS];
  int32_t max_blocks[DSA_MAX_SHARDS];
  int32_t fp8;
};
struct CacheWriteLaunch {
  CacheWriteSide kv, idx;
  const uint16_t* kv_in;   // [N][576] bf16
  const uint16_t* idx_in;  // [N][128] bf16 or NULL
  const int32_t* tok_req;
  const int32_t* tok_pos;
  int32_t num_tokens, num_reqs, W, page_size;
  double theta[32];        // rope_base^(-i/32), i < 32: the rotation rates
  int32_t* d_err;
};
cudaError_t launch_cache_write(const CacheWriteLaunch& p, cudaStream_t stream);

// ------------------------------------------------------------- LSE merge

// max_parts / out_max (optional, both or neither): out_max = the largest of
// the parts' maxima, per (row, head)
cudaError_t launch_lse_merge(const float* O_parts, const float* lse_parts, int parts,
                             int rows, int heads, int dv, float* out, float* out_lse,
                             cudaStream_t stream, bool pdl = false,
                             const float* max_parts = nullptr, float* out_max = nullptr);

// one CTA that waits on an mbarrier phase nothing completes, with the
// kernels' bounded wait and the given limit; sets DSA_DEVERR_TIMEOUT in d_err
// and the time it waited (ns) in *waited_ns
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* d_err, uint64_t* waited_ns,
                                         cudaStream_t stream);

int num_sms();

}  // namespace dsa
