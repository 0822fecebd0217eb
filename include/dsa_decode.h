/*
 * dsa_decode.h -- C ABI of the GB300 (sm_103a) DSA sparse-attention decode
 * library.
 *
 * What the library computes (sources are named by page title and section):
 *
 *   "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2"
 *   (sgl-project/sglang pull request 42618):
 *     - Motivation: DSA scores the whole cached sequence with an indexer and
 *       keeps the top 2048 tokens before attention.
 *     - Modifications / Writes: token slot t lives on shard t % W
 *       (interleave size 1).
 *     - Modifications / Indexer decode: every shard takes a local top-k over
 *       its own tokens; the (score, global position) candidates are merged
 *       into the exact global top-k; the merge directly emits the local rows
 *       each shard owns.
 *     - Modifications / Sparse decode: each shard attends only the selected
 *       tokens it owns with a split-K kernel that also returns the
 *       natural-log LSE; partial results are merged by LSE.  Commit "store a
 *       lone split's output and LSE in place": with one split the partial is
 *       the final result and is written directly.
 *   "Harden DeepSeek V4 DSpark DP2 serving" (shiftup-ai/sglang pull request
 *   1), section 6.3: outputs and LSE go to caller-owned buffers; the
 *   optimized path fails closed instead of falling back.
 *
 * Readings of points the pages leave open (fixed by this library):
 *   - indexer: 64 heads x 128 dims, score(t) = sum_h w[h] * relu(q[h] . k[t]);
 *   - selection: the k tokens first in the order (score descending, token
 *     position ascending), so a tie at the k-th place goes to the lower
 *     position; the selected positions are written in ascending order (the
 *     pages fix which tokens are kept, not the order of the list); rows with
 *     fewer visible tokens than k keep all of them and pad the list with -1;
 *   - MLA latent rows are 576 wide; logits z = sm_scale * (q . kv) over all
 *     576 dims; the value is the first 512 dims of the same row;
 *   - fp8 caches hold OCP E4M3 codes with one fp32 scale per token
 *     (value = code value * scale);
 *   - a query row at position pos sees tokens 0..pos of its request.
 *
 * Conventions shared by every entry point:
 *   - every pointer argument named d_* or documented "device" is device
 *     memory; descriptor structs themselves are read on the host during the
 *     call and may be freed after it returns;
 *   - the caller owns every buffer; the library allocates nothing and keeps
 *     no state between calls; inputs are read-only; outputs are overwritten
 *     as documented;
 *   - every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and never synchronizes the host;
 *   - a call first validates its host-visible arguments and returns a status
 *     without launching anything if they are bad; launch failures return
 *     DSA_ERR_CUDA;
 *   - faults only visible on the device (a request row range out of order, a
 *     position past its block table, a -1 or out-of-range page id inside a
 *     span, a selected index outside the row's tokens, a NaN score, a bounded
 *     wait that gave up) are OR-ed as DSA_DEVERR_* bits into the caller's
 *     int32 error word `d_err` (device memory, zeroed by the caller) and the
 *     affected work is skipped; kernels never trap.  dsa_read_error() fetches
 *     the word;
 *   - every launch stays on `stream` with fixed buffer addresses, so a
 *     sequence of calls can be captured in a CUDA graph.
 */
#ifndef DSA_DECODE_H_
#define DSA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 3

/* fixed geometry */
#define DSA_INDEX_HEADS 64   /* indexer heads per query row */
#define DSA_INDEX_DIM 128    /* indexer key / query width */
#define DSA_KV_DIM 576       /* MLA latent row width (512 value + 64 rope) */
#define DSA_V_DIM 512        /* value width */
#define DSA_MAX_SHARDS 8     /* token shards of the emulated DCP group */
#define DSA_MAX_ROWS_PER_REQ 1024 /* query rows of one request (MTP, multi-query extend) */

/* status codes returned by every entry point */
enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,         /* bad pointer, size or descriptor */
  DSA_ERR_UNSUPPORTED = 2,         /* valid but not built (e.g. head count) */
  DSA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the query */
  DSA_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed */
  DSA_ERR_DEVICE_CHECK = 5,        /* dsa_read_error found device error bits */
  DSA_ERR_TIMEOUT = 6              /* reserved for host-side waits */
};

/* bits of the device error word */
enum {
  DSA_DEVERR_ROWS = 1 << 0,     /* row_start not monotone or out of range */
  DSA_DEVERR_POS = 1 << 1,      /* row position beyond the block table */
  DSA_DEVERR_PAGE = 1 << 2,     /* -1 / out-of-range page id inside a span */
  DSA_DEVERR_INDEX = 1 << 3,    /* selected index or count out of range */
  DSA_DEVERR_NAN = 1 << 4,      /* NaN indexer score */
  DSA_DEVERR_TIMEOUT = 1 << 5,  /* a bounded on-chip wait gave up */
  DSA_DEVERR_GROUP = 1 << 6     /* a request has more rows than declared */
};

/* storage type of a cache */
enum { DSA_DTYPE_BF16 = 0, DSA_DTYPE_FP8_E4M3 = 1 };

/*
 * A paged token cache (index keys or MLA latent rows).
 *   data:        device, [num_pages][page_size][row_elems] elements of dtype
 *                (bf16: 2 bytes, fp8: 1 byte), 16-byte aligned;
 *   scale:       device, fp8 only: [num_pages][page_size] fp32 per-token
 *                scales, 16-byte aligned; NULL for bf16;
 *   block_table: device, [num_reqs][max_blocks] int32 physical page ids of
 *                each request's logical pages, -1 past its span; NULL means
 *                contiguous: logical page j of request b is physical page
 *                b * max_blocks + j;
 *   page_size:   tokens per page, a multiple of 64.
 * Token t of request b lives in page block_table[b][t / page_size], slot
 * t % page_size.
 */
typedef struct {
  const void* data;
  const float* scale;
  const int32_t* block_table;
  int32_t dtype;
  int32_t row_elems;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_blocks;
} dsa_paged_cache;

/*
 * The query rows of a decode batch.
 *   row_start:  device [num_reqs + 1], rows of request b are
 *               row_start[b] .. row_start[b+1]-1 (non-decreasing, row_start[0]
 *               = 0, row_start[num_reqs] = num_rows);
 *   row_pos:    device [num_rows], position of each row's query; the row sees
 *               tokens 0..row_pos[r] of its request;
 *   max_rows_per_req: host bound on rows of one request
 *               (1..DSA_MAX_ROWS_PER_REQ); the indexer scores a request's
 *               rows in groups of up to 8, each group streaming the
 *               request's keys once;
 *   max_len:    host bound with row_pos[r] < max_len for every row; sizes the
 *               score rows and the workspace.
 * Several rows of one request (MTP / EAGLE verify: one row per draft token)
 * share that request's cache stream.
 */
typedef struct {
  int32_t num_rows;
  int32_t num_reqs;
  int32_t max_rows_per_req;
  int32_t max_len;
  const int32_t* row_start;
  const int32_t* row_pos;
} dsa_rows;

/* ABI version this library was built with (DSA_ABI_VERSION). */
int dsa_abi_version(void);

/* Static, human-readable name of a status code. */
const char* dsa_status_string(int status);

/*
 * Copy the device error word to *h_err (synchronizes `stream`).  Returns
 * DSA_ERR_DEVICE_CHECK when any bit is set, DSA_OK otherwise.
 */
int dsa_read_error(const int32_t* d_err, int32_t* h_err, void* stream);

/*
 * dsa_selftest_bounded_wait -- run, in one CTA with nothing else in flight,
 * the bounded on-chip wait every kernel of this library uses (DSpark page,
 * fail-closed convention: a wait that cannot complete ends in a reported
 * error, not a hang) on an mbarrier phase that nothing completes, giving up
 * after limit_us microseconds (0 .. 2000000; the kernels use 2 s).
 *   d_err:       device int32, OR-ed with DSA_DEVERR_TIMEOUT when the wait
 *                gives up (it always does)
 *   d_waited_ns: device uint64, the time the wait took (ns of %globaltimer)
 * Errors: DSA_ERR_INVALID_ARG for a bad limit or NULL pointers.
 */
int dsa_selftest_bounded_wait(int32_t limit_us, int32_t* d_err, uint64_t* d_waited_ns,
                              void* stream);

/*
 * dsa_indexer_scores -- DSA indexer over one (shard of a) paged index-K
 * cache.  DCP page, Motivation (score the whole sequence before selecting)
 * and Modifications / Indexer decode (each shard scores its own index-K
 * shard).
 *
 *   q_idx:  device bf16 [num_rows][64][128]
 *   w_idx:  device fp32 [num_rows][64] head weights
 *   idx_k:  index-K cache of this shard (row_elems = 128; bf16 or fp8)
 *   shard, num_shards: this cache holds the tokens t with t % num_shards ==
 *           shard at local position t / num_shards (1 shard: the whole
 *           sequence); a row at position pos sees local positions
 *           0 .. valid-1, valid = pos < shard ? 0 : (pos - shard) / W + 1
 *   scores: device fp32 [num_rows][ld_scores]; scores[r][j] is written for
 *           j < valid(r), other entries are left untouched;
 *           ld_scores >= ceil(rows->max_len / num_shards), a multiple of 4.
 *
 * Errors: DSA_ERR_INVALID_ARG for NULL pointers, bad sizes, a cache that is
 * not 128 wide, ld_scores too small; DSA_ERR_UNSUPPORTED for
 * max_rows_per_req > DSA_MAX_ROWS_PER_REQ.  Device: DSA_DEVERR_ROWS/POS/PAGE/GROUP
 * (GROUP: a request with more than max_rows_per_req rows).
 */
int dsa_indexer_scores(const uint16_t* q_idx, const float* w_idx,
                       const dsa_paged_cache* idx_k, const dsa_rows* rows,
                       int32_t shard, int32_t num_shards, float* scores,
                       int64_t ld_scores, int32_t* d_err, void* stream);

/*
 * Workspace bytes dsa_topk uses for its segment-parallel form on num_rows
 * score rows of stride ld_scores (0 for num_rows <= 0 or a bad stride).
 */
size_t dsa_topk_workspace_size(int32_t num_rows, int64_t ld_scores);

/*
 * dsa_topk -- exact top-k of every score row (DCP page, Motivation: the top
 * 2048 tokens of the whole sequence).
 *
 *   scores:    device fp32 [num_rows][ld_scores]; row r has valid_len[r]
 *              valid entries
 *   valid_len: device int32 [num_rows], 0 <= valid_len[r] <= ld_scores
 *   k:         1..4096
 *   out_idx:   device int32 [num_rows][k]: the selected j (the k first in
 *              the order score desc, j asc), mapped to j * index_stride +
 *              index_offset, listed by ascending j; entries past
 *              out_count[r] are -1
 *   out_score: device fp32 [num_rows][k] or NULL: the selected scores, same
 *              order (entries past the count are -inf)
 *   out_count: device int32 [num_rows]: min(k, valid_len[r])
 *   workspace: device, >= dsa_topk_workspace_size(num_rows, ld_scores)
 *              bytes, 16-byte aligned, or NULL.  With it the passes over the
 *              scores are split into segments spread over every SM (three
 *              launches; the call first clears the workspace's histograms
 *              on `stream`); without it one CTA per row does every pass
 *              (one launch, slower when rows are few or long).  The result
 *              is the same.  DSA_ERR_WORKSPACE_TOO_SMALL when workspace_bytes
 *              is below the size.
 * -0.0 and +0.0 are equal scores (a selected -0.0 is listed in out_score as
 * +0.0).  A NaN score sets DSA_DEVERR_NAN.
 * index_stride/index_offset turn shard-local positions into global ones
 * (stride = W, offset = shard); pass 1 and 0 otherwise.
 */
int dsa_topk(const float* scores, int64_t ld_scores, const int32_t* valid_len,
             int32_t num_rows, int32_t k, int32_t index_stride,
             int32_t index_offset, int32_t* out_idx, float* out_score,
             int32_t* out_count, void* workspace, size_t workspace_bytes,
             int32_t* d_err, void* stream);

/*
 * dsa_shard_topk_merge -- exact global top-k from per-shard local top-k
 * candidate lists, plus each shard's owned selection (DCP page,
 * Modifications / Indexer decode: the all-gathered (score, global position)
 * candidates are merged and the merge emits the local rows every shard owns).
 *
 *   cand_score: device fp32 [W][num_rows][k]: each shard's local top-k
 *               scores, listed by ascending position as dsa_topk writes them
 *   cand_pos:   device int32 [W][num_rows][k] global positions (ascending in
 *               each list); shard w's positions are == w mod W
 *   cand_count: device int32 [W][num_rows]
 *   pos_bound:  0, or a bound every candidate position is below (the
 *               requests' longest length); with one of at most 262144 the
 *               merge marks the selection in a bitmap of positions instead
 *               of ranking every candidate by searches in the other lists
 *               (same result; a position at or above the bound sets
 *               DSA_DEVERR_INDEX and is left out)
 *   out_idx:    device int32 [num_rows][k] global top-k of the union (ties at
 *               the k-th place to the lower position), ascending, -1 pad
 *   out_count:  device int32 [num_rows] = min(k, sum_w cand_count)
 *   owned_local: device int32 [W][num_rows][k]: local positions (pos / W) of
 *               the selected tokens shard w owns, ascending, -1 pad
 *   owned_count: device int32 [W][num_rows]
 */
int dsa_shard_topk_merge(const float* cand_score, const int32_t* cand_pos,
                         const int32_t* cand_count, int32_t num_shards,
                         int32_t num_rows, int32_t k, int32_t pos_bound, int32_t* out_idx,
                         int32_t* out_count, int32_t* owned_local,
                         int32_t* owned_count, int32_t* d_err, void* stream);

/*
 * Workspace bytes dsa_sparse_mla_decode needs for these sizes (num_splits 0
 * = the automatic choice on the current device).
 */
size_t dsa_sparse_mla_decode_workspace_size(int32_t num_rows, int32_t heads,
                                            int32_t k, int32_t num_splits);

/*
 * dsa_sparse_mla_decode -- absorbed-MLA attention of every query row over
 * its selected latent rows, split-K with LSE (DCP page, Modifications /
 * Sparse decode; commit "store a lone split's output and LSE in place").
 *
 *   q:        device bf16 [num_rows][heads][576]; heads 16 or 32
 *   sm_scale: logit scale (1/sqrt(576) for the configurations here)
 *   kv:       latent cache (row_elems = 576; bf16 or fp8)
 *   rows:     row -> request mapping (row_pos is not read here)
 *   idx:      device int32 [num_rows][k]: positions in `kv` to attend,
 *             first count[r] entries used
 *   count:    device int32 [num_rows], 0..k
 *   num_splits: 0 = automatic, else 1..k/64 splits of the list
 *   out:      device fp32 [num_rows][heads][512]
 *   out_lse:  device fp32 [num_rows][heads], natural log of the softmax
 *             denominator of the scaled logits; -inf for an empty row (out
 *             is then 0)
 *   workspace: device, >= dsa_sparse_mla_decode_workspace_size() bytes (may
 *             be NULL when that size is 0)
 */
int dsa_sparse_mla_decode(const uint16_t* q, int32_t heads, float sm_scale,
                          const dsa_paged_cache* kv, const dsa_rows* rows,
                          const int32_t* idx, const int32_t* count, int32_t k,
                          int32_t num_splits, float* out, float* out_lse,
                          void* workspace, size_t workspace_bytes,
                          int32_t* d_err, void* stream);

/*
 * Workspace bytes dsa_sparse_mla_prefill_into needs for these sizes (num_splits
 * 0 = the automatic choice on the current device): the split-K partial
 * outputs, LSEs and maxima; 0 with a single split.
 */
size_t dsa_sparse_mla_prefill_into_workspace_size(int32_t num_rows, int32_t heads,
                                                  int32_t k, int32_t num_splits);

/*
 * dsa_sparse_mla_prefill_into -- sparse attention of many query rows (a
 * prefill or extend chunk: each row with its own selected positions, e.g.
 * from dsa_topk over its causal prefix) that writes all three outputs into
 * caller-owned buffers (DSpark page, section 6.3 "Reserve sparse-prefill
 * outputs before allocator fragmentation": the output, max-logit and LSE
 * tensors are reserved once by the caller and the kernel writes into them).
 * Nothing is allocated; the split-K partials go to the caller's workspace.
 *
 * Same arguments, checks and errors as dsa_sparse_mla_decode, plus:
 *   out_max_logit: device fp32 [num_rows][heads], the largest scaled logit
 *             sm_scale * q.kv over the row's selected rows (natural units,
 *             not exponentiated); -inf for an empty row.  Required: NULL with
 *             num_rows > 0 is DSA_ERR_INVALID_ARG.  For every row,
 *             out_lse - ln(count) <= out_max_logit <= out_lse.
 *   workspace: device, >= dsa_sparse_mla_prefill_into_workspace_size() bytes
 *             (may be NULL when that size is 0); DSA_ERR_WORKSPACE_TOO_SMALL
 *             otherwise, before any launch.
 * Rows of one request are independent here: each reads only its own list
 * idx[r][0 .. count[r]) through its request's block table.
 */
int dsa_sparse_mla_prefill_into(const uint16_t* q, int32_t heads, float sm_scale,
                                const dsa_paged_cache* kv, const dsa_rows* rows,
                                const int32_t* idx, const int32_t* count, int32_t k,
                                int32_t num_splits, float* out, float* out_max_logit,
                                float* out_lse, void* workspace, size_t workspace_bytes,
                                int32_t* d_err, void* stream);

/*
 * Size of the fixed device array behind dsa_sparse_mla_decode_noalloc.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * dsa_sparse_mla_decode_noalloc -- dsa_sparse_mla_decode without a caller
 * workspace, for callers that cannot allocate device memory (a serving
 * runtime that reserved nearly all HBM for its KV pools, a plugin whose host
 * framework owns every allocation, a path where a synchronizing
 * cudaMalloc/cudaFree is not affordable).  The pages have no counterpart of
 * this entry point; it is a convenience of this library.
 *
 * Same arguments, results and errors as dsa_sparse_mla_decode.  The split-K
 * partials go to one fixed device array of DSA_NOALLOC_SCRATCH_BYTES that the
 * library's device image carries, and the call itself never allocates or
 * frees device memory.
 *   - The array is reserved on a device when the library's device code loads
 *     there; with CUDA's default lazy loading that is the first call of this
 *     entry point on the device.  Make that first call at start-up, before
 *     reserving the KV pools and before any stream capture.  The device then
 *     holds the array until the process exits.
 *   - Sizes whose partials do not fit (dsa_sparse_mla_decode_workspace_size()
 *     > DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE_TOO_SMALL before
 *     any launch.
 *   - Every call looks up the array's device address with the call's device
 *     current (after a context reset the address may change).
 *   - All calls share the one array: calls whose kernels overlap on a GPU
 *     (other streams, other threads) race on it and give wrong results; order
 *     them on one stream.  The array keeps the last call's contents; nothing in
 *     it needs to start at zero.
 */
int dsa_sparse_mla_decode_noalloc(const uint16_t* q, int32_t heads, float sm_scale,
                                  const dsa_paged_cache* kv, const dsa_rows* rows,
                                  const int32_t* idx, const int32_t* count, int32_t k,
                                  int32_t num_splits, float* out, float* out_lse,
                                  int32_t* d_err, void* stream);

/*
 * dsa_lse_merge -- merge num_parts partial attention results over disjoint
 * token sets (DCP page, Modifications / Sparse decode: partial results are
 * merged by their LSE):  lse = ln sum_p exp(lse_p),
 * out = sum_p exp(lse_p - lse) * O_p; parts with lse_p = -inf are skipped.
 *
 *   O_parts:   device fp32 [num_parts][num_rows][heads][dv]
 *   lse_parts: device fp32 [num_parts][num_rows][heads]
 *   out, out_lse: device fp32 [num_rows][heads][dv], [num_rows][heads]
 *   dv: a multiple of 4, <= 1024
 */
int dsa_lse_merge(const float* O_parts, const float* lse_parts,
                  int32_t num_parts, int32_t num_rows, int32_t heads,
                  int32_t dv, float* out, float* out_lse, void* stream);

/*
 * The whole decode path in one call.
 *   num_shards: W (1 = unsharded); idx_k[w], kv[w] are shard w's caches
 *               (token t of a request on shard t % W at local t / W)
 *   rows, q_idx, w_idx: as dsa_indexer_scores
 *   q, heads, sm_scale: as dsa_sparse_mla_decode
 *   topk: k (2048 for the configurations here)
 *   num_splits: 0 = automatic
 *   out, out_lse: as dsa_sparse_mla_decode
 *   out_topk_idx, out_topk_count: optional device [num_rows][k] /
 *               [num_rows]: the global selection (NULL = keep it in the
 *               workspace)
 */
typedef struct {
  int32_t num_shards;
  const dsa_paged_cache* idx_k;
  const dsa_paged_cache* kv;
  dsa_rows rows;
  const uint16_t* q_idx;
  const float* w_idx;
  const uint16_t* q;
  int32_t heads;
  float sm_scale;
  int32_t topk;
  int32_t num_splits;
  float* out;
  float* out_lse;
  int32_t* out_topk_idx;
  int32_t* out_topk_count;
} dsa_decode_desc;

/*
 * dsa_cache_write -- one decode step's cache write: every new token's latent
 * KV row and index-K row, RoPE applied, stored (quantized for fp8 caches) in
 * the cache of the shard that owns the token.  DCP page, Modifications /
 * Writes (MLA KV and indexer K land only on the owner rank, slot % W ==
 * rank; the fused RoPE + KV-cache write) and the decode-gap analysis (the
 * owner-rule write location computed once per step inside the write kernel
 * instead of by many small kernels).
 *
 * Token j < num_tokens belongs to request tok_req[j] (< num_reqs) at logical
 * position tok_pos[j] (>= 0):
 *   kv_in:   device bf16 [num_tokens][576], the latent row; its last 64 dims
 *            are given before RoPE
 *   idx_in:  device bf16 [num_tokens][128], the index-K row; its last 64
 *            dims are given before RoPE (NULL: no index-K write)
 *   RoPE:    on the last 64 dims of each row, pairs (2i, 2i+1), i < 32:
 *            a = pos * rope_base^(-i/32) (the angle is formed in double),
 *            (x, y) -> (x cos a - y sin a, x sin a + y cos a)
 *   kv, idx_k: [num_shards] caches (row_elems 576 and 128, one dtype per
 *            array, the same page size); token j goes to shard w = pos % W
 *            at local position p = pos / W: page
 *            block_table_w[req * max_blocks_w + p / page_size] (req *
 *            max_blocks_w + p / page_size when block_table is NULL), slot
 *            p % page_size.  The caches' data and scale arrays are written.
 *   bf16 caches store the RNE bf16 of every value.  fp8 caches store the
 *   e4m3 codes (round to nearest even, saturating at +-448) of value / s,
 *   s = max|value| / 448 over the row (fp32; s = 1 for an all-zero row), and
 *   s in the token's scale slot.
 *
 * Only each token's owner slot is written; nothing else is touched.  Two
 * tokens with the same (request, position) write the same slot in no
 * defined order.
 * Errors: DSA_ERR_INVALID_ARG for NULL pointers, bad sizes, num_shards
 * outside 1..DSA_MAX_SHARDS, caches of the wrong width or of mixed dtype or
 * page size.  Device: DSA_DEVERR_ROWS (request out of range), DSA_DEVERR_POS
 * (negative position or one past the block table), DSA_DEVERR_PAGE (page id
 * out of range); such a token is not written.
 */
int dsa_cache_write(const uint16_t* kv_in, const uint16_t* idx_in, const int32_t* tok_req,
                    const int32_t* tok_pos, int32_t num_tokens, int32_t num_reqs,
                    float rope_base, const dsa_paged_cache* kv,
                    const dsa_paged_cache* idx_k, int32_t num_shards, int32_t* d_err,
                    void* stream);

/* Where dsa_decode keeps its intermediates inside the workspace (byte
 * offsets; -1 = not used).  scores is [W][num_rows][ld_scores] fp32. */
typedef struct {
  int64_t scores;
  int64_t ld_scores;
  int64_t cand_idx, cand_score, cand_count;
  int64_t topk_idx, topk_count;
  int64_t topk_ws;  /* the top-k's own workspace (histograms, candidates, bitmaps) */
  int64_t owned_local, owned_count;
  int64_t part_out, part_lse;
  int32_t num_splits;
  int32_t num_parts;
  int32_t launches;  /* kernels one dsa_decode call launches with this layout */
  int32_t reserved;
  int64_t total_bytes;
} dsa_decode_layout;

/* Workspace bytes for dsa_decode (0 on an invalid descriptor). */
size_t dsa_decode_workspace_size(const dsa_decode_desc* desc);

/* Fill *layout for this descriptor; returns a status. */
int dsa_decode_workspace_layout(const dsa_decode_desc* desc,
                                dsa_decode_layout* layout);

/*
 * dsa_decode -- indexer -> top-k (-> per-shard local top-k and exact merge)
 * -> sparse MLA split-K -> LSE merge, all on `stream`, intermediates in the
 * caller's workspace.  Errors as the entry points above, plus
 * DSA_ERR_WORKSPACE_TOO_SMALL.
 */
int dsa_decode(const dsa_decode_desc* desc, void* workspace,
               size_t workspace_bytes, int32_t* d_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_DECODE_H_ */
