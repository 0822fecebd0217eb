// C ABI of the library: argument validation, TMA descriptors, workspace
// layout and the order of launches of the fused decode.  Everything here runs
// on the host and only enqueues kernels on the caller's stream.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_decode.h"
#include "dsa_internal.h"

namespace dsa {

int mla_smem_bytes(int heads, int fp8, int chunk);
int merge_smem_bytes(int W, int k);

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

constexpr int64_t kAlign = 256;
int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cache(const dsa_paged_cache* c, int row_elems) {
  if (c == nullptr || c->data == nullptr) return DSA_ERR_INVALID_ARG;
  if (c->row_elems != row_elems) return DSA_ERR_INVALID_ARG;
  if (c->dtype != DSA_DTYPE_BF16 && c->dtype != DSA_DTYPE_FP8_E4M3) return DSA_ERR_INVALID_ARG;
  if (c->page_size <= 0 || (c->page_size % 64) != 0) return DSA_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->max_blocks <= 0) return DSA_ERR_INVALID_ARG;
  if (!aligned16(c->data)) return DSA_ERR_INVALID_ARG;
  if (c->dtype == DSA_DTYPE_FP8_E4M3 && (c->scale == nullptr || !aligned16(c->scale)))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

int check_rows(const dsa_rows* rw) {
  if (rw == nullptr) return DSA_ERR_INVALID_ARG;
  if (rw->num_rows < 0 || rw->num_reqs < 1 || rw->max_len < 1) return DSA_ERR_INVALID_ARG;
  if (rw->max_rows_per_req < 1) return DSA_ERR_INVALID_ARG;
  if (rw->max_rows_per_req > DSA_MAX_ROWS_PER_REQ) return DSA_ERR_UNSUPPORTED;
  if (rw->num_rows > 0 && (rw->row_start == nullptr || rw->row_pos == nullptr))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

int resolve_splits(int num_splits, int work_rows, int k, int expected) {
  int s = num_splits > 0 ? num_splits : auto_mla_splits(work_rows, k, expected);
  if (s > (k + 63) / 64) s = (k + 63) / 64;
  if (s < 1) s = 1;
  int chunk = (k + s - 1) / s;
  chunk = (chunk + 63) / 64 * 64;
  return (k + chunk - 1) / chunk;  // splits that the rounded chunk gives
}
int split_chunk(int splits, int k) {
  int chunk = (k + splits - 1) / splits;
  return (chunk + 63) / 64 * 64;
}

// The rows of a request are scored in groups of at most kRowsPerGroup
// (the query rows one CTA holds in shared memory); each group streams the
// request's keys once.
void set_row_groups(IndexerLaunch& L, int max_rows_per_req) {
  L.max_rows = max_rows_per_req < kRowsPerGroup ? max_rows_per_req : kRowsPerGroup;
  L.groups = (max_rows_per_req + kRowsPerGroup - 1) / kRowsPerGroup;
}

void fill_indexer_shard(IndexerLaunch& L, int i, const dsa_paged_cache& c) {
  L.block_table[i] = c.block_table;
  L.kscale[i] = c.scale;
  L.num_pages[i] = c.num_pages;
  L.max_blocks[i] = c.max_blocks;
}

void fill_mla_shard(MlaLaunch& L, int i, const dsa_paged_cache& c) {
  L.kv[i] = c.data;
  L.kscale[i] = c.scale;
  L.block_table[i] = c.block_table;
  L.num_pages[i] = c.num_pages;
  L.max_blocks[i] = c.max_blocks;
}

}  // namespace

cudaError_t make_index_k_tmap(CUtensorMap* map, const dsa_paged_cache& c) {
  auto enc = get_encode();
  if (enc == nullptr) return cudaErrorNotSupported;
  const bool fp8 = c.dtype == DSA_DTYPE_FP8_E4M3;
  const cuuint64_t esz = fp8 ? 1 : 2;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(c.page_size),
                        static_cast<cuuint64_t>(c.num_pages)};
  cuuint64_t gstride[2] = {kIdxDim * esz, static_cast<cuuint64_t>(c.page_size) * kIdxDim * esz};
  cuuint32_t box[3] = {fp8 ? 128u : 64u, 64u, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(c.data), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_kv_fp8_tmap(CUtensorMap* map, const void* data, int num_pages, int page_size) {
  auto enc = get_encode();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the cache as [pages * page_size rows][576] e4m3; 128-byte column boxes of
  // one row, gathered four rows at a time
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kKvDim),
                        static_cast<cuuint64_t>(num_pages) * static_cast<cuuint64_t>(page_size)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kKvDim)};
  cuuint32_t box[2] = {128u, 1u};
  cuuint32_t estride[2] = {1u, 1u};
  // no L2 promotion: a 576-byte row starts 64 bytes off a 128-byte line for
  // every other row, so wider fetches would read bytes of neighbouring rows
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(data), gdim, gstride,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace dsa

using namespace dsa;

namespace {

// Workspace bytes of a sparse MLA call: the split-K partial outputs and LSEs,
// and with_max the partial maxima (none with a single split)
size_t mla_workspace_bytes(int32_t num_rows, int32_t heads, int32_t k, int32_t num_splits,
                           bool with_max) {
  if (num_rows < 0 || heads < 1 || k < 1 || num_splits < 0) return 0;
  const int S = resolve_splits(num_splits, num_rows, k, k);
  if (S <= 1) return 0;
  const int64_t o = align_up(static_cast<int64_t>(S) * num_rows * heads * kVDim * 4, kAlign);
  const int64_t l = align_up(static_cast<int64_t>(S) * num_rows * heads * 4, kAlign);
  return static_cast<size_t>(o + l + (with_max ? l : 0));
}

// dsa_sparse_mla_decode, and with out_max != nullptr dsa_sparse_mla_prefill_into
int run_sparse_mla(const uint16_t* q, int32_t heads, float sm_scale, const dsa_paged_cache* kv,
                   const dsa_rows* rows, const int32_t* idx, const int32_t* count, int32_t k,
                   int32_t num_splits, float* out, float* out_max, float* out_lse,
                   void* workspace, size_t workspace_bytes, int32_t* d_err, void* stream) {
  int st = check_rows(rows);
  if (st != DSA_OK) return st;
  st = check_cache(kv, kKvDim);
  if (st != DSA_OK) return st;
  if (heads != 16 && heads != 32) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > 4096 || num_splits < 0 || d_err == nullptr) return DSA_ERR_INVALID_ARG;
  const int R = rows->num_rows;
  if (R == 0) return DSA_OK;
  if (!q || !idx || !count || !out || !out_lse || !aligned16(q) || !aligned16(out))
    return DSA_ERR_INVALID_ARG;
  const bool with_max = out_max != nullptr;
  const int S = resolve_splits(num_splits, R, k, k);
  const int chunk = split_chunk(S, k);
  if (mla_smem_bytes(heads, kv->dtype == DSA_DTYPE_FP8_E4M3, chunk) > 227 * 1024)
    return DSA_ERR_UNSUPPORTED;
  const size_t need = mla_workspace_bytes(R, heads, k, num_splits, with_max);
  if (workspace_bytes < need || (need > 0 && workspace == nullptr))
    return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (static_cast<long long>(kv->num_pages) * kv->page_size > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  MlaLaunch L{};
  fill_mla_shard(L, 0, *kv);
  L.page_size = kv->page_size;
  L.fp8 = kv->dtype == DSA_DTYPE_FP8_E4M3;
  L.nshards = 1;
  L.q = q;
  L.heads = heads;
  L.sm_scale = sm_scale;
  L.row_start = rows->row_start;
  L.num_reqs = rows->num_reqs;
  L.rows = R;
  L.idx = idx;
  L.count = count;
  L.k = k;
  L.num_splits = S;
  L.chunk = chunk;
  L.out = out;
  L.out_lse = out_lse;
  L.out_max = out_max;
  L.d_err = d_err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (S > 1) {
    const int64_t o = align_up(static_cast<int64_t>(S) * R * heads * kVDim * 4, kAlign);
    const int64_t l = align_up(static_cast<int64_t>(S) * R * heads * 4, kAlign);
    L.part_out = reinterpret_cast<float*>(ws);
    L.part_lse = reinterpret_cast<float*>(ws + o);
    if (with_max) L.part_max = reinterpret_cast<float*>(ws + o + l);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_sparse_mla(L, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  if (S > 1)
    e = launch_lse_merge(L.part_out, L.part_lse, S, R, heads, kVDim, out, out_lse, s, false,
                         L.part_max, out_max);
  return cuda_status(e);
}

}  // namespace

extern "C" {

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

int dsa_selftest_bounded_wait(int32_t limit_us, int32_t* d_err, uint64_t* d_waited_ns,
                              void* stream) {
  if (limit_us < 0 || limit_us > 2000000 || d_err == nullptr || d_waited_ns == nullptr)
    return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_bounded_wait_selftest(static_cast<uint64_t>(limit_us) * 1000u, d_err,
                                                  d_waited_ns, static_cast<cudaStream_t>(stream)));
}

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: bad pointer, size or descriptor";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: valid but not supported by this build";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "DSA_ERR_WORKSPACE_TOO_SMALL";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA call failed";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK: the device error word is set";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    default: return "unknown dsa status";
  }
}

int dsa_read_error(const int32_t* d_err, int32_t* h_err, void* stream) {
  if (d_err == nullptr || h_err == nullptr) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(h_err, d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  return *h_err != 0 ? DSA_ERR_DEVICE_CHECK : DSA_OK;
}

int dsa_indexer_scores(const uint16_t* q_idx, const float* w_idx, const dsa_paged_cache* idx_k,
                       const dsa_rows* rows, int32_t shard, int32_t num_shards, float* scores,
                       int64_t ld_scores, int32_t* d_err, void* stream) {
  int st = check_rows(rows);
  if (st != DSA_OK) return st;
  st = check_cache(idx_k, kIdxDim);
  if (st != DSA_OK) return st;
  if (d_err == nullptr || num_shards < 1 || num_shards > kMaxShards || shard < 0 ||
      shard >= num_shards)
    return DSA_ERR_INVALID_ARG;
  if (rows->num_rows == 0) return DSA_OK;
  if (q_idx == nullptr || w_idx == nullptr || scores == nullptr || !aligned16(q_idx))
    return DSA_ERR_INVALID_ARG;
  const int64_t need = (static_cast<int64_t>(rows->max_len) + num_shards - 1) / num_shards;
  if (ld_scores < need) return DSA_ERR_INVALID_ARG;
  IndexerLaunch L{};
  cudaError_t e = make_index_k_tmap(&L.kmap[0], *idx_k);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  fill_indexer_shard(L, 0, *idx_k);
  L.page_size = idx_k->page_size;
  L.fp8 = idx_k->dtype == DSA_DTYPE_FP8_E4M3;
  L.W = num_shards;
  L.shard_base = shard;
  L.nshards = 1;
  L.q_idx = q_idx;
  L.w_idx = w_idx;
  L.row_start = rows->row_start;
  L.row_pos = rows->row_pos;
  L.num_rows = rows->num_rows;
  L.num_reqs = rows->num_reqs;
  set_row_groups(L, rows->max_rows_per_req);
  L.scores = scores;
  L.ld = ld_scores;
  L.shard_stride = 0;
  L.d_err = d_err;
  return cuda_status(launch_indexer(L, static_cast<cudaStream_t>(stream)));
}

size_t dsa_topk_workspace_size(int32_t num_rows, int64_t ld_scores) {
  if (num_rows <= 0 || ld_scores < 0 || ld_scores > INT32_MAX) return 0;
  return topk_workspace_bytes(num_rows, ld_scores);
}

int dsa_topk(const float* scores, int64_t ld_scores, const int32_t* valid_len, int32_t num_rows,
             int32_t k, int32_t index_stride, int32_t index_offset, int32_t* out_idx,
             float* out_score, int32_t* out_count, void* workspace, size_t workspace_bytes,
             int32_t* d_err, void* stream) {
  if (num_rows < 0 || k < 1 || k > 4096 || d_err == nullptr || ld_scores < 0)
    return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (scores == nullptr || valid_len == nullptr || out_idx == nullptr || out_count == nullptr)
    return DSA_ERR_INVALID_ARG;
  if (ld_scores > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (workspace != nullptr) {
    if (workspace_bytes < topk_workspace_bytes(num_rows, ld_scores))
      return DSA_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return DSA_ERR_INVALID_ARG;
  }
  TopkLaunch L{};
  L.scores = scores;
  L.ld = ld_scores;
  L.shard_stride = 0;
  L.valid_len = valid_len;
  L.row_pos = nullptr;
  L.W = 1;
  L.shard_offset = 0;
  L.rows = num_rows;
  L.nshards = 1;
  L.k = k;
  L.index_stride = index_stride;
  L.index_offset = index_offset;
  L.offset_per_shard = 0;
  L.out_idx = out_idx;
  L.out_score = out_score;
  L.out_count = out_count;
  L.d_err = d_err;
  topk_set_workspace(L, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (workspace != nullptr && topk_uses_workspace(num_rows, ld_scores) &&
      cudaMemsetAsync(workspace, 0, topk_workspace_clear_bytes(num_rows), s) != cudaSuccess)
    return DSA_ERR_CUDA;
  return cuda_status(launch_topk(L, s));
}

int dsa_shard_topk_merge(const float* cand_score, const int32_t* cand_pos,
                         const int32_t* cand_count, int32_t num_shards, int32_t num_rows,
                         int32_t k, int32_t pos_bound, int32_t* out_idx, int32_t* out_count,
                         int32_t* owned_local, int32_t* owned_count, int32_t* d_err,
                         void* stream) {
  if (num_shards < 1 || num_shards > kMaxShards || num_rows < 0 || k < 1 || k > 4096 ||
      pos_bound < 0 || d_err == nullptr)
    return DSA_ERR_INVALID_ARG;
  if (merge_smem_bytes(num_shards, k) > 227 * 1024) return DSA_ERR_UNSUPPORTED;
  if (num_rows == 0) return DSA_OK;
  if (!cand_score || !cand_pos || !cand_count || !out_idx || !out_count || !owned_local ||
      !owned_count)
    return DSA_ERR_INVALID_ARG;
  MergeTopkLaunch L{cand_score, cand_pos, cand_count, num_shards, num_rows, k,
                    out_idx,    out_count, owned_local, owned_count, d_err, pos_bound};
  return cuda_status(launch_shard_topk_merge(L, static_cast<cudaStream_t>(stream)));
}

size_t dsa_sparse_mla_decode_workspace_size(int32_t num_rows, int32_t heads, int32_t k,
                                            int32_t num_splits) {
  return mla_workspace_bytes(num_rows, heads, k, num_splits, false);
}

int dsa_sparse_mla_decode(const uint16_t* q, int32_t heads, float sm_scale,
                          const dsa_paged_cache* kv, const dsa_rows* rows, const int32_t* idx,
                          const int32_t* count, int32_t k, int32_t num_splits, float* out,
                          float* out_lse, void* workspace, size_t workspace_bytes,
                          int32_t* d_err, void* stream) {
  return run_sparse_mla(q, heads, sm_scale, kv, rows, idx, count, k, num_splits, out, nullptr,
                        out_lse, workspace, workspace_bytes, d_err, stream);
}

size_t dsa_sparse_mla_prefill_into_workspace_size(int32_t num_rows, int32_t heads, int32_t k,
                                                  int32_t num_splits) {
  return mla_workspace_bytes(num_rows, heads, k, num_splits, true);
}

int dsa_sparse_mla_prefill_into(const uint16_t* q, int32_t heads, float sm_scale,
                                const dsa_paged_cache* kv, const dsa_rows* rows,
                                const int32_t* idx, const int32_t* count, int32_t k,
                                int32_t num_splits, float* out, float* out_max_logit,
                                float* out_lse, void* workspace, size_t workspace_bytes,
                                int32_t* d_err, void* stream) {
  if (rows != nullptr && rows->num_rows > 0 && out_max_logit == nullptr) return DSA_ERR_INVALID_ARG;
  return run_sparse_mla(q, heads, sm_scale, kv, rows, idx, count, k, num_splits, out,
                        out_max_logit, out_lse, workspace, workspace_bytes, d_err, stream);
}

int dsa_lse_merge(const float* O_parts, const float* lse_parts, int32_t num_parts,
                  int32_t num_rows, int32_t heads, int32_t dv, float* out, float* out_lse,
                  void* stream) {
  if (num_parts < 1 || num_rows < 0 || heads < 1 || dv < 4 || (dv % 4) != 0 || dv > 1024)
    return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!O_parts || !lse_parts || !out || !out_lse || !aligned16(O_parts) || !aligned16(out))
    return DSA_ERR_INVALID_ARG;
  return cuda_status(launch_lse_merge(O_parts, lse_parts, num_parts, num_rows, heads, dv, out,
                                      out_lse, static_cast<cudaStream_t>(stream)));
}

static int check_decode(const dsa_decode_desc* d) {
  if (d == nullptr) return DSA_ERR_INVALID_ARG;
  if (d->num_shards < 1 || d->num_shards > kMaxShards) return DSA_ERR_INVALID_ARG;
  if (d->idx_k == nullptr || d->kv == nullptr) return DSA_ERR_INVALID_ARG;
  int st = check_rows(&d->rows);
  if (st != DSA_OK) return st;
  for (int w = 0; w < d->num_shards; ++w) {
    st = check_cache(&d->idx_k[w], kIdxDim);
    if (st != DSA_OK) return st;
    st = check_cache(&d->kv[w], kKvDim);
    if (st != DSA_OK) return st;
    if (static_cast<long long>(d->kv[w].num_pages) * d->kv[w].page_size > INT32_MAX)
      return DSA_ERR_UNSUPPORTED;
    if (d->idx_k[w].dtype != d->idx_k[0].dtype || d->kv[w].dtype != d->kv[0].dtype ||
        d->idx_k[w].page_size != d->idx_k[0].page_size ||
        d->kv[w].page_size != d->kv[0].page_size)
      return DSA_ERR_INVALID_ARG;
  }
  if (d->heads != 16 && d->heads != 32) return DSA_ERR_UNSUPPORTED;
  if (d->topk < 1 || d->topk > 4096 || d->num_splits < 0) return DSA_ERR_INVALID_ARG;
  if (d->num_shards > 1 && merge_smem_bytes(d->num_shards, d->topk) > 227 * 1024)
    return DSA_ERR_UNSUPPORTED;
  if (d->rows.num_rows > 0) {
    if (!d->q_idx || !d->w_idx || !d->q || !d->out || !d->out_lse) return DSA_ERR_INVALID_ARG;
    if (!aligned16(d->q_idx) || !aligned16(d->q) || !aligned16(d->out)) return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

int dsa_cache_write(const uint16_t* kv_in, const uint16_t* idx_in, const int32_t* tok_req,
                    const int32_t* tok_pos, int32_t num_tokens, int32_t num_reqs,
                    float rope_base, const dsa_paged_cache* kv, const dsa_paged_cache* idx_k,
                    int32_t num_shards, int32_t* d_err, void* stream) {
  if (num_tokens < 0 || num_reqs < 1 || num_shards < 1 || num_shards > kMaxShards ||
      !(rope_base > 0.0f) || d_err == nullptr || kv == nullptr)
    return DSA_ERR_INVALID_ARG;
  if (num_tokens == 0) return DSA_OK;
  if (kv_in == nullptr || tok_req == nullptr || tok_pos == nullptr || !aligned16(kv_in))
    return DSA_ERR_INVALID_ARG;
  if (idx_in != nullptr && (idx_k == nullptr || !aligned16(idx_in))) return DSA_ERR_INVALID_ARG;
  CacheWriteLaunch L{};
  const int page = kv[0].page_size;
  for (int w = 0; w < num_shards; ++w) {
    int st = check_cache(&kv[w], kKvDim);
    if (st != DSA_OK) return st;
    if (kv[w].dtype != kv[0].dtype || kv[w].page_size != page) return DSA_ERR_INVALID_ARG;
    L.kv.data[w] = const_cast<void*>(kv[w].data);
    L.kv.scale[w] = const_cast<float*>(kv[w].scale);
    L.kv.block_table[w] = kv[w].block_table;
    L.kv.num_pages[w] = kv[w].num_pages;
    L.kv.max_blocks[w] = kv[w].max_blocks;
    if (idx_in != nullptr) {
      st = check_cache(&idx_k[w], kIdxDim);
      if (st != DSA_OK) return st;
      if (idx_k[w].dtype != idx_k[0].dtype || idx_k[w].page_size != page)
        return DSA_ERR_INVALID_ARG;
      L.idx.data[w] = const_cast<void*>(idx_k[w].data);
      L.idx.scale[w] = const_cast<float*>(idx_k[w].scale);
      L.idx.block_table[w] = idx_k[w].block_table;
      L.idx.num_pages[w] = idx_k[w].num_pages;
      L.idx.max_blocks[w] = idx_k[w].max_blocks;
    }
  }
  L.kv.fp8 = kv[0].dtype == DSA_DTYPE_FP8_E4M3;
  L.idx.fp8 = idx_in != nullptr && idx_k[0].dtype == DSA_DTYPE_FP8_E4M3;
  L.kv_in = kv_in;
  L.idx_in = idx_in;
  L.tok_req = tok_req;
  L.tok_pos = tok_pos;
  L.num_tokens = num_tokens;
  L.num_reqs = num_reqs;
  L.W = num_shards;
  L.page_size = page;
  for (int i = 0; i < 32; ++i) L.theta[i] = std::pow(static_cast<double>(rope_base), -i / 32.0);
  L.d_err = d_err;
  return cuda_status(launch_cache_write(L, static_cast<cudaStream_t>(stream)));
}

int dsa_decode_workspace_layout(const dsa_decode_desc* d, dsa_decode_layout* lay) {
  if (lay == nullptr) return DSA_ERR_INVALID_ARG;
  const int st = check_decode(d);
  if (st != DSA_OK) return st;
  const int64_t W = d->num_shards, R = d->rows.num_rows, k = d->topk, H = d->heads;
  dsa_decode_layout L;
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  L.ld_scores = align_up((d->rows.max_len + W - 1) / W, 4);
  L.scores = take(W * R * L.ld_scores * 4);
  if (W > 1) {
    L.cand_idx = take(W * R * k * 4);
    L.cand_score = take(W * R * k * 4);
    L.cand_count = take(W * R * 4);
    L.owned_local = take(W * R * k * 4);
    L.owned_count = take(W * R * 4);
  } else {
    L.cand_idx = L.cand_score = L.cand_count = L.owned_local = L.owned_count = -1;
  }
  L.topk_idx = d->out_topk_idx ? -1 : take(R * k * 4);
  L.topk_count = d->out_topk_count ? -1 : take(R * 4);
  L.topk_ws = take(static_cast<int64_t>(topk_workspace_bytes(static_cast<int>(W * R), L.ld_scores)));
  const int64_t expected = (k < d->rows.max_len ? k : d->rows.max_len) / W;
  const int S = resolve_splits(d->num_splits, static_cast<int>(W * R), static_cast<int>(k),
                               static_cast<int>(expected > 0 ? expected : 1));
  L.num_splits = S;
  L.num_parts = static_cast<int32_t>(W * S);
  if (L.num_parts > 1) {
    L.part_out = take(L.num_parts * R * H * kVDim * 4);
    L.part_lse = take(L.num_parts * R * H * 4);
  } else {
    L.part_out = L.part_lse = -1;
  }
  L.total_bytes = off;
  // indexer, top-k (three launches in its segment form), the shard merge,
  // the attention and the LSE merge of its parts
  L.launches = 1 + (topk_uses_workspace(static_cast<int>(W * R), L.ld_scores) ? 3 : 1) +
               (W > 1 ? 1 : 0) + 1 + (L.num_parts > 1 ? 1 : 0);
  L.reserved = 0;
  if (mla_smem_bytes(static_cast<int>(H), d->kv[0].dtype == DSA_DTYPE_FP8_E4M3,
                     split_chunk(S, static_cast<int>(k))) > 227 * 1024)
    return DSA_ERR_UNSUPPORTED;
  *lay = L;
  return DSA_OK;
}

size_t dsa_decode_workspace_size(const dsa_decode_desc* d) {
  dsa_decode_layout L;
  if (dsa_decode_workspace_layout(d, &L) != DSA_OK) return 0;
  return static_cast<size_t>(L.total_bytes);
}

int dsa_decode(const dsa_decode_desc* d, void* workspace, size_t workspace_bytes, int32_t* d_err,
               void* stream) {
  dsa_decode_layout lay;
  int st = dsa_decode_workspace_layout(d, &lay);
  if (st != DSA_OK) return st;
  if (d_err == nullptr) return DSA_ERR_INVALID_ARG;
  if (workspace_bytes < static_cast<size_t>(lay.total_bytes) ||
      (lay.total_bytes > 0 && workspace == nullptr))
    return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (d->rows.num_rows == 0) return DSA_OK;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int W = d->num_shards, R = d->rows.num_rows, k = d->topk;

  // The kernels after the indexer are programmatic dependents of the one
  // before them: each starts launching while its predecessor runs and waits
  // for it before touching the predecessor's outputs.  The indexer follows
  // the caller's work and is launched plainly.
  // 0. the top-k histograms and candidate counts start at zero
  if (topk_uses_workspace(W * R, lay.ld_scores) &&
      cudaMemsetAsync(ws + lay.topk_ws, 0, topk_workspace_clear_bytes(W * R), s) != cudaSuccess)
    return DSA_ERR_CUDA;
  // 1. indexer over every shard's cache, one launch
  {
    IndexerLaunch L{};
    for (int w = 0; w < W; ++w) {
      if (make_index_k_tmap(&L.kmap[w], d->idx_k[w]) != cudaSuccess) return DSA_ERR_CUDA;
      fill_indexer_shard(L, w, d->idx_k[w]);
    }
    L.page_size = d->idx_k[0].page_size;
    L.fp8 = d->idx_k[0].dtype == DSA_DTYPE_FP8_E4M3;
    L.W = W;
    L.shard_base = 0;
    L.nshards = W;
    L.q_idx = d->q_idx;
    L.w_idx = d->w_idx;
    L.row_start = d->rows.row_start;
    L.row_pos = d->rows.row_pos;
    L.num_rows = R;
    L.num_reqs = d->rows.num_reqs;
    set_row_groups(L, d->rows.max_rows_per_req);
    L.scores = reinterpret_cast<float*>(ws + lay.scores);
    L.ld = lay.ld_scores;
    L.shard_stride = static_cast<int64_t>(R) * lay.ld_scores;
    L.d_err = d_err;
    if (launch_indexer(L, s) != cudaSuccess) return DSA_ERR_CUDA;
  }
  int32_t* topk_idx =
      d->out_topk_idx ? d->out_topk_idx : reinterpret_cast<int32_t*>(ws + lay.topk_idx);
  int32_t* topk_cnt =
      d->out_topk_count ? d->out_topk_count : reinterpret_cast<int32_t*>(ws + lay.topk_count);
  // 2. (local) top-k of every shard's rows, global positions out
  {
    TopkLaunch L{};
    L.scores = reinterpret_cast<const float*>(ws + lay.scores);
    L.ld = lay.ld_scores;
    L.shard_stride = static_cast<int64_t>(R) * lay.ld_scores;
    L.valid_len = nullptr;
    L.row_pos = d->rows.row_pos;
    L.W = W;
    L.shard_offset = 0;
    L.rows = R;
    L.nshards = W;
    L.k = k;
    L.index_stride = W;
    L.index_offset = 0;
    L.offset_per_shard = 1;
    if (W > 1) {
      L.out_idx = reinterpret_cast<int32_t*>(ws + lay.cand_idx);
      L.out_score = reinterpret_cast<float*>(ws + lay.cand_score);
      L.out_count = reinterpret_cast<int32_t*>(ws + lay.cand_count);
    } else {
      L.out_idx = topk_idx;
      L.out_score = nullptr;
      L.out_count = topk_cnt;
    }
    L.d_err = d_err;
    topk_set_workspace(L, ws + lay.topk_ws);
    if (launch_topk(L, s, true) != cudaSuccess) return DSA_ERR_CUDA;
  }
  // 3. exact merge of the shards' candidates; owned local rows per shard
  if (W > 1) {
    MergeTopkLaunch L{reinterpret_cast<const float*>(ws + lay.cand_score),
                      reinterpret_cast<const int32_t*>(ws + lay.cand_idx),
                      reinterpret_cast<const int32_t*>(ws + lay.cand_count),
                      W,
                      R,
                      k,
                      topk_idx,
                      topk_cnt,
                      reinterpret_cast<int32_t*>(ws + lay.owned_local),
                      reinterpret_cast<int32_t*>(ws + lay.owned_count),
                      d_err,
                      d->rows.max_len};
    if (launch_shard_topk_merge(L, s, true) != cudaSuccess) return DSA_ERR_CUDA;
  }
  // 4. sparse MLA over each shard's owned rows, split-K
  {
    MlaLaunch L{};
    for (int w = 0; w < W; ++w) fill_mla_shard(L, w, d->kv[w]);
    L.page_size = d->kv[0].page_size;
    L.fp8 = d->kv[0].dtype == DSA_DTYPE_FP8_E4M3;
    L.nshards = W;
    L.q = d->q;
    L.heads = d->heads;
    L.sm_scale = d->sm_scale;
    L.row_start = d->rows.row_start;
    L.num_reqs = d->rows.num_reqs;
    L.rows = R;
    L.idx = W > 1 ? reinterpret_cast<const int32_t*>(ws + lay.owned_local) : topk_idx;
    L.count = W > 1 ? reinterpret_cast<const int32_t*>(ws + lay.owned_count) : topk_cnt;
    L.k = k;
    L.num_splits = lay.num_splits;
    L.chunk = split_chunk(lay.num_splits, k);
    L.out = d->out;
    L.out_lse = d->out_lse;
    if (lay.num_parts > 1) {
      L.part_out = reinterpret_cast<float*>(ws + lay.part_out);
      L.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
    }
    L.d_err = d_err;
    if (launch_sparse_mla(L, s, true) != cudaSuccess) return DSA_ERR_CUDA;
    // 5. LSE merge of the W * S partials
    if (lay.num_parts > 1 &&
        launch_lse_merge(L.part_out, L.part_lse, lay.num_parts, R, d->heads, kVDim, d->out,
                         d->out_lse, s, true) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // extern "C"
