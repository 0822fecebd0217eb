"""Python binding of the C ABI: the same entry points, taking torch CUDA
tensors.  This module only marshals arguments (pointers, sizes, the current
stream); every step of the decode runs in the library's kernels.  Non-OK
statuses raise DsaError."""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import _lib as C


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = C.lib().dsa_status_string(status).decode()
        super().__init__(f"{where}: {msg} ({status})")


def _check(status: int, where: str):
    if status != C.DSA_OK:
        raise DsaError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class PagedCache:
    """Device view of one paged cache (see dsa_paged_cache)."""

    data: torch.Tensor                   # [pages, page, row] int16/uint16 (bf16 bits) or uint8
    scale: Optional[torch.Tensor]        # [pages, page] fp32 (fp8 only)
    block_table: Optional[torch.Tensor]  # [B, max_blocks] int32 or None (contiguous)
    dtype: int
    page_size: int
    max_blocks: int

    def c(self) -> C.DsaPagedCache:
        return C.DsaPagedCache(
            data=_ptr(self.data), scale=_ptr(self.scale), block_table=_ptr(self.block_table),
            dtype=self.dtype, row_elems=int(self.data.shape[2]), page_size=self.page_size,
            num_pages=int(self.data.shape[0]), max_blocks=self.max_blocks)


@dataclass
class Rows:
    row_start: torch.Tensor   # [B+1] int32
    row_pos: torch.Tensor     # [R] int32
    max_rows_per_req: int
    max_len: int

    @property
    def num_rows(self) -> int:
        return int(self.row_pos.shape[0])

    @property
    def num_reqs(self) -> int:
        return int(self.row_start.shape[0]) - 1

    def c(self) -> C.DsaRows:
        return C.DsaRows(num_rows=self.num_rows, num_reqs=self.num_reqs,
                         max_rows_per_req=self.max_rows_per_req, max_len=self.max_len,
                         row_start=_ptr(self.row_start), row_pos=_ptr(self.row_pos))


def dsa_abi_version() -> int:
    return C.lib().dsa_abi_version()


def dsa_status_string(status: int) -> str:
    return C.lib().dsa_status_string(status).decode()


def dsa_read_error(d_err: torch.Tensor, stream=None) -> int:
    h = ctypes.c_int32(0)
    st = C.lib().dsa_read_error(_ptr(d_err), ctypes.byref(h), _stream(stream))
    if st not in (C.DSA_OK, C.DSA_ERR_DEVICE_CHECK):
        _check(st, "dsa_read_error")
    return int(h.value)


def dsa_selftest_bounded_wait(limit_us: int, d_err, d_waited_ns, stream=None):
    """The library's bounded on-chip wait on a phase nothing completes (see
    the header): sets DSA_DEVERR_TIMEOUT in d_err and the time waited (ns) in
    d_waited_ns (a one-element int64 tensor)."""
    _check(C.lib().dsa_selftest_bounded_wait(int(limit_us), _ptr(d_err), _ptr(d_waited_ns),
                                             _stream(stream)), "dsa_selftest_bounded_wait")


def dsa_indexer_scores(q_idx, w_idx, idx_k: PagedCache, rows: Rows, scores, d_err,
                       shard: int = 0, num_shards: int = 1, stream=None):
    c, r = idx_k.c(), rows.c()
    _check(C.lib().dsa_indexer_scores(_ptr(q_idx), _ptr(w_idx), ctypes.byref(c), ctypes.byref(r),
                                      shard, num_shards, _ptr(scores), int(scores.shape[1]),
                                      _ptr(d_err), _stream(stream)), "dsa_indexer_scores")


def dsa_topk_workspace_size(num_rows: int, ld_scores: int) -> int:
    return int(C.lib().dsa_topk_workspace_size(num_rows, ld_scores))


def dsa_topk(scores, valid_len, k: int, out_idx, out_count, d_err, out_score=None,
             index_stride: int = 1, index_offset: int = 0, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(C.lib().dsa_topk(_ptr(scores), int(scores.shape[1]), _ptr(valid_len),
                            int(scores.shape[0]), k, index_stride, index_offset, _ptr(out_idx),
                            _ptr(out_score), _ptr(out_count), _ptr(workspace), ws_bytes,
                            _ptr(d_err), _stream(stream)),
           "dsa_topk")


def dsa_cache_write(kv_in, tok_req, tok_pos, num_reqs: int, kv: Sequence[PagedCache], d_err,
                    idx_in=None, idx_k: Optional[Sequence[PagedCache]] = None,
                    rope_base: float = 10000.0, stream=None):
    """One decode step's cache write: the new tokens' latent rows (kv_in
    [N, 576] bf16 bits) and index-K rows (idx_in [N, 128]), RoPE on their last
    64 dims, stored on the owner shard (pos % W) of `kv` / `idx_k`."""
    W = len(kv)
    kvc = (C.DsaPagedCache * W)(*[c.c() for c in kv])
    ixc = (C.DsaPagedCache * W)(*[c.c() for c in idx_k]) if idx_k is not None else None
    _check(C.lib().dsa_cache_write(_ptr(kv_in), _ptr(idx_in), _ptr(tok_req), _ptr(tok_pos),
                                   int(tok_pos.shape[0]), int(num_reqs), float(rope_base), kvc,
                                   ixc, W, _ptr(d_err), _stream(stream)), "dsa_cache_write")


def dsa_shard_topk_merge(cand_score, cand_pos, cand_count, out_idx, out_count, owned_local,
                         owned_count, d_err, pos_bound: int = 0, stream=None):
    W, R, k = (int(x) for x in cand_score.shape)
    _check(C.lib().dsa_shard_topk_merge(_ptr(cand_score), _ptr(cand_pos), _ptr(cand_count), W, R,
                                        k, int(pos_bound), _ptr(out_idx), _ptr(out_count), _ptr(owned_local),
                                        _ptr(owned_count), _ptr(d_err), _stream(stream)),
           "dsa_shard_topk_merge")


def dsa_sparse_mla_decode_workspace_size(num_rows: int, heads: int, k: int,
                                         num_splits: int = 0) -> int:
    return int(C.lib().dsa_sparse_mla_decode_workspace_size(num_rows, heads, k, num_splits))


def dsa_sparse_mla_decode(q, sm_scale: float, kv: PagedCache, rows: Rows, idx, count, out,
                          out_lse, d_err, workspace=None, num_splits: int = 0, stream=None):
    c, r = kv.c(), rows.c()
    k = int(idx.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(C.lib().dsa_sparse_mla_decode(_ptr(q), int(q.shape[1]), float(sm_scale),
                                         ctypes.byref(c), ctypes.byref(r), _ptr(idx), _ptr(count),
                                         k, num_splits, _ptr(out), _ptr(out_lse),
                                         _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)),
           "dsa_sparse_mla_decode")


def dsa_sparse_mla_prefill_into_workspace_size(num_rows: int, heads: int, k: int,
                                               num_splits: int = 0) -> int:
    return int(C.lib().dsa_sparse_mla_prefill_into_workspace_size(num_rows, heads, k, num_splits))


def dsa_sparse_mla_prefill_into(q, sm_scale: float, kv: PagedCache, rows: Rows, idx, count, out,
                                out_max_logit, out_lse, d_err, workspace=None,
                                num_splits: int = 0, stream=None):
    """Sparse attention of many query rows into caller-owned O, max-logit and
    LSE buffers (see the header)."""
    c, r = kv.c(), rows.c()
    k = int(idx.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(C.lib().dsa_sparse_mla_prefill_into(_ptr(q), int(q.shape[1]), float(sm_scale),
                                               ctypes.byref(c), ctypes.byref(r), _ptr(idx),
                                               _ptr(count), k, num_splits, _ptr(out),
                                               _ptr(out_max_logit), _ptr(out_lse), _ptr(workspace),
                                               ws_bytes, _ptr(d_err), _stream(stream)),
           "dsa_sparse_mla_prefill_into")


def dsa_sparse_mla_decode_noalloc(q, sm_scale: float, kv: PagedCache, rows: Rows, idx, count,
                                  out, out_lse, d_err, num_splits: int = 0, stream=None):
    """dsa_sparse_mla_decode for callers that cannot allocate device memory:
    the split-K partials live in the library's fixed device array (see the
    header); calls that overlap on the GPU race on it."""
    c, r = kv.c(), rows.c()
    k = int(idx.shape[1])
    _check(C.lib().dsa_sparse_mla_decode_noalloc(_ptr(q), int(q.shape[1]), float(sm_scale),
                                                 ctypes.byref(c), ctypes.byref(r), _ptr(idx),
                                                 _ptr(count), k, num_splits, _ptr(out),
                                                 _ptr(out_lse), _ptr(d_err), _stream(stream)),
           "dsa_sparse_mla_decode_noalloc")


def dsa_lse_merge(O_parts, lse_parts, out, out_lse, stream=None):
    P, R, H, dv = (int(x) for x in O_parts.shape)
    _check(C.lib().dsa_lse_merge(_ptr(O_parts), _ptr(lse_parts), P, R, H, dv, _ptr(out),
                                 _ptr(out_lse), _stream(stream)), "dsa_lse_merge")


class DecodeDesc:
    """Holds a dsa_decode_desc and everything it points to."""

    def __init__(self, idx_k: Sequence[PagedCache], kv: Sequence[PagedCache], rows: Rows,
                 q_idx, w_idx, q, sm_scale: float, topk: int, out, out_lse,
                 num_splits: int = 0, out_topk_idx=None, out_topk_count=None):
        W = len(idx_k)
        assert len(kv) == W
        self._idx = (C.DsaPagedCache * W)(*[c.c() for c in idx_k])
        self._kv = (C.DsaPagedCache * W)(*[c.c() for c in kv])
        self._keep = (idx_k, kv, rows, q_idx, w_idx, q, out, out_lse, out_topk_idx, out_topk_count)
        self.desc = C.DsaDecodeDesc(
            num_shards=W,
            idx_k=ctypes.cast(self._idx, ctypes.POINTER(C.DsaPagedCache)),
            kv=ctypes.cast(self._kv, ctypes.POINTER(C.DsaPagedCache)),
            rows=rows.c(), q_idx=_ptr(q_idx), w_idx=_ptr(w_idx), q=_ptr(q),
            heads=int(q.shape[1]), sm_scale=float(sm_scale), topk=topk, num_splits=num_splits,
            out=_ptr(out), out_lse=_ptr(out_lse), out_topk_idx=_ptr(out_topk_idx),
            out_topk_count=_ptr(out_topk_count))


def dsa_decode_workspace_size(d: DecodeDesc) -> int:
    return int(C.lib().dsa_decode_workspace_size(ctypes.byref(d.desc)))


def dsa_decode_workspace_layout(d: DecodeDesc) -> C.DsaDecodeLayout:
    lay = C.DsaDecodeLayout()
    _check(C.lib().dsa_decode_workspace_layout(ctypes.byref(d.desc), ctypes.byref(lay)),
           "dsa_decode_workspace_layout")
    return lay


def dsa_decode(d: DecodeDesc, workspace, d_err, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(C.lib().dsa_decode(ctypes.byref(d.desc), _ptr(workspace), ws_bytes, _ptr(d_err),
                              _stream(stream)), "dsa_decode")
