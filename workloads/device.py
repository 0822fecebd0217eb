"""Copy a generated workload to device tensors in the binding's layout (the
KV / index-K caches, block tables, row metadata and queries).  Pure data
movement; used by the GPU tests and the benchmark."""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

from dsa_sparse_attention_decode_gb300 import api
from dsa_sparse_attention_decode_gb300._lib import DSA_DTYPE_BF16, DSA_DTYPE_FP8_E4M3

from .synth import PagedCache, Workload


def _t(a: Optional[np.ndarray], device, pin=False):
    if a is None:
        return None
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(np.ascontiguousarray(a))
    if pin:
        t = t.pin_memory()
    return t.to(device, non_blocking=False)


def cache_to_device(c: PagedCache, device) -> api.PagedCache:
    return api.PagedCache(
        data=_t(c.data, device), scale=_t(c.scale, device),
        block_table=_t(c.block_table, device),
        dtype=DSA_DTYPE_BF16 if c.dtype == "bf16" else DSA_DTYPE_FP8_E4M3,
        page_size=c.page_size, max_blocks=c.max_blocks)


@dataclass
class DeviceWorkload:
    wl: Workload
    rows: api.Rows
    q_idx: torch.Tensor
    w_idx: torch.Tensor
    q: torch.Tensor
    idx_k: api.PagedCache
    kv: api.PagedCache
    idx_k_shards: List[api.PagedCache]
    kv_shards: List[api.PagedCache]


def upload(wl: Workload, device="cuda", shards: bool = True, unsharded: bool = True) -> DeviceWorkload:
    rows = api.Rows(row_start=_t(wl.row_start, device), row_pos=_t(wl.row_pos, device),
                    max_rows_per_req=wl.spec.rows_per_req, max_len=int(wl.row_pos.max()) + 1)
    idx_k = cache_to_device(wl.idx_k, device) if unsharded or wl.W == 1 else None
    kv = cache_to_device(wl.kv, device) if unsharded or wl.W == 1 else None
    if wl.W == 1:
        idx_sh, kv_sh = [idx_k], [kv]
    elif shards:
        idx_sh = [cache_to_device(c, device) for c in wl.idx_k_shards]
        kv_sh = [cache_to_device(c, device) for c in wl.kv_shards]
    else:
        idx_sh, kv_sh = [], []
    return DeviceWorkload(wl=wl, rows=rows, q_idx=_t(wl.q_idx, device),
                          w_idx=_t(wl.w_idx, device), q=_t(wl.q, device), idx_k=idx_k, kv=kv,
                          idx_k_shards=idx_sh, kv_shards=kv_sh)


def decode_args(dw: DeviceWorkload, sharded: bool, out, out_lse, out_topk_idx=None,
                out_topk_count=None, num_splits: int = 0) -> api.DecodeDesc:
    if sharded:
        ik, kv = dw.idx_k_shards, dw.kv_shards
    else:
        ik, kv = [dw.idx_k], [dw.kv]
    return api.DecodeDesc(ik, kv, dw.rows, dw.q_idx, dw.w_idx, dw.q, dw.wl.sm_scale,
                          dw.wl.topk, out, out_lse, num_splits=num_splits,
                          out_topk_idx=out_topk_idx, out_topk_count=out_topk_count)
