"""ctypes view of ``include/dsa_decode.h``: structs and prototypes."""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

from ._build import LIB_PATH

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_WORKSPACE_TOO_SMALL = 3
DSA_ERR_CUDA = 4
DSA_ERR_DEVICE_CHECK = 5
DSA_ERR_TIMEOUT = 6

DSA_DEVERR_ROWS = 1 << 0
DSA_DEVERR_POS = 1 << 1
DSA_DEVERR_PAGE = 1 << 2
DSA_DEVERR_INDEX = 1 << 3
DSA_DEVERR_NAN = 1 << 4
DSA_DEVERR_TIMEOUT = 1 << 5
DSA_DEVERR_GROUP = 1 << 6

DSA_DTYPE_BF16 = 0
DSA_DTYPE_FP8_E4M3 = 1
DSA_MAX_ROWS_PER_REQ = 1024

INDEX_HEADS = 64
INDEX_DIM = 128
KV_DIM = 576
V_DIM = 512
MAX_SHARDS = 8
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class DsaPagedCache(ctypes.Structure):
    _fields_ = [
        ("data", c_void_p),
        ("scale", c_void_p),
        ("block_table", c_void_p),
        ("dtype", c_int32),
        ("row_elems", c_int32),
        ("page_size", c_int32),
        ("num_pages", c_int32),
        ("max_blocks", c_int32),
    ]


class DsaRows(ctypes.Structure):
    _fields_ = [
        ("num_rows", c_int32),
        ("num_reqs", c_int32),
        ("max_rows_per_req", c_int32),
        ("max_len", c_int32),
        ("row_start", c_void_p),
        ("row_pos", c_void_p),
    ]


class DsaDecodeDesc(ctypes.Structure):
    _fields_ = [
        ("num_shards", c_int32),
        ("idx_k", POINTER(DsaPagedCache)),
        ("kv", POINTER(DsaPagedCache)),
        ("rows", DsaRows),
        ("q_idx", c_void_p),
        ("w_idx", c_void_p),
        ("q", c_void_p),
        ("heads", c_int32),
        ("sm_scale", c_float),
        ("topk", c_int32),
        ("num_splits", c_int32),
        ("out", c_void_p),
        ("out_lse", c_void_p),
        ("out_topk_idx", c_void_p),
        ("out_topk_count", c_void_p),
    ]


class DsaDecodeLayout(ctypes.Structure):
    _fields_ = [
        ("scores", c_int64),
        ("ld_scores", c_int64),
        ("cand_idx", c_int64),
        ("cand_score", c_int64),
        ("cand_count", c_int64),
        ("topk_idx", c_int64),
        ("topk_count", c_int64),
        ("topk_ws", c_int64),
        ("owned_local", c_int64),
        ("owned_count", c_int64),
        ("part_out", c_int64),
        ("part_lse", c_int64),
        ("num_splits", c_int32),
        ("num_parts", c_int32),
        ("launches", c_int32),
        ("reserved", c_int32),
        ("total_bytes", c_int64),
    ]


# name -> (restype, argtypes), in the order of the header
PROTOTYPES = {
    "dsa_abi_version": (c_int, []),
    "dsa_status_string": (c_char_p, [c_int]),
    "dsa_read_error": (c_int, [c_void_p, POINTER(c_int32), c_void_p]),
    "dsa_selftest_bounded_wait": (c_int, [c_int32, c_void_p, c_void_p, c_void_p]),
    "dsa_indexer_scores": (c_int, [c_void_p, c_void_p, POINTER(DsaPagedCache), POINTER(DsaRows),
                                   c_int32, c_int32, c_void_p, c_int64, c_void_p, c_void_p]),
    "dsa_topk_workspace_size": (c_size_t, [c_int32, c_int64]),
    "dsa_topk": (c_int, [c_void_p, c_int64, c_void_p, c_int32, c_int32, c_int32, c_int32,
                         c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    "dsa_shard_topk_merge": (c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                     c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dsa_sparse_mla_decode_workspace_size": (c_size_t, [c_int32, c_int32, c_int32, c_int32]),
    "dsa_sparse_mla_decode": (c_int, [c_void_p, c_int32, c_float, POINTER(DsaPagedCache),
                                      POINTER(DsaRows), c_void_p, c_void_p, c_int32, c_int32,
                                      c_void_p, c_void_p, c_void_p, c_size_t, c_void_p,
                                      c_void_p]),
    "dsa_sparse_mla_prefill_into_workspace_size": (c_size_t, [c_int32, c_int32, c_int32, c_int32]),
    "dsa_sparse_mla_prefill_into": (c_int, [c_void_p, c_int32, c_float, POINTER(DsaPagedCache),
                                            POINTER(DsaRows), c_void_p, c_void_p, c_int32, c_int32,
                                            c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                            c_void_p, c_void_p]),
    "dsa_sparse_mla_decode_noalloc": (c_int, [c_void_p, c_int32, c_float, POINTER(DsaPagedCache),
                                              POINTER(DsaRows), c_void_p, c_void_p, c_int32,
                                              c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dsa_lse_merge": (c_int, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p,
                              c_void_p, c_void_p]),
    "dsa_cache_write": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float,
                                POINTER(DsaPagedCache), POINTER(DsaPagedCache), c_int32, c_void_p,
                                c_void_p]),
    "dsa_decode_workspace_size": (c_size_t, [POINTER(DsaDecodeDesc)]),
    "dsa_decode_workspace_layout": (c_int, [POINTER(DsaDecodeDesc), POINTER(DsaDecodeLayout)]),
    "dsa_decode": (c_int, [POINTER(DsaDecodeDesc), c_void_p, c_size_t, c_void_p, c_void_p]),
}

_LIB = None


def lib(path: str = LIB_PATH):
    """Load the library (once).  Raises if it has not been built: there is no
    fallback implementation."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L
