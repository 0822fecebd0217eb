"""The C-ABI library without a GPU: it builds, loads, exports every symbol
the header declares, and rejects bad host arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

import dsa_sparse_attention_decode_gb300 as pkg
from dsa_sparse_attention_decode_gb300 import _lib as C

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dsa_decode.h")


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return pkg.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(dsa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_documented_entry_points():
    names = _declared()
    for n in ("dsa_indexer_scores", "dsa_topk", "dsa_shard_topk_merge", "dsa_sparse_mla_decode",
              "dsa_lse_merge", "dsa_decode", "dsa_decode_workspace_size", "dsa_abi_version"):
        assert n in names
    assert set(names) == set(C.PROTOTYPES), "binding prototypes out of sync with the header"


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.dsa_abi_version() == 3
    for s in range(7):
        assert lib.dsa_status_string(s).startswith(b"DSA_")
    assert lib.dsa_status_string(99) == b"unknown dsa status"


def test_host_validation_rejects_bad_arguments(lib):
    err = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # k out of range
    assert lib.dsa_topk(ctypes.c_void_p(16), 10, ctypes.c_void_p(16), 1, 0, 1, 0,
                        ctypes.c_void_p(16), None, ctypes.c_void_p(16), None, 0, err,
                        None) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_topk(ctypes.c_void_p(16), 10, ctypes.c_void_p(16), 1, 5000, 1, 0,
                        ctypes.c_void_p(16), None, ctypes.c_void_p(16), None, 0, err,
                        None) == C.DSA_ERR_INVALID_ARG
    # a workspace below the size
    need = lib.dsa_topk_workspace_size(3, 5000)
    assert need > 0
    assert lib.dsa_topk(ctypes.c_void_p(16), 5000, ctypes.c_void_p(16), 3, 64, 1, 0,
                        ctypes.c_void_p(16), None, ctypes.c_void_p(16), ctypes.c_void_p(256),
                        need - 1, err, None) == C.DSA_ERR_WORKSPACE_TOO_SMALL
    # zero rows: nothing to do, no CUDA call
    assert lib.dsa_topk(None, 10, None, 0, 64, 1, 0, None, None, None, None, 0, err,
                        None) == C.DSA_OK
    # unsupported head count
    cache = C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=0, row_elems=576,
                            page_size=64, num_pages=4, max_blocks=4)
    rows = C.DsaRows(num_rows=1, num_reqs=1, max_rows_per_req=1, max_len=10, row_start=16,
                     row_pos=16)
    st = lib.dsa_sparse_mla_decode(ctypes.c_void_p(16), 64, 0.1, ctypes.byref(cache),
                                   ctypes.byref(rows), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   2048, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None, 0,
                                   err, None)
    assert st == C.DSA_ERR_UNSUPPORTED
    # page size not a multiple of 64
    cache.page_size = 48
    st = lib.dsa_sparse_mla_decode(ctypes.c_void_p(16), 32, 0.1, ctypes.byref(cache),
                                   ctypes.byref(rows), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   2048, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None, 0,
                                   err, None)
    assert st == C.DSA_ERR_INVALID_ARG
    # fp8 cache without scales
    cache.page_size, cache.dtype = 64, 1
    st = lib.dsa_indexer_scores(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.byref(
        C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=1, row_elems=128,
                        page_size=64, num_pages=4, max_blocks=4)), ctypes.byref(rows), 0, 1,
        ctypes.c_void_p(16), 16, err, None)
    assert st == C.DSA_ERR_INVALID_ARG
    # more rows per request than supported
    rows.max_rows_per_req = C.DSA_MAX_ROWS_PER_REQ + 1
    st = lib.dsa_indexer_scores(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.byref(
        C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=0, row_elems=128,
                        page_size=64, num_pages=4, max_blocks=4)), ctypes.byref(rows), 0, 1,
        ctypes.c_void_p(16), 16, err, None)
    assert st == C.DSA_ERR_UNSUPPORTED


def test_prefill_into_host_checks(lib):
    """The sparse-prefill entry point's caller-owned contract, without a GPU:
    the max-logit buffer is required, the workspace holds the partial maxima
    beside the partial outputs and LSEs, and a short workspace is refused
    before any launch."""
    err = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    cache = C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=0, row_elems=576,
                            page_size=64, num_pages=64, max_blocks=64)
    rows = C.DsaRows(num_rows=3, num_reqs=1, max_rows_per_req=3, max_len=4096, row_start=16,
                     row_pos=16)
    args = (ctypes.c_void_p(16), 32, 0.1, ctypes.byref(cache), ctypes.byref(rows),
            ctypes.c_void_p(16), ctypes.c_void_p(16), 2048, 4, ctypes.c_void_p(16))
    # no max-logit buffer
    assert lib.dsa_sparse_mla_prefill_into(*args, None, ctypes.c_void_p(16), None, 0, err,
                                           None) == C.DSA_ERR_INVALID_ARG
    # 4 splits: decode's partials plus 4 x rows x heads maxima (256-byte aligned)
    dec = lib.dsa_sparse_mla_decode_workspace_size(3, 32, 2048, 4)
    pre = lib.dsa_sparse_mla_prefill_into_workspace_size(3, 32, 2048, 4)
    assert dec > 0 and pre - dec == -(-(4 * 3 * 32 * 4) // 256) * 256
    assert lib.dsa_sparse_mla_prefill_into_workspace_size(3, 32, 2048, 1) == 0
    assert lib.dsa_sparse_mla_prefill_into(*args, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                           ctypes.c_void_p(256), pre - 1, err,
                                           None) == C.DSA_ERR_WORKSPACE_TOO_SMALL
    # zero rows: nothing to do
    rows.num_rows = 0
    assert lib.dsa_sparse_mla_prefill_into(*args, None, None, None, 0, err, None) == C.DSA_OK


def test_decode_workspace_layout_host_only(lib):
    ik = (C.DsaPagedCache * 2)(
        *[C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=0, row_elems=128,
                          page_size=64, num_pages=8, max_blocks=4) for _ in range(2)])
    kv = (C.DsaPagedCache * 2)(
        *[C.DsaPagedCache(data=16, scale=None, block_table=None, dtype=0, row_elems=576,
                          page_size=64, num_pages=8, max_blocks=4) for _ in range(2)])
    d = C.DsaDecodeDesc(num_shards=2, idx_k=ctypes.cast(ik, ctypes.POINTER(C.DsaPagedCache)),
                        kv=ctypes.cast(kv, ctypes.POINTER(C.DsaPagedCache)),
                        rows=C.DsaRows(num_rows=3, num_reqs=3, max_rows_per_req=1, max_len=501,
                                       row_start=16, row_pos=16),
                        q_idx=16, w_idx=16, q=16, heads=32, sm_scale=0.04, topk=256,
                        num_splits=2, out=16, out_lse=16, out_topk_idx=None,
                        out_topk_count=None)
    lay = C.DsaDecodeLayout()
    assert lib.dsa_decode_workspace_layout(ctypes.byref(d), ctypes.byref(lay)) == C.DSA_OK
    assert lay.ld_scores == 252  # ceil(501 / 2) rounded up to 4
    assert lay.num_splits == 2 and lay.num_parts == 4
    regions = sorted((getattr(lay, f), f) for f in ("scores", "cand_idx", "cand_score",
                                                      "cand_count", "topk_idx", "topk_count",
                                                      "owned_local", "owned_count", "part_out",
                                                      "part_lse"))
    assert all(off % 256 == 0 for off, _ in regions)
    assert lib.dsa_decode_workspace_size(ctypes.byref(d)) == lay.total_bytes
    # a workspace that is too small is refused before any launch
    assert lib.dsa_decode(ctypes.byref(d), ctypes.c_void_p(256), lay.total_bytes - 1,
                          ctypes.c_void_p(16), None) == C.DSA_ERR_WORKSPACE_TOO_SMALL


def test_selftest_bounded_wait_rejects_bad_limits(lib):
    assert lib.dsa_selftest_bounded_wait(-1, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_selftest_bounded_wait(3_000_000, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_selftest_bounded_wait(10, None, ctypes.c_void_p(16), None) == C.DSA_ERR_INVALID_ARG


def test_shard_merge_host_checks(lib):
    """The candidate merge's argument checks, before any launch: shard count,
    k, a negative position bound, the error word; zero rows is a no-op."""
    p = ctypes.c_void_p(16)
    args = lambda W, k, bound, err=p: (p, p, p, W, 4, k, bound, p, p, p, p, err, None)  # noqa: E731
    assert lib.dsa_shard_topk_merge(*args(0, 256, 0)) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_shard_topk_merge(*args(C.MAX_SHARDS + 1, 256, 0)) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_shard_topk_merge(*args(2, 0, 0)) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_shard_topk_merge(*args(2, 5000, 0)) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_shard_topk_merge(*args(2, 256, -1)) == C.DSA_ERR_INVALID_ARG
    assert lib.dsa_shard_topk_merge(*args(2, 256, 0, None)) == C.DSA_ERR_INVALID_ARG
    # no rows: nothing to launch
    assert lib.dsa_shard_topk_merge(p, p, p, 2, 0, 256, 1000, p, p, p, p, p, None) == C.DSA_OK
