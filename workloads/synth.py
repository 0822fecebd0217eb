"""Seeded synthetic decode batches shaped like the DCP/DSA serving workloads.

Recipe (the same for every configuration; only the sizes change):

* indexer query ``q_idx`` [R, 64, 128]: N(0, 1) drawn in fp32, stored as bf16
  (round to nearest even);
* indexer head weights ``w_idx`` [R, 64]: U(0, 1) / 8, fp32;
* indexer keys, one 128-wide row per cached token: N(0, 1);
* MLA query ``q`` [R, H, 576] and latent cache rows (576 = 512 + 64 rope):
  N(0, 0.5) (0.5 is the standard deviation);
* bf16 caches store the draws rounded to bf16; fp8 caches store e4m3 codes of
  ``x / s`` with the per-token fp32 scale ``s = amax(|x|) / 448``;
* paged caches have 64-token pages; a request's logical page j lives in the
  physical page ``block_table[b, j]`` (a seeded random permutation of all
  pages), entries past the request's span are -1;
* a request with ``rows_per_req`` query rows (MTP/EAGLE verify) has them at the
  consecutive positions L-rows .. L-1; row r attends tokens 0..pos[r];
* a sharded workload (decode context parallel) keeps token t on shard
  ``t % W`` at shard-local position ``t // W`` with its own block table, and
  also carries the unsharded cache holding the very same stored values.

Random numbers come from numpy's PCG64 streams keyed by
(seed, stream id, chunk id), so every value is independent of the thread count
used to fill the arrays.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np

PAGE = 64
IDX_HEADS = 64
IDX_DIM = 128
KV_DIM = 576
V_DIM = 512
TOPK = 2048
FP8_MAX = 448.0

_CHUNK_PAGES = 128  # pages drawn per random stream chunk

# stream ids (keep stable: they define the data)
_S_LEN, _S_PERM, _S_QIDX, _S_W, _S_Q, _S_IDXK, _S_KV, _S_SHARDPERM = range(8)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, chunk])


# ----------------------------------------------------------------------------
# storage encodings (input synthesis only)
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def to_e4m3_codes(v: np.ndarray) -> np.ndarray:
    """fp32 -> OCP fp8 E4M3 (E4M3FN) code, round to nearest even, saturating
    at +-448.  Inputs are expected to be finite."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    bits = v.view(np.uint32).astype(np.int64)
    sign = (bits >> 24) & 0x80
    mag = bits & 0x7FFFFFFF
    # normal results: keep 3 mantissa bits with round-half-even, then move the
    # exponent bias from 127 to 7
    r = mag + 0x7FFFF + ((mag >> 20) & 1)
    code_n = np.minimum((r >> 20) - (120 << 3), 0x7E)
    # subnormal results (|v| < 2^-6): multiples of 2^-9
    a = np.abs(v)
    code_s = np.rint(a * np.float32(512.0)).astype(np.int64)
    code = np.where(a < np.float32(2.0 ** -6), code_s, code_n)
    return (code | sign).astype(np.uint8)


# ----------------------------------------------------------------------------
# data classes
# ----------------------------------------------------------------------------

@dataclass
class PagedCache:
    """One paged cache: ``data[page, slot, :]`` holds one token row."""

    data: np.ndarray                 # uint16 (bf16 bits) or uint8 (e4m3 codes)
    scale: Optional[np.ndarray]      # fp32 [num_pages, page] for fp8, else None
    dtype: str                       # "bf16" | "fp8_e4m3"
    block_table: Optional[np.ndarray]  # int32 [B, max_blocks]; None = contiguous
    max_blocks: int
    seq_len: np.ndarray              # int32 [B]: tokens stored per request
    page_size: int = PAGE

    @property
    def num_pages(self) -> int:
        return int(self.data.shape[0])

    @property
    def row_elems(self) -> int:
        return int(self.data.shape[2])

    def physical_page(self, b: int, j: int) -> int:
        if self.block_table is None:
            return b * self.max_blocks + j
        return int(self.block_table[b, j])

    def nbytes(self) -> int:
        n = self.data.nbytes
        if self.scale is not None:
            n += self.scale.nbytes
        if self.block_table is not None:
            n += self.block_table.nbytes
        return n


@dataclass
class Spec:
    name: str
    seed: int
    B: int
    length_law: str = "fixed"        # fixed | uniform | loguniform
    L: int = 4096                    # fixed length
    L_lo: int = 4096                 # uniform / loguniform bounds (inclusive)
    L_hi: int = 4096
    rows_per_req: int = 1
    H: int = 32
    dtype: str = "bf16"              # bf16 | fp8_e4m3
    shards: int = 1
    paged: bool = True
    page_size: int = PAGE
    topk: int = TOPK
    seq_lens: Optional[tuple] = None  # explicit per-request lengths

    @property
    def R(self) -> int:
        return self.B * self.rows_per_req


@dataclass
class Workload:
    spec: Spec
    seq_len: np.ndarray        # int32 [B]
    row_start: np.ndarray      # int32 [B+1]
    row_pos: np.ndarray        # int32 [R]
    row_req: np.ndarray        # int32 [R]
    q_idx: np.ndarray          # uint16 bf16 bits [R, 64, 128]
    w_idx: np.ndarray          # fp32 [R, 64]
    q: np.ndarray              # uint16 bf16 bits [R, H, 576]
    idx_k: PagedCache          # unsharded index-K cache
    kv: PagedCache             # unsharded latent cache
    idx_k_shards: List[PagedCache] = field(default_factory=list)
    kv_shards: List[PagedCache] = field(default_factory=list)
    sm_scale: float = KV_DIM ** -0.5

    @property
    def R(self) -> int:
        return int(self.row_pos.shape[0])

    @property
    def B(self) -> int:
        return int(self.seq_len.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def W(self) -> int:
        return len(self.idx_k_shards)

    @property
    def topk(self) -> int:
        return self.spec.topk

    @property
    def max_len(self) -> int:
        return int(self.seq_len.max())


# ----------------------------------------------------------------------------
# the five configurations
# ----------------------------------------------------------------------------

CONFIG_NAMES = {
    0: "tiny-1row-L4096-bf16-H16-contiguous",
    1: "B32-L32768-bf16-H32-paged",
    2: "B64x6mtp-L16K..64K-fp8-H32-paged",
    3: "B4-L80000-bf16-H32-W4-sharded",
    4: "ragged-B{B}-L4K..128K-loguniform-fp8-H32-paged",
}


def config_spec(i: int, **overrides) -> Spec:
    """Spec of configuration ``i`` (0..4); keyword overrides shrink it for
    tests (e.g. ``B=2``)."""
    if i == 0:
        s = Spec(name=CONFIG_NAMES[0], seed=0, B=1, L=4096, H=16, paged=False)
    elif i == 1:
        s = Spec(name=CONFIG_NAMES[1], seed=1, B=32, L=32768, H=32)
    elif i == 2:
        s = Spec(name=CONFIG_NAMES[2], seed=2, B=64, length_law="uniform",
                 L_lo=16384, L_hi=65536, rows_per_req=6, H=32, dtype="fp8_e4m3")
    elif i == 3:
        s = Spec(name=CONFIG_NAMES[3], seed=3, B=4, L=80000, H=32, shards=4)
    elif i == 4:
        B = overrides.pop("B", 64)
        s = Spec(name=CONFIG_NAMES[4].format(B=B), seed=4, B=B,
                 length_law="loguniform", L_lo=4096, L_hi=131072, H=32,
                 dtype="fp8_e4m3")
    else:
        raise ValueError(f"no configuration {i}")
    return replace(s, **overrides)


# ----------------------------------------------------------------------------
# generation
# ----------------------------------------------------------------------------

def _draw_lengths(spec: Spec) -> np.ndarray:
    if spec.seq_lens is not None:
        L = np.asarray(spec.seq_lens, dtype=np.int64)
        assert L.shape == (spec.B,)
    elif spec.length_law == "fixed":
        L = np.full(spec.B, spec.L, dtype=np.int64)
    else:
        rng = _rng(spec.seed, _S_LEN)
        if spec.length_law == "uniform":
            L = rng.integers(spec.L_lo, spec.L_hi + 1, size=spec.B)
        elif spec.length_law == "loguniform":
            u = rng.uniform(math.log(spec.L_lo), math.log(spec.L_hi), size=spec.B)
            L = np.rint(np.exp(u)).astype(np.int64)
            L = np.clip(L, spec.L_lo, spec.L_hi)
        else:
            raise ValueError(spec.length_law)
    if np.any(L < spec.rows_per_req):
        raise ValueError("every request needs at least rows_per_req tokens")
    return L.astype(np.int32)


def _block_table(lens: np.ndarray, page: int, paged: bool, seed: int,
                 stream: int):
    nblk = (lens.astype(np.int64) + page - 1) // page
    max_blocks = int(nblk.max())
    B = len(lens)
    if not paged:
        return None, max_blocks, B * max_blocks
    total = int(nblk.sum())
    perm = _rng(seed, stream).permutation(total).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, max_blocks, total


def _fill_pool(num_pages: int, page: int, dim: int, std: float, dtype: str,
               seed: int, stream: int):
    """Draw ``num_pages`` pages of N(0, std) token rows and store them."""
    if dtype == "bf16":
        data = np.empty((num_pages, page, dim), dtype=np.uint16)
        scale = None
    elif dtype == "fp8_e4m3":
        data = np.empty((num_pages, page, dim), dtype=np.uint8)
        scale = np.empty((num_pages, page), dtype=np.float32)
    else:
        raise ValueError(dtype)

    def work(c):
        p0 = c * _CHUNK_PAGES
        p1 = min(num_pages, p0 + _CHUNK_PAGES)
        x = _rng(seed, stream, c).standard_normal((p1 - p0, page, dim),
                                                  dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if dtype == "bf16":
            data[p0:p1] = to_bf16_bits(x)
        else:
            amax = np.abs(x).max(axis=2)
            s = (amax / np.float32(FP8_MAX)).astype(np.float32)
            scale[p0:p1] = s
            data[p0:p1] = to_e4m3_codes(x / s[:, :, None])

    nchunks = (num_pages + _CHUNK_PAGES - 1) // _CHUNK_PAGES
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(nchunks)))
    return data, scale


def _make_cache(lens, spec: Spec, dim: int, std: float, dtype: str,
                stream: int) -> PagedCache:
    bt, max_blocks, num_pages = _block_table(lens, spec.page_size, spec.paged,
                                             spec.seed, stream * 16 + _S_PERM)
    data, scale = _fill_pool(num_pages, spec.page_size, dim, std, dtype,
                             spec.seed, stream)
    return PagedCache(data=data, scale=scale, dtype=dtype, block_table=bt,
                      max_blocks=max_blocks, seq_len=lens.astype(np.int32),
                      page_size=spec.page_size)


def _logical_rows(c: PagedCache, b: int, n: int):
    """Stored rows (and scales) of request b's first n logical tokens."""
    P = c.page_size
    nblk = (n + P - 1) // P
    pages = np.array([c.physical_page(b, j) for j in range(nblk)], dtype=np.int64)
    rows = c.data[pages].reshape(nblk * P, c.row_elems)[:n]
    sc = None
    if c.scale is not None:
        sc = c.scale[pages].reshape(nblk * P)[:n]
    return rows, sc


def _shard_cache(full: PagedCache, W: int, w: int, spec: Spec,
                 stream: int) -> PagedCache:
    """Owner rule: token t lives on shard t % W at local position t // W."""
    lens = full.seq_len.astype(np.int64)
    loc = np.maximum(0, (lens - w + W - 1) // W).astype(np.int32)
    bt, max_blocks, num_pages = _block_table(
        np.maximum(loc, 1), spec.page_size, spec.paged, spec.seed,
        stream * 16 + _S_SHARDPERM)
    P = spec.page_size
    data = np.zeros((num_pages, P, full.row_elems), dtype=full.data.dtype)
    scale = None
    if full.scale is not None:
        scale = np.ones((num_pages, P), dtype=np.float32)
    c = PagedCache(data=data, scale=scale, dtype=full.dtype, block_table=bt,
                   max_blocks=max_blocks, seq_len=loc, page_size=P)
    for b in range(len(lens)):
        rows, sc = _logical_rows(full, b, int(lens[b]))
        rows = rows[w::W]
        n = rows.shape[0]
        for j0 in range(0, n, P):
            j1 = min(n, j0 + P)
            p = c.physical_page(b, j0 // P)
            data[p, : j1 - j0] = rows[j0:j1]
            if scale is not None:
                scale[p, : j1 - j0] = sc[w::W][j0:j1]
    return c


def make_workload(spec: Spec) -> Workload:
    lens = _draw_lengths(spec)
    B, rpr, H = spec.B, spec.rows_per_req, spec.H
    R = B * rpr
    row_start = (np.arange(B + 1, dtype=np.int32) * rpr).astype(np.int32)
    row_req = np.repeat(np.arange(B, dtype=np.int32), rpr)
    row_pos = (np.repeat(lens, rpr) - rpr
               + np.tile(np.arange(rpr, dtype=np.int32), B)).astype(np.int32)

    q_idx = to_bf16_bits(_rng(spec.seed, _S_QIDX).standard_normal(
        (R, IDX_HEADS, IDX_DIM), dtype=np.float32))
    w_idx = (_rng(spec.seed, _S_W).random((R, IDX_HEADS), dtype=np.float32)
             / np.float32(8.0)).astype(np.float32)
    q = to_bf16_bits(np.float32(0.5) * _rng(spec.seed, _S_Q).standard_normal(
        (R, H, KV_DIM), dtype=np.float32))

    idx_k = _make_cache(lens, spec, IDX_DIM, 1.0, spec.dtype, _S_IDXK)
    kv = _make_cache(lens, spec, KV_DIM, 0.5, spec.dtype, _S_KV)

    if spec.shards > 1:
        W = spec.shards
        idx_sh = [_shard_cache(idx_k, W, w, spec, 100 + w) for w in range(W)]
        kv_sh = [_shard_cache(kv, W, w, spec, 200 + w) for w in range(W)]
    else:
        idx_sh, kv_sh = [idx_k], [kv]

    return Workload(spec=spec, seq_len=lens, row_start=row_start,
                    row_pos=row_pos, row_req=row_req, q_idx=q_idx, w_idx=w_idx,
                    q=q, idx_k=idx_k, kv=kv, idx_k_shards=idx_sh,
                    kv_shards=kv_sh)
