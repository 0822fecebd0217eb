"""Float64 CPU oracle of DSA sparse-attention decode.

TEST INFRASTRUCTURE.  Imported only by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It shares
no code with the CUDA library; both read the same seeded inputs.

Sources (page title, section):

* "[ROCm] Support decode context parallel (DCP) for GLM-5 / DeepSeek-V3.2"
  (sgl-project/sglang pull request 42618) -- Motivation: DSA selects the top
  2048 tokens of the whole sequence before attention; Modifications (Writes,
  Indexer decode, Sparse decode): owner rule ``slot % W``, per-shard local
  top-k, exact merge of (score, global position) candidates into the global
  top-k, owned-slot attention returning a natural-log LSE, LSE merge of the
  partial results; commit "Triton sparse decode: store a lone split's output
  and LSE in place".
* "Harden DeepSeek V4 DSpark DP2 serving" (shiftup-ai/sglang pull request 1),
  section 6.3: caller-owned output / LSE buffers.

Readings where the pages say nothing (each is listed with its reason in the
design notes):

* indexer score of token t for a query row:
  ``s_t = sum_h w_h * max(0, q_h . k_t)`` over 64 heads of width 128, no
  extra scale;
* fp8 caches: stored value = e4m3 code value * per-token fp32 scale;
* attention logits ``z_t = tau * (q . kv_t)`` over all 576 latent dims with
  ``tau = 1/sqrt(576)``; the value vector is the first 512 dims of the same row;
* selection order: score descending, then token position ascending (a tie
  at the k-th place goes to the lower position); the selected positions are
  listed in ascending order; with fewer valid tokens than k all are kept;
* a row at position ``pos`` sees tokens 0..pos;
* an empty partial (no tokens) has LSE = -inf and contributes nothing;
* cache write (Modifications / Writes and the fused RoPE + cache write the
  page names): RoPE on the last 64 dims of each row in consecutive pairs,
  pair i rotated counter-clockwise by pos * base^(-i/32); a token is stored
  only on shard pos % W at local position pos // W; fp8 rows store e4m3 codes
  of value / s with s = max|value| / 448, both decided in fp32.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms, brute force, library routines,
invariants); none is "parity unpinned".
"""

from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

NEG_INF = -math.inf

# ----------------------------------------------------------------------------
# stored-value decoding
# ----------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper half of an IEEE-754 binary32: widen and read."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def e4m3_code_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent 0 is subnormal (2^-6 * m/8); the only
    NaN encodings are S.1111.111; there is no infinity."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = s * (2.0 ** -6) * (m / 8.0)
    nrm = s * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    v = np.where(e == 0, sub, nrm)
    return np.where((e == 15) & (c & 0x7 == 7), np.nan, v)


def decode_rows(data: np.ndarray, scale: Optional[np.ndarray], dtype: str) -> np.ndarray:
    """Stored cache rows -> float64 values (fp8 rows times their token scale)."""
    if dtype == "bf16":
        return bf16_bits_to_f64(data)
    if dtype == "fp8_e4m3":
        v = e4m3_code_to_f64(data)
        return v * np.asarray(scale, dtype=np.float64)[..., None]
    raise ValueError(dtype)


def cache_rows(cache, b: int, positions: np.ndarray) -> np.ndarray:
    """Float64 rows of request b's logical tokens ``positions`` of a paged
    cache (page = position // page_size through the block table)."""
    positions = np.asarray(positions, dtype=np.int64)
    P = cache.page_size
    if cache.block_table is None:
        pages = b * cache.max_blocks + positions // P
    else:
        pages = cache.block_table[b, positions // P].astype(np.int64)
        if np.any(pages < 0):
            raise ValueError("block table holds -1 inside the request's span")
    slots = positions % P
    data = cache.data[pages, slots]
    scale = cache.scale[pages, slots] if cache.scale is not None else None
    return decode_rows(data, scale, cache.dtype)


# ----------------------------------------------------------------------------
# indexer scoring
# ----------------------------------------------------------------------------


def indexer_scores(q_idx: np.ndarray, w: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Indexer score of every token row of K for one query row:
    ``s_t = sum_h w_h * max(0, q_h . k_t)``.

    q_idx: [heads, d] float64, w: [heads], K: [n, d]  ->  [n] float64.
    The DCP page (Motivation) only says that the indexer scores the whole
    sequence so that the top 2048 can be picked before attention; the formula
    is the reading stated in the module docstring."""
    q_idx = np.asarray(q_idx, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    logits = K @ q_idx.T                    # [n, heads]
    return np.maximum(logits, 0.0) @ w      # [n]


# ----------------------------------------------------------------------------
# exact top-k
# ----------------------------------------------------------------------------


def topk_select(scores: np.ndarray, k: int, positions: Optional[np.ndarray] = None
                ) -> np.ndarray:
    """Exact top-k (DCP page, Motivation: "the top 2048 tokens of the whole
    sequence").  Full sort by score descending, then position ascending; the
    first min(k, n) entries are the selection.  The pages fix which tokens
    are kept, not the order of the list: it is reported in ascending position
    order.  Returns the positions (default positions 0..n-1)."""
    s = np.asarray(scores, dtype=np.float64)
    if np.any(np.isnan(s)):
        raise ValueError("NaN score")
    n = s.shape[0]
    pos = np.arange(n, dtype=np.int64) if positions is None else np.asarray(positions, dtype=np.int64)
    order = np.lexsort((pos, -s))           # last key is the primary key
    return np.sort(pos[order[: min(k, n)]])


# ----------------------------------------------------------------------------
# absorbed-MLA attention over a selected set, LSE, LSE merge
# ----------------------------------------------------------------------------


def mla_attention(q: np.ndarray, KV: np.ndarray, tau: float, dv: int = 512
                  ) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of every head of one query row over the selected
    latent rows (DCP page, Modifications - Sparse decode: the kernel returns
    the output and the LSE).

    q: [H, D], KV: [m, D] (value = first dv dims of each row).
    z = tau * q . kv; lse = max z + ln sum exp(z - max z) (natural log);
    O = sum exp(z - lse) * v.  m = 0 gives O = 0 and lse = -inf."""
    q = np.asarray(q, dtype=np.float64)
    KV = np.asarray(KV, dtype=np.float64)
    H = q.shape[0]
    if KV.shape[0] == 0:
        return np.zeros((H, dv)), np.full(H, NEG_INF)
    z = tau * (q @ KV.T)                     # [H, m]
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
    p = np.exp(z - lse[:, None])
    return p @ KV[:, :dv], lse


def mla_attention_into(q: np.ndarray, KV: np.ndarray, tau: float, dv: int = 512
                       ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The three outputs of a sparse-prefill call that writes into caller-owned
    buffers (DSpark page, section 6.3: output, max-logit and LSE together):
    O and lse as in mla_attention, and max_logit = max over the selected rows
    of z = tau * q . kv (natural units, the scaled logit itself), -inf when
    nothing is selected.  lse - ln(m) <= max_logit <= lse for m rows."""
    O, lse = mla_attention(q, KV, tau, dv)
    H = np.asarray(q).shape[0]
    if np.asarray(KV).shape[0] == 0:
        return O, np.full(H, NEG_INF), lse
    z = tau * (np.asarray(q, dtype=np.float64) @ np.asarray(KV, dtype=np.float64).T)
    return O, z.max(axis=1), lse


def lse_merge(O_parts: np.ndarray, lse_parts: np.ndarray
              ) -> Tuple[np.ndarray, np.ndarray]:
    """Merge partial attention results that each cover a disjoint part of the
    selected set (DCP page, Modifications - Sparse decode and the LSE merge
    commits): lse = ln sum_p exp(lse_p); O = sum_p exp(lse_p - lse) O_p.
    Parts with lse = -inf (no tokens) contribute nothing.

    O_parts: [P, H, dv], lse_parts: [P, H]."""
    O_parts = np.asarray(O_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)                           # [H]
    safe_m = np.where(np.isfinite(m), m, 0.0)
    wts = np.where(np.isfinite(lse_parts), np.exp(lse_parts - safe_m), 0.0)  # [P, H]
    tot = wts.sum(axis=0)
    lse = np.where(tot > 0, safe_m + np.log(np.where(tot > 0, tot, 1.0)), NEG_INF)
    coef = np.where(tot > 0, wts / np.where(tot > 0, tot, 1.0), 0.0)
    O = np.einsum("ph,phd->hd", coef, O_parts)
    return O, lse


# ----------------------------------------------------------------------------
# sharded (decode context parallel) pieces
# ----------------------------------------------------------------------------


def shard_of(t, W: int):
    """Owner rule (DCP page, Modifications - Writes: slot % W == rank)."""
    return np.asarray(t) % W


def shard_local(t, W: int):
    """Local position of token t on its owner shard (interleave size 1)."""
    return np.asarray(t) // W


def shard_valid_len(pos: int, W: int, w: int) -> int:
    """Number of tokens 0..pos owned by shard w."""
    return 0 if pos < w else (pos - w) // W + 1


def merge_candidates(cand_scores: Sequence[np.ndarray], cand_pos: Sequence[np.ndarray],
                     k: int, W: int):
    """Exact global top-k from the per-shard local top-k lists of
    (score, global position) (DCP page, Modifications - Indexer decode).
    Returns (global positions in selection order, [owned local positions of
    shard w in the same order for w in 0..W-1])."""
    s = np.concatenate([np.asarray(c, dtype=np.float64) for c in cand_scores])
    p = np.concatenate([np.asarray(c, dtype=np.int64) for c in cand_pos])
    sel = topk_select(s, k, positions=p)
    owned = [shard_local(sel[shard_of(sel, W) == w], W) for w in range(W)]
    return sel, owned


# ----------------------------------------------------------------------------
# whole rows
# ----------------------------------------------------------------------------


def row_scores(wl, r: int, cache=None, W: int = 1, w: int = 0) -> np.ndarray:
    """Indexer scores of query row r over the tokens it sees (positions
    0..pos, or shard w's local positions of those tokens)."""
    b = int(wl.row_req[r])
    pos = int(wl.row_pos[r])
    cache = wl.idx_k if cache is None else cache
    n = shard_valid_len(pos, W, w)
    K = cache_rows(cache, b, np.arange(n))
    q = bf16_bits_to_f64(wl.q_idx[r])
    return indexer_scores(q, wl.w_idx[r], K)


def row_attention(wl, r: int, positions: np.ndarray, cache=None):
    b = int(wl.row_req[r])
    cache = wl.kv if cache is None else cache
    KV = cache_rows(cache, b, positions)
    q = bf16_bits_to_f64(wl.q[r])
    return mla_attention(q, KV, wl.sm_scale)


def row_attention_into(wl, r: int, positions: np.ndarray, cache=None):
    """mla_attention_into for query row r of workload wl."""
    b = int(wl.row_req[r])
    cache = wl.kv if cache is None else cache
    KV = cache_rows(cache, b, positions)
    q = bf16_bits_to_f64(wl.q[r])
    return mla_attention_into(q, KV, wl.sm_scale)


def decode_row(wl, r: int, scores: Optional[np.ndarray] = None):
    """Unsharded DSA decode of query row r: score the whole visible sequence,
    take the exact top-k, attend the selected latent rows.  ``scores`` may be
    given (e.g. the GPU's own fp32 scores) to run selection and attention on
    them instead of the oracle's."""
    if scores is None:
        scores = row_scores(wl, r)
    sel = topk_select(scores, wl.topk)
    O, lse = row_attention(wl, r, sel)
    return dict(scores=scores, idx=sel, O=O, lse=lse)


def decode_row_sharded(wl, r: int, W: Optional[int] = None):
    """Sharded DSA decode of query row r, following the DCP page
    (Modifications - Indexer decode and Sparse decode) step by step: each
    shard scores its own tokens and keeps a local top-k; the (score, global
    position) candidates of all shards are merged into the exact global top-k;
    each shard attends only the selected tokens it owns and returns (O, LSE);
    the partial results are LSE-merged."""
    W = wl.W if W is None else W
    k = wl.topk
    pos = int(wl.row_pos[r])
    cs, cp = [], []
    for w in range(W):
        s_loc = row_scores(wl, r, wl.idx_k_shards[w], W, w)
        j = topk_select(s_loc, k)
        cs.append(s_loc[j])
        cp.append(j * W + w)
    sel, owned = merge_candidates(cs, cp, k, W)
    Os, ls = [], []
    for w in range(W):
        O_w, l_w = row_attention(wl, r, owned[w], wl.kv_shards[w])
        Os.append(O_w)
        ls.append(l_w)
    O, lse = lse_merge(np.stack(Os), np.stack(ls))
    return dict(idx=sel, owned=owned, O=O, lse=lse, cand_scores=cs, cand_pos=cp)


# ----------------------------------------------------------------------------
# cache write (the step that appends new tokens to the caches)
# ----------------------------------------------------------------------------
#
# DCP page, Modifications / Writes: MLA KV and indexer K land only on the
# owner rank (slot % W); the page names a fused RoPE + KV-cache write.  The
# page gives no RoPE convention; the reading used here (and in the library):
# the last 64 dims of each row are the rope dims, taken in consecutive pairs
# (2i, 2i + 1), i < 32, rotated counter-clockwise by pos * base^(-i/32).
# fp8 rows: scale s = max|value| / 448 (1 for an all-zero row) and codes
# e4m3(value / s), both taken in fp32 (the kernel's precision), round to
# nearest even, saturating at +-448.

_E4M3_POS = None


def _e4m3_positive_values() -> np.ndarray:
    """Values of the 127 finite non-negative e4m3 codes 0x00..0x7E, in code
    order (which is value order)."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_code_to_f64(np.arange(127, dtype=np.uint8))
    return _E4M3_POS


def e4m3_encode_rne(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code of every value (ties to the even code, i.e. the even
    mantissa), magnitudes above 448 saturating to 448.  The sign goes to bit 7
    (a negative value that rounds to zero keeps its sign)."""
    x = np.asarray(x, dtype=np.float64)
    vals = _e4m3_positive_values()
    m = np.minimum(np.abs(x), vals[-1])
    hi = np.searchsorted(vals, m, side="left")        # first value >= m
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    dl = m - vals[lo]
    dh = vals[hi] - m
    pick_hi = (dh < dl) | ((dh == dl) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(vals[hi] == m, hi, code)           # exact hits
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def bf16_round_rne(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (bits) of float64 values, ties to even: the two bf16
    neighbours of x come from truncating its float32 pattern."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32) & np.uint32(0xFFFF0000)
    lo = u.view(np.float32).astype(np.float64)
    up = (u + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    # lo is the neighbour towards zero, up the one away from it
    dlo = np.abs(x - lo)
    dup = np.abs(up - x)
    even_lo = ((u >> np.uint32(16)) & np.uint32(1)) == 0
    take_up = (dup < dlo) | ((dup == dlo) & ~even_lo)
    bits = np.where(take_up, (u + np.uint32(0x10000)), u) >> np.uint32(16)
    return bits.astype(np.uint16)


def rope_last64(row: np.ndarray, pos: int, base: float) -> np.ndarray:
    """The row with its last 64 dims rotated pairwise: pair i = (x, y) at
    dims (D-64+2i, D-64+2i+1) becomes (x cos a - y sin a, x sin a + y cos a),
    a = pos * base^(-i/32)."""
    out = np.array(row, dtype=np.float64, copy=True)
    D = out.shape[-1]
    i = np.arange(32)
    a = float(pos) * np.power(float(base), -i / 32.0)
    x = out[..., D - 64::2].copy()
    y = out[..., D - 63::2].copy()
    out[..., D - 64::2] = x * np.cos(a) - y * np.sin(a)
    out[..., D - 63::2] = x * np.sin(a) + y * np.cos(a)
    return out


def cache_write_row(row_bits: np.ndarray, pos: int, base: float, dtype: str):
    """What the cache write stores for one token's row: (stored bf16 bits or
    e4m3 codes, fp32 scale or None, the exact post-RoPE values in float64)."""
    exact = rope_last64(bf16_bits_to_f64(row_bits), pos, base)
    if dtype == "bf16":
        return bf16_round_rne(exact), None, exact
    if dtype == "fp8_e4m3":
        x32 = exact.astype(np.float32)
        amax = np.float32(np.abs(x32).max())
        s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        q = (x32 / s).astype(np.float32)
        return e4m3_encode_rne(q), s, exact
    raise ValueError(dtype)
