"""dsa_cache_write through the C ABI against the CPU oracle: RoPE, bf16
rounding / e4m3 quantization with the per-token scale, the owner-rule
placement into shard caches through their block tables, and that nothing
but the owner slot of each token changes."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dsa_sparse_attention_decode_gb300 import api  # noqa: E402
from dsa_sparse_attention_decode_gb300 import _lib as C  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
BASE = 10000.0
PAGE = 64


def _cache(rng, W_pages, max_blocks, num_reqs, row, fp8):
    """A shard cache full of sentinel bytes, with a permuted block table."""
    if fp8:
        data = torch.from_numpy(rng.integers(0, 256, (W_pages, PAGE, row), dtype=np.uint8))
        scale = torch.from_numpy(rng.standard_normal((W_pages, PAGE)).astype(np.float32))
    else:
        data = torch.from_numpy(rng.integers(0, 65536, (W_pages, PAGE, row), dtype=np.uint16).view(np.int16))
        scale = None
    bt = torch.from_numpy(rng.permutation(W_pages)[: num_reqs * max_blocks].reshape(num_reqs, max_blocks).astype(np.int32))
    return api.PagedCache(data=data.to(DEV), scale=None if scale is None else scale.to(DEV),
                          block_table=bt.to(DEV),
                          dtype=C.DSA_DTYPE_FP8_E4M3 if fp8 else C.DSA_DTYPE_BF16,
                          page_size=PAGE, max_blocks=max_blocks)


def _close_rounding(got_vals, ref_vals, exact, budget):
    """got is the reference rounding of the exact value, or the other
    neighbour when the exact value lies within the arithmetic's error budget
    of their midpoint (a value the kernel may legitimately compute)."""
    same = got_vals == ref_vals
    tie = np.abs(np.abs(got_vals - exact) - np.abs(ref_vals - exact)) <= 2 * budget
    return same | tie


def _rope_budget(row_bits, scale=1.0):
    """Absolute error budget of the fp32 rotation of each rope pair (a few
    roundings of products of inputs of size |x| + |y|), zero elsewhere."""
    v = orc.bf16_bits_to_f64(row_bits)
    D = v.shape[0]
    mag = np.abs(v[D - 64::2]) + np.abs(v[D - 63::2])
    b = np.zeros(D)
    b[D - 64::2] = mag
    b[D - 63::2] = mag
    return 1e-6 * b / scale


def _check_row(stored, scale, row_bits, pos, fp8):
    ref, s_ref, exact = orc.cache_write_row(row_bits, pos, BASE, "fp8_e4m3" if fp8 else "bf16")
    if not fp8:
        got = np.asarray(stored).view(np.uint16)
        assert np.array_equal(got[:-64], row_bits[:-64]), "nope dims are copied exactly"
        ok = _close_rounding(orc.bf16_bits_to_f64(got), orc.bf16_bits_to_f64(ref), exact,
                             _rope_budget(row_bits))
        assert ok.all(), (pos, np.nonzero(~ok))
        return int((got != ref).sum())
    assert abs(float(scale) - float(s_ref)) <= 1e-6 * float(s_ref), (scale, s_ref)
    got = np.asarray(stored).view(np.uint8)
    x = exact.astype(np.float32).astype(np.float64) / float(s_ref)
    # x / s in fp32 adds a rounding of its own (relative 2^-24)
    ok = _close_rounding(orc.e4m3_code_to_f64(got), orc.e4m3_code_to_f64(ref), x,
                         _rope_budget(row_bits, float(s_ref)) + 1e-7 * np.abs(x))
    assert ok.all(), (pos, np.nonzero(~ok))
    return int((got != ref).sum())


def _run(W, kv_fp8, idx_fp8, N=48, num_reqs=2, max_pos=131072, seed=0, with_idx=True):
    rng = np.random.default_rng(seed)
    max_blocks = (max_pos // W + PAGE - 1) // PAGE + 1
    pages = num_reqs * max_blocks + 5
    kv = [_cache(rng, pages, max_blocks, num_reqs, 576, kv_fp8) for _ in range(W)]
    ix = [_cache(rng, pages, max_blocks, num_reqs, 128, idx_fp8) for _ in range(W)]
    before = [(c.data.clone(), None if c.scale is None else c.scale.clone()) for c in kv + ix]
    req = rng.integers(0, num_reqs, N).astype(np.int32)
    pos = np.concatenate([[0, 1, 63, 64, 65, max_pos - 1], rng.integers(0, max_pos, N - 6)]).astype(np.int32)
    # one write per (request, position)
    _, first = np.unique(req.astype(np.int64) * (1 << 32) + pos, return_index=True)
    req, pos = req[np.sort(first)], pos[np.sort(first)]
    N = len(pos)
    kv_in = orc.bf16_round_rne(rng.standard_normal((N, 576)) * 0.5)
    kv_in[0, :] = 0                                       # an all-zero row
    ix_in = orc.bf16_round_rne(rng.standard_normal((N, 128)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    api.dsa_cache_write(t(kv_in.view(np.int16)), t(req), t(pos), num_reqs, kv, err,
                        idx_in=t(ix_in.view(np.int16)) if with_idx else None,
                        idx_k=ix if with_idx else None, rope_base=BASE)
    assert api.dsa_read_error(err) == 0
    flips = 0
    expect = [(d.cpu().numpy().copy(), None if s is None else s.cpu().numpy().copy()) for d, s in before]
    for j in range(N):
        w, p = int(pos[j]) % W, int(pos[j]) // W
        for kind, caches, rows, fp8, off in (("kv", kv, kv_in, kv_fp8, 0), ("idx", ix, ix_in, idx_fp8, W)):
            if kind == "idx" and not with_idx:
                continue
            c = caches[w]
            pg = int(c.block_table[req[j], p // PAGE])
            stored = c.data[pg, p % PAGE].cpu().numpy()
            scale = None if c.scale is None else c.scale[pg, p % PAGE].item()
            flips += _check_row(stored, scale, rows[j], int(pos[j]), fp8)
            expect[off + w][0][pg, p % PAGE] = stored
            if scale is not None:
                expect[off + w][1][pg, p % PAGE] = scale
    # nothing but the owner slots changed
    for (d, s), c in zip(expect, kv + ix):
        assert np.array_equal(d, c.data.cpu().numpy())
        if s is not None:
            assert np.array_equal(s, c.scale.cpu().numpy())
    return flips


@pytest.mark.parametrize("W", [1, 3])
@pytest.mark.parametrize("fp8", [False, True])
def test_cache_write_against_oracle(W, fp8):
    flips = _run(W, fp8, fp8, seed=W * 10 + fp8)
    assert flips <= 8, "only near-tie roundings may differ from the oracle's"


def test_cache_write_mixed_dtypes_and_no_index_rows():
    _run(2, True, False, seed=7)
    _run(2, False, True, seed=8, with_idx=False)


def test_cache_write_bad_position_and_page():
    rng = np.random.default_rng(9)
    kv = [_cache(rng, 10, 4, 2, 576, False)]
    before = kv[0].data.clone()
    kv[0].block_table[1, 2] = -1                          # a missing page
    req = torch.tensor([0, 1, 0], dtype=torch.int32, device=DEV)
    pos = torch.tensor([4 * PAGE, 2 * PAGE + 3, -1], dtype=torch.int32, device=DEV)
    kv_in = torch.zeros((3, 576), dtype=torch.int16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.dsa_cache_write(kv_in, req, pos, 2, kv, err)
    e = api.dsa_read_error(err)
    assert e & C.DSA_DEVERR_POS and e & C.DSA_DEVERR_PAGE
    assert torch.equal(before, kv[0].data), "no row of a rejected token is written"
