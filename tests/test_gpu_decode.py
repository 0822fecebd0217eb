"""Parity of the fused dsa_decode path against the CPU oracle on all five
workload configurations, at reduced sizes and at full sizes (the ragged fp8
sweep at B = 64, 128 and 256), every row checked, plus sharded == unsharded."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dsa_oracle as orc  # noqa: E402
from workloads import config_spec, make_workload  # noqa: E402
from workloads.device import upload  # noqa: E402

from gpu_util import DecodeRun, check_decode_rows  # noqa: E402

pytestmark = pytest.mark.gpu


def _run(spec, sharded=False, num_splits=0, rows=None):
    wl = make_workload(spec)
    dw = upload(wl, "cuda")
    run = DecodeRun(dw, sharded=sharded, num_splits=num_splits)
    assert run.run() == 0
    rows = range(wl.R) if rows is None else rows
    return wl, run, check_decode_rows(run, rows)


def test_config0_full():
    _run(config_spec(0))


@pytest.mark.parametrize("L", [300, 2048, 2049, 5000])
def test_config1_reduced(L):
    _run(config_spec(1, B=3, L=L))


def test_config2_reduced_mtp_fp8():
    _run(config_spec(2, B=3, L_lo=1500, L_hi=6000))


@pytest.mark.parametrize("W,L", [(2, 5001), (3, 6007), (4, 9001)])
def test_config3_reduced_sharded(W, L):
    _run(config_spec(3, B=2, L=L, shards=W), sharded=True)


@pytest.mark.parametrize("W,L", [(2, 5001), (4, 9001)])
def test_sharded_fp8_caches(W, L):
    """The sharded path on fp8 index-K and latent caches: each shard's own
    scales, and the tensor-core attention over W shard caches at once."""
    _run(config_spec(3, B=2, L=L, shards=W, dtype="fp8_e4m3"), sharded=True)


def test_config4_reduced_ragged_fp8():
    _run(config_spec(4, B=9, L_lo=300, L_hi=12000))


@pytest.mark.parametrize("cfg,kw,page", [(1, dict(B=3, L=2500), 128),
                                         (4, dict(B=4, L_lo=300, L_hi=9000), 128),
                                         (2, dict(B=2, L_lo=1500, L_hi=5000), 128),
                                         (1, dict(B=3, L=2500), 192),
                                         (4, dict(B=3, L_lo=300, L_hi=9000), 192)])
def test_pages_of_128_and_192_tokens(cfg, kw, page):
    """Pages of 128 and 192 tokens: the indexer's 64-token boxes start inside
    a page, gathers resolve slots beyond 64, and 192 takes the division path
    instead of the shift; bf16 and fp8, MTP rows."""
    _run(config_spec(cfg, page_size=page, **kw))


@pytest.mark.parametrize("rpr,dtype", [(9, "bf16"), (20, "fp8_e4m3"), (33, "bf16")])
def test_multi_query_extend_rows(rpr, dtype):
    """More query rows per request than one indexer row group (8) holds, at
    consecutive positions (a multi-query extend): the rows are scored in
    groups of 8 that each stream the request's keys, and every row keeps its
    own causal window, top-k and attention."""
    _run(config_spec(2, B=2, L_lo=2500, L_hi=5000, rows_per_req=rpr, dtype=dtype))


def test_multi_query_extend_rows_sharded():
    _run(config_spec(3, B=2, L=3001, shards=2, rows_per_req=12), sharded=True)


def test_more_rows_than_declared_sets_error_bit():
    import dataclasses

    from dsa_sparse_attention_decode_gb300 import _lib as C
    wl = make_workload(config_spec(2, B=2, L_lo=2500, L_hi=3000, rows_per_req=20,
                                   dtype="bf16"))
    dw = upload(wl, "cuda")
    dw.rows = dataclasses.replace(dw.rows, max_rows_per_req=16)  # two groups of 8 < 20 rows
    run = DecodeRun(dw)
    assert run.run() & C.DSA_DEVERR_GROUP


@pytest.mark.parametrize("k", [1, 100, 1000, 4096])
def test_decode_other_k(k):
    """k other than 2048: a single token, fewer than a tile, not a multiple
    of 64, and the largest k the entry points accept."""
    _run(config_spec(1, B=2, L=5000, topk=k))


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_cache_write_then_decode(dtype):
    """One decode step's cache write feeds the decode: new rows (RoPE'd, and
    quantized for fp8 caches) go to each request's last 5 positions through
    the block tables; the decode at the last position then matches the oracle
    run on the caches as written."""
    from dsa_sparse_attention_decode_gb300 import api
    from workloads.device import upload as _upload
    from workloads.synth import to_bf16_bits
    wl = make_workload(config_spec(1, B=2, L=4000, dtype=dtype))
    dw = _upload(wl, "cuda")
    rng = np.random.default_rng(21)
    n_new = 5
    req = np.repeat(np.arange(wl.B, dtype=np.int32), n_new)
    pos = np.concatenate([np.arange(int(wl.row_pos[b]) - n_new + 1, int(wl.row_pos[b]) + 1)
                          for b in range(wl.B)]).astype(np.int32)
    kv_in = to_bf16_bits(rng.standard_normal((len(pos), 576)) * 0.5)
    ix_in = to_bf16_bits(rng.standard_normal((len(pos), 128)))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dsa_cache_write(t(kv_in.view(np.int16)), t(req), t(pos), wl.B, [dw.kv], err,
                        idx_in=t(ix_in.view(np.int16)), idx_k=[dw.idx_k])
    assert api.dsa_read_error(err) == 0
    # the oracle reads the caches exactly as the kernel wrote them
    for host, dev in ((wl.kv, dw.kv), (wl.idx_k, dw.idx_k)):
        host.data[...] = dev.data.cpu().numpy().view(host.data.dtype)
        if host.scale is not None:
            host.scale[...] = dev.scale.cpu().numpy()
    run = DecodeRun(dw)
    assert run.run() == 0
    check_decode_rows(run, range(wl.R))


def test_many_rows_read_metadata_from_global():
    """2400 query rows: the row metadata no longer fits the indexer's shared-
    memory copy, and the schedule reads it from global memory instead."""
    wl, run, _ = _run(config_spec(2, B=400, L_lo=300, L_hi=700, rows_per_req=6),
                      rows=range(0, 2400, 97))
    assert wl.R == 2400


def test_wide_block_table_reads_global():
    """A block table wider than the MLA's shared-memory copy (4096 entries per
    request): the gather reads the global table."""
    import dataclasses
    wl = make_workload(config_spec(1, B=2, L=3000))
    dw = upload(wl, "cuda")
    wide = 5000
    for name in ("kv", "idx_k"):
        c = getattr(dw, name)
        bt = torch.full((c.block_table.shape[0], wide), -1, dtype=torch.int32, device="cuda")
        bt[:, : c.block_table.shape[1]] = c.block_table
        setattr(dw, name, dataclasses.replace(c, block_table=bt, max_blocks=wide))
    run = DecodeRun(dw)
    assert run.run() == 0
    check_decode_rows(run, range(wl.R))


@pytest.mark.parametrize("S", [1, 2, 7, 32])
def test_split_counts_agree(S):
    _run(config_spec(1, B=2, L=4500), num_splits=S)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_sharded_equals_unsharded_bit_exact(W):
    wl = make_workload(config_spec(3, B=2, L=7777, shards=W))
    dw = upload(wl, "cuda")
    a = DecodeRun(dw, sharded=False)
    b = DecodeRun(dw, sharded=True)
    assert a.run() == 0 and b.run() == 0
    for r in range(wl.R):
        full = a.scores(r)
        for w in range(W):
            assert np.array_equal(b.scores(r, w).view(np.uint32), full[w::W].view(np.uint32))
    assert torch.equal(a.idx, b.idx) and torch.equal(a.cnt, b.cnt)
    o_a, o_b = a.out.cpu().numpy(), b.out.cpu().numpy()
    rel = np.abs(o_a - o_b).max(axis=-1) / np.abs(o_a).max(axis=-1)
    assert rel.max() <= 2e-3
    assert np.abs(a.lse.cpu().numpy() - b.lse.cpu().numpy()).max() <= 1e-4


def test_deterministic():
    wl = make_workload(config_spec(2, B=2, L_lo=3000, L_hi=5000))
    dw = upload(wl, "cuda")
    a = DecodeRun(dw)
    assert a.run() == 0
    o1, l1, i1 = a.out.clone(), a.lse.clone(), a.idx.clone()
    assert a.run() == 0
    assert torch.equal(o1, a.out) and torch.equal(l1, a.lse) and torch.equal(i1, a.idx)


# ------------------------------------------------------------- full sizes


def test_config1_full_size_every_row():
    """B=32, L=32768, bf16, paged: every row checked."""
    _run(config_spec(1))


def test_config2_full_size_every_row():
    """B=64 x 6 MTP rows, L 16K..64K, fp8: all 384 rows checked."""
    _run(config_spec(2))


def test_config3_full_size():
    _run(config_spec(3), sharded=True)


@pytest.mark.parametrize("B", [64, 128, 256])
def test_config4_full_size_every_row(B):
    """The ragged fp8 sweep at full size (L log-uniform in 4K..128K), every
    row checked: scores, bit-exact top-k on the GPU's scores, O and LSE."""
    wl, run, _ = _run(config_spec(4, B=B))
    assert int(wl.seq_len.max()) > 100_000 and int(wl.seq_len.min()) < 8192
