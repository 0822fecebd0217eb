"""The seeded input generator: encodings, layouts and the oracle's whole-row
paths on small workloads (CPU only)."""

import numpy as np
import pytest

from oracle import dsa_oracle as orc
from workloads import config_spec, make_workload
from workloads.synth import to_bf16_bits, to_e4m3_codes


def test_bf16_encoder_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 10
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(to_bf16_bits(x), ref)


def test_e4m3_encoder_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.uniform(-448, 448, 200000),
        rng.uniform(-2 ** -5, 2 ** -5, 200000),          # subnormal range
        np.array([448.0, -448.0, 0.0, 2 ** -10, 3 * 2 ** -10, 1.0625, 232.0]),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = to_e4m3_codes(x)
    # torch keeps the sign of a value that rounds to zero; so do we
    assert np.array_equal(got, ref)


def test_config_shapes_small():
    wl = make_workload(config_spec(2, B=3, L_lo=200, L_hi=300, topk=64))
    assert wl.R == 18 and wl.q_idx.shape == (18, 64, 128) and wl.q.shape == (18, 32, 576)
    assert wl.idx_k.data.dtype == np.uint8 and wl.idx_k.scale.shape[1] == 64
    for b in range(wl.B):
        L = int(wl.seq_len[b])
        assert np.array_equal(wl.row_pos[6 * b: 6 * b + 6], np.arange(L - 6, L))
        n = (L + 63) // 64
        assert np.all(wl.idx_k.block_table[b, :n] >= 0)
        assert np.all(wl.idx_k.block_table[b, n:] == -1)
    used = wl.kv.block_table[wl.kv.block_table >= 0]
    assert np.array_equal(np.sort(used), np.arange(wl.kv.num_pages))


def test_generator_is_deterministic():
    a = make_workload(config_spec(1, B=2, L=300))
    b = make_workload(config_spec(1, B=2, L=300))
    assert np.array_equal(a.kv.data, b.kv.data)
    assert np.array_equal(a.idx_k.block_table, b.idx_k.block_table)
    assert np.array_equal(a.q, b.q)


def test_fp8_scale_recipe():
    wl = make_workload(config_spec(4, B=2, L_lo=100, L_hi=200))
    v = orc.e4m3_code_to_f64(wl.kv.data)
    assert np.isfinite(v).all()
    amax = np.abs(v).max(axis=2)
    # amax / 448 scaling: every token's largest code is 448 (or rounds to it)
    assert np.all(amax == 448.0)


@pytest.mark.parametrize("W,L", [(2, 301), (3, 200), (4, 257)])
def test_shard_caches_hold_the_same_tokens(W, L):
    wl = make_workload(config_spec(3, B=2, L=L, shards=W, topk=32))
    for b in range(2):
        full = orc.cache_rows(wl.kv, b, np.arange(L))
        fullk = orc.cache_rows(wl.idx_k, b, np.arange(L))
        for w in range(W):
            n = int(wl.kv_shards[w].seq_len[b])
            assert n == len(range(w, L, W))
            loc = orc.cache_rows(wl.kv_shards[w], b, np.arange(n))
            assert np.array_equal(loc, full[w::W])
            lk = orc.cache_rows(wl.idx_k_shards[w], b, np.arange(n))
            assert np.array_equal(lk, fullk[w::W])


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_oracle_sharded_equals_unsharded(W):
    wl = make_workload(config_spec(3, B=2, L=517, shards=W, topk=64))
    for r in range(wl.R):
        u = orc.decode_row(wl, r)
        s = orc.decode_row_sharded(wl, r)
        assert np.array_equal(u["idx"], s["idx"])
        assert np.allclose(u["O"], s["O"], rtol=1e-12, atol=1e-13)
        assert np.allclose(u["lse"], s["lse"], rtol=1e-13)


def test_oracle_fp8_mtp_rows_are_causal():
    wl = make_workload(config_spec(2, B=1, L_lo=300, L_hi=300, topk=64))
    outs = [orc.decode_row(wl, r) for r in range(6)]
    for j, o in enumerate(outs):
        assert o["scores"].shape == (300 - 6 + j + 1,)
        assert o["idx"].max() <= 300 - 6 + j
    # the scores of a shared token are the same for all rows only if the rows
    # share the query; they do not, but every row sees the same cache values
    assert outs[0]["O"].shape == (32, 512)
