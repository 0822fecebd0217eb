"""Pins of the CPU oracle to things other than itself: the OFP8 table, a
hand-worked decode, closed forms, brute force on tiny inputs, library
routines and invariants.  CPU only."""

import json
import math
import os
import random

import numpy as np
import pytest

from oracle import dsa_oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _expr(s):
    if isinstance(s, (int, float)):
        return float(s)
    try:
        return float(s)  # keeps the sign of "-0"
    except ValueError:
        pass
    env = {"log": math.log, "exp": math.exp, "nan": float("nan")}
    return float(eval(s, {"__builtins__": {}}, env))


# ---------------------------------------------------------------- decoding


def test_e4m3_against_ofp8_table():
    rows = []
    with open(os.path.join(GOLD, "e4m3_ofp8_table.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, val = line.split()
                rows.append((int(code.replace(".", ""), 2), val))
    for code, val in rows:
        got = orc.e4m3_code_to_f64(np.array([code], dtype=np.uint8))[0]
        want = _expr(val)
        if math.isnan(want):
            assert math.isnan(got), hex(code)
        else:
            assert got == want, (hex(code), got, want)
            assert math.copysign(1.0, got) == math.copysign(1.0, want)


def test_e4m3_all_codes_against_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_code_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_bf16_against_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=20000, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]  # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.bf16_bits_to_f64(bits), ref)


def test_fp8_rows_carry_token_scale():
    codes = np.array([[0x38, 0xB8, 0x40]], dtype=np.uint8)  # 1, -1, 2
    v = orc.decode_rows(codes, np.array([0.25]), "fp8_e4m3")
    assert np.array_equal(v, [[0.25, -0.25, 0.5]])


# ---------------------------------------------------------------- indexer


def test_indexer_hand_worked():
    g = json.load(open(os.path.join(GOLD, "hand_worked_decode.json")))["indexer"]
    s = orc.indexer_scores(np.array(g["q"], float), np.array(g["w"], float),
                           np.array(g["K"], float))
    assert np.allclose(s, [_expr(x) for x in g["scores"]], rtol=0, atol=1e-15)
    for k, want in g["topk"].items():
        assert orc.topk_select(s, int(k)).tolist() == want


def test_indexer_brute_force_loops():
    rng = random.Random(1)
    Hh, d, n = 3, 5, 7
    q = [[rng.uniform(-1, 1) for _ in range(d)] for _ in range(Hh)]
    w = [rng.uniform(0, 1) for _ in range(Hh)]
    K = [[rng.uniform(-1, 1) for _ in range(d)] for _ in range(n)]
    want = []
    for t in range(n):
        acc = 0.0
        for h in range(Hh):
            dot = sum(q[h][i] * K[t][i] for i in range(d))
            acc += w[h] * (dot if dot > 0 else 0.0)
        want.append(acc)
    got = orc.indexer_scores(np.array(q), np.array(w), np.array(K))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)


def test_indexer_closed_forms():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((64, 128))
    w = rng.random(64) / 8
    K = rng.standard_normal((50, 128))
    s_pos = orc.indexer_scores(q, w, K)
    s_neg = orc.indexer_scores(-q, w, K)
    dots = K @ q.T
    # relu(x) + relu(-x) = |x| and relu(x) - relu(-x) = x
    assert np.allclose(s_pos + s_neg, np.abs(dots) @ w)
    assert np.allclose(s_pos - s_neg, dots @ w)
    # all q.k < 0 -> 0
    Kneg = -np.abs(K)
    assert np.all(orc.indexer_scores(np.abs(q), w, Kneg) == 0.0)
    # one head, w = 1, K = e_i -> relu(q_i)
    q1 = rng.standard_normal((1, 128))
    s = orc.indexer_scores(q1, np.array([1.0]), np.eye(128))
    assert np.array_equal(s, np.maximum(q1[0], 0))
    # positive scale of K scales the score
    assert np.allclose(orc.indexer_scores(q, w, 3.0 * K), 3.0 * s_pos)


# ---------------------------------------------------------------- top-k


def _brute_topk(s, k):
    return sorted([t for _, t in sorted(((-float(v), t) for t, v in enumerate(s)))][:k])


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    s = rng.integers(0, 6, size=n).astype(np.float64)  # heavy ties
    k = int(rng.integers(1, 300))
    assert orc.topk_select(s, k).tolist() == _brute_topk(s, k)


def test_topk_special_cases():
    assert orc.topk_select(np.zeros(5000), 2048).tolist() == list(range(2048))
    s = np.array([3.0, 1.0, 2.0])
    assert orc.topk_select(s, 2048).tolist() == [0, 1, 2]
    assert orc.topk_select(s, 2).tolist() == [0, 2]
    # ties straddling the k-th place: the lower positions win
    s = np.array([1.0, 5.0, 2.0, 2.0, 2.0, 0.0])
    assert orc.topk_select(s, 3).tolist() == [1, 2, 3]
    s = np.array([2.0, 5.0, 2.0, 9.0, 2.0, 0.0])
    assert orc.topk_select(s, 3).tolist() == [0, 1, 3]
    # -0.0 and +0.0 are the same score
    s = np.array([-0.0, 0.0, -0.0, 1.0])
    assert orc.topk_select(s, 3).tolist() == [0, 1, 3]
    with pytest.raises(ValueError):
        orc.topk_select(np.array([1.0, np.nan]), 1)


# ---------------------------------------------------------------- attention


def test_attention_hand_worked():
    g = json.load(open(os.path.join(GOLD, "hand_worked_decode.json")))["attention"]
    KV = np.array([[_expr(x) for x in row] for row in g["KV"]])
    O, lse = orc.mla_attention(np.array(g["q"], float), KV, g["tau"], dv=g["dv"])
    assert np.allclose(O, [[_expr(x) for x in r] for r in g["O"]], rtol=1e-14)
    assert np.allclose(lse, [_expr(x) for x in g["lse"]], rtol=1e-14)


def test_attention_brute_force_loops():
    rng = random.Random(3)
    H, D, dv, m, tau = 2, 4, 3, 5, 0.7
    q = [[rng.uniform(-1, 1) for _ in range(D)] for _ in range(H)]
    KV = [[rng.uniform(-1, 1) for _ in range(D)] for _ in range(m)]
    O, lse = orc.mla_attention(np.array(q), np.array(KV), tau, dv=dv)
    for h in range(H):
        z = [tau * sum(q[h][i] * KV[t][i] for i in range(D)) for t in range(m)]
        den = sum(math.exp(x) for x in z)
        assert abs(lse[h] - math.log(den)) < 1e-13
        for c in range(dv):
            num = sum(math.exp(z[t]) * KV[t][c] for t in range(m))
            assert abs(O[h, c] - num / den) < 1e-13


def test_attention_closed_forms():
    rng = np.random.default_rng(4)
    tau = 576 ** -0.5
    q = rng.standard_normal((16, 576)) * 0.5
    kv = rng.standard_normal((1, 576)) * 0.5
    O, lse = orc.mla_attention(q, kv, tau)
    assert np.allclose(O, np.broadcast_to(kv[0, :512], O.shape))
    assert np.allclose(lse, tau * (q @ kv[0]))
    # m identical rows: O = v, lse = z + ln m
    O2, lse2 = orc.mla_attention(q, np.repeat(kv, 9, axis=0), tau)
    assert np.allclose(O2, O)
    assert np.allclose(lse2, lse + math.log(9))
    # empty set
    O3, lse3 = orc.mla_attention(q, np.zeros((0, 576)), tau)
    assert np.all(O3 == 0) and np.all(np.isneginf(lse3))


def test_attention_equals_masked_dense_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(6)
    L, tau = 300, 576 ** -0.5
    q = rng.standard_normal((8, 576)) * 0.5
    KV = rng.standard_normal((L, 576)) * 0.5
    sel = rng.choice(L, size=64, replace=False)
    O, lse = orc.mla_attention(q, KV[sel], tau)
    z = tau * (q @ KV.T)
    mask = np.full(L, -np.inf)
    mask[sel] = 0.0
    zm = z + mask
    p = scipy_special.softmax(zm, axis=1)
    assert np.allclose(lse, scipy_special.logsumexp(zm, axis=1), rtol=1e-13)
    assert np.allclose(O, p @ KV[:, :512], rtol=1e-12, atol=1e-14)


def test_attention_into_hand_worked():
    g = json.load(open(os.path.join(GOLD, "hand_worked_decode.json")))["attention"]
    KV = np.array([[_expr(x) for x in row] for row in g["KV"]])
    O, mx, lse = orc.mla_attention_into(np.array(g["q"], float), KV, g["tau"], dv=g["dv"])
    assert np.allclose(mx, [_expr(x) for x in g["max_logit"]], rtol=1e-14)
    assert np.allclose(O, [[_expr(x) for x in r] for r in g["O"]], rtol=1e-14)
    assert np.allclose(lse, [_expr(x) for x in g["lse"]], rtol=1e-14)


def test_attention_into_max_logit_brute_force_and_bounds():
    rng = random.Random(11)
    H, D, m, tau = 3, 5, 7, 0.6
    q = [[rng.uniform(-2, 2) for _ in range(D)] for _ in range(H)]
    KV = [[rng.uniform(-2, 2) for _ in range(D)] for _ in range(m)]
    _, mx, lse = orc.mla_attention_into(np.array(q), np.array(KV), tau, dv=2)
    for h in range(H):
        z = [tau * sum(q[h][i] * KV[t][i] for i in range(D)) for t in range(m)]
        assert abs(mx[h] - max(z)) < 1e-13
        # lse - ln m <= max <= lse
        assert lse[h] - math.log(m) - 1e-13 <= mx[h] <= lse[h] + 1e-13


def test_attention_into_closed_forms():
    rng = np.random.default_rng(12)
    tau = 576 ** -0.5
    q = rng.standard_normal((16, 576)) * 0.5
    kv = rng.standard_normal((1, 576)) * 0.5
    # one row: max logit = lse = z
    _, mx, lse = orc.mla_attention_into(q, kv, tau)
    assert np.allclose(mx, tau * (q @ kv[0])) and np.allclose(mx, lse)
    # identical rows: the max is z, the lse z + ln m
    _, mx2, lse2 = orc.mla_attention_into(q, np.repeat(kv, 5, axis=0), tau)
    assert np.allclose(mx2, mx) and np.allclose(lse2, mx + math.log(5))
    # nothing selected
    O3, mx3, lse3 = orc.mla_attention_into(q, np.zeros((0, 576)), tau)
    assert np.all(O3 == 0) and np.all(np.isneginf(mx3)) and np.all(np.isneginf(lse3))
    # splits: the largest split maximum is the maximum over the union
    KV = rng.standard_normal((40, 576)) * 0.5
    _, mxa, _ = orc.mla_attention_into(q, KV, tau)
    parts = [orc.mla_attention_into(q, KV[p], tau)[1] for p in np.array_split(np.arange(40), 3)]
    assert np.array_equal(np.max(np.stack(parts), axis=0), mxa)


@pytest.mark.parametrize("S", [1, 2, 7, 64])
def test_split_then_merge_equals_single_pass(S):
    rng = np.random.default_rng(7)
    tau = 576 ** -0.5
    q = rng.standard_normal((4, 576)) * 0.5
    KV = rng.standard_normal((64, 576)) * 0.5
    O, lse = orc.mla_attention(q, KV, tau)
    parts = np.array_split(np.arange(64), S)
    Os, ls = zip(*[orc.mla_attention(q, KV[p], tau) for p in parts])
    # add an empty part: it must not change anything
    Os = list(Os) + [np.zeros_like(O)]
    ls = list(ls) + [np.full(4, -np.inf)]
    Om, lm = orc.lse_merge(np.stack(Os), np.stack(ls))
    assert np.allclose(Om, O, rtol=1e-12, atol=1e-14)
    assert np.allclose(lm, lse, rtol=1e-13)


def test_merge_hand_worked():
    g = json.load(open(os.path.join(GOLD, "hand_worked_decode.json")))["merge"]
    Op = np.array(g["O_parts"], float)
    lp = np.array([[_expr(x) for x in r] for r in g["lse_parts"]])
    O, lse = orc.lse_merge(Op, lp)
    assert np.allclose(O, [[_expr(x) for x in r] for r in g["O"]], rtol=1e-14)
    assert np.allclose(lse, [_expr(x) for x in g["lse"]], rtol=1e-14)


def test_merge_all_empty():
    O, lse = orc.lse_merge(np.zeros((3, 2, 5)), np.full((3, 2), -np.inf))
    assert np.all(O == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- sharding


def test_owner_rule_and_local_positions():
    t = np.arange(23)
    for W in (1, 2, 3, 4):
        assert np.array_equal(orc.shard_local(t, W) * W + orc.shard_of(t, W), t)
        for pos in (0, 1, 5, 22):
            for w in range(W):
                want = sum(1 for x in range(pos + 1) if x % W == w)
                assert orc.shard_valid_len(pos, W, w) == want


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_candidate_merge_equals_global_topk(W):
    rng = np.random.default_rng(8 + W)
    n, k = 997, 100
    s = rng.integers(0, 40, size=n).astype(np.float64)  # ties across shards
    want = orc.topk_select(s, k)
    cs, cp = [], []
    for w in range(W):
        pos = np.arange(w, n, W)
        j = orc.topk_select(s[pos], k)
        cs.append(s[pos][j])
        cp.append(pos[j])
    sel, owned = orc.merge_candidates(cs, cp, k, W)
    assert np.array_equal(sel, want)
    for w in range(W):
        assert np.array_equal(owned[w], want[want % W == w] // W)


# ----------------------------------------------------------------------------
# cache write: e4m3 / bf16 rounding, RoPE, the stored row
# ----------------------------------------------------------------------------


def test_e4m3_encoder_roundtrip_ties_and_saturation():
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_code_to_f64(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(orc.e4m3_encode_rne(vals[fin]), codes[fin])
    pos = orc.e4m3_code_to_f64(np.arange(127, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    got = orc.e4m3_encode_rne(mids).astype(np.int64)
    lo = np.arange(126)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1)), "ties go to the even code"
    assert np.array_equal(orc.e4m3_encode_rne(-mids).astype(np.int64), got | 0x80)
    assert list(orc.e4m3_encode_rne(np.array([448.0, 449.0, 1e30, -1e30]))) == [0x7E, 0x7E, 0x7E, 0xFE]
    assert orc.e4m3_encode_rne(np.array([2.0 ** -10]))[0] == 0   # half the smallest step: even (0)
    assert orc.e4m3_encode_rne(np.array([2.0 ** -10 * 1.01]))[0] == 1


def test_e4m3_encoder_against_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8 in this torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 60, rng.standard_normal(5000) * 1e-2])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode_rne(x.astype(np.float64)), ref)


def test_bf16_rounding_against_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-20, 20, 50000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_round_rne(x.astype(np.float64)), ref)


def test_rope_closed_forms():
    base = 10000.0
    rng = np.random.default_rng(7)
    row = rng.standard_normal(576)
    assert np.array_equal(orc.rope_last64(row, 0, base), row)          # position 0: identity
    out = orc.rope_last64(row, 12345, base)
    assert np.array_equal(out[:512], row[:512])                         # nope dims untouched
    n0 = row[512::2] ** 2 + row[513::2] ** 2
    n1 = out[512::2] ** 2 + out[513::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-13, atol=0)                      # rotations keep norms
    # pair 0 turns by pos radians; pair 16 by pos / sqrt(base); (1, 0) -> (cos, sin)
    e = np.zeros(128)
    e[64] = 1.0
    e[64 + 32] = 1.0
    r = orc.rope_last64(e, 3, base)
    assert math.isclose(r[64], math.cos(3.0), abs_tol=1e-15) and math.isclose(r[65], math.sin(3.0), abs_tol=1e-15)
    a16 = 3.0 / math.sqrt(base)
    assert math.isclose(r[96], math.cos(a16), abs_tol=1e-15) and math.isclose(r[97], math.sin(a16), abs_tol=1e-15)
    e2 = np.zeros(128)
    e2[65] = 1.0                                                        # (0, 1) -> (-sin, cos)
    r2 = orc.rope_last64(e2, 3, base)
    assert math.isclose(r2[64], -math.sin(3.0), abs_tol=1e-15) and math.isclose(r2[65], math.cos(3.0), abs_tol=1e-15)
    # composition: positions add
    ab = orc.rope_last64(orc.rope_last64(row, 700, base), 41, base)
    assert np.allclose(ab, orc.rope_last64(row, 741, base), rtol=0, atol=1e-12)


def _bits(x):
    return orc.bf16_round_rne(np.asarray(x, dtype=np.float64))


def test_cache_write_row_bf16_and_fp8():
    rng = np.random.default_rng(8)
    row = _bits(rng.standard_normal(576) * 0.5)
    stored, s, exact = orc.cache_write_row(row, 777, 10000.0, "bf16")
    assert s is None and np.array_equal(stored[:512], row[:512])         # copies are exact
    assert np.array_equal(stored, orc.bf16_round_rne(exact))
    codes, s, exact = orc.cache_write_row(row, 777, 10000.0, "fp8_e4m3")
    x32 = exact.astype(np.float32)
    assert s == np.float32(np.abs(x32).max() / np.float32(448.0))
    j = int(np.argmax(np.abs(x32)))
    assert codes[j] in (0x7E, 0xFE)                                      # the row's max -> +-448
    deq = orc.e4m3_code_to_f64(codes) * float(s)
    pos = orc.e4m3_code_to_f64(np.arange(127, dtype=np.uint8))
    step = np.diff(pos)[np.clip(np.searchsorted(pos, np.abs(x32 / s)) - 1, 0, 125)] * float(s)
    assert np.all(np.abs(deq - x32) <= step / 2 * (1 + 1e-6))            # nearest code
    z, sz, _ = orc.cache_write_row(np.zeros(128, dtype=np.uint16), 5, 10000.0, "fp8_e4m3")
    assert sz == np.float32(1.0) and np.all((z & 0x7F) == 0)            # +-0 codes only
