"""The individual entry points through the C ABI against the CPU oracle, and
the edge cases: ties, short rows, single tokens, device-side error checks."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dsa_sparse_attention_decode_gb300 import api  # noqa: E402
from dsa_sparse_attention_decode_gb300 import _lib as C  # noqa: E402
from oracle import dsa_oracle as orc  # noqa: E402
from workloads import config_spec, make_workload  # noqa: E402
from workloads.device import upload  # noqa: E402

from gpu_util import DecodeRun, attn_err, check_decode_rows, score_ok  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("cfg,kw", [(1, dict(B=3, L=1000)), (2, dict(B=2, L_lo=700, L_hi=1500)),
                                    (0, {})])
def test_indexer_scores(cfg, kw):
    wl = make_workload(config_spec(cfg, **kw))
    dw = upload(wl, DEV)
    ld = dw.rows.max_len + 3
    scores = torch.full((wl.R, ld), 12345.0, device=DEV)
    err = _err()
    api.dsa_indexer_scores(dw.q_idx, dw.w_idx, dw.idx_k, dw.rows, scores, err)
    assert api.dsa_read_error(err) == 0
    s = scores.cpu().numpy()
    for r in range(wl.R):
        n = int(wl.row_pos[r]) + 1
        ok, e = score_ok(s[r, :n], orc.row_scores(wl, r))
        assert ok, (r, e)
        assert np.all(s[r, n:] == 12345.0), "wrote past the row's valid length"


def test_indexer_single_shard_call():
    wl = make_workload(config_spec(3, B=2, L=3001, shards=3))
    dw = upload(wl, DEV)
    for w in range(3):
        n = (dw.rows.max_len + 2) // 3
        scores = torch.zeros((wl.R, n), device=DEV)
        err = _err()
        api.dsa_indexer_scores(dw.q_idx, dw.w_idx, dw.idx_k_shards[w], dw.rows, scores, err,
                               shard=w, num_shards=3)
        assert api.dsa_read_error(err) == 0
        for r in range(wl.R):
            m = orc.shard_valid_len(int(wl.row_pos[r]), 3, w)
            ok, e = score_ok(scores[r, :m].cpu().numpy(),
                             orc.row_scores(wl, r, wl.idx_k_shards[w], 3, w))
            assert ok, (w, r, e)


def _topk_case(s: np.ndarray, valid: np.ndarray, k: int, stride=1, offset=0):
    """Both forms of dsa_topk (with a workspace: segments over every SM; without:
    one CTA per row) against the oracle's selection; returns the OR of the
    two calls' device error words."""
    R = s.shape[0]
    st = torch.from_numpy(s.astype(np.float32)).to(DEV)
    vt = torch.from_numpy(valid.astype(np.int32)).to(DEV)
    want = [orc.topk_select(s[r, : int(valid[r])].astype(np.float32).astype(np.float64), k)
            for r in range(R)]
    e = 0
    for with_ws in (True, False):
        oi = torch.full((R, k), -5, dtype=torch.int32, device=DEV)
        os_ = torch.zeros((R, k), dtype=torch.float32, device=DEV)
        oc = torch.zeros(R, dtype=torch.int32, device=DEV)
        err = _err()
        ws = None
        if with_ws:
            # stale contents: the call must clear what has to start at zero
            ws = torch.full((api.dsa_topk_workspace_size(R, s.shape[1]),), 0x5A,
                            dtype=torch.uint8, device=DEV)
        api.dsa_topk(st, vt, k, oi, oc, err, out_score=os_, index_stride=stride,
                     index_offset=offset, workspace=ws)
        e |= api.dsa_read_error(err)
        oi_h, os_h, oc_h = oi.cpu().numpy(), os_.cpu().numpy(), oc.cpu().numpy()
        for r in range(R):
            assert oc_h[r] == len(want[r]), (with_ws, r)
            assert np.array_equal(oi_h[r, : oc_h[r]], want[r] * stride + offset), (with_ws, r)
            assert np.all(oi_h[r, oc_h[r]:] == -1), (with_ws, r)
            assert np.array_equal(os_h[r, : oc_h[r]], s[r, want[r]].astype(np.float32)), (with_ws, r)
    return e


def _topk_both_forms(s: np.ndarray, valid: np.ndarray, k: int, stride=1, offset=0):
    """The rows as given (few rows: the cluster form), then repeated to 80 or
    more rows (the segment form and its one-CTA-per-row variant)."""
    e = _topk_case(s, valid, k, stride, offset)
    rep = -(-80 // s.shape[0])
    return e | _topk_case(np.tile(s, (rep, 1)), np.tile(valid, rep), k, stride, offset)


def test_topk_random_rows():
    rng = np.random.default_rng(0)
    R, L = 6, 70000
    s = rng.standard_normal((R, L)).astype(np.float32) * 3
    valid = np.array([L, 1, 2047, 2048, 2049, 50000])
    assert _topk_both_forms(s, valid, 2048) == 0


def test_topk_wide_and_narrow_key_ranges():
    """Rows whose keys span many octaves, a very narrow band, a few huge
    outliers over a narrow band, and negatives; lengths on both sides of the
    row length whose keys still fit in shared memory."""
    rng = np.random.default_rng(2)
    R, L = 5, 60000
    s = np.empty((R, L), dtype=np.float32)
    s[0] = np.exp(rng.normal(0.0, 8.0, L))
    s[1] = 20.0 + rng.normal(0.0, 1e-3, L)
    s[2] = 20.0 + rng.normal(0.0, 1e-3, L)
    s[2, ::997] = 1e30
    s[3] = -np.exp(rng.normal(0.0, 3.0, L))
    s[4] = rng.standard_normal(L)
    valid = np.array([L, 55296, 55297, 40000, 2049])
    assert _topk_both_forms(s, valid, 2048) == 0
    assert _topk_both_forms(s, valid, 37) == 0


@pytest.mark.parametrize("R", [50, 100, 400])
def test_topk_many_rows(R):
    """Many rows of mixed lengths: several rows share an SM, and the launch
    runs more rows than the GPU holds at once (400)."""
    rng = np.random.default_rng(3)
    L = 40000
    s = (rng.standard_normal((R, L)) * 2 + 10).astype(np.float32)
    valid = rng.integers(1, L + 1, R)
    valid[:4] = [L, 2048, 2049, 1]
    assert _topk_case(s, valid, 2048) == 0


@pytest.mark.parametrize("R", [2, 45, 80])
def test_topk_rows_too_long_for_the_bitmaps(R):
    """Score rows of 800000 positions: the position bitmaps of one row do not
    fit in shared memory, so a cluster of 4 (2 rows), 2 (45 rows) or 1 CTA
    (80 rows) selects each row."""
    rng = np.random.default_rng(5)
    L = 800_000
    s = (rng.standard_normal((R, L)) * 2 + 10).astype(np.float32)
    valid = rng.integers(1, 60_000, R)
    valid[0] = L
    valid[1] = 2049
    assert _topk_case(s, valid, 2048) == 0


def test_topk_crowded_threshold_bin():
    """Three score values over 30000 positions: the bin holding the k-th
    largest key has about 10000 keys, more than the candidate list holds."""
    rng = np.random.default_rng(4)
    R, L = 3, 30000
    s = rng.integers(0, 3, (R, L)).astype(np.float32)
    s[2] = np.where(rng.random(L) < 0.5, 7.0, 7.000001)
    valid = np.array([L, L, L])
    assert _topk_both_forms(s, valid, 2048) == 0
    assert _topk_both_forms(s, valid, 4096) == 0


def test_topk_ties_and_signed_zero():
    rng = np.random.default_rng(1)
    R, L = 5, 9000
    s = np.zeros((R, L), dtype=np.float32)
    s[1] = rng.integers(0, 3, L)               # heavy ties
    s[2] = rng.integers(-2, 3, L).astype(np.float32) * 0.0  # +0 / -0 mix
    s[3, :] = 1.0
    s[3, ::7] = 2.0                             # 1286 twos, ties at the k-th place
    s[4] = np.round(rng.standard_normal(L), 1)
    valid = np.full(R, L)
    assert _topk_both_forms(s, valid, 2048) == 0
    assert _topk_both_forms(s, valid, 100, stride=4, offset=3) == 0


def test_topk_nan_flag():
    s = np.ones((1, 3000), dtype=np.float32)
    s[0, 17] = np.nan
    st = torch.from_numpy(s).to(DEV)
    vt = torch.tensor([3000], dtype=torch.int32, device=DEV)
    oi = torch.zeros((1, 64), dtype=torch.int32, device=DEV)
    oc = torch.zeros(1, dtype=torch.int32, device=DEV)
    err = _err()
    api.dsa_topk(st, vt, 64, oi, oc, err)
    assert api.dsa_read_error(err) & C.DSA_DEVERR_NAN


@pytest.mark.parametrize("W,k,n,levels,bounded", [
    (3, 256, 2000, 50, False), (3, 256, 2000, 50, True),         # many ties at the k-th place
    (4, 2048, 40000, 1 << 30, False), (4, 2048, 40000, 1 << 30, True),
    (8, 2048, 9000, 7, True),                                     # few distinct scores, 8 shards
    (2, 2048, 3000, 1 << 30, True),                               # short rows: the union < k
    (5, 512, 262144, 1000, True),                                 # the largest bitmap
])
def test_shard_merge_against_oracle(W, k, n, levels, bounded):
    """Both forms of the merge (bitmap over positions when a position bound
    is given, ranking searches otherwise) against the oracle's merge."""
    rng = np.random.default_rng(2)
    R = 4
    cs = np.zeros((W, R, k), np.float32)
    cp = np.full((W, R, k), -1, np.int32)
    cc = np.zeros((W, R), np.int32)
    s_full = rng.integers(0, levels, (R, n)).astype(np.float32)
    if levels > 1000:
        s_full = rng.standard_normal((R, n)).astype(np.float32)
    for r in range(R):
        for w in range(W):
            pos = np.arange(w, n - r * (n // 7), W)
            j = orc.topk_select(s_full[r, pos].astype(np.float64), k)
            cc[w, r] = len(j)
            cs[w, r, : len(j)] = s_full[r, pos[j]]
            cp[w, r, : len(j)] = pos[j]
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    oi = torch.zeros((R, k), dtype=torch.int32, device=DEV)
    oc = torch.zeros(R, dtype=torch.int32, device=DEV)
    ol = torch.zeros((W, R, k), dtype=torch.int32, device=DEV)
    ocnt = torch.zeros((W, R), dtype=torch.int32, device=DEV)
    err = _err()
    api.dsa_shard_topk_merge(t(cs), t(cp), t(cc), oi, oc, ol, ocnt, err,
                             pos_bound=n if bounded else 0)
    assert api.dsa_read_error(err) == 0
    for r in range(R):
        sel, owned = orc.merge_candidates([cs[w, r, : cc[w, r]] for w in range(W)],
                                          [cp[w, r, : cc[w, r]] for w in range(W)], k, W)
        assert int(oc[r]) == len(sel)
        assert np.array_equal(oi[r, : len(sel)].cpu().numpy(), sel)
        for w in range(W):
            m = int(ocnt[w, r])
            assert np.array_equal(ol[w, r, :m].cpu().numpy(), owned[w])
            assert np.all(ol[w, r, m:].cpu().numpy() == -1)


@pytest.mark.parametrize("cfg", [1, 2])
def test_sparse_mla_alone(cfg):
    wl = make_workload(config_spec(cfg, B=2, L=3000, L_lo=2500, L_hi=4000))
    dw = upload(wl, DEV)
    rng = np.random.default_rng(3)
    k = 2048
    idx = np.full((wl.R, k), -1, np.int32)
    cnt = np.zeros(wl.R, np.int32)
    for r in range(wl.R):
        n = [2048, 5, 1, 700, 2048, 64, 65, 1000, 2048, 3, 128, 2000][r % 12]
        n = min(n, int(wl.row_pos[r]) + 1)
        idx[r, :n] = rng.choice(int(wl.row_pos[r]) + 1, n, replace=False)
        cnt[r] = n
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    for S in (0, 1, 3):
        out = torch.zeros((wl.R, wl.H, 512), device=DEV)
        lse = torch.zeros((wl.R, wl.H), device=DEV)
        wsz = api.dsa_sparse_mla_decode_workspace_size(wl.R, wl.H, k, S)
        ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
        err = _err()
        api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, t(idx), t(cnt), out, lse,
                                  err, workspace=ws, num_splits=S)
        assert api.dsa_read_error(err) == 0
        for r in range(wl.R):
            O_ref, l_ref = orc.row_attention(wl, r, idx[r, : cnt[r]])
            eo, el = attn_err(out[r].cpu().numpy(), lse[r].cpu().numpy(), O_ref, l_ref)
            assert eo <= (2e-3 if cfg == 1 else 5e-3) and el <= 1e-4, (S, r, eo, el)


def test_sparse_mla_many_rows_split_forms_agree():
    """420 rows on an fp8 cache with selections of every size from 0 to 2048:
    the automatic split choice (one split per row here: the output written
    in place) against four splits merged by their LSEs, every row, and
    sampled rows against the oracle."""
    wl = make_workload(config_spec(2, B=70, L_lo=2500, L_hi=4000))
    dw = upload(wl, DEV)
    rng = np.random.default_rng(17)
    k = 2048
    sizes = [2048, 0, 1, 127, 128, 129, 700, 2047, 64, 2048, 1500, 3]
    idx = np.full((wl.R, k), -1, np.int32)
    cnt = np.zeros(wl.R, np.int32)
    for r in range(wl.R):
        n = min(sizes[r % len(sizes)], int(wl.row_pos[r]) + 1)
        idx[r, :n] = rng.choice(int(wl.row_pos[r]) + 1, n, replace=False)
        cnt[r] = n
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    res = {}
    for S in (0, 4):
        out = torch.full((wl.R, wl.H, 512), float("nan"), device=DEV)
        lse = torch.full((wl.R, wl.H), float("nan"), device=DEV)
        ws = torch.zeros(max(1, api.dsa_sparse_mla_decode_workspace_size(wl.R, wl.H, k, S)),
                         dtype=torch.uint8, device=DEV)
        err = _err()
        api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, t(idx), t(cnt), out, lse,
                                  err, workspace=ws, num_splits=S)
        assert api.dsa_read_error(err) == 0
        res[S] = (out.cpu().numpy(), lse.cpu().numpy())
    (o0, l0), (o4, l4) = res[0], res[4]
    assert np.isfinite(o0).all()
    both_inf = np.isneginf(l0) & np.isneginf(l4)
    assert np.array_equal(np.isneginf(l0), np.isneginf(l4))
    assert np.all(np.where(both_inf, 0.0, np.abs(l0 - l4)) <= 1e-4)
    den = np.abs(o4).max(axis=-1)
    rel = np.abs(o0 - o4).max(axis=-1) / np.where(den > 0, den, 1.0)
    assert rel.max() <= 5e-3
    for r in list(range(0, 24)) + list(range(wl.R - 12, wl.R)) + list(rng.choice(wl.R, 24)):
        O_ref, l_ref = orc.row_attention(wl, r, idx[r, : cnt[r]])
        eo, el = attn_err(o0[r], l0[r], O_ref, l_ref)
        assert eo <= 5e-3 and el <= 1e-4, (r, int(cnt[r]), eo, el)


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_sparse_mla_prefill_into(cfg):
    """Sparse attention of a prefill chunk (two requests of 40 query rows at
    consecutive positions, each row with its own selection from its causal
    prefix, some empty) into caller-owned O, max-logit and LSE buffers."""
    wl = make_workload(config_spec(cfg, B=2, L=3000, L_lo=2500, L_hi=4000, rows_per_req=40))
    dw = upload(wl, DEV)
    rng = np.random.default_rng(31)
    k = 2048
    idx = np.full((wl.R, k), -1, np.int32)
    cnt = np.zeros(wl.R, np.int32)
    for r in range(wl.R):
        n = [2048, 0, 1, 700, 2048, 64, 65, 1000, 3, 2047][r % 10]
        n = min(n, int(wl.row_pos[r]) + 1)
        idx[r, :n] = np.sort(rng.choice(int(wl.row_pos[r]) + 1, n, replace=False))
        cnt[r] = n
    t = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    for S in (0, 1, 3):
        out = torch.full((wl.R, wl.H, 512), 7.0, device=DEV)
        mx = torch.full((wl.R, wl.H), 7.0, device=DEV)
        lse = torch.full((wl.R, wl.H), 7.0, device=DEV)
        wsz = api.dsa_sparse_mla_prefill_into_workspace_size(wl.R, wl.H, k, S)
        ws = torch.zeros(max(wsz, 1), dtype=torch.uint8, device=DEV)
        err = _err()
        api.dsa_sparse_mla_prefill_into(dw.q, wl.sm_scale, dw.kv, dw.rows, t(idx), t(cnt), out,
                                        mx, lse, err, workspace=ws, num_splits=S)
        assert api.dsa_read_error(err) == 0
        O_all, m_all, l_all = out.cpu().numpy(), mx.cpu().numpy(), lse.cpu().numpy()
        for r in range(wl.R):
            O_ref, m_ref, l_ref = orc.row_attention_into(wl, r, idx[r, : cnt[r]])
            if cnt[r] == 0:
                assert np.all(O_all[r] == 0) and np.all(np.isneginf(m_all[r]))
                assert np.all(np.isneginf(l_all[r]))
                continue
            eo, el = attn_err(O_all[r], l_all[r], O_ref, l_ref)
            assert eo <= (5e-3 if cfg == 2 else 2e-3) and el <= 1e-4, (S, r, eo, el)
            assert np.max(np.abs(m_all[r] - m_ref)) <= 1e-4, (S, r)
            # the bound the three outputs satisfy together
            assert np.all(m_all[r] <= l_all[r] + 1e-5)
            assert np.all(m_all[r] >= l_all[r] - np.log(cnt[r]) - 1e-5)


def test_sparse_mla_running_max_moves_fp8():
    """fp8 latent rows whose token scales are multiplied by 1, 10 and 30 in
    runs of 128 selected rows (one tensor-core tile): the maximum logit of
    every head jumps by several nats from one tile to the next, so the
    running maxima must move and the accumulated output be rescaled."""
    wl = make_workload(config_spec(2, B=2, L_lo=2500, L_hi=4000))
    rng = np.random.default_rng(12)
    k = 2048
    idx = np.zeros((wl.R, k), np.int32)
    cnt = np.zeros(wl.R, np.int32)
    c = wl.kv
    for r in range(wl.R):
        n = min(k, int(wl.row_pos[r]) + 1)
        idx[r, :n] = rng.choice(int(wl.row_pos[r]) + 1, n, replace=False).astype(np.int32)
        cnt[r] = n
    # the same token is selected by several rows of a request: scale tokens by
    # their rank in row 0 of the request, so every row sees jumps
    for b in range(wl.B):
        r0 = int(wl.row_start[b])
        for rank, t in enumerate(idx[r0, : cnt[r0]]):
            f = (1.0, 10.0, 30.0)[(rank // 128) % 3]
            pg, sl = c.physical_page(b, int(t) // c.page_size), int(t) % c.page_size
            c.scale[pg, sl] *= np.float32(f)
    dw = upload(wl, DEV)
    t_ = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    for S in (0, 1, 3):
        out = torch.zeros((wl.R, wl.H, 512), device=DEV)
        lse = torch.zeros((wl.R, wl.H), device=DEV)
        ws = torch.zeros(max(api.dsa_sparse_mla_decode_workspace_size(wl.R, wl.H, k, S), 1),
                         dtype=torch.uint8, device=DEV)
        err = _err()
        api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, t_(idx), t_(cnt), out, lse,
                                  err, workspace=ws, num_splits=S)
        assert api.dsa_read_error(err) == 0
        for r in range(wl.R):
            O_ref, l_ref = orc.row_attention(wl, r, idx[r, : cnt[r]])
            eo, el = attn_err(out[r].cpu().numpy(), lse[r].cpu().numpy(), O_ref, l_ref)
            assert eo <= 5e-3 and el <= 1e-4, (S, r, eo, el)


@pytest.mark.parametrize("cfg", [0, 1])
def test_sparse_mla_running_max_moves(cfg):
    """Selected rows scaled by 1, 10 and 30 tile by tile (64 tokens, in list
    order): every head's maximum logit jumps by several nats from one tile to
    the next, so the kernel must move its running maxima and rescale the
    accumulated output (the lazy rule moves a maximum only past 2^8)."""
    from workloads.synth import to_bf16_bits
    wl = make_workload(config_spec(cfg, B=2, L=3000))
    rng = np.random.default_rng(11)
    k = 2048
    idx = np.zeros((wl.R, k), np.int32)
    cnt = np.zeros(wl.R, np.int32)
    c = wl.kv
    for r in range(wl.R):
        b = int(wl.row_req[r])
        n = min(k, int(wl.row_pos[r]) + 1)
        sel = rng.choice(int(wl.row_pos[r]) + 1, n, replace=False).astype(np.int32)
        idx[r, :n] = sel
        cnt[r] = n
        for rank, t in enumerate(sel):
            f = (1.0, 10.0, 30.0)[(rank // 64) % 3]
            pg, sl = c.physical_page(b, int(t) // c.page_size), int(t) % c.page_size
            c.data[pg, sl] = to_bf16_bits(orc.bf16_bits_to_f64(c.data[pg, sl]) * f)
    dw = upload(wl, DEV)
    t_ = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
    for S in (1, 3):
        out = torch.zeros((wl.R, wl.H, 512), device=DEV)
        lse = torch.zeros((wl.R, wl.H), device=DEV)
        ws = torch.zeros(max(api.dsa_sparse_mla_decode_workspace_size(wl.R, wl.H, k, S), 1),
                         dtype=torch.uint8, device=DEV)
        err = _err()
        api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, t_(idx), t_(cnt), out, lse,
                                  err, workspace=ws, num_splits=S)
        assert api.dsa_read_error(err) == 0
        for r in range(wl.R):
            O_ref, l_ref = orc.row_attention(wl, r, idx[r, : cnt[r]])
            assert l_ref.max() > 10.0, "the scaled tiles dominate"
            eo, el = attn_err(out[r].cpu().numpy(), lse[r].cpu().numpy(), O_ref, l_ref)
            assert eo <= 2e-3 and el <= 1e-4, (S, r, eo, el)


@pytest.mark.parametrize("P,dv", [(5, 512), (9, 512), (40, 512), (128, 512), (128, 96),
                                  (1030, 512)])
def test_lse_merge_against_oracle(P, dv):
    """All three forms of the merge: up to 8 parts (every load at once), the
    live-list form (9..1024 parts, split between thread groups), and the
    sequential form beyond; many empty parts (LSE -inf) among them."""
    rng = np.random.default_rng(4)
    R, H = 3, 4
    Op = rng.standard_normal((P, R, H, dv)).astype(np.float32)
    lp = (rng.standard_normal((P, R, H)) * 3).astype(np.float32)
    lp[1, 0, :] = -np.inf
    lp[:, 2, 1] = -np.inf  # a fully empty (row, head)
    if P > 8:
        lp[rng.random((P, R, H)) < 0.7] = -np.inf  # most parts empty, as split-K leaves them
    out = torch.zeros((R, H, dv), device=DEV)
    ol = torch.zeros((R, H), device=DEV)
    api.dsa_lse_merge(torch.from_numpy(Op).to(DEV), torch.from_numpy(lp).to(DEV), out, ol)
    torch.cuda.synchronize()
    for r in range(R):
        O_ref, l_ref = orc.lse_merge(Op[:, r].astype(np.float64), lp[:, r].astype(np.float64))
        assert np.allclose(out[r].cpu().numpy(), O_ref, rtol=1e-5, atol=1e-6)
        got = ol[r].cpu().numpy()
        assert np.array_equal(np.isneginf(got), np.isneginf(l_ref))
        fin = np.isfinite(l_ref)
        assert np.allclose(got[fin], l_ref[fin], atol=1e-5)


# ------------------------------------------------------------- edge cases


def test_single_token_rows():
    """pos = 0: the only token is selected; O = its value, LSE = its logit."""
    wl = make_workload(config_spec(1, B=3, L=1))
    dw = upload(wl, DEV)
    run = DecodeRun(dw)
    assert run.run() == 0
    check_decode_rows(run, range(wl.R))
    assert np.all(run.cnt.cpu().numpy() == 1)


def test_all_equal_scores_pick_first_positions():
    wl = make_workload(config_spec(1, B=2, L=5000))
    wl.idx_k.data[:] = 0  # every key 0 -> every score 0 -> ties everywhere
    dw = upload(wl, DEV)
    run = DecodeRun(dw)
    assert run.run() == 0
    idx = run.idx.cpu().numpy()
    assert np.array_equal(idx[0], np.arange(2048)) and np.array_equal(idx[1], np.arange(2048))
    check_decode_rows(run, range(wl.R))


def test_bad_page_sets_error_bit():
    wl = make_workload(config_spec(1, B=2, L=3000))
    wl.idx_k.block_table = wl.idx_k.block_table.copy()
    wl.idx_k.block_table[1, 3] = -1
    dw = upload(wl, DEV)
    run = DecodeRun(dw)
    e = run.run()
    assert e & C.DSA_DEVERR_PAGE


def test_position_past_block_table_sets_error_bit():
    wl = make_workload(config_spec(1, B=2, L=300))
    wl.row_pos = wl.row_pos.copy()
    wl.row_pos[0] = 64 * wl.idx_k.max_blocks + 5
    dw = upload(wl, DEV)
    run = DecodeRun(dw)
    e = run.run()
    assert e & C.DSA_DEVERR_POS


def test_empty_batch_is_a_no_op():
    wl = make_workload(config_spec(1, B=1, L=100))
    dw = upload(wl, DEV)
    dw.rows.row_pos = dw.rows.row_pos[:0]
    dw.rows.row_start = torch.zeros(2, dtype=torch.int32, device=DEV)
    out = torch.zeros((0, 32, 512), device=DEV)
    lse = torch.zeros((0, 32), device=DEV)
    d = api.DecodeDesc([dw.idx_k], [dw.kv], dw.rows, dw.q_idx, dw.w_idx, dw.q, wl.sm_scale,
                       2048, out, lse)
    ws = torch.zeros(max(1, api.dsa_decode_workspace_size(d)), dtype=torch.uint8, device=DEV)
    api.dsa_decode(d, ws, _err())
    torch.cuda.synchronize()


def test_long_single_row_max_length():
    """One 131072-token row (the longest cfg 4 length), fp8."""
    wl = make_workload(config_spec(4, B=1, seq_lens=(131072,)))
    dw = upload(wl, DEV)
    run = DecodeRun(dw)
    assert run.run() == 0
    check_decode_rows(run, [0])


@pytest.mark.parametrize("limit_us", [0, 1000, 20000])
def test_bounded_wait_gives_up_and_reports(limit_us):
    """The kernels' bounded mbarrier wait, on a phase nothing completes: it
    returns after its limit (not before, and within a few ms after), sets
    DSA_DEVERR_TIMEOUT in the error word, and the context stays usable."""
    err = _err()
    waited = torch.zeros(1, dtype=torch.int64, device=DEV)
    api.dsa_selftest_bounded_wait(limit_us, err, waited)
    assert api.dsa_read_error(err) & C.DSA_DEVERR_TIMEOUT
    w_ns = int(waited.item())
    assert limit_us * 1000 <= w_ns <= limit_us * 1000 + 5_000_000
    # the device still runs work after the timeout
    x = torch.arange(1000, device=DEV)
    assert int(x.sum().item()) == 999 * 1000 // 2
