"""The allocation-free sparse MLA entry point, for callers that cannot
allocate device memory (its split-K partials live in a fixed device array of
the library): through the C ABI it must give the same results as the
workspace entry point, call after call, and refuse sizes the array cannot
hold.  Collected last on purpose, so that a failure here leaves every other
test already run."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dsa_sparse_attention_decode_gb300 import _lib as C  # noqa: E402
from dsa_sparse_attention_decode_gb300 import api  # noqa: E402
from workloads import config_spec, make_workload  # noqa: E402
from workloads.device import upload  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(cfg=1):
    wl = make_workload(config_spec(cfg, B=6, L=3000, L_lo=2500, L_hi=4000, rows_per_req=1))
    dw = upload(wl, DEV)
    rng = np.random.default_rng(11)
    k = 2048
    idx = np.full((wl.R, k), -1, np.int32)
    cnt = np.zeros(wl.R, np.int32)
    for r in range(wl.R):
        n = [2048, 700, 1, 2048, 65, 1500][r]
        idx[r, :n] = np.sort(rng.choice(int(wl.row_pos[r]) + 1, n, replace=False))
        cnt[r] = n
    return wl, dw, torch.from_numpy(idx).to(DEV), torch.from_numpy(cnt).to(DEV)


def _compare(wl, dw, idx, cnt, S, calls, tol):
    """The allocation-free entry point against the workspace one on the same
    inputs, `calls` times in a row."""
    R, H, k = wl.R, wl.H, 2048
    need = api.dsa_sparse_mla_decode_workspace_size(R, H, k, S)
    assert 0 < need <= C.NOALLOC_SCRATCH_BYTES  # the fixed array is really used
    ref_o = torch.zeros((R, H, 512), device=DEV)
    ref_l = torch.zeros((R, H), device=DEV)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, idx, cnt, ref_o, ref_l, err,
                              workspace=ws, num_splits=S)
    assert api.dsa_read_error(err) == 0
    ref_o, ref_l = ref_o.cpu().numpy(), ref_l.cpu().numpy()
    for _ in range(calls):
        out = torch.full((R, H, 512), float("nan"), device=DEV)
        lse = torch.full((R, H), float("nan"), device=DEV)
        api.dsa_sparse_mla_decode_noalloc(dw.q, wl.sm_scale, dw.kv, dw.rows, idx, cnt, out, lse,
                                          err, num_splits=S)
        assert api.dsa_read_error(err) == 0
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        den = np.abs(ref_o).max(axis=-1)
        rel = np.abs(o - ref_o).max(axis=-1) / np.where(den > 0, den, 1.0)
        assert rel.max() <= tol
        both_inf = np.isneginf(l) & np.isneginf(ref_l)
        assert np.all(np.where(both_inf, 0.0, np.abs(l - ref_l)) <= 1e-4)


@pytest.mark.parametrize("cfg,tol,S", [(1, 2e-3, 4), (2, 5e-3, 4), (2, 5e-3, 0)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cfg, tol, S):
    """bf16 and fp8 caches, four splits and the automatic choice (16 splits
    for these six rows); full selections, then (after the array holds a full
    call's partials) other selections whose later splits are empty, so that
    partials left by the earlier call must not reach the result."""
    wl, dw, idx, cnt = _case(cfg)
    _compare(wl, dw, idx, cnt, S, 2, tol)
    rng = np.random.default_rng(5)
    k = 2048
    idx2 = np.full((wl.R, k), -1, np.int32)
    cnt2 = np.zeros(wl.R, np.int32)
    for r in range(wl.R):
        n = [1, 65, 1, 2048, 65, 1][r]
        idx2[r, :n] = np.sort(rng.choice(int(wl.row_pos[r]) + 1, n, replace=False))
        cnt2[r] = n
    _compare(wl, dw, torch.from_numpy(idx2).to(DEV), torch.from_numpy(cnt2).to(DEV), S, 2, tol)


def test_noalloc_refuses_sizes_beyond_the_array():
    """4096 rows x 32 heads x 32 splits of partials need far more than the
    fixed array holds: the call fails on the host, before any launch."""
    import ctypes

    wl, dw, idx, cnt = _case()
    assert api.dsa_sparse_mla_decode_workspace_size(4096, 32, 2048, 32) > C.NOALLOC_SCRATCH_BYTES
    c = dw.kv.c()
    r = C.DsaRows(num_rows=4096, num_reqs=dw.rows.num_reqs, max_rows_per_req=1,
                  max_len=dw.rows.max_len, row_start=None, row_pos=None)
    st = C.lib().dsa_sparse_mla_decode_noalloc(
        ctypes.c_void_p(dw.q.data_ptr()), 32, wl.sm_scale, ctypes.byref(c), ctypes.byref(r),
        ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()), 2048, 32,
        ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert st == C.DSA_ERR_WORKSPACE_TOO_SMALL
