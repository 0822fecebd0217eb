"""Helpers of the GPU parity tests: run the library through the C ABI and
compare with the CPU oracle under the stated tolerances."""

from __future__ import annotations

import numpy as np
import torch

from dsa_sparse_attention_decode_gb300 import api
from oracle import dsa_oracle as orc
from workloads.device import decode_args, upload

# tolerances
SCORE_RTOL = 1e-4
O_RTOL = {"bf16": 2e-3, "fp8_e4m3": 5e-3}
LSE_ATOL = 1e-4


def score_ok(s_gpu: np.ndarray, s_ref: np.ndarray):
    """|s_gpu - s_ref| <= 1e-4 * max(|s_ref|, 1e-3 * max_t |s_ref|)."""
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    floor = 1e-3 * np.abs(s_ref).max() if s_ref.size else 0.0
    tol = SCORE_RTOL * np.maximum(np.abs(s_ref), floor)
    bad = np.abs(s_gpu - s_ref) > tol
    return not bad.any(), (np.abs(s_gpu - s_ref) / np.maximum(np.abs(s_ref), floor + 1e-300)).max()


def attn_err(O_gpu, lse_gpu, O_ref, lse_ref):
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    den = np.abs(O_ref).max(axis=-1)
    rel = np.abs(O_gpu - O_ref).max(axis=-1) / np.where(den > 0, den, 1.0)
    dl = np.abs(np.asarray(lse_gpu, dtype=np.float64) - lse_ref)
    dl = np.where(np.isneginf(lse_ref) & np.isneginf(lse_gpu), 0.0, dl)
    return rel.max(), dl.max()


class DecodeRun:
    """dsa_decode on one workload; keeps outputs and the workspace."""

    def __init__(self, dw, sharded=False, num_splits=0, device="cuda"):
        wl = dw.wl
        R, H, k = wl.R, wl.H, wl.topk
        self.dw = dw
        self.out = torch.full((R, H, 512), float("nan"), device=device)
        self.lse = torch.full((R, H), float("nan"), device=device)
        self.idx = torch.full((R, k), -7, dtype=torch.int32, device=device)
        self.cnt = torch.full((R,), -7, dtype=torch.int32, device=device)
        self.desc = decode_args(dw, sharded, self.out, self.lse, self.idx, self.cnt,
                                num_splits=num_splits)
        self.lay = api.dsa_decode_workspace_layout(self.desc)
        self.ws = torch.zeros(max(1, self.lay.total_bytes), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.W = len(self.desc._keep[0])

    def run(self):
        api.dsa_decode(self.desc, self.ws, self.err)
        torch.cuda.synchronize()
        return api.dsa_read_error(self.err)

    def scores(self, r: int, w: int = 0, n: int = None) -> np.ndarray:
        wl = self.dw.wl
        W = self.W
        if n is None:
            n = orc.shard_valid_len(int(wl.row_pos[r]), W, w)
        ld = int(self.lay.ld_scores)
        off = self.lay.scores + ((w * wl.R + r) * ld) * 4
        return self.ws[off: off + n * 4].view(torch.float32).cpu().numpy()


def check_decode_rows(run: DecodeRun, rows, check_scores=True):
    """Parity of the fused path on the given rows; returns worst errors."""
    wl = run.dw.wl
    k = wl.topk
    worst_o = worst_l = worst_s = 0.0
    idx = run.idx.cpu().numpy()
    cnt = run.cnt.cpu().numpy()
    out = run.out.cpu().numpy()
    lse = run.lse.cpu().numpy()
    for r in rows:
        r = int(r)
        if run.W == 1:
            s_gpu = run.scores(r)
            if check_scores:
                s_ref = orc.row_scores(wl, r)
                ok, e = score_ok(s_gpu, s_ref)
                assert ok, f"row {r}: scores off by {e:.3e} relative"
                worst_s = max(worst_s, e)
            sel = orc.topk_select(s_gpu.astype(np.float64), k)
        else:
            # sharded: per-shard local top-k of the GPU's shard scores, merged
            cs, cp = [], []
            for w in range(run.W):
                s_loc = run.scores(r, w).astype(np.float64)
                if check_scores:
                    s_ref = orc.row_scores(wl, r, wl.idx_k_shards[w], run.W, w)
                    ok, e = score_ok(s_loc, s_ref)
                    assert ok, f"row {r} shard {w}: scores off by {e:.3e}"
                    worst_s = max(worst_s, e)
                j = orc.topk_select(s_loc, k)
                cs.append(s_loc[j])
                cp.append(j * run.W + w)
            sel, _ = orc.merge_candidates(cs, cp, k, run.W)
        assert cnt[r] == len(sel), f"row {r}: count {cnt[r]} != {len(sel)}"
        assert np.array_equal(idx[r, : cnt[r]], sel), f"row {r}: top-k indices differ"
        assert np.all(idx[r, cnt[r]:] == -1), f"row {r}: padding not -1"
        O_ref, lse_ref = orc.row_attention(wl, r, sel)
        eo, el = attn_err(out[r], lse[r], O_ref, lse_ref)
        assert eo <= O_RTOL[wl.spec.dtype], f"row {r}: O rel err {eo:.3e}"
        assert el <= LSE_ATOL, f"row {r}: LSE err {el:.3e}"
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    return worst_s, worst_o, worst_l
