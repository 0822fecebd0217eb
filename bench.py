#!/usr/bin/env python
"""Benchmark of the DSA sparse-attention decode path on GB300.

Default workload: the ragged throughput sweep's largest batch, B = 256
requests x 1 query row, per-request cached length drawn log-uniform in
[4K, 128K], fp8_e4m3 index keys and latent rows with one fp32 scale per token,
64 x 128 indexer, 32 MLA heads x 576-wide latent rows, top-2048, 64-token
pages with seeded random block tables (synthetic data).  `--config N`
(`--batch B` for configuration 4) selects another configuration of the
same contract line.

A step is one dsa_decode call (indexer -> top-k -> sparse MLA split-K ->
LSE merge) over the whole batch, inputs resident in HBM.  Between timed steps
L2 is flushed by writing a 512 MB buffer and then reading a 256 MB one (the
step's own HBM stream is also larger than L2 for every configuration but the
tiny one).  Each step is timed with CUDA events on the launching stream;
`value` = rows of all ranks / max over ranks of the summed step time.

`--impl reference` times the CPU oracle instead (the only other place that
runs it is the `cpu_baseline` leg): same workload, same metric, each step a
bounded sample of rows.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# the CPU oracle's BLAS uses every visible core; fix the count before numpy loads
_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np  # noqa: E402

METRIC = "DSA decode query-rows/sec at 1 GB300; HBM GB/s as fraction of ~8 TB/s roofline"
UNIT = "rows/s"
DEFAULT_CONFIG = 4
DEFAULT_BATCH = 256
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="product", choices=["product", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (host copies through the C ABI)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG,
                    help="workload: configuration 0..4 (default 4, the ragged fp8 sweep)")
    ap.add_argument("--batch", type=int, default=None,
                    help=f"requests of configuration 4 (default {DEFAULT_BATCH})")
    ap.add_argument("--rows-per-req", type=int, default=None,
                    help="query rows per request at consecutive positions "
                         "(MTP verify or a multi-query extend)")
    ap.add_argument("--kernel", default=None,
                    choices=["indexer", "topk", "mla", "cache_write", "prefill_into"],
                    help="time one kernel of the step alone on the same workload (a short "
                         "run for profilers: W warm-up launches, then K timed ones); "
                         "prefill_into: the sparse attention of every query row into "
                         "caller-owned O, max-logit and LSE (with --rows-per-req, a chunk of "
                         "that many rows per request)")
    return ap.parse_args()


def workload_spec(args):
    from workloads import config_spec

    kw = {}
    if args.config == 4:
        kw["B"] = args.batch or DEFAULT_BATCH
    elif args.batch:
        kw["B"] = args.batch
    if args.rows_per_req:
        kw["rows_per_req"] = args.rows_per_req
    return config_spec(args.config, **kw)


def describe(wl) -> dict:
    """The workload's name and shape for the JSON line's `config`."""
    s = wl.spec
    L = wl.seq_len
    law = (f"L={int(L[0])}" if s.length_law == "fixed" and s.seq_lens is None else
           f"L {s.length_law} in [{s.L_lo}, {s.L_hi}] (drawn: min {int(L.min())}, "
           f"mean {float(L.mean()):.0f}, max {int(L.max())})")
    store = "bf16" if s.dtype == "bf16" else "fp8_e4m3 (one fp32 scale per token)"
    paging = "page 64, random block tables" if s.paged else "contiguous"
    text = (f"{s.name}: decode B={s.B} x {s.rows_per_req} row(s), {law}, {store} index-K and "
            f"latent caches ({paging}), indexer 64x128, MLA {s.H} heads x 576, "
            f"top-{s.topk}" + (f", W={s.shards} token shards emulated on one GPU"
                               if s.shards > 1 else ""))
    return {"workload": text, "global_batch": int(wl.R), "seq_len_mean": float(L.mean()),
            "seq_len_max": int(L.max()), "kv_dtype": s.dtype, "topk": s.topk,
            "mla_heads": s.H, "shards": s.shards}


# ----------------------------------------------------------------- ranks


def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n:
        raise SystemExit(f"--gpus {n} but WORLD_SIZE={world}")
    return rank, world, local


def aggregate(rows_local: float, seconds_local: float, group=None, device=None):
    """Whole-job throughput: the rows of all ranks over the slowest rank's
    time.  Returns (value, max_seconds, total_rows)."""
    import torch
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        t = torch.tensor([seconds_local], dtype=torch.float64, device=device)
        n = torch.tensor([rows_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
        sec, rows = float(t.item()), float(n.item())
    else:
        sec, rows = seconds_local, rows_local
    return rows / sec, sec, rows


# ----------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the sampled clocks of this run (a git-ignored build folder)
        self.path = os.path.join(ROOT, "_build", f"clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            ident = str(self.gpu)
            try:
                import torch
                u = str(torch.cuda.get_device_properties(self.gpu).uuid)
                ident = u if u.startswith("GPU-") else "GPU-" + u
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        try:
            lines = [l.strip() for l in open(self.path) if l.strip()]
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- helpers


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def kernel_source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dsa_sparse_attention_decode_gb300", "csrc")
    for n in names:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summaries, if one was
    taken of this kernel on this workload with the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            entries = json.load(f)
    except Exception:
        return None
    for d in entries:
        if d.get("kernel") != kernel or d.get("workload") != workload:
            continue
        if d.get("source_hash") != kernel_source_hash(d.get("sources", [])):
            return None
        return d.get("dram_bytes_per_launch")
    return None


def algorithmic_bytes(wl):
    """Bytes the method must move per step, per kernel:
    indexer: key stream (+ fp8 scales) + block tables + queries/weights;
    top-k: the valid scores read + the selection written;
    MLA (+ LSE merge): selected latent rows (+ fp8 scales) + indices + query
    + output/LSE; with W shards also the W partials the merge reads and the
    result it writes (H * 513 * 4 B each)."""
    R, H = wl.R, wl.H
    k = wl.topk
    W = max(1, wl.W)
    esz = 2 if wl.spec.dtype == "bf16" else 1
    per_tok_idx = 128 * esz + (0 if esz == 2 else 4)
    per_tok_kv = 576 * esz + (0 if esz == 2 else 4)
    idx = 0
    for b in range(wl.B):
        L = int(wl.row_pos[wl.row_start[b + 1] - 1]) + 1
        idx += L * per_tok_idx + ((L + 63) // 64) * 4
    idx += R * (64 * 128 * 2 + 64 * 4)
    topk = 0
    mla = 0
    for r in range(R):
        valid = int(wl.row_pos[r]) + 1
        n = min(k, valid)
        topk += valid * 4 + k * 4 + 4
        mla += n * per_tok_kv + k * 4 + H * 576 * 2 + H * 512 * 4 + H * 4
        if W > 1:
            mla += (W + 1) * H * 513 * 4
    return {"indexer": idx, "topk": topk, "mla": mla}


# ----------------------------------------------------------------- product arm


def run_kernel_only(args):
    """One kernel of the step on the benchmark's workload: `warmup` untimed
    launches, then `steps` timed ones with the L2 flush between them.  The
    launches a profiler should capture are the last `steps` of that kernel."""
    import torch

    import dsa_sparse_attention_decode_gb300 as pkg
    from dsa_sparse_attention_decode_gb300 import api
    from workloads import make_workload
    from workloads.device import decode_args, upload

    pkg.build()
    pkg.lib()
    dev = torch.device("cuda", 0)
    spec = workload_spec(args)
    if spec.shards > 1:
        raise SystemExit("--kernel times the unsharded path; configuration 3 is sharded")
    wl = make_workload(spec)
    dw = upload(wl, dev)
    R, H, k = wl.R, wl.H, wl.topk
    out = torch.empty(R, H, 512, device=dev)
    lse = torch.empty(R, H, device=dev)
    tidx = torch.empty(R, k, dtype=torch.int32, device=dev)
    tcnt = torch.empty(R, dtype=torch.int32, device=dev)
    desc = decode_args(dw, False, out, lse, tidx, tcnt)
    lay = api.dsa_decode_workspace_layout(desc)
    ws = torch.zeros(lay.total_bytes, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dsa_decode(desc, ws, err)  # produces the scores and selections the kernels read
    scores = ws[lay.scores: lay.scores + R * lay.ld_scores * 4].view(torch.float32).view(
        R, lay.ld_scores)
    valid = (dw.rows.row_pos + 1).to(torch.int32)
    mla_ws = torch.empty(max(1, api.dsa_sparse_mla_decode_workspace_size(R, H, k, lay.num_splits)),
                         dtype=torch.uint8, device=dev)
    if args.kernel == "cache_write":
        return time_cache_write(args, dw, spec, dev, err)
    topk_ws = torch.empty(max(1, api.dsa_topk_workspace_size(R, lay.ld_scores)), dtype=torch.uint8,
                          device=dev)
    pre_ws = torch.empty(max(1, api.dsa_sparse_mla_prefill_into_workspace_size(R, H, k, 0)),
                         dtype=torch.uint8, device=dev)
    out_max = torch.empty(R, H, device=dev)
    fn = {
        "indexer": lambda: api.dsa_indexer_scores(dw.q_idx, dw.w_idx, dw.idx_k, dw.rows, scores,
                                                  err),
        "topk": lambda: api.dsa_topk(scores, valid, k, tidx, tcnt, err, workspace=topk_ws),
        "mla": lambda: api.dsa_sparse_mla_decode(dw.q, wl.sm_scale, dw.kv, dw.rows, tidx, tcnt,
                                                 out, lse, err, workspace=mla_ws,
                                                 num_splits=lay.num_splits),
        "prefill_into": lambda: api.dsa_sparse_mla_prefill_into(
            dw.q, wl.sm_scale, dw.kv, dw.rows, tidx, tcnt, out, out_max, lse, err,
            workspace=pre_ws, num_splits=0),
    }[args.kernel]
    flush_w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    ms = []
    for i in range(args.warmup + args.steps):
        flush_w.zero_()
        flush_r.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            ms.append(a.elapsed_time(b))
    if api.dsa_read_error(err) != 0:
        raise SystemExit("device error word set")
    line = {"kernel": args.kernel, "workload": spec.name, "launches": args.steps,
            "us_mean": round(1e3 * float(np.mean(ms)), 2)}
    if args.kernel in ("mla", "prefill_into"):
        # rows attended per second, and the gathered latent rows' bytes per
        # second (a row's selections overlap its neighbours' in a chunk, so
        # part of them come from L2)
        row_b = 576 * (1 if spec.dtype == "fp8_e4m3" else 2) + (4 if spec.dtype == "fp8_e4m3" else 0)
        gathered = float(tcnt.sum().item()) * row_b
        sec = float(np.mean(ms)) * 1e-3
        line.update({"rows": R, "rows_per_req": spec.rows_per_req,
                     "rows_per_s": round(R / sec, 1),
                     "gathered_gbs": round(gathered / sec / 1e9, 1)})
    print(json.dumps(line), flush=True)


def time_cache_write(args, dw, spec, dev, err):
    """The cache write of one decode step (one new token per request, at the
    row's position) and of a 1024-token append per request, into the
    workload's own caches (their contents change: this mode times only)."""
    import torch

    from dsa_sparse_attention_decode_gb300 import api

    B = dw.rows.num_reqs
    flush_w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(11)
    res = {}
    for name, per_req in (("decode_step", 1), ("append_1024", 1024)):
        N = B * per_req
        req = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(per_req)
        last = dw.rows.row_pos[dw.rows.row_start[1:].long() - 1]
        pos = (last.repeat_interleave(per_req) -
               torch.arange(per_req, dtype=torch.int32, device=dev).repeat(B)).to(torch.int32)
        kv_in = torch.randn((N, 576), generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
        ix_in = torch.randn((N, 128), generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
        ms = []
        for i in range(args.warmup + args.steps):
            flush_w.zero_()
            flush_r.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            api.dsa_cache_write(kv_in, req, pos, B, [dw.kv], err, idx_in=ix_in, idx_k=[dw.idx_k])
            b.record()
            torch.cuda.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        us = 1e3 * float(np.median(ms))
        esz = 2 if spec.dtype == "bf16" else 1
        byts = N * (576 * 2 + 128 * 2 + 576 * esz + 128 * esz + (8 if esz == 1 else 0) + 8)
        res[name] = {"tokens": N, "us": round(us, 2), "tokens_per_s": round(N / (us * 1e-6), 1),
                     "algorithmic_bytes": byts, "gbs": round(byts / (us * 1e-6) / 1e9, 1)}
    if api.dsa_read_error(err) != 0:
        raise SystemExit("device error word set")
    print(json.dumps({"kernel": "cache_write", "workload": spec.name, "launches": args.steps,
                      **res}), flush=True)


def run_product(args):
    import torch

    rank, world, local = dist_init(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import dsa_sparse_attention_decode_gb300 as pkg
    from dsa_sparse_attention_decode_gb300 import api
    from workloads import make_workload
    from workloads.device import decode_args, upload

    pkg.build()
    pkg.lib()
    spec = workload_spec(args)
    sharded = spec.shards > 1
    wl = make_workload(spec)
    dw = upload(wl, dev, shards=sharded, unsharded=not sharded)
    R, H, k = wl.R, wl.H, wl.topk
    out = torch.empty(R, H, 512, device=dev)
    lse = torch.empty(R, H, device=dev)
    tidx = torch.empty(R, k, dtype=torch.int32, device=dev)
    tcnt = torch.empty(R, dtype=torch.int32, device=dev)
    desc = decode_args(dw, sharded, out, lse, tidx, tcnt)
    lay = api.dsa_decode_workspace_layout(desc)
    ws = torch.zeros(lay.total_bytes, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        # write 512 MB (> L2), then read 256 MB so that L2 is left holding clean
        # lines: no write-back of the flush competes with the next timed kernel
        flush_w.zero_()
        flush_r.sum()

    def step():
        api.dsa_decode(desc, ws, err, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if api.dsa_read_error(err) != 0:
        raise SystemExit("device error word set during warm-up")

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        # a head start for the host: the GPU spins for a few milliseconds while
        # every step is queued, so no bracketed step waits on the host
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(20_000_000)
        for a, b in evs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed(step, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_sec = sum(ms) / 1e3
    value, max_sec, total_rows = aggregate(R * args.steps, step_sec, device=dev)
    ms_per_step = max_sec * 1e3 / args.steps

    # ---- per-kernel timing of the same path (live, CUDA events, same stream),
    # through the single-step entry points on the step's own intermediates
    alg = algorithmic_bytes(wl)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    kern_us = {}
    if not sharded:
        scores = ws[lay.scores: lay.scores + R * lay.ld_scores * 4].view(torch.float32).view(
            R, lay.ld_scores)
        valid = (dw.rows.row_pos + 1).to(torch.int32)
        kern = {}
        kern["indexer"] = timed(lambda: api.dsa_indexer_scores(
            dw.q_idx, dw.w_idx, dw.idx_k, dw.rows, scores, err, stream=stream), args.steps)
        topk_ws = torch.empty(max(1, api.dsa_topk_workspace_size(R, lay.ld_scores)),
                              dtype=torch.uint8, device=dev)
        kern["topk"] = timed(lambda: api.dsa_topk(scores, valid, k, tidx, tcnt, err,
                                                  workspace=topk_ws, stream=stream), args.steps)
        mla_ws = torch.empty(max(1, api.dsa_sparse_mla_decode_workspace_size(
            R, H, k, lay.num_splits)), dtype=torch.uint8, device=dev)
        kern["mla"] = timed(lambda: api.dsa_sparse_mla_decode(
            dw.q, wl.sm_scale, dw.kv, dw.rows, tidx, tcnt, out, lse, err, workspace=mla_ws,
            num_splits=lay.num_splits, stream=stream), args.steps)
        torch.cuda.synchronize()
        if api.dsa_read_error(err) != 0:
            raise SystemExit("device error word set")
        # median: one launch delayed by the host (the events bracket it) must
        # not skew the per-kernel figures
        kern_us = {n: 1e3 * float(np.median(v)) for n, v in kern.items()}
    kernel_names = {"indexer": "indexer_kernel (dsa_indexer_scores)",
                    "topk": "topk_kernel (dsa_topk)",
                    "mla": "sparse_mla_kernel + lse_merge_kernel (dsa_sparse_mla_decode)"}
    kernels = {}
    for n, us in kern_us.items():
        gbs = alg[n] / (us * 1e-6) / 1e9
        kernels[n] = {"us": round(us, 2), "algorithmic_bytes": alg[n], "gbs": round(gbs, 1),
                      "frac_of_measured_hbm": round(gbs / hbm, 4)}
    if "topk" in kernels:
        kernels["topk"]["note"] = "reads the indexer's scores from L2 where they fit"

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its inputs (queries, weights, row metadata, block tables) from one pinned
    # staging buffer into one device buffer that the descriptor points into,
    # runs the decode, and copies O and LSE (one device allocation) back; the
    # caches stay resident in HBM.  The steps are pipelined the way a serving
    # loop would run them: device inputs and outputs are double-buffered, the
    # input copy of step i + 1 runs on one copy stream and the result copy of
    # step i - 1 on another while step i computes, ordered by events.  One
    # timed region spans all steps, from the first input copy to the last
    # result copy (no L2 flush inside it: every step streams its caches,
    # more than the 129 MB L2 for every configuration but the tiny one).
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(args, api, dw, wl, sharded, ws, err, stream, out, lse, tidx, tcnt, dev)

    # ---- roofline of the dominant kernel (the longest one of the step)
    path_bytes = sum(alg.values())
    path_gbs = path_bytes / (ms_per_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "peak": hbm, "unit": "GB/s", "peak_source": peak_kind,
                "path_algorithmic_bytes_per_step": path_bytes,
                "path_achieved_gbs": round(path_gbs, 1),
                "path_frac": round(path_gbs / hbm, 4),
                "path_frac_of_nominal_8tbs": round(path_gbs / NOMINAL_HBM_GBS, 4)}
    if kern_us:
        dom = max(("indexer", "mla"), key=lambda n: kern_us[n])
        ach = alg[dom] / (kern_us[dom] * 1e-6) / 1e9
        roofline.update({"kernel": kernel_names[dom], "achieved": round(ach, 1),
                         "frac": round(ach / hbm, 4), "algorithmic_bytes_per_launch": alg[dom],
                         "traffic": ncu_traffic(dom, spec.name)})
    else:
        roofline.update({"kernel": "whole dsa_decode step (sharded: no single-kernel timing)",
                         "achieved": round(path_gbs, 1), "frac": round(path_gbs / hbm, 4),
                         "algorithmic_bytes_per_launch": path_bytes, "traffic": None})

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank == 0:
        launches_per_step = int(lay.launches)  # the library's own count for this layout
        cfg = describe(wl)
        cfg["parallelism"] = f"dp{world} (independent request batches per GPU)"
        cfg["l2"] = ("flushed between timed steps (512 MB write, then 256 MB read); "
                     f"the step streams {path_bytes / 1e6:.0f} MB")
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3 caches, fp32 accumulate" if spec.dtype != "bf16" else "bf16",
            "data": "synthetic (seeded N(0,1)/N(0,0.5) caches and queries, U(0,1)/8 weights)",
            "config": cfg,
            "roofline": roofline,
            "num_splits": lay.num_splits,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_leg(args, api, dw, wl, sharded, ws, err, stream, out, lse, tidx, tcnt, dev):
    """The decode through the C ABI with host buffers (see run_product)."""
    import dataclasses

    import torch

    from dsa_sparse_attention_decode_gb300.api import DecodeDesc

    R, H, k = wl.R, wl.H, wl.topk
    ik = dw.idx_k_shards if sharded else [dw.idx_k]
    kv = dw.kv_shards if sharded else [dw.kv]
    W = len(ik)
    in_src = [dw.q_idx, dw.w_idx, dw.q, dw.rows.row_start, dw.rows.row_pos]
    bt_at = []
    for c in list(ik) + list(kv):
        if c.block_table is not None:
            bt_at.append(len(in_src))
            in_src.append(c.block_table)
        else:
            bt_at.append(None)
    offs, total = [], 0
    for t in in_src:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_pack = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for t, o in zip(in_src, offs):
        nb = t.numel() * t.element_size()
        h_pack[o:o + nb].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
    o_elems = R * H * 512
    d_pack, d_res, h_res, desc_e = [], [], [], []
    for _ in range(2):
        dp = torch.empty(total, dtype=torch.uint8, device=dev)
        views = []
        for t, o in zip(in_src, offs):
            nb = t.numel() * t.element_size()
            views.append(dp[o:o + nb].view(t.dtype).view(t.shape))
        rows_e = dataclasses.replace(dw.rows, row_start=views[3], row_pos=views[4])
        caches = [c if j is None else dataclasses.replace(c, block_table=views[j])
                  for c, j in zip(list(ik) + list(kv), bt_at)]
        dr = torch.empty(o_elems + R * H, dtype=torch.float32, device=dev)
        d_pack.append(dp)
        d_res.append(dr)
        h_res.append(torch.empty(o_elems + R * H, dtype=torch.float32, pin_memory=True))
        desc_e.append(DecodeDesc(caches[:W], caches[W:], rows_e, views[0], views[1], views[2],
                                 wl.sm_scale, k, dr[:o_elems].view(R, H, 512),
                                 dr[o_elems:].view(R, H), out_topk_idx=tidx, out_topk_count=tcnt))
    h2d = sum(t.numel() * t.element_size() for t in in_src)
    d2h = d_res[0].numel() * 4
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_run(n, head_start=True):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_in):
            if head_start and hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(20_000_000)  # the host queues every step meanwhile
            t0.record(s_in)
        stream.wait_event(t0)
        s_out.wait_event(t0)
        for i in range(n):
            bsel = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])  # step i - 2 is done with this input buffer
                d_pack[bsel].copy_(h_pack, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # this result buffer has been copied out
            api.dsa_decode(desc_e[bsel], ws, err, stream=stream)
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                h_res[bsel].copy_(d_res[bsel], non_blocking=True)
                ev_out[i].record(s_out)
        t1.record(s_out)  # after the last result copy, which follows every other step
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_run(2, head_start=False)
    e2e_ms = e2e_run(args.steps)
    e2e_value, _, _ = aggregate(R * args.steps, e2e_ms / 1e3, device=dev)
    torch.cuda.synchronize()
    if api.dsa_read_error(err) != 0:
        raise SystemExit("device error word set in the end-to-end leg")
    # the device leg's last full step left its O and LSE in `out` / `lse`
    # (the per-kernel timing rewrote them with the same values)
    last = (args.steps - 1) & 1
    got = torch.from_numpy(h_res[last].numpy().copy())
    if not (torch.equal(got[:o_elems].view(R, H, 512), out.cpu())
            and torch.equal(got[o_elems:].view(R, H), lse.cpu())):
        raise SystemExit("the end-to-end leg and the device leg disagree")
    return {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "note": "per-step inputs (queries, weights, rows, block tables) from pinned host "
                    "memory and O/LSE back; caches stay resident in HBM; steps pipelined "
                    "(input copy of step i+1 and result copy of step i-1 on two copy streams "
                    "while step i computes, double-buffered device inputs/outputs), one timed "
                    "region over all steps, no L2 flush inside it"}


# ----------------------------------------------------------------- CPU oracle


def cpu_baseline(wl, seconds: float):
    from oracle import dsa_oracle as orc

    rows, t0 = 0, time.perf_counter()
    r = 0
    toks = 0
    while True:
        orc.decode_row(wl, r % wl.R)
        toks += int(wl.row_pos[r % wl.R]) + 1
        rows += 1
        r += 1
        el = time.perf_counter() - t0
        if el >= seconds and rows >= 2:
            break
    return {"value": round(rows / el, 3), "unit": UNIT, "cores": _CORES, "kind": "oracle",
            "sample": f"{rows} query rows of the same workload (rows 0..{min(rows, wl.R) - 1} in "
                      f"order, {toks / rows:.0f} cached tokens per row on average), one after "
                      f"another, full path (indexer over the row's tokens, exact "
                      f"top-{wl.topk}, MLA) in float64 numpy, {el:.1f} s",
            "single_thread_config0": single_thread_config0()}


# The oracle on the tiny workload (configuration 0: one row over 4096 tokens,
# 16 heads) with one BLAS thread, in a child process (the thread count of
# numpy's BLAS is fixed when it loads).
_SINGLE = """
import sys, time
sys.path.insert(0, sys.argv[1])
from oracle import dsa_oracle as orc
from workloads import config_spec, make_workload
wl = make_workload(config_spec(0))
orc.decode_row(wl, 0)
t0, n = time.perf_counter(), 0
while n < 2 or time.perf_counter() - t0 < float(sys.argv[2]):
    orc.decode_row(wl, 0)
    n += 1
print(n / (time.perf_counter() - t0))
"""


def single_thread_config0(seconds: float = 3.0):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", _SINGLE, ROOT, str(seconds)], env=env,
                           capture_output=True, text=True, timeout=120)
        value = float(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the GPU line does not depend on it
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    return {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "workload": "configuration 0 (one row, L=4096, bf16, 16 heads), one BLAS thread"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import dsa_oracle as orc
    from workloads import make_workload

    wl = make_workload(workload_spec(args))
    for i in range(args.warmup):
        orc.decode_row(wl, i % wl.R)
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.decode_row(wl, i % wl.R)  # each step: one sampled row of the batch
    el = time.perf_counter() - t0
    value = args.steps / el
    cfg = describe(wl)
    cfg["parallelism"] = f"dp{args.gpus} (independent request batches per GPU)"
    cfg["l2"] = "not applicable: the oracle runs on the host cores"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": _CORES,
                         "kind": "oracle",
                         "sample": "one query row of the batch per step, rows 0, 1, 2, ... "
                                   "(full path, float64 numpy)"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.kernel is not None:
        run_kernel_only(a)
        sys.exit(0)
    if a.warmup < 3 and a.impl == "product":
        a.warmup = 3
    if a.impl == "reference":
        run_reference(a)
    else:
        run_product(a)
