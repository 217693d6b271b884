#!/usr/bin/env python3
"""Benchmark of the MFA decode hot path on GB300.

One step = one decode step of a whole batch through the C ABI:
    mfa_decode_attention (split-KV kernel + LSE combine) over the cache,
preceded by mfa_kv_append (one new token per sequence) for the workload
that appends before attending (ragged); the others attend over a cache of
fixed length.
Inputs are seeded synthetic data with the workload's shapes (64 query heads
sharing one K/V head, d = 256, 64-token pages in a random page permutation).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ctx4k]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on the host

Prints one JSON line (rank 0).  `value` is achieved HBM throughput in TB/s:
algorithmic bytes (KV rows attended, queries, outputs, page-table entries and
the append traffic, each counted once) divided by device time, with every
input resident in HBM.  The timed region replays CUDA graphs of the steps.
To defeat the 135 MB L2, steps rotate over device-resident copies of the
cache, so a step never finds its cache in L2; with an append each copy grows
by one token per visit, and the mean attended length is reported.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_mfa_gb300 import accounting as acc  # noqa: E402
from decode_attention_mfa_gb300 import dist as mdist  # noqa: E402
from decode_attention_mfa_gb300 import workloads as wl  # noqa: E402

METRIC = "MFA decode-attn achieved HBM TB/s (% of peak) and decode steps/s at B×L"
UNIT = "TB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 135_528_448
COPY_MEM_BUDGET = 100e9
DRIFT = 0.03              # with an append, each cache copy grows by at most about this fraction of its length
MAX_HEADLINE_STEPS = 20000
MIN_GRAPH_STEPS = 32      # steps per captured graph (graph launches amortised over at least this many)
E2E_GROUP = 16            # end to end: steps per stream synchronisation (two sets of per-step buffers)
E2E_GRAPH_STEPS = 512     # end to end: steps per captured graph (its first group's inputs are copied in at its start)
EXTRA_WORKLOADS = ("long", "fp8", "ragged")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(wl.WORKLOADS) + ["qproj"], default="ctx4k",
                    help="a decode workload, or qproj: the low-rank query path at the Step-3 shape")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (debug runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--region-seconds", type=float, default=0.5,
                    help="device time the headline's repeated K-step regions add up to (median region reported)")
    ap.add_argument("--no-extra", action="store_true",
                    help="with the default workload, skip the extra workloads timed after the headline")
    ap.add_argument("--copies", type=int, default=0,
                    help="device-resident cache copies to rotate over (default: enough to defeat L2 "
                         "and keep the per-copy length growth near 1%%; small values suit ncu captures)")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (every 20 ms) while running."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="mfa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=open(self.path + ".err", "w"))
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
                except (ValueError, IndexError):
                    continue
            os.unlink(self.path)
        if not rows:
            err = ""
            if self.path and os.path.exists(self.path + ".err"):
                err = open(self.path + ".err").read().strip()[:200]
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"no nvidia-smi samples {err}".strip()],
                    "samples": 0}
        inside = [r for r in rows if t0 - 0.03 <= r[0] <= t1 + 0.03] or rows[-3:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ workload
def appends(w: wl.Workload) -> bool:
    """Whether a step of the workload appends one token per sequence first."""
    return w.append_tokens > 0


def arm_config(w: wl.Workload, world: int) -> dict:
    """The workload's identity, the same dict in both arms of the benchmark."""
    app = appends(w)
    blocks = w.select_blocks > 0
    return {"workload": w.name, "description": w.description, "batch": w.batch, "heads": wl.HEADS,
            "head_dim": wl.HEAD_DIM, "page_size": wl.PAGE_SIZE, "kv_dtype": w.kv_dtype,
            "queries_per_sequence": w.queries,
            "step": ("mfa_kv_append(1 token/seq) + " if app else "") +
                    (("mfa_decode_attention_blocks_fp8" if w.kv_dtype == "fp8" else "mfa_decode_attention_blocks")
                     if blocks else
                     ("mfa_decode_attention_mtp" + {"fp8": "_fp8", "fp4": "_fp4"}.get(w.kv_dtype, "")
                      + f" (n_query={w.queries})") if w.queries > 1 else
                     "mfa_decode_attention_fp4" if w.kv_dtype == "fp4" else
                     "mfa_decode_attention_fp8" if w.kv_dtype == "fp8" else "mfa_decode_attention") +
                    " (split + LSE combine)",
            "l2": "steps rotate over device-resident copies of the cache, together more than 3x the 135 MB L2, "
                  "so no step finds its cache in L2",
            "parallelism": f"dp{world} (independent batch per GPU)"}


def bench_lengths(w: wl.Workload) -> np.ndarray:
    """Cache lengths when the benchmark starts (the workload's own lengths)."""
    return wl.draw_lengths(w)


def first_attended(w: wl.Workload) -> np.ndarray:
    """Lengths the first step attends over."""
    return bench_lengths(w) + (1 if appends(w) else 0)


def choose_copies(w: wl.Workload, lens: np.ndarray, total_steps: int) -> int:
    kv_copy = float(lens.sum()) * acc.kv_bytes_per_token(w.kv_dtype)
    need_l2 = math.ceil(3 * L2_BYTES / kv_copy) + 1
    need_drift = math.ceil(total_steps / max(1.0, DRIFT * float(lens.mean()))) if appends(w) else 0
    cap = max(2, int(COPY_MEM_BUDGET // (2.2 * kv_copy)))
    return int(max(2, min(cap, max(need_l2, need_drift))))


def est_step_seconds(w: wl.Workload, lens) -> float:
    """Rough step time (algorithmic bytes at 5 TB/s), used only to size the timed regions."""
    L = np.asarray(lens, dtype=np.int64)
    if w.select_blocks:
        return max(5e-6, 1024.0 * (8 * w.select_blocks + 8) * L.size / 5e12)
    return max(5e-6, acc.decode_step_bytes(L, w.kv_dtype, appended_tokens=w.append_tokens, n_query=w.queries) / 5e12)


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_mfa_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("decode_split") or f.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, tokens_per_launch: float):
    """DRAM bytes per split-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source; scaled by tokens when the capture
    ran a smaller case."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    entry = d.get("workloads", {}).get(workload)
    if not entry or entry.get("source_sha") != kernel_source_sha():
        return None
    return float(entry["dram_bytes_per_token"]) * tokens_per_launch


def ncu_step_share(workload: str):
    """The split kernel's share of a step's device time in the committed ncu launch list of this workload
    (cold, serialised launches), if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path)).get("step_share", {}).get(workload)
    if not entry or entry.get("source_sha") != kernel_source_sha():
        return None
    return float(entry["split_share"])


def query_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_mfa_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("query_lowrank") or f.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def query_traffic():
    """DRAM bytes of one query-path call (both launches) from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "query_lowrank_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    return float(d["dram_bytes_per_call"]) if d.get("source_sha") == query_source_sha() else None


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local, workload=None, region_s=None, with_e2e=None):
    """One workload through the C ABI. The headline times K steps in each of several
    regions (about `region_s` seconds of them in all, so the clock sampler sees the load);
    its value is the median region."""
    import torch
    from decode_attention_mfa_gb300 import capi
    from decode_attention_mfa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[workload or args.workload]
    e2e_on = (not args.no_e2e) if with_e2e is None else with_e2e
    region_s = args.region_seconds if region_s is None else region_s
    lens0 = bench_lengths(w)
    B = int(lens0.size)
    est_step_s = est_step_seconds(w, lens0)
    n_reg = max(3, min(math.ceil(region_s / (args.steps * est_step_s)), max(3, MAX_HEADLINE_STEPS // args.steps)))
    total_steps = args.warmup + args.steps * (n_reg + (1 if e2e_on else 0)) + 2
    total_steps += max(2, min(args.steps, 512))  # the region that times the split kernel alone
    blocks = w.select_blocks > 0
    if blocks:  # block gather: the caller's selection, the same every step
        bidx_h, nblk_h = wl.draw_blocks(lens0, w.select_blocks, [w.seed + 1000 * rank])
    # L2 sizing by the rows a step reads (block gather: the selected ones)
    R = args.copies if args.copies > 0 else choose_copies(
        w, acc.blocks_attended(lens0, nblk_h) if blocks else lens0, total_steps)
    headroom = math.ceil(total_steps / R) + 2
    # inputs: seeded on the host, one copy moved to HBM, cloned R times there
    wr = wl.Workload(w.name, w.batch, w.lengths, w.kv_dtype, w.permute_pages, 0, w.seed + 1000 * rank,
                     queries=w.queries)
    nq = w.queries
    case = wl.make_case(wr, lengths=lens0, headroom_tokens=headroom)
    max_pages = case.page_table.shape[1]
    num_pages = case.num_pages
    page_table = torch.from_numpy(case.page_table).to(dev)
    fp8 = w.kv_dtype in ("fp8", "fp4")  # quantised cache with per-token scales (E4M3, or packed E2M1)
    fp4 = w.kv_dtype == "fp4"
    row_bytes = wl.HEAD_DIM // 2 if fp4 else wl.HEAD_DIM
    append_q = capi.mfa_kv_append_fp4 if fp4 else capi.mfa_kv_append_fp8
    decode_q = capi.mfa_decode_attention_fp4 if fp4 else capi.mfa_decode_attention_fp8
    mtp_q = capi.mfa_decode_attention_mtp_fp4 if fp4 else capi.mfa_decode_attention_mtp_fp8
    stream = torch.cuda.Stream(device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    ws_hint = int(acc.blocks_attended(lens0, nblk_h).max()) if blocks else int(lens0.max()) + headroom
    ws_bytes = (capi.mfa_decode_mtp_workspace_bytes(B, nq, ws_hint) if nq > 1
                else capi.mfa_decode_workspace_bytes(B, ws_hint))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    capi.mfa_workspace_init(workspace, ws_bytes)
    with torch.cuda.stream(stream):
        if fp8:
            k0 = torch.zeros((num_pages, wl.PAGE_SIZE, row_bytes), dtype=torch.uint8, device=dev)
            v0 = torch.zeros_like(k0)
            ks0 = torch.ones((num_pages, wl.PAGE_SIZE), dtype=torch.float32, device=dev)
            vs0 = torch.ones_like(ks0)
            sl_tmp = torch.zeros(B, dtype=torch.int32, device=dev)
            kr, vr = case.k_rows.to(dev), case.v_rows.to(dev)
            off = 0
            for b, n in enumerate(lens0):   # quantise on the device, one append per sequence
                n = int(n)
                append_q(kr[off:off + n], vr[off:off + n], n, k0, v0, ks0, vs0,
                                       page_table.data_ptr() + 4 * b * max_pages, sl_tmp.data_ptr() + 4 * b,
                                       1, max_pages, num_pages, workspace, stream)
                off += n
            del kr, vr
        else:
            k0 = wl.scatter_rows(case.k_rows, lens0, case.page_table, num_pages, fill=0.0).to(dev)
            v0 = wl.scatter_rows(case.v_rows, lens0, case.page_table, num_pages, fill=0.0).to(dev)
            ks0 = vs0 = None
        k_caches = [k0] + [k0.clone() for _ in range(R - 1)]
        v_caches = [v0] + [v0.clone() for _ in range(R - 1)]
        k_scales = [ks0] + [ks0.clone() for _ in range(R - 1)] if fp8 else [None] * R
        v_scales = [vs0] + [vs0.clone() for _ in range(R - 1)] if fp8 else [None] * R
        seq_lens = torch.from_numpy(np.tile(lens0.astype(np.int32), (R, 1))).to(dev)
        if nq > 1:  # [B, nq, 64, 256]: the step's query tokens
            q1 = wl.draw_rows(B * nq * wl.HEADS, wl.HEAD_DIM, [wr.seed, 90], 0).view(B, nq, wl.HEADS, wl.HEAD_DIM)
        else:
            q1 = case.q
        q = q1.to(dev).unsqueeze(0).repeat(R, *([1] * q1.dim())).contiguous()
        newkv = wl.draw_rows(2 * B, wl.HEAD_DIM, [w.seed, rank], 11).view(2, B, 1, wl.HEAD_DIM).to(dev)
        if blocks:
            block_idx = torch.from_numpy(bidx_h).to(dev)
            n_blocks = torch.from_numpy(nblk_h).to(dev)
        qshape = (B, nq) if nq > 1 else (B,)
        out_main = torch.empty(qshape + (wl.HEADS, wl.HEAD_DIM), dtype=torch.bfloat16, device=dev)
        lse_main = torch.empty(qshape + (wl.HEADS,), dtype=torch.float32, device=dev)
    stream.synchronize()
    del case
    host_len = np.tile(lens0.astype(np.int64), (R, 1))  # host mirror of every copy's length
    step_bytes, split_bytes = [], []

    app = appends(w)

    def step(r, qsrc=None, kvsrc=None, outs=None):
        kn = newkv[0] if kvsrc is None else kvsrc[0]
        vn = newkv[1] if kvsrc is None else kvsrc[1]
        qq = q[r] if qsrc is None else qsrc
        out, lse = (out_main, lse_main) if outs is None else outs
        sl = seq_lens[r]
        if fp8:
            if app:
                append_q(kn, vn, 1, k_caches[r], v_caches[r], k_scales[r], v_scales[r], page_table,
                                       sl, B, max_pages, num_pages, workspace, stream)
            if blocks:
                capi.mfa_decode_attention_blocks_fp8(qq, k_caches[r], v_caches[r], k_scales[r], v_scales[r],
                                                     page_table, sl, block_idx, n_blocks, block_idx.shape[1], out,
                                                     lse, wl.SCALE, B, max_pages, num_pages, ws_hint, workspace,
                                                     ws_bytes, stream)
            elif nq > 1:
                mtp_q(qq, k_caches[r], v_caches[r], k_scales[r], v_scales[r], page_table, sl, out, lse, wl.SCALE, B,
                      nq, max_pages, num_pages, ws_hint, workspace, ws_bytes, stream)
            else:
                decode_q(qq, k_caches[r], v_caches[r], k_scales[r], v_scales[r], page_table, sl,
                         out, lse, wl.SCALE, B, max_pages, num_pages, ws_hint, workspace, ws_bytes, stream)
        else:
            if app:
                capi.mfa_kv_append(kn, vn, 1, k_caches[r], v_caches[r], page_table, sl, B, max_pages, num_pages,
                                   workspace, stream)
            if blocks:
                capi.mfa_decode_attention_blocks(qq, k_caches[r], v_caches[r], page_table, sl, block_idx, n_blocks,
                                                 block_idx.shape[1], out, lse, wl.SCALE, B, max_pages, num_pages,
                                                 ws_hint, workspace, ws_bytes, stream)
            elif nq > 1:
                capi.mfa_decode_attention_mtp(qq, k_caches[r], v_caches[r], page_table, sl, out, lse, wl.SCALE, B,
                                              nq, max_pages, num_pages, ws_hint, workspace, ws_bytes, stream)
            else:
                capi.mfa_decode_attention(qq, k_caches[r], v_caches[r], page_table, sl, out, lse, wl.SCALE, B,
                                          max_pages, num_pages, ws_hint, workspace, ws_bytes, stream)

    def account(r):
        if app:
            host_len[r] += 1
        L = host_len[r].copy()
        if blocks:  # the split kernel reads everything but the outputs
            sb = acc.decode_blocks_step_bytes(L, nblk_h, w.kv_dtype)
            step_bytes.append(sb)
            split_bytes.append(sb - B * wl.HEADS * (wl.HEAD_DIM * 2 + 4))
            return acc.blocks_attended(L, nblk_h)
        step_bytes.append(acc.decode_step_bytes(L, w.kv_dtype, appended_tokens=1 if app else 0, n_query=nq))
        split_bytes.append(int(L.sum()) * acc.kv_bytes_per_token(w.kv_dtype) + nq * B * wl.HEADS * wl.HEAD_DIM * 2
                           + int(((L + 63) // 64).sum()) * 4 + B * 4)
        return L

    # warm-up (eager)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % R)
            account(i % R)
    stream.synchronize()
    capi.mfa_check_device_errors(workspace, clear=True, stream=stream)
    cursor = args.warmup

    def capture(indices, with_events, e2e_bufs=None):
        g = torch.cuda.CUDAGraph()
        evs = []
        if with_events:
            for _ in indices:
                pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                pair[0].record(stream); pair[1].record(stream)  # create the handles outside capture
                evs.append(pair)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for j, r in enumerate(indices):
                if with_events:
                    capi.mfa_profile_split_events(*evs[j])
                if e2e_bufs is None:
                    step(r)
            if e2e_bufs is not None:
                e2e_pipeline(indices, e2e_bufs)
            capi.mfa_profile_split_events(None, None)
        return g, evs

    def e2e_pipeline(indices, bufs):
        """Every step copies its own inputs in from pinned host memory and its result back out, on a copy
        stream. The copies are per step, but the streams synchronise once per group of E2E_GROUP steps: a
        wait on the copy stream in front of a step's first launch costs that launch its programmatic
        overlap with the previous step (4.2 us a step on the 4K configuration), so the compute stream
        waits for a whole group's inputs at once, and the copy stream waits for a whole group's results.
        Two sets of per-step device buffers: group g + 1's inputs go in while group g computes."""
        hq, hkv, hout, hlse, dq, dkv, dout, dlse = bufs
        cs = copy_stream
        n = len(indices)
        G = E2E_GROUP
        groups = [list(range(k, min(n, k + G))) for k in range(0, n, G)]
        ev_in = [torch.cuda.Event() for _ in groups]
        ev_done = [torch.cuda.Event() for _ in groups]
        cs.wait_stream(stream)

        def buf(j):  # group parity, then position in the group
            return ((j // G) % 2) * G + j % G

        def copy_in(gi):
            with torch.cuda.stream(cs):
                for j in groups[gi]:
                    dq[buf(j)].copy_(hq, non_blocking=True)
                    if app:
                        dkv[buf(j)].copy_(hkv, non_blocking=True)
                ev_in[gi].record(cs)

        for gi in range(min(2, len(groups))):
            copy_in(gi)
        for gi, members in enumerate(groups):
            stream.wait_event(ev_in[gi])
            for j in members:
                step(indices[j], qsrc=dq[buf(j)], kvsrc=dkv[buf(j)], outs=(dout[buf(j)], dlse[buf(j)]))
            ev_done[gi].record(stream)
            cs.wait_event(ev_done[gi])
            with torch.cuda.stream(cs):
                for j in members:
                    hout.copy_(dout[buf(j)], non_blocking=True)
                    hlse.copy_(dlse[buf(j)], non_blocking=True)
            if gi + 2 < len(groups):
                copy_in(gi + 2)  # after group gi's steps and their results left its buffer set
        stream.wait_stream(cs)

    def timed(n_steps, with_events, e2e_bufs=None, regions=1):
        """Times `regions` regions of n_steps steps each (the same captured graphs replayed); returns
        the device ms of every region, the split-launch event times (with_events), the lengths of the
        last R steps, the wall-clock span, and the algorithmic bytes of every region."""
        nonlocal cursor
        order = [(cursor + i) % R for i in range(n_steps)]
        # one graph holds at least MIN_GRAPH_STEPS steps (a whole number of passes over the R copies), so
        # that graph launches are amortised; end to end, at least 16, so the copy pipeline rarely drains
        grp = R * max(1, -(-(MIN_GRAPH_STEPS if e2e_bufs is None else E2E_GRAPH_STEPS) // R))
        if with_events:
            grp = R
        full = order[:grp] if n_steps >= grp else []
        reps = n_steps // grp if full else 0
        tail = order[reps * grp:]
        g_full, ev_full = capture(full, with_events, e2e_bufs) if full else (None, [])
        g_tail, ev_tail = capture(tail, with_events, e2e_bufs) if tail else (None, [])
        region_ms, region_bytes, lens_seen = [], [], []
        t_first = None
        for _ in range(regions):
            # the captures did not run: lengths are unchanged; account in execution order
            n0 = len(step_bytes)
            lens_seen = [account(r) for r in order]
            region_bytes.append(float(sum(step_bytes[n0:])))
            torch.cuda.synchronize()
            mdist.barrier()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.time()
            t_first = t0 if t_first is None else t_first
            with torch.cuda.stream(stream):  # replay() launches on the current stream
                e0.record(stream)
                for _ in range(reps):
                    g_full.replay()
                if g_tail is not None:
                    g_tail.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            t1 = time.time()
            mdist.barrier()
            cursor += n_steps
            region_ms.append(e0.elapsed_time(e1))
        evs = ev_full if ev_full else ev_tail
        split_ms = [a.elapsed_time(b) for a, b in evs]
        last_lens = lens_seen[(reps - 1) * grp:(reps - 1) * grp + R] if reps else lens_seen[-len(tail):]
        return region_ms, split_ms, last_lens, (t_first, t1), region_bytes

    clocks = ClockSampler(local)
    clocks.start()
    # headline: n_reg regions of K steps, no events in the graphs (an event node between the
    # kernels of a step would break their programmatic overlap)
    reg_ms, _, last_lens, (t0, t1), reg_bytes = timed(args.steps, with_events=False, regions=n_reg)
    time.sleep(0.15)
    clocks.stop()
    clk = clocks.summary(t0, t1)
    capi.mfa_check_device_errors(workspace, clear=True, stream=stream)
    mean_len = float(np.mean([float(np.mean(L)) for L in last_lens]))
    # split-kernel device time: the same steps again, with an event pair
    # recorded around every split launch on its stream
    n_ev = max(2, min(args.steps, 512))
    n_before = len(split_bytes)
    _, split_ms, _, _, _ = timed(n_ev, with_events=True)
    split_bytes_last = split_bytes[n_before:][-len(split_ms):]
    capi.mfa_check_device_errors(workspace, clear=True, stream=stream)

    tot_b, max_s = mdist.aggregate_many(reg_bytes, [m / 1e3 for m in reg_ms])
    reg_val = [b / t / 1e12 for b, t in zip(tot_b, max_s)]
    med = int(np.argsort(reg_val)[len(reg_val) // 2])  # the median region
    value = reg_val[med]
    max_s = max_s[med]
    peak_gbs, peak_kind = measured_peaks()
    avg_split_s = float(np.mean(split_ms)) / 1e3 if split_ms else float("nan")
    achieved = float(np.mean(split_bytes_last)) / avg_split_s / 1e9 if split_ms else None
    tokens_per_launch = float(np.mean([float(np.sum(L)) for L in last_lens]))
    share = ncu_step_share(w.name)
    in_step = None
    if share is not None and split_ms:
        us = share * max_s * 1e6 / args.steps
        ach = float(np.mean(split_bytes_last)) / (us * 1e-6) / 1e9
        in_step = {"share_of_step": share, "us": us, "achieved": ach, "frac": ach / peak_gbs,
                   "how": "the split kernel's share of the step's device time in the committed ncu launch list "
                          "(profiles/), times this run's step time: the kernel as it runs inside the step, "
                          "overlapped with its neighbours"}

    e2e = None
    if e2e_on:
        hq = torch.empty(q[0].shape, dtype=torch.bfloat16).pin_memory()
        hq.copy_(q[0].cpu())
        hkv = torch.empty((2, B, 1, wl.HEAD_DIM), dtype=torch.bfloat16).pin_memory()
        hkv.copy_(newkv.cpu())
        hout = torch.empty(out_main.shape, dtype=torch.bfloat16).pin_memory()
        hlse = torch.empty(lse_main.shape, dtype=torch.float32).pin_memory()
        dq = [torch.empty_like(q[0]) for _ in range(2 * E2E_GROUP)]
        dkv = [torch.empty_like(newkv) for _ in range(2 * E2E_GROUP)]
        dout = [torch.empty_like(out_main) for _ in range(2 * E2E_GROUP)]
        dlse = [torch.empty_like(lse_main) for _ in range(2 * E2E_GROUP)]
        n_before = len(step_bytes)
        e_ms, _, _, _, e_reg_b = timed(args.steps, with_events=False,
                                       e2e_bufs=(hq, hkv, hout, hlse, dq, dkv, dout, dlse))
        e_bytes, e_s = mdist.aggregate(e_reg_b[0], e_ms[0] / 1e3)
        capi.mfa_check_device_errors(workspace, clear=True, stream=stream)
        e2e = {"value": e_bytes / e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(hq.numel() * 2 + (hkv.numel() * 2 if app else 0)),
               "d2h_bytes_per_step": int(hout.numel() * 2 + hlse.numel() * 4),
               "ms_per_step": e_ms[0] / args.steps,
               "how": f"CUDA graphs of {E2E_GRAPH_STEPS} C-ABI calls; each step's inputs copied in from pinned host "
                      f"memory and its result copied back, on a copy stream that overlaps the computing steps; the "
                      f"streams synchronise once per group of {E2E_GROUP} steps (two sets of per-step buffers)"}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1" if fp4 else "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), bf16)",
        "config": arm_config(w, world),
        "mean_attended_len": mean_len,
        "cache_copies": R,
        "regions": {"count": len(reg_val), "steps_each": args.steps, "value_of_each": "median reported",
                    "min": min(reg_val), "max": max(reg_val)},
        "steps_per_s": args.steps * world / max_s,
        "decoded_tokens_per_s": args.steps * world * B * nq / max_s,
        "pct_of_measured_peak": 100.0 * value * 1e3 / peak_gbs,
        "pct_of_8TBps": 100.0 * value * 1e3 / NOMINAL_HBM_GBS,
        "gpu_launches": (3 if app else 2) * args.steps,
        "clocks": clk,
        "roofline": {"bound": "hbm", "kernel": "decode split (mfa_decode_attention)",
                     "achieved": achieved, "peak": peak_gbs, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": (achieved / peak_gbs) if achieved else None,
                     "traffic": ncu_traffic(w.name, tokens_per_launch),
                     "algorithmic_bytes_per_launch": float(np.mean(split_bytes_last)) if split_ms else None,
                     "avg_launch_us": avg_split_s * 1e6, "launches_averaged": len(split_ms),
                     "how": "CUDA events around each split launch on its stream, in a timed region of "
                            "the same steps run right after the headline region; the events keep the split "
                            "kernel from overlapping its neighbours (programmatic dependent launch), so this is "
                            "the kernel's stand-alone duration, which can exceed the overlapped step time",
                     "in_step": in_step},
        "e2e": e2e,
    }
    return result, lens0


def extra_workloads(args, rank, world, local) -> dict:
    """After the headline, the other full-size configurations timed the same way (no
    end-to-end leg, no CPU baseline): step time, throughput, split-kernel time, clocks."""
    import torch
    out = {}
    for name in EXTRA_WORKLOADS:
        r, _ = run_ours(args, rank, world, local, workload=name, region_s=min(args.region_seconds, 0.2),
                        with_e2e=False)
        rf = r["roofline"]
        out[name] = {"description": r["config"]["description"], "value": r["value"], "unit": r["unit"],
                     "ms_per_step": r["ms_per_step"], "steps_per_s": r["steps_per_s"],
                     "pct_of_measured_peak": r["pct_of_measured_peak"], "pct_of_8TBps": r["pct_of_8TBps"],
                     "mean_attended_len": r["mean_attended_len"], "regions": r["regions"],
                     "split_kernel": {"avg_launch_us": rf["avg_launch_us"], "achieved_gbs": rf["achieved"],
                                      "frac": rf["frac"], "traffic": rf["traffic"]},
                     "clocks": r["clocks"], "dtype": r["dtype"]}
        del r
        gc.collect()
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle
class OracleSampler:
    """The fp64 CPU oracle on a bounded sample of (sequence, head) rows of one
    step of the workload; inputs are drawn once and kept on the host."""

    def __init__(self, w: wl.Workload, lens_attended, threads: int):
        import oracle

        oracle.build()
        self.oracle = oracle
        self.w = w
        self.threads = threads
        case = wl.make_case(w, lengths=lens_attended, headroom_tokens=0)
        if w.kv_dtype in ("fp8", "fp4"):
            quant = oracle.quantize_tokens_e2m1 if w.kv_dtype == "fp4" else oracle.quantize_tokens_e4m3
            width = wl.HEAD_DIM // 2 if w.kv_dtype == "fp4" else wl.HEAD_DIM
            kc_, ks_ = quant(wl.bits(case.k_rows))
            vc_, vs_ = quant(wl.bits(case.v_rows))
            slots = wl.slots_of(case.lengths0, case.page_table)
            n = case.num_pages * wl.PAGE_SIZE
            kc = np.zeros((n, width), np.uint8); kc[slots] = kc_
            vc = np.zeros((n, width), np.uint8); vc[slots] = vc_
            ks = np.ones(n, np.float32); ks[slots] = ks_
            vs = np.ones(n, np.float32); vs[slots] = vs_
            self.kc, self.vc = kc.reshape(-1, wl.PAGE_SIZE, width), vc.reshape(-1, wl.PAGE_SIZE, width)
            self.ks, self.vs = ks.reshape(-1, wl.PAGE_SIZE), vs.reshape(-1, wl.PAGE_SIZE)
        else:
            self.kc = wl.bits(wl.scatter_rows(case.k_rows, case.lengths0, case.page_table, case.num_pages, fill=0.0))
            self.vc = wl.bits(wl.scatter_rows(case.v_rows, case.lengths0, case.page_table, case.num_pages, fill=0.0))
            self.ks = self.vs = None
        nq = w.queries
        self.step_bytes = acc.decode_step_bytes(case.lengths0, w.kv_dtype, appended_tokens=w.append_tokens,
                                                n_query=nq)
        if nq > 1:  # token t of sequence b: a single-token decode over its first L - nq + 1 + t positions
            q = wl.draw_rows(case.batch * nq * wl.HEADS, wl.HEAD_DIM, [w.seed, 90], 0)
            self.q = wl.bits(q.view(case.batch * nq, wl.HEADS, wl.HEAD_DIM))
            self.page_table = np.repeat(case.page_table, nq, axis=0)
            L = case.lengths0.astype(np.int64)
            self.sl = np.maximum(L[:, None] - nq + 1 + np.arange(nq)[None, :], 0).astype(np.int32).reshape(-1)
        else:
            self.q = wl.bits(case.q)
            self.page_table = case.page_table
            self.sl = case.lengths0.astype(np.int32)
        self.total_rows = self.sl.size * wl.HEADS
        self.order = np.random.default_rng(0).permutation(self.total_rows)

    def run(self, nrows: int) -> float:
        rows = self.order[:nrows]
        t = time.perf_counter()
        self.oracle.mfa_decode(self.q, self.kc, self.vc, self.page_table, self.sl, wl.SCALE, k_scale=self.ks,
                               v_scale=self.vs, rows=(rows // wl.HEADS, rows % wl.HEADS), threads=self.threads)
        return time.perf_counter() - t

    def rows_for(self, budget_s: float) -> int:
        probe = min(self.total_rows, max(self.threads, 8))
        dt = self.run(probe)
        return int(min(self.total_rows, max(probe, probe * budget_s / max(dt, 1e-6))))

    def bytes_of(self, nrows: int) -> float:
        return self.step_bytes * nrows / self.total_rows


class BlockOracleSampler:
    """The fp64 oracle of block-gather decode (gather of the selected rows, then
    the fp64 decode) on the first n sequences of the workload, all heads; the
    inputs of the largest sample are drawn once."""

    def __init__(self, w: wl.Workload, lens, threads: int):
        import oracle

        oracle.build()
        self.oracle = oracle
        self.w = w
        self.threads = threads
        self.lens = np.asarray(lens, dtype=np.int64)
        self.bi, self.nb = wl.draw_blocks(self.lens, w.select_blocks, [w.seed])
        self.total_rows = int(self.lens.size)  # sequences
        self.inputs = None

    def _prepare(self, n):
        if self.inputs is None or self.inputs[0] < n:
            case = wl.make_case(self.w, lengths=self.lens[:n], headroom_tokens=0)
            ks = vs = None
            if self.w.kv_dtype == "fp8":  # the oracle's own per-token E4M3 quantiser
                kcodes, kscale = self.oracle.quantize_tokens_e4m3(wl.bits(case.k_rows))
                vcodes, vscale = self.oracle.quantize_tokens_e4m3(wl.bits(case.v_rows))
                slots = wl.slots_of(case.lengths0, case.page_table)
                rows = case.num_pages * wl.PAGE_SIZE
                kc = np.zeros((rows, wl.HEAD_DIM), np.uint8); kc[slots] = kcodes
                vc = np.zeros((rows, wl.HEAD_DIM), np.uint8); vc[slots] = vcodes
                ks = np.ones(rows, np.float32); ks[slots] = kscale
                vs = np.ones(rows, np.float32); vs[slots] = vscale
                shape = (case.num_pages, wl.PAGE_SIZE)
                kc, vc, ks, vs = kc.reshape(shape + (-1,)), vc.reshape(shape + (-1,)), ks.reshape(shape), vs.reshape(shape)
            else:
                kc = wl.bits(wl.scatter_rows(case.k_rows, case.lengths0, case.page_table, case.num_pages, fill=0.0))
                vc = wl.bits(wl.scatter_rows(case.v_rows, case.lengths0, case.page_table, case.num_pages, fill=0.0))
            self.inputs = (n, wl.bits(case.q), kc, vc, ks, vs, case.page_table)
        return self.inputs

    def run(self, n: int) -> float:
        _, q, kc, vc, ks, vs, pt = self._prepare(n)
        t = time.perf_counter()
        self.oracle.mfa_decode_blocks(q[:n], kc, vc, pt[:n], self.lens[:n].astype(np.int32), self.bi[:n],
                                      self.nb[:n], wl.SCALE, k_scale=ks, v_scale=vs, threads=self.threads)
        return time.perf_counter() - t

    def rows_for(self, budget_s: float) -> int:
        dt = self.run(1)
        return int(min(self.total_rows, max(1, budget_s / max(dt, 1e-6))))

    def bytes_of(self, n: int) -> float:
        return float(acc.decode_blocks_step_bytes(self.lens[:n], self.nb[:n], self.w.kv_dtype))


def make_sampler(w: wl.Workload, lens, threads):
    return BlockOracleSampler(w, lens, threads) if w.select_blocks else OracleSampler(w, lens, threads)


def sample_unit(w: wl.Workload) -> str:
    return "sequences (all 64 heads)" if w.select_blocks else "(sequence, head) rows"


def cpu_baseline(w: wl.Workload, lens_attended, budget_s=12.0):
    threads = len(os.sched_getaffinity(0))
    sampler = make_sampler(w, lens_attended, threads)
    rows = sampler.rows_for(budget_s)
    dt = sampler.run(rows)
    return {"value": sampler.bytes_of(rows) / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {sampler.total_rows} {sample_unit(w)} of one {w.name} step "
                      f"(fp64 C oracle, {threads} OpenMP threads, {dt:.2f} s)"}


def run_reference(args):
    rank, world, _ = mdist.env_rank()
    if rank != 0:
        return None
    if args.workload == "qproj":  # the fp64 oracle of the query path on a bounded sample of rows
        import torch
        g = torch.Generator().manual_seed(1234)
        B, Dm, R_, N = QPROJ["batch"], QPROJ["d_model"], QPROJ["rank"], QPROJ["n_out"]
        x = torch.randn(B, Dm, generator=g).to(torch.bfloat16)
        w_down = (torch.randn(Dm, R_, generator=g) / Dm ** 0.5).to(torch.bfloat16)
        gamma = (1.0 + 0.1 * torch.randn(R_, generator=g)).to(torch.bfloat16)
        w_up = (torch.randn(R_, N, generator=g) / R_ ** 0.5).to(torch.bfloat16)
        cb = qproj_cpu_baseline(x, w_down, gamma, w_up, budget_s=max(0.05, 150.0 / max(1, args.steps + args.warmup)))
        return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
                "config": {"workload": "qproj", "batch": B, "d_model": Dm, "rank": R_, "n_out": N},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
    w = wl.WORKLOADS[args.workload]
    lens = first_attended(w)   # lengths attended in the first step of our arm
    threads = len(os.sched_getaffinity(0))
    sampler = make_sampler(w, lens, threads)
    rows = sampler.rows_for(max(0.05, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sampler.run(rows)
    secs = sum(sampler.run(rows) for _ in range(args.steps))
    value = sampler.bytes_of(rows) * args.steps / secs / 1e12
    sample = (f"{rows} of {sampler.total_rows} {sample_unit(w)} per step of {w.name} "
              f"(fp64 C oracle, {threads} OpenMP threads)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1), bf16)",
            "config": arm_config(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ query path
QPROJ = {"batch": 32, "d_model": 7168, "rank": 2048, "n_out": 64 * 256, "eps": 1e-6}


def qproj_bytes(B, d_model, rank, n_out):
    """Algorithmic bytes of one query-path call: both weights and the gain once,
    x read, q written (the fp32/bf16 scratch rows are not counted)."""
    return 2 * (d_model * rank + rank * n_out + rank + B * d_model + B * n_out)


def run_qproj(args, rank_id, world, local):
    import torch
    from decode_attention_mfa_gb300 import capi
    from decode_attention_mfa_gb300.build import build

    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, Dm, R_, N = QPROJ["batch"], QPROJ["d_model"], QPROJ["rank"], QPROJ["n_out"]
    g = torch.Generator(device=dev).manual_seed(1234 + rank_id)
    copies = args.copies if args.copies > 0 else 3  # 3 x 96 MB of weights >> the 135 MB L2
    w_down = [(torch.randn(Dm, R_, device=dev, generator=g) / Dm ** 0.5).to(torch.bfloat16) for _ in range(copies)]
    w_up = [(torch.randn(R_, N, device=dev, generator=g) / R_ ** 0.5).to(torch.bfloat16) for _ in range(copies)]
    gamma = (1.0 + 0.1 * torch.randn(R_, device=dev, generator=g)).to(torch.bfloat16)
    x = torch.randn(B, Dm, device=dev, generator=g).to(torch.bfloat16)
    q = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    ws_bytes = capi.mfa_query_lowrank_workspace_bytes(B, R_, N)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    capi.mfa_workspace_init(ws, ws_bytes)
    stream = torch.cuda.Stream(device=dev)

    copy_stream = torch.cuda.Stream(device=dev)

    def call(i, xs=None, qs=None):
        capi.mfa_query_lowrank(x if xs is None else xs, w_down[i], gamma, w_up[i], q if qs is None else qs, B, Dm, R_,
                               N, QPROJ["eps"], ws, ws_bytes, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i % copies)
    stream.synchronize()
    capi.mfa_check_device_errors(ws, clear=True, stream=stream)

    def pipeline(calls, bufs):
        """Every call copies its x in from pinned host memory and its q back, on a copy stream that overlaps
        the computing calls; the streams synchronise once per group of E2E_GROUP calls, as in the decode
        pipeline (a wait in front of a call's first launch costs it the overlap with the previous call)."""
        hx, hq, dx, dq = bufs
        G = E2E_GROUP
        groups = [list(range(k, min(len(calls), k + G))) for k in range(0, len(calls), G)]
        ev_in = [torch.cuda.Event() for _ in groups]
        ev_done = [torch.cuda.Event() for _ in groups]
        copy_stream.wait_stream(stream)

        def buf(j):
            return ((j // G) % 2) * G + j % G

        def copy_in(gi):
            with torch.cuda.stream(copy_stream):
                for j in groups[gi]:
                    dx[buf(j)].copy_(hx, non_blocking=True)
                ev_in[gi].record(copy_stream)

        for gi in range(min(2, len(groups))):
            copy_in(gi)
        for gi, members in enumerate(groups):
            stream.wait_event(ev_in[gi])
            for j in members:
                call(calls[j], dx[buf(j)], dq[buf(j)])
            ev_done[gi].record(stream)
            copy_stream.wait_event(ev_done[gi])
            with torch.cuda.stream(copy_stream):
                for j in members:
                    hq.copy_(dq[buf(j)], non_blocking=True)
            if gi + 2 < len(groups):
                copy_in(gi + 2)
        stream.wait_stream(copy_stream)

    def timed(n, e2e=None):
        gr = torch.cuda.CUDAGraph()
        stream.synchronize()
        # a whole number of passes over the weight copies, at least MIN_GRAPH_STEPS calls (end to end:
        # E2E_GRAPH_STEPS), so that graph launches are amortised
        grp = copies * max(1, -(-(MIN_GRAPH_STEPS if e2e is None else E2E_GRAPH_STEPS) // copies))
        with torch.cuda.graph(gr, stream=stream):
            if e2e is None:
                for j in range(grp):
                    call(j % copies)
            else:
                pipeline([j % copies for j in range(grp)], e2e)
        reps = max(1, n // grp)
        torch.cuda.synchronize()
        mdist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        mdist.barrier()
        return e0.elapsed_time(e1), reps * grp, (t0, t1)

    clocks = ClockSampler(local)
    clocks.start()
    ms, n, (t0, t1) = timed(args.steps)
    time.sleep(0.15)
    clocks.stop()
    clk = clocks.summary(t0, t1)
    # per-call device time: an event pair around each call, issued eagerly (the
    # host enqueues far ahead of the GPU, so the stream never waits on it)
    n_ev = min(args.steps, 64)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            call(i % copies)
            b.record(stream)
    torch.cuda.synchronize()
    per_call = [a.elapsed_time(b) for a, b in evs]
    capi.mfa_check_device_errors(ws, clear=True, stream=stream)
    step_bytes = qproj_bytes(B, Dm, R_, N)
    total_bytes, max_s = mdist.aggregate(float(step_bytes) * n, ms / 1e3)
    value = total_bytes / max_s / 1e12
    peak_gbs, peak_kind = measured_peaks()
    avg_us = float(np.mean(per_call)) * 1e3
    achieved = step_bytes / (avg_us * 1e-6) / 1e9
    e2e = None
    if not args.no_e2e:
        hx = torch.empty(x.shape, dtype=torch.bfloat16).pin_memory()
        hx.copy_(x.cpu())
        hq = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        dx = [torch.empty_like(x) for _ in range(2 * E2E_GROUP)]
        dq = [torch.empty_like(q) for _ in range(2 * E2E_GROUP)]
        e_ms, e_n, _ = timed(args.steps, (hx, hq, dx, dq))
        e_bytes, e_s = mdist.aggregate(float(step_bytes) * e_n, e_ms / 1e3)
        e2e = {"value": e_bytes / e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(hx.numel() * 2),
               "d2h_bytes_per_step": int(hq.numel() * 2), "ms_per_step": e_ms / e_n,
               "how": f"CUDA graphs of {E2E_GRAPH_STEPS} C-ABI calls; each call's x copied in from pinned host "
                      f"memory and its q copied back, on a copy stream that overlaps the computing calls; the streams "
                      f"synchronise once per group of {E2E_GROUP} calls (two sets of per-call buffers)"}
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": max_s * 1e3 / n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights, bf16)",
        "config": {"workload": "qproj", "description": "low-rank query path, Step-3 shape: x[32][7168] W_down[7168][2048] "
                   "-> RMSNorm -> W_up[2048][16384]", "batch": B, "d_model": Dm, "rank": R_, "n_out": N,
                   "step": "mfa_query_lowrank (two tensor-core GEMM launches + RMSNorm in their epilogues)",
                   "l2": f"weights rotate over {copies} device-resident copies "
                         f"({copies * 2 * (Dm * R_ + R_ * N) / 1e9:.2f} GB >> 135 MB L2)",
                   "parallelism": f"dp{world} (independent batch per GPU)"},
        "steps_per_s": n * world / max_s,
        "pct_of_measured_peak": 100.0 * value * 1e3 / peak_gbs,
        "gpu_launches": 2 * n,
        "clocks": clk,
        "roofline": {"bound": "hbm", "kernel": "query path (down GEMM, then up GEMM with the RMSNorm scale)",
                     "achieved": achieved, "peak": peak_gbs, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak_gbs, "traffic": query_traffic(), "algorithmic_bytes_per_launch": float(step_bytes), "avg_launch_us": avg_us,
                     "launches_averaged": len(per_call),
                     "how": "CUDA events around each call on its stream, eager calls after the headline region"},
        "e2e": e2e,
    }
    if rank_id == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = qproj_cpu_baseline(x.cpu(), w_down[0].cpu(), gamma.cpu(), w_up[0].cpu())
    return result


def qproj_cpu_baseline(x, w_down, gamma, w_up, budget_s=10.0):
    import oracle
    threads = len(os.sched_getaffinity(0))
    B = x.shape[0]
    bx, bd, bg, bu = wl.bits(x), wl.bits(w_down), wl.bits(gamma), wl.bits(w_up)
    t = time.perf_counter()
    oracle.query_lowrank(bx[:1], bd, bg, bu, QPROJ["eps"])
    one = time.perf_counter() - t
    rows = int(max(1, min(B, budget_s / max(one, 1e-6))))
    t = time.perf_counter()
    oracle.query_lowrank(bx[:rows], bd, bg, bu, QPROJ["eps"])
    dt = time.perf_counter() - t
    step_bytes = qproj_bytes(B, *w_down.shape, w_up.shape[1])
    return {"value": step_bytes * rows / B / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {B} rows of one query-path call (fp64 numpy oracle, {dt:.2f} s), bytes scaled "
                      "by the rows"}


def main():
    args = parse_args()
    if args.workload == "qproj" and args.impl == "ours":
        rank, world, local = mdist.init()
        res = run_qproj(args, rank, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        mdist.finalize()
        return
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, local = mdist.init()
    res, lens0 = run_ours(args, rank, world, local)
    if args.workload == "ctx4k" and not args.no_extra:
        res["workloads"] = extra_workloads(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl.WORKLOADS[args.workload], first_attended(wl.WORKLOADS[args.workload]))
        print(json.dumps(res), flush=True)
    mdist.finalize()


if __name__ == "__main__":
    main()
