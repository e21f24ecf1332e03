#!/usr/bin/env python3
"""Benchmark of the fused KDA RecoverSSM replay + verify step on GB300.

One step = one kda_replay_verify launch over the large-batch workload
(H=64 heads, B=512 requests, Q=8 verified tokens each, FP32 state pool of
1024 slots, pending ~ U{0..8}, 5% padding rows) with every input resident
in HBM.  Prints one JSON line (rank 0):

  value       verify tokens/s (live requests x Q per step / time), summed
              over ranks (replicas: each GPU runs its own copy)
  roofline    algorithmic bytes of one launch / its CUDA-event duration,
              against the measured HBM copy bandwidth
  e2e         the same metric through the C ABI with the step's inputs in
              pinned host memory: per step the activations and request
              metadata are copied in and the outputs copied out
  cpu_baseline the FP64 oracle on a bounded sample of the same items, over
              every host core (one worker process per core, forked before
              any CUDA call), with the one-core figure beside it

`--impl reference` times the oracle alone (every host core, a bounded sample
of items per step) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import os

# each oracle worker runs on exactly one core
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "replay-verify-f32-h64-b512-q8"
METRIC = "fused replay+verify tokens/s and state HBM GB/s (% of GB300 peak), 1 GPU"
DIM = 128


# ---------------------------------------------------------------------------
# algorithmic traffic of one step (bytes that must cross HBM at least once)
# ---------------------------------------------------------------------------

def algorithmic_bytes(case):
    """Bytes one replay + verify launch must move, from the workload itself.

    Per live item (request b with a live slot, head h): the 64 KB FP32 state
    page read; written back iff n > 0; n recorded corrections (512 B each)
    and key/gate records (512 B each) read; this window's q, k, v, raw_g
    (4 x Q x 256 B) and raw_beta (2 B per token) read; the outputs (Q x 256 B)
    written; with a record row, Q corrections and Q key/gate records
    (512 + 512 B per token) written.  Per inert item: its outputs (zeros)
    written.  Plus the per-request indices and the per-head gate
    parameters, read once.  With windows of different lengths (``q_lens``)
    each request's q_b replaces Q.
    """
    B, H, Q, RQ = case["B"], case["H"], case["Q"], case["RQ"]
    slots, rows, pending = case["state_slots"], case["record_rows"], case["pending"]
    q_lens = case.get("q_lens")
    page = DIM * DIM * 4
    total = 0
    state = 0
    live_items = 0
    for b in range(B):
        Q = int(q_lens[b]) if q_lens is not None else case["Q"]
        if slots[b] <= case["null_slot"]:
            total += H * Q * DIM * 2
            continue
        rec = rows[b]
        n = min(max(int(pending[rec]), 0), RQ) if rec >= 0 else 0
        per = page + (page if n > 0 else 0)
        state += H * per
        per += n * (DIM * 4 + 2 * DIM * 2)
        per += 4 * Q * DIM * 2 + Q * 2 + Q * DIM * 2
        if rec >= 0:
            per += Q * (DIM * 4 + 2 * DIM * 2)
        total += H * per
        live_items += H
    total += B * 4 * 2 + len(pending) * 0 + H * (4 + DIM * 4)
    if q_lens is not None:
        total += (B + 1) * 4
        live_tokens = int(q_lens[slots > case["null_slot"]].sum())
    else:
        live_tokens = int((slots > case["null_slot"]).sum()) * case["Q"]
    return dict(total=total, state=state, live_items=live_items, live_tokens=live_tokens)


# ---------------------------------------------------------------------------
# DRAM traffic measured by ncu for the step kernel (reported only while the
# kernel sources are the ones it was measured on)
# ---------------------------------------------------------------------------

PROFILED = {
    # one kda_step_ws launch of the profiling workload, scaled by live items
    "step": dict(
        sources=("kda_step_ws.cuh", "kda_step.cuh", "kda_device.cuh", "kda_step_launch.cuh",
                 "kda_step_q8.cu"),
        sha256="620c2da2457db0fec740a53211ff563ccb89fcdc57b68328b2aee8a9961c19eb",
        workload=WORKLOAD,
        bytes_per_launch=(608.2 + 464.5) * 1e6 * 31104 / 7808,
        how="dram__bytes_read.sum + dram__bytes_write.sum of one kda_step_ws launch on "
            "replay-verify-f32-h64-b128-q8 (608.2 + 464.5 MB, 7808 live items), scaled by "
            "live items to this workload's 31104"),
    # one kda_commit_ws launch of the standalone-commit workload itself
    "commit": dict(
        sources=("kda_commit.cu", "kda_device.cuh"),
        sha256="70b1471b3c91c16867767ed36da7dd9315f40df30e911fd48f86ac5d8891f448",
        workload="commit-bf16-l4-h32-b64-q4-align",
        bytes_per_launch=(194.8 + 167.1) * 1e6,
        how="dram__bytes_read.sum + dram__bytes_write.sum of one kda_commit_ws launch of "
            "this workload"),
}


def sources_digest(names):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_speculative_recoverssm_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(row, workload):
    """ncu DRAM bytes per launch of a row's kernel, or None when the workload
    differs or the kernel sources changed since they were measured."""
    e = PROFILED[row]
    if workload != e["workload"] or sources_digest(e["sources"]) != e["sha256"]:
        return None
    return e["bytes_per_launch"]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the oracle (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_rate(case, seconds, seed=0):
    """Times the FP64 oracle on a bounded random sample of live items; returns
    (tokens/s equivalent of a whole step, items timed, seconds)."""
    from oracle import kda_oracle as ko
    B, H, Q = case["B"], case["H"], case["Q"]
    live = np.flatnonzero(case["state_slots"] > case["null_slot"])
    all_items = (live[:, None] * H + np.arange(H)[None, :]).ravel()
    rng = np.random.default_rng(seed)
    order = rng.permutation(all_items)
    state = case["state"]
    corr, kg = case["corr"].copy(), case["key_gate"].copy()
    out = np.zeros((0,), dtype=np.uint16)
    done = 0
    t0 = time.perf_counter()
    chunk = 16
    while done < len(order):
        items = order[done:done + chunk]
        saved = {}
        for i in items:
            b, h = divmod(int(i), H)
            s = int(case["state_slots"][b])
            saved[(s, h)] = state[s, h].copy()
        out = np.zeros(case["v"].shape, dtype=np.uint16) if out.size == 0 else out
        ko.replay_verify(q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"],
                         raw_beta=case["raw_beta"], A_log=case["A_log"],
                         dt_bias=case["dt_bias"], lower_bound=case["lower_bound"],
                         q_scale=case["q_scale"], state=state, state_slots=case["state_slots"],
                         record_rows=case["record_rows"], corr=corr, key_gate=kg, out=out,
                         B=B, H=H, Q=Q, pending=case["pending"], items=items)
        for (s, h), page in saved.items():  # leave the host pool as it was
            state[s, h] = page
        done += len(items)
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    live_tokens = len(live) * Q
    step_equiv = dt * len(all_items) / done
    return live_tokens / step_equiv, done, dt


# ---------------------------------------------------------------------------
# the oracle over every host core: worker processes forked before any CUDA
# call, each running the unchanged oracle on its own share of the items; the
# workload's arrays are inherited copy-on-write, and each worker restores the
# pages it replays into, so every timed sample starts from the same state
# ---------------------------------------------------------------------------

_POOL_CASE = None


def _oracle_share(task):
    """One worker: the oracle on its items, 16 at a time, until the deadline
    (a time.time() value); returns (items done, seconds busy)."""
    from oracle import kda_oracle as ko
    items, deadline = task
    case = _POOL_CASE
    H = case["H"]
    state, corr, kg = case["state"], case["corr"], case["key_gate"]
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    done = 0
    t0 = time.perf_counter()
    while done < len(items) and time.time() < deadline:
        chunk = items[done:done + 16]
        saved = {}
        for i in chunk:
            b, h = divmod(int(i), H)
            s = int(case["state_slots"][b])
            saved[(s, h)] = state[s, h].copy()
        ko.replay_verify(q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"],
                         raw_beta=case["raw_beta"], A_log=case["A_log"],
                         dt_bias=case["dt_bias"], lower_bound=case["lower_bound"],
                         q_scale=case["q_scale"], state=state, state_slots=case["state_slots"],
                         record_rows=case["record_rows"], corr=corr, key_gate=kg, out=out,
                         B=case["B"], H=H, Q=case["Q"], pending=case["pending"], items=chunk)
        for (s, h), page in saved.items():
            state[s, h] = page
        done += len(chunk)
    return done, time.perf_counter() - t0


class OraclePool:
    """A pool of oracle workers, one per host core, forked from a process
    that has not touched CUDA (a pool forked after the first GPU call can
    hang).  The records the oracle writes land in each worker's own copy."""

    def __init__(self, case, workers=None):
        import multiprocessing as mp
        global _POOL_CASE
        _POOL_CASE = case
        self.case = case
        self.workers = workers or os.cpu_count() or 1
        self.pool = mp.get_context("fork").Pool(self.workers)

    def rate(self, seconds, seed=0):
        """(tokens/s equivalent of a whole step, items done, wall seconds)
        of the oracle on every worker for about `seconds`."""
        case = self.case
        H, Q = case["H"], case["Q"]
        live = np.flatnonzero(case["state_slots"] > case["null_slot"])
        all_items = (live[:, None] * H + np.arange(H)[None, :]).ravel()
        order = np.random.default_rng(seed).permutation(all_items)
        shares = [order[w::self.workers] for w in range(self.workers)]
        deadline = time.time() + seconds
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_share, [(sh, deadline) for sh in shares])
        wall = time.perf_counter() - t0
        done = sum(r[0] for r in res)
        step_equiv = wall * len(all_items) / max(done, 1)
        return len(live) * Q / step_equiv, done, wall

    def close(self):
        self.pool.terminate()
        self.pool.join()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from linear_attention_speculative_recoverssm_gb300 import synth
    case = synth.make(args.workload)
    pool = OraclePool(case)
    per_step = args.ref_step_seconds
    for _ in range(args.warmup):
        pool.rate(per_step)
    rates, items, secs = [], 0, 0.0
    for i in range(args.steps):
        r, n, dt = pool.rate(per_step, seed=i + 1)
        rates.append(r)
        items += n
        secs += dt
    pool.close()
    value = float(statistics.median(rates))
    ab = algorithmic_bytes(case)
    line = dict(
        impl="reference", metric=METRIC, value=value, unit="tok/s", n_gpus=args.gpus,
        steps=args.steps, warmup=args.warmup,
        ms_per_step=1e3 * ab["live_tokens"] / value, higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
        config=workload_config(case, args.workload),
        cpu_baseline=dict(value=value, unit="tok/s", cores=pool.workers, kind="oracle",
                          sample=f"{items} random live (request, head) items over "
                                 f"{args.steps} steps ({secs:.1f} s of FP64 numpy on "
                                 f"{pool.workers} worker processes), scaled to the whole step"),
        e2e=dict(value=value, unit="tok/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
    )
    print(json.dumps(line))


def max_over_ranks(value, device="cpu"):
    """The largest of one float across the ranks of the default process group
    (the job's time is its slowest replica's); the value itself on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(live_tokens_per_rank, world, steps, ms):
    """Whole-job throughput: every replica processes the same workload."""
    return live_tokens_per_rank * world * steps / (ms / 1e3)


def workload_config(case, name):
    return dict(workload=name, B=case["B"], H=case["H"], Q=case["Q"], RQ=case["RQ"],
                state_slots=int(case["state"].shape[0]), state_dtype="f32", K=DIM, V=DIM,
                padding_rows=int((case["state_slots"] <= case["null_slot"]).sum()),
                l2="inputs larger than L2: ~2 GB of state pages touched per step vs 129 MB L2",
                parallelism="replicas")


# ---------------------------------------------------------------------------
# the other rows of the step: standalone commit, mid-size batch, the cluster
# split's small-batch latencies, the bookkeeping kernels
# ---------------------------------------------------------------------------

def commit_algorithmic_bytes(c):
    """Bytes one standalone commit must move: per live (layer, request, head)
    item the source page read, the destination page written, the boundary
    page written when the boundary is live, and the n recorded corrections
    (FP32) and key / gate rows (BF16) read."""
    L, B, H, Q = c["L"], c["B"], c["H"], c["Q"]
    esz = c["layers"][0]["state"].dtype.itemsize
    page = DIM * DIM * esz
    total = 0
    for b in range(B):
        n = min(max(int(c["commit_lens"][b]), 0), Q)
        live = n > 0 and c["sources"][b] > c["null_slot"] and c["destinations"][b] > c["null_slot"]
        if not live:
            continue
        per = 2 * page + n * (DIM * 4 + 2 * DIM * 2)
        if c["boundaries"][b] > c["null_slot"] and c["boundary_lens"][b] > 0:
            per += page
        total += L * H * per
    return total


def verify_algorithmic_bytes(case):
    """Bytes one verify-only launch (the checkpoint is read, never written)
    must move: per live item the state page, this window's inputs and
    outputs, and with a record row the new records; per inert item its
    zero outputs."""
    B, H, Q = case["B"], case["H"], case["Q"]
    page = DIM * DIM * case["state"].dtype.itemsize
    total = 0
    for b in range(B):
        if case["state_slots"][b] <= case["null_slot"]:
            total += H * Q * DIM * 2
            continue
        per = page + 4 * Q * DIM * 2 + Q * 2 + Q * DIM * 2
        if case["record_rows"][b] >= 0:
            per += Q * (DIM * 4 + 2 * DIM * 2)
        total += H * per
    return total


def _event_ms(stream, fn, iters):
    """Device milliseconds per call of ``fn``, from CUDA events on ``stream``.
    A device-side sleep is queued first, so the host enqueues all ``iters``
    calls while it runs and the events bracket back-to-back device work: a
    short kernel is timed on the device, not at the host's launch rate."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(_HEAD_START_CYCLES)
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


# ~5 ms at the SM clock: longer than the host takes to enqueue any timed
# loop below
_HEAD_START_CYCLES = 10_000_000

ROW_GROUPS = ("commit", "mid_batch", "layers", "varlen", "latency", "bookkeeping", "decode_loop",
              "layer")


def measure_rows(dev, stream, peak, cpu_seconds, only=None, layer_workload=None):
    """Timings of the step's other rows (CUDA events on the launching stream;
    every pool below is larger than L2 except the latency sweep's, which is a
    latency measurement by design).  ``only``: the row groups to run (all
    when None)."""
    want = lambda group: only is None or group in only
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_BF16, kda_commit,
                                                               kda_defer_commit, kda_flush_plan,
                                                               kda_replay_verify, layer_tables,
                                                               synth)
    rows = {}
    names = ("q", "k", "v", "raw_g", "raw_beta", "A_log", "dt_bias", "state", "state_slots",
             "record_rows", "pending", "corr", "key_gate")

    def dt(a):
        return (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
                else torch.from_numpy(a)).to(dev)

    if want('commit'):
        # standalone commit, BF16 pools, 4 layers
        name = "commit-bf16-l4-h32-b64-q4-align"
        c = synth.make(name)
        states = [dt(lay["state"]) for lay in c["layers"]]
        corrs = [dt(lay["corr"]) for lay in c["layers"]]
        kgs = [dt(lay["key_gate"]) for lay in c["layers"]]
        tabs = layer_tables(states, corrs, kgs, dev)
        ct = {k: dt(c[k]) for k in ("A_log", "dt_bias", "sources", "commit_lens", "destinations",
                                    "boundaries", "boundary_lens")}

        def commit():
            kda_commit(*tabs, ct["A_log"], ct["dt_bias"], ct["sources"], ct["commit_lens"],
                       ct["destinations"], state_dtype=KDA_STATE_BF16, lower_bound=c["lower_bound"],
                       L=c["L"], H=c["H"], B=c["B"], Q=c["Q"], n_slots=states[0].shape[0],
                       n_rows=corrs[0].shape[0], boundaries=ct["boundaries"],
                       boundary_lens=ct["boundary_lens"], stream=stream)
        for _ in range(5):
            commit()
        ms = _event_ms(stream, commit, 50)
        nbytes = commit_algorithmic_bytes(c)
        row = dict(workload=name, ms=ms, bytes_per_launch=nbytes,
                   roofline=dict(bound="hbm", achieved=nbytes / ms / 1e6, peak=peak, unit="GB/s",
                                 frac=nbytes / ms / 1e6 / peak,
                                 traffic=profiled_traffic("commit", name)))
        if cpu_seconds > 0:
            from oracle import kda_oracle as ko
            L, B, H = c["L"], c["B"], c["H"]
            items = np.random.default_rng(0).permutation(L * B * H)
            ref = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
            t0, done = time.perf_counter(), 0
            while done < len(items) and time.perf_counter() - t0 < cpu_seconds:
                ko.commit(layers=ref, A_log=c["A_log"], dt_bias=c["dt_bias"], sources=c["sources"],
                          commit_lens=c["commit_lens"], destinations=c["destinations"],
                          lower_bound=c["lower_bound"], Q=c["Q"], B=B, H=H,
                          boundaries=c["boundaries"], boundary_lens=c["boundary_lens"],
                          items=items[done:done + 64])
                done += len(items[done:done + 64])
            secs = time.perf_counter() - t0
            row["cpu_baseline"] = dict(ms=1e3 * secs * len(items) / done, cores=1, kind="oracle",
                                       sample=f"{done} of {len(items)} (layer, request, head) items, "
                                              f"{secs:.1f} s on one core, scaled to the launch")
        rows["commit"] = row
        del states, corrs, kgs, tabs

    if want('mid_batch'):
        # fused step on the mid-size batch
        name = "replay-verify-f32-h32-b128-q4"
        c = synth.make(name)
        d = {n: dt(c[n]) for n in names}
        out = torch.zeros(c["v"].shape, dtype=torch.bfloat16, device=dev)

        def step():
            kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                              d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                              d["pending"], d["corr"], d["key_gate"], out, Q=c["Q"],
                              lower_bound=c["lower_bound"], q_scale=c["q_scale"], split=0,
                              stream=stream)
        for _ in range(5):
            step()
        ms = _event_ms(stream, step, 50)
        ab = algorithmic_bytes(c)
        row = dict(workload=name, ms=ms, tok_s=ab["live_tokens"] / (ms / 1e3),
                   bytes_per_launch=ab["total"],
                   roofline=dict(bound="hbm", achieved=ab["total"] / ms / 1e6, peak=peak, unit="GB/s",
                                 frac=ab["total"] / ms / 1e6 / peak))
        if cpu_seconds > 0:
            rate, items, secs = oracle_rate(c, cpu_seconds)
            row["cpu_baseline"] = dict(value=rate, unit="tok/s", cores=1, kind="oracle",
                                       sample=f"{items} live items, {secs:.1f} s on one core")
        rows["replay_verify_mid_batch"] = row

        # the stock verify (checkpoint read-only) on the same batch
        from linear_attention_speculative_recoverssm_gb300 import kda_verify

        def verify():
            kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
                       d["state"], d["state_slots"], d["corr"], d["key_gate"], out, Q=c["Q"],
                       lower_bound=c["lower_bound"], q_scale=c["q_scale"],
                       record_rows=d["record_rows"], stream=stream)
        for _ in range(5):
            verify()
        ms = _event_ms(stream, verify, 50)
        nbytes = verify_algorithmic_bytes(c)
        rows["verify_mid_batch"] = dict(
            workload=name, ms=ms, tok_s=ab["live_tokens"] / (ms / 1e3), bytes_per_launch=nbytes,
            roofline=dict(bound="hbm", achieved=nbytes / ms / 1e6, peak=peak, unit="GB/s",
                          frac=nbytes / ms / 1e6 / peak))
        del d, out

    if want('layers'):
        rows["replay_verify_layers"] = measure_layers(dev, stream, dt, peak)

    if want('varlen'):
        # the large batch with windows of 1..8 tokens (query_start_loc)
        name = "replay-verify-varlen-f32-h64-b512-q8"
        c = synth.make(name)
        d = {n: dt(c[n]) for n in names + ("query_start_loc",)}
        out = torch.zeros(c["v"].shape, dtype=torch.bfloat16, device=dev)
        st_v = torch.zeros(1, dtype=torch.int32, device=dev)

        def step_varlen():
            kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                              d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                              d["pending"], d["corr"], d["key_gate"], out, Q=c["Q"],
                              lower_bound=c["lower_bound"], q_scale=c["q_scale"], split=0,
                              query_start_loc=d["query_start_loc"], status=st_v, stream=stream)
        for _ in range(5):
            step_varlen()
        ms = _event_ms(stream, step_varlen, 50)
        if int(st_v.item()) != 0:
            raise RuntimeError(f"variable-window step: device status {int(st_v.item())}")
        ab_v = algorithmic_bytes(c)
        rows["replay_verify_varlen"] = dict(
            workload=name, ms=ms, tok_s=ab_v["live_tokens"] / (ms / 1e3),
            mean_window=float(c["q_lens"][c["state_slots"] > c["null_slot"]].mean()),
            bytes_per_launch=ab_v["total"],
            roofline=dict(bound="hbm", achieved=ab_v["total"] / ms / 1e6, peak=peak, unit="GB/s",
                          frac=ab_v["total"] / ms / 1e6 / peak))
        del d, out, c

    if want('latency'):
        # small batches: per-launch device time (a CUDA graph of 20 launches)
        lat = {}
        for B in (1, 4, 16):
            for Q in (1, 2, 4, 8):
                c = synth.latency_case(B=B, Q=Q)
                d = {n: dt(c[n]) for n in names}
                out = torch.zeros(c["v"].shape, dtype=torch.bfloat16, device=dev)
                res = {}
                for split in (1, 2, 4):
                    def one(split=split):
                        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"],
                                          d["A_log"], d["dt_bias"], d["state"], d["state_slots"],
                                          d["record_rows"], d["pending"], d["corr"], d["key_gate"],
                                          out, Q=Q, lower_bound=c["lower_bound"],
                                          q_scale=c["q_scale"], split=split,
                                          stream=torch.cuda.current_stream())
                    for _ in range(3):
                        one()
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        for _ in range(20):
                            one()
                    g.replay()
                    torch.cuda.synchronize()
                    res[f"split{split}"] = 1e3 * _event_ms(torch.cuda.current_stream(), g.replay,
                                                           10) / 20
                lat[f"B{B}_q{Q}"] = res
        rows["latency_us_h32"] = lat

    if want('bookkeeping'):
        # bookkeeping (defer, then flush plan) for 512 requests
        rng = np.random.default_rng(7)
        B = 512
        slots = torch.from_numpy(rng.integers(-1, 1024, B).astype(np.int32)).to(dev)
        rrows = torch.from_numpy(rng.permutation(B).astype(np.int32)).to(dev)
        pend = torch.zeros(B, dtype=torch.int32, device=dev)
        lens = torch.from_numpy(rng.integers(0, 9, B).astype(np.int32)).to(dev)
        plan = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(4)]

        def book():
            kda_defer_commit(slots, lens, rrows, pend, stream=stream)
            kda_flush_plan(slots, rrows, pend, *plan, Q=8, stream=stream)
        for _ in range(5):
            book()
        rows["bookkeeping_us_b512"] = 1e3 * _event_ms(stream, book, 50)
        del slots, rrows, pend, lens, plan

    if want("decode_loop"):
        rows["decode_loop"] = measure_decode_loop(dev, dt, peak)
    if want("layer"):
        rows["layer"] = measure_layer(dev, stream, dt, peak,
                                      **({} if layer_workload is None else
                                         dict(name=layer_workload)))
    return rows


def measure_layers(dev, stream, dt, peak, L=4):
    """The fused step over L = 4 layers of the mid-size batch's shapes (H=32,
    B=128, q=4, a 512-slot FP32 pool per layer), as one multi-layer launch
    and as L single-layer launches back to back; the bytes are the L
    layers' algorithmic bytes."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (kda_replay_verify,
                                                               kda_replay_verify_layers, synth)
    spec = dict(synth.WORKLOADS["replay-verify-f32-h32-b128-q4"])
    spec.pop("kind")
    c = synth.layers_case(L=L, **spec)
    st = {key: dt(c[key]) for key in synth.LAYER_STACKED + synth.SHARED_INDEX}
    pools = [dt(lay["state"]) for lay in c["layers"]]
    corrs = [dt(lay["corr"]) for lay in c["layers"]]
    kgs = [dt(lay["key_gate"]) for lay in c["layers"]]
    out = torch.zeros(c["q"].shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    common = dict(Q=c["Q"], lower_bound=c["lower_bound"], q_scale=c["q_scale"], status=status,
                  stream=stream)

    def fused():
        kda_replay_verify_layers(st["q"], st["k"], st["v"], st["raw_g"], st["raw_beta"],
                                 st["A_log"], st["dt_bias"], pools, st["state_slots"],
                                 st["record_rows"], st["pending"], corrs, kgs, out, **common)

    def per_layer():
        for l in range(L):
            kda_replay_verify(st["q"][l], st["k"][l], st["v"][l], st["raw_g"][l],
                              st["raw_beta"][l], st["A_log"][l], st["dt_bias"][l], pools[l],
                              st["state_slots"], st["record_rows"], st["pending"], corrs[l],
                              kgs[l], out[l], split=1, **common)
    for _ in range(5):
        fused()
        per_layer()
    ms_fused = _event_ms(stream, fused, 30)
    ms_single = _event_ms(stream, per_layer, 30)
    if int(status.item()) != 0:
        raise RuntimeError(f"multi-layer step: device status {int(status.item())}")
    abs_ = [algorithmic_bytes(lay) for lay in c["layers"]]
    nbytes = sum(a["total"] for a in abs_)
    tokens = sum(a["live_tokens"] for a in abs_)
    row = dict(workload=f"replay-verify-layers-f32-l{L}-h32-b128-q4", L=L, ms=ms_fused,
               ms_single_layer_launches=ms_single, tok_s=tokens / (ms_fused / 1e3),
               bytes_per_launch=nbytes,
               roofline=dict(bound="hbm", achieved=nbytes / ms_fused / 1e6, peak=peak,
                             unit="GB/s", frac=nbytes / ms_fused / 1e6 / peak))
    del pools, corrs, kgs, st, out
    return row


def layer_algorithmic_bytes(c):
    """Bytes the layer's prologue and epilogue must move for one step (the
    step's own are ``algorithmic_bytes``).  Prologue, per live (request,
    head) item: its q, k, v input channels (3 * Q * 256 B), three window
    values read and Q + 2 written per channel (384 channels, BF16), and the
    step inputs q, k, v, raw_g written (4 * Q * 256 B); once: f_a, f_b and
    the convolution weights.  Epilogue, per (token, head): the step output
    and the gate read and the layer output written (3 * 256 B)."""
    B, H, Q = c["B"], c["H"], c["Q"]
    live = int((c["state_slots"] > c["null_slot"]).sum()) * H
    per_item = 3 * Q * 256 + 384 * (3 + Q + 2) * 2 + 4 * Q * 256
    once = c["f_a"].nbytes + c["f_b"].nbytes + c["conv_weight"].nbytes
    once += 0 if c["conv_bias"] is None else c["conv_bias"].nbytes
    prologue = live * per_item + once
    epilogue = B * Q * H * 3 * 256 + c["norm_weight"].nbytes
    return prologue, epilogue


def measure_layer(dev, stream, dt, peak, name="layer-f32-h64-b512-q8"):
    """The model layer around the large-batch step: the prologue
    (convolution + SiLU, gate projection, window rewrite), the fused
    replay + verify on its outputs, and the gated-norm epilogue."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (kda_layer_epilogue,
                                                               kda_layer_prologue,
                                                               kda_replay_verify, synth)
    c = synth.make(name)
    keys = ("x", "conv_weight", "conv_bias", "conv_state", "f_a", "f_b", "gate", "norm_weight",
            "raw_beta", "A_log", "dt_bias", "state", "state_slots", "record_rows", "pending",
            "corr", "key_gate")
    d = {k: None if c[k] is None else dt(c[k]) for k in keys}
    T = c["B"] * c["Q"]
    shape = (T, c["H"], 128)
    for k in ("q", "k", "v", "raw_g", "o"):
        d[k] = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    out = torch.zeros((T, c["H"] * 128), dtype=torch.bfloat16, device=dev)

    def prologue():
        kda_layer_prologue(d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"],
                           d["f_b"], d["state_slots"], d["record_rows"], d["pending"], d["q"],
                           d["k"], d["v"], d["raw_g"], Q=c["Q"], stream=stream)

    def core():
        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], d["o"], Q=c["Q"],
                          lower_bound=c["lower_bound"], q_scale=c["q_scale"], split=0,
                          stream=stream)

    def epilogue():
        kda_layer_epilogue(d["o"], d["gate"], d["norm_weight"], out, eps=c["eps"],
                           stream=stream)

    def layer():
        prologue()
        core()
        epilogue()

    # the fused layer entry point: the same prologue into a workspace, then
    # the step with the gated RMSNorm folded into its row solve
    from linear_attention_speculative_recoverssm_gb300 import (kda_layer_step,
                                                               kda_layer_step_workspace_bytes)
    workspace = torch.empty(kda_layer_step_workspace_bytes(c["B"], c["H"], c["Q"]),
                            dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def fused_layer():
        kda_layer_step(d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"],
                       d["f_b"], d["raw_beta"], d["A_log"], d["dt_bias"], d["state"],
                       d["state_slots"], d["record_rows"], d["pending"], d["corr"],
                       d["key_gate"], d["gate"], d["norm_weight"], out, workspace, Q=c["Q"],
                       lower_bound=c["lower_bound"], q_scale=c["q_scale"], eps=c["eps"],
                       status=status, stream=stream)
    for _ in range(3):
        layer()
        fused_layer()
    ms = {"layer": _event_ms(stream, layer, 20), "prologue": _event_ms(stream, prologue, 20),
          "step": _event_ms(stream, core, 20), "epilogue": _event_ms(stream, epilogue, 20),
          "fused_layer": _event_ms(stream, fused_layer, 20)}
    if int(status.item()) != 0:
        raise RuntimeError(f"fused layer step: device status {int(status.item())}")
    pro_b, epi_b = layer_algorithmic_bytes(c)
    step_b = algorithmic_bytes(c)
    total = pro_b + step_b["total"] + epi_b
    gbs = total / ms["layer"] / 1e6
    # fused: the epilogue's read of o and write of the output are gone; the
    # step reads the gate and writes the normed output in place of o
    fused_b = pro_b + step_b["total"] + c["gate"].nbytes
    fused_gbs = fused_b / ms["fused_layer"] / 1e6
    return dict(
        workload=name, ms=ms, tok_s=step_b["live_tokens"] / (ms["layer"] / 1e3),
        bytes_per_launch=dict(prologue=pro_b, step=step_b["total"], epilogue=epi_b,
                              fused_layer=fused_b),
        roofline=dict(bound="hbm", achieved=gbs, peak=peak, unit="GB/s", frac=gbs / peak),
        prologue_roofline_frac=pro_b / ms["prologue"] / 1e6 / peak,
        epilogue_roofline_frac=epi_b / ms["epilogue"] / 1e6 / peak,
        fused_layer=dict(ms=ms["fused_layer"],
                         tok_s=step_b["live_tokens"] / (ms["fused_layer"] / 1e3),
                         roofline=dict(bound="hbm", achieved=fused_gbs, peak=peak, unit="GB/s",
                                       frac=fused_gbs / peak)))


def decode_loop_bytes(c, eager):
    """Algorithmic bytes of one graph of the decode workload.  Deferred:
    the stock verify, then fused steps whose pending counts are the previous
    step's accepted counts, then the flush's in-place commit of the last
    step's.  Eager: every step the stock verify and a commit of its accepted
    tokens.  The bookkeeping's few bytes per request are left out."""
    steps, live = c["steps"], c["state_slots"] > c["null_slot"]

    def commit_bytes(lens):
        return commit_algorithmic_bytes(dict(
            L=1, B=c["B"], H=c["H"], Q=c["RQ"], layers=[dict(state=c["state"])],
            commit_lens=np.where(live & (c["record_rows"] >= 0), lens, 0),
            sources=c["state_slots"], destinations=c["state_slots"],
            boundaries=np.zeros(c["B"], np.int32), boundary_lens=np.zeros(c["B"], np.int32),
            null_slot=c["null_slot"]))
    total = 0
    for s in range(steps):
        if eager or s == 0:
            total += verify_algorithmic_bytes(c)
        else:
            step = dict(c)
            step["pending"] = np.zeros_like(c["pending"])
            has = live & (c["record_rows"] >= 0)
            step["pending"][c["record_rows"][has]] = c["accepted"][s - 1][has]
            total += algorithmic_bytes(step)["total"]
        if eager:
            total += commit_bytes(c["accepted"][s])
    if not eager:
        total += commit_bytes(c["accepted"][steps - 1])
    return total


def measure_decode_loop(dev, dt, peak):
    """Eight decode steps of the large batch as one CUDA graph, in two
    schedules: deferred (the fused replay + verify; the stock verify after
    each flush; defer after sampling; a flush after the eighth step) and
    eager (the stock verify, then a commit of the accepted tokens every
    step, which reads and writes every live checkpoint once more)."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import DeferredRecoverSSM, synth
    name = "decode-loop-f32-h64-b512-q8"
    c = synth.make(name)
    steps, B, H, Q = c["steps"], c["B"], c["H"], c["Q"]
    keys = ("q", "k", "v", "raw_g", "raw_beta")
    d = {n: dt(c[n]) for n in ("A_log", "dt_bias", "state", "state_slots", "record_rows",
                               "pending", "corr", "key_gate")}
    win = {key: dt(c["windows"][key]) for key in keys}
    acc0 = dt(c["accepted"])
    acc = acc0.clone()
    eager_all = torch.ones(B, dtype=torch.uint8, device=dev)
    out = torch.zeros(c["windows"]["v"].shape[1:], dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream()  # graphs are captured on a side stream
    loop = DeferredRecoverSSM(d["state"], d["state_slots"], d["record_rows"], d["pending"],
                              d["corr"], d["key_gate"], d["A_log"], d["dt_bias"], Q=Q,
                              lower_bound=c["lower_bound"], q_scale=c["q_scale"],
                              stream=stream)

    def cycle(eager):
        acc.copy_(acc0)
        loop.flushed = True
        for s in range(steps):
            w = int(c["window_of_step"][s])
            if eager:
                loop.flushed = True
            loop.verify(*(win[key][w] for key in keys), out)
            loop.accept(acc[s], eager_all if eager else None)
        if not eager:
            loop.flush()

    live = c["state_slots"] > 0
    tokens = int(live.sum()) * Q
    accepted = int(c["accepted"][:, live].sum()) / steps
    row = dict(workload=name, steps_per_graph=steps,
               launches_per_graph=dict(deferred=2 * steps + 2, eager=3 * steps))
    torch.cuda.synchronize()
    for eager in (False, True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            cycle(eager)  # warm-up outside the graph
            with torch.cuda.graph(g, stream=stream):
                cycle(eager)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ms = _event_ms(torch.cuda.current_stream(), g.replay, 5) / steps
        nbytes = decode_loop_bytes(c, eager)
        gbs = nbytes / (ms * steps) / 1e6
        row["eager" if eager else "deferred"] = dict(
            ms_per_step=ms, verify_tok_s=tokens / (ms / 1e3),
            accepted_tok_s=accepted / (ms / 1e3), bytes_per_graph=nbytes,
            roofline=dict(bound="hbm", achieved=gbs, peak=peak, unit="GB/s", frac=gbs / peak))
    row["eager_over_deferred"] = row["eager"]["ms_per_step"] / row["deferred"]["ms_per_step"]
    return row


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # the oracle's workers are forked now, before this process touches CUDA
    pool = None
    pre_case = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from linear_attention_speculative_recoverssm_gb300 import synth as _synth
        pre_case = _synth.make(args.workload)
        pool = OraclePool(pre_case)

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify, synth

    case = pre_case if pre_case is not None else synth.make(args.workload)
    ab = algorithmic_bytes(case)

    def dt(a, pin=False):
        t = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
             else torch.from_numpy(a))
        return t.pin_memory() if pin else t.to(dev)

    names = ("q", "k", "v", "raw_g", "raw_beta", "A_log", "dt_bias", "state", "state_slots",
             "record_rows", "pending", "corr", "key_gate")
    d = {n: dt(case[n]) for n in names}
    out = torch.zeros(case["v"].shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    Q = case["Q"]

    def step(dd):
        kda_replay_verify(dd["q"], dd["k"], dd["v"], dd["raw_g"], dd["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], dd["state_slots"], dd["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], dd["out"], Q=Q,
                          lower_bound=case["lower_bound"], q_scale=case["q_scale"], split=1,
                          status=status, stream=stream)

    dd = dict(d, out=out)
    for _ in range(args.warmup):
        step(dd)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    sampler.start()
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record(stream)
    for i in range(args.steps):
        ev_s[i].record(stream)
        step(dd)
        ev_e[i].record(stream)
    t_end.record(stream)
    barrier()
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    kern_ms = [a.elapsed_time(b) for a, b in zip(ev_s, ev_e)]
    avg_kernel_ms = sum(kern_ms) / len(kern_ms)

    total_ms = max_over_ranks(total_ms, dev)
    value = job_tokens_per_s(ab["live_tokens"], world, args.steps, total_ms)

    # ---- end to end through the C ABI, inputs from pinned host memory ----
    e2e = None
    if not args.no_e2e:
        # Every step copies its activations and request indices in from pinned
        # host memory and reads its outputs back; as in a decoding loop, step
        # i + 1's inputs are copied while step i computes (two device input
        # sets, copies on their own streams), and the state pool and records
        # stay resident.  Kernels run in step order on one stream.
        host_names = ("q", "k", "v", "raw_g", "raw_beta", "state_slots", "record_rows")
        host = {n: dt(case[n], pin=True) for n in host_names}
        dev_in = [{n: torch.empty_like(host[n], device=dev) for n in host_names} for _ in range(2)]
        dev_out = [out, torch.empty_like(out)]
        out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host[0].numel() * out_host[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        returned = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n_steps):
            for i in range(n_steps):
                bsel = i & 1
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(computed[bsel])  # step i - 2 done with this input set
                    for n in host_names:
                        dev_in[bsel][n].copy_(host[n], non_blocking=True)
                    copied[bsel].record(s_in)
                stream.wait_event(copied[bsel])
                if i >= 2:
                    stream.wait_event(returned[bsel])  # step i - 2's outputs read back
                step(dict(dev_in[bsel], out=dev_out[bsel]))
                computed[bsel].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(computed[bsel])
                    out_host[bsel].copy_(dev_out[bsel], non_blocking=True)
                    returned[bsel].record(s_out)
            for ev in returned[:min(n_steps, 2)]:
                stream.wait_event(ev)

        e2e_run(max(2, args.warmup))
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)  # the timed region starts before the first copy
        e2e_run(args.steps)
        e1.record(stream)
        barrier()
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, dev)
        e2e = dict(value=job_tokens_per_s(ab["live_tokens"], world, args.steps, e_ms), unit="tok/s",
                   h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                   overlap="step i + 1's host-to-device copies run during step i's kernel")

    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = ab["total"] / (avg_kernel_ms / 1e3) / 1e9
    state_gbs = ab["state"] / (avg_kernel_ms / 1e3) / 1e9

    rows = None
    if rank == 0 and not args.no_rows:
        rows = measure_rows(dev, stream, peak, 0.0 if args.no_cpu_baseline else 3.0,
                            only=None if args.rows is None else set(args.rows.split(",")),
                            layer_workload=args.layer_workload)

    cpu = None
    if pool is not None:
        rate, items, secs = pool.rate(args.cpu_seconds)
        rate1, items1, secs1 = oracle_rate(case, args.cpu_seconds / 2)
        cpu = dict(value=rate, unit="tok/s", cores=pool.workers, kind="oracle",
                   sample=f"{items} random live (request, head) items of this workload "
                          f"({secs:.1f} s of FP64 numpy on {pool.workers} worker processes, "
                          "one per host core), scaled to the whole step",
                   single_core=dict(value=rate1, unit="tok/s", cores=1,
                                    sample=f"{items1} items, {secs1:.1f} s on one core"))
        pool.close()

    if rank == 0:
        line = dict(
            metric=METRIC, value=value, unit="tok/s", n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=total_ms / args.steps, higher_is_better=True,
            scaling="weak", vs_baseline=None, dtype="f32", data="synthetic",
            config=workload_config(case, args.workload),
            state_gbs=state_gbs, algorithmic_gbs=achieved,
            hbm_frac=achieved / peak,
            kernel_ms=avg_kernel_ms,
            roofline=dict(bound="hbm", achieved=achieved, peak=peak, unit="GB/s",
                          frac=achieved / peak,
                          traffic=args.traffic if args.traffic is not None
                          else profiled_traffic("step", args.workload),
                          peak_source="MEASURED_PEAKS.json hbm_gbs" if "hbm_gbs" in peaks
                          else "fallback 6.8 TB/s",
                          bytes_per_launch=ab["total"], state_bytes_per_launch=ab["state"]),
            cpu_baseline=cpu, e2e=e2e, gpu_launches=args.steps, clocks=clocks, rows=rows,
        )
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the commit / mid-batch / latency / bookkeeping timings")
    ap.add_argument("--rows", default=None,
                    help="comma-separated row groups to run (default all): "
                         + ", ".join(ROW_GROUPS))
    ap.add_argument("--layer-workload", default=None,
                    help="the model-layer row's workload (default layer-f32-h64-b512-q8)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=1.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the current kernel, if measured")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
