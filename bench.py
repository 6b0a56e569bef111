"""Benchmark of the QSA hot path: one step = qsa_prep + qsa_score + qsa_attn.

Workload: prompt attention, long context -- T = 1984 query tokens at
pos0 = 30000 over a 31984-cell int8 K/V cache (fp16 scales per 32 dims),
12 query heads sharing one KV head, head_dim 128, 2048 evenly spaced causal
selected ids per token (W = 2048).  The step normalises/rotates the queries
and quantises the new K/V rows into the cache, scores every causal cell
(from the head sum of the rotated fp32 queries, which prep writes into the
score's workspace; 61.5 M scores written) and runs the selected-id attention;
the score runs on a second stream beside the attention, since both depend
only on prep.

With --select the step also runs qsa_select between the score and the
attention: each token keeps 64 sink cells, the previous 256 cells and its own
cell, plus the best-scoring other causal cells up to 2048, and the attention
reads those ids instead of the evenly spaced ones.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--select]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "query tokens/s and achieved HBM GB/s (% of roofline) for QSA attention at T=1984"
UNIT = "tokens/s"
NTOK, POS0, WIDTH, HQ, D, G = 1984, 30000, 2048, 12, 128, 32
SCORE_CTAS = 0  # 0: the overlapped score fills the attention's tail (a fixed SM share measured slower)
WORKLOAD = ("prompt attention long context: T=1984 query tokens, pos0=30000, int8 K/V cache of 31984 cells "
            "with fp16 per-32 scales, 12 q heads / 1 KV head, head_dim 128, 2048 evenly spaced causal ids per "
            "token; step = qsa_prep + qsa_score (all causal cells, from the head sum of the fp32 rotated queries that "
            "qsa_prep writes) + qsa_attn")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
KERNELS = ("prep", "score", "attn")
KERNELS_SELECT = ("prep", "score", "select", "attn")
WORKLOAD_SELECT = WORKLOAD.replace("2048 evenly spaced causal ids per token",
                                   "2048 ids per token chosen by qsa_select (64 sink + 256 local + current + "
                                   "top-scoring causal cells)").replace("+ qsa_attn", "+ qsa_select + qsa_attn")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--ntok", type=int, default=NTOK, help="fewer tokens: for small profiling captures only")
    p.add_argument("--pos0", type=int, default=POS0, help="another context length: for profiling captures only")
    p.add_argument("--select", action="store_true",
                   help="step = prep + score + select + attention on the selected ids")
    p.add_argument("--pages-shape", action="store_true",
                   help="time the attention alone at the pages' own shape (2 KV x 12 heads, head_dim 256, "
                        "per-64 scales) on the same token / id workload")
    p.add_argument("--decode", action="store_true",
                   help="latency of the attention alone on the decode windows: 1 token at pos0=320 and the "
                        "8-token MTP window at pos0=30000 (64 sink + 256 local + own cell, width 384)")
    p.add_argument("--score-sweep", action="store_true",
                   help="the score pass alone from fp32 queries (head-sum pass + tcgen05 score) at T=1984 and "
                        "pos0 = 0, 2048, 8192, 30000")
    p.add_argument("--score-ctas", type=int, default=SCORE_CTAS,
                   help="SMs the overlapped score takes (0: it fills the attention's tail instead)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-workload block (decode windows, short prompt, score sweep)")
    p.add_argument("--cpu-sample-seconds", type=float, default=8.0)
    return p.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work per launch (bytes the method must move, flops it must do)
# ---------------------------------------------------------------------------

def attn_bytes(ids_np, ntok, hkv=1, hq=HQ, d=D):
    """Gathered bytes: per valid id and KV head 2 * (d + 8) (K and V codes plus
    four fp16 scales each; 272 B at d = 128), every id slot read (4 B), q read
    and out written (fp16)."""
    valid = int((ids_np >= 0).sum())
    return valid * hkv * 2 * (d + 8) + ids_np.size * 4 + 2 * ntok * hq * d * 2, valid


def score_pairs(ntok, pos0):
    return sum(pos0 + t + 1 for t in range(ntok))


def score_bytes(ntok, pos0, cells):
    """The head sum read (fp16 hi/lo rows and one int32 exponent per token,
    prep writes them), int8 codes + fp16 scales of every cell read, one fp32
    score written per causal (token, cell) pair."""
    ntok_pad = -(-ntok // 64) * 64
    return ntok_pad * (2 * D * 2 + 4) + cells * (D + 2 * (D // G)) + 4 * score_pairs(ntok, pos0)


def select_bytes(ntok, pos0, sink=64, local=256):
    """Algorithmic bytes of one qsa_select launch: each token's free causal
    scores (after the sink, before the local run), read once as fp32, and its
    W int32 ids written."""
    free = sum(max(min(max(sink, p - local), p) - sink, 0) for p in range(pos0, pos0 + ntok))
    return 4 * free + 4 * ntok * WIDTH


def prep_bytes(ntok):
    """fp32 q, k, v rows read, fp16 q written, int8 K/V codes and fp16 scales
    written, the score's head sum (fp16 hi/lo rows and an int32 exponent per
    token) written, the norm weight."""
    ntok_pad = -(-ntok // 64) * 64
    return (ntok * HQ * D * (4 + 2) + 2 * ntok * D * 4 + 2 * ntok * (D + 2 * (D // G)) + ntok_pad * (2 * D * 2 + 4)
            + D * 4)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def l2_copy_gbs(dev, nbytes=32 << 20, reps=200):
    """Measured L2 bandwidth: a device-to-device copy of a 32 MiB buffer into
    another (64 MiB live, well inside the 129 MB L2), repeated after a
    warm-up; bytes read plus bytes written per second."""
    import torch
    src = torch.ones(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    for _ in range(10):
        dst.copy_(src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e9 * 2e-6 * reps))  # the copies queue behind it and then run back to back
    e0.record()
    for _ in range(reps):
        dst.copy_(src)
    e1.record()
    e1.synchronize()
    return 2 * nbytes * reps / (e0.elapsed_time(e1) / 1e3) / 1e9


def l2_gather_gbs(dev, reps=20):
    """Measured L2 read rate for the attention's access pattern: 128-byte rows
    gathered by id from an L2-resident 8.2 MB table (the K and V rows of the
    long-context cache), eight lanes per row, over a grid that fills every SM
    (libqsa_l2probe.so).  Row bytes plus id bytes per second; None if the
    probe library was not built."""
    import ctypes
    import torch
    from sparse_selected_attention_gb300 import build as qsa_build
    if not os.path.exists(qsa_build.PROBE_LIB):
        return None
    L = ctypes.CDLL(qsa_build.PROBE_LIB)
    L.qsa_l2_gather_probe.restype = ctypes.c_int
    L.qsa_l2_gather_probe.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_longlong,
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    nrows, nids = 2 * 31984, 2 * 1984 * 2048
    g = torch.Generator(device=dev).manual_seed(7)
    table = torch.randint(0, 255, (nrows * 128,), dtype=torch.uint8, device=dev, generator=g)
    ids = torch.randint(0, nrows, (nids,), dtype=torch.int32, device=dev, generator=g)
    blocks = 8 * torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.empty(blocks * 256, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)

    def launch():
        rc = L.qsa_l2_gather_probe(table.data_ptr(), nrows, ids.data_ptr(), nids, sink.data_ptr(), blocks, sp)
        if rc != 0:
            raise RuntimeError(f"qsa_l2_gather_probe failed ({rc})")

    for _ in range(3):
        launch()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e9 * 80e-6 * reps))  # the launches queue behind it and then run back to back
    e0.record(stream)
    for _ in range(reps):
        launch()
    e1.record(stream)
    e1.synchronize()
    return nids * (128 + 4) * reps / (e0.elapsed_time(e1) / 1e3) / 1e9


def traffic_l2_record(kernel):
    """lts (L2) bytes per launch from the committed ncu summary, if current."""
    if traffic_record(kernel) is None:
        return None
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        return json.load(f)[kernel].get("lts_bytes")


def traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; None otherwise."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    src = os.path.join(ROOT, "sparse_selected_attention_gb300", "csrc", rec["source"])
    try:
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
    except OSError:
        return None
    return rec["dram_bytes_per_launch"]


# ---------------------------------------------------------------------------
# multi-rank aggregation (one process per GPU; replicas, no data exchange)
# ---------------------------------------------------------------------------

def max_over_ranks(x, device=None):
    """The largest per-rank value (every rank gets it); x itself at world size 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, world, slowest_ms):
    """Whole-job tokens/s: every rank processes its own batch of
    `tokens_per_rank` tokens; the job takes as long as the slowest rank."""
    return world * tokens_per_rank / (slowest_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------
#
# The oracle runs in a pool of single-threaded worker processes (started with
# `spawn`, so no worker inherits the parent's CUDA state).  Each worker makes
# the workload's inputs once; a task is a list of token rows, for which it
# runs prep on those rows, their score rows over every causal cell and their
# attention, and returns its own compute time.

_ORACLE = None


def _oracle_worker_init(ntok, pos0, width):
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    sys.path.insert(0, ROOT)
    from sparse_selected_attention_gb300 import workloads as wl
    global _ORACLE
    _ORACLE = {"inp": wl.prep_inputs(ntok, seed=5), "cache": wl.make_cache(pos0 + ntok, seed=5),
               "ids": wl.even_ids(ntok, pos0, width), "pos0": pos0}


def _oracle_rows(rows):
    import numpy as np

    from oracle import attention, prep, score
    w = _ORACLE
    inp, cache, rows = w["inp"], w["cache"], np.asarray(rows, dtype=np.int64)
    t0 = time.perf_counter()
    q64, q16, q32 = prep(inp.q_in[rows], inp.k_in[rows], inp.v_in[rows], inp.norm_w, w["pos0"], cache.kq,
                         cache.vq, cache.ksc, cache.vsc)
    score(q32, cache.kq, cache.ksc, w["pos0"])
    attention(q16, cache.kq, cache.vq, cache.ksc, cache.vsc, w["ids"][rows], 1 / math.sqrt(128))
    return len(rows), time.perf_counter() - t0


class OraclePool:
    """`cores` single-threaded oracle workers on this host."""

    def __init__(self, cores, ntok=NTOK, pos0=POS0):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        self.cores, self.ntok = cores, ntok
        self.ex = ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn"),
                                      initializer=_oracle_worker_init, initargs=(ntok, pos0, WIDTH))
        list(self.ex.map(_oracle_rows, [[0]] * cores))  # start every worker and warm it

    def rows(self, n, offset=0):
        """n token rows spread evenly over the workload, starting at an offset."""
        return [int((offset + i * self.ntok / n)) % self.ntok for i in range(n)]

    def run(self, rows, workers):
        """Rows dealt to `workers` workers at once; (rows done, wall seconds)."""
        parts = [rows[i::workers] for i in range(workers)]
        t0 = time.perf_counter()
        done = sum(n for n, _ in self.ex.map(_oracle_rows, parts))
        return done, time.perf_counter() - t0

    def close(self):
        self.ex.shutdown()


def cpu_baseline(target_seconds, pool=None):
    """The oracle's throughput on one thread and on every host core, each
    over a sample of about `target_seconds`."""
    own = pool is None
    pool = pool or OraclePool(os.cpu_count() or 1)
    try:
        n, dt = pool.run(pool.rows(4), 1)
        per_row = dt / n
        n1 = int(max(4, min(NTOK, target_seconds / per_row)))
        d1, t1 = pool.run(pool.rows(n1), 1)
        nc = int(max(pool.cores, min(NTOK, target_seconds * pool.cores / per_row)))
        dc, tc = pool.run(pool.rows(nc, offset=1), pool.cores)
    finally:
        if own:
            pool.close()
    return {"value": dc / tc, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
            "single_thread_value": d1 / t1,
            "sample": f"{dc} evenly spaced token rows of the workload on {pool.cores} single-threaded worker "
                      f"processes ({tc:.1f} s wall); each row: prep of its q/k/v rows, its score row over all "
                      f"causal cells, its attention over its ids.  One thread: {d1} rows in {t1:.1f} s"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from sparse_selected_attention_gb300 import (qsa_attn, qsa_prep, qsa_score, qsa_score_workspace_bytes,
                                                 qsa_select)
    from sparse_selected_attention_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    T, pos0 = args.ntok, args.pos0
    C = pos0 + T
    inp = wl.prep_inputs(T, seed=5 + rank)
    cache = wl.make_cache(C, seed=5 + rank)
    ids_np = wl.even_ids(T, pos0, WIDTH)

    def d(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    q_in, k_in, v_in, norm_w = d(inp.q_in), d(inp.k_in), d(inp.v_in), d(inp.norm_w)
    kq, vq, ksc, vsc = d(cache.kq), d(cache.vq), d(cache.ksc), d(cache.vsc)
    ids = d(ids_np)
    q16 = torch.empty((T, HQ, D), dtype=torch.float16, device=dev)
    scores = torch.empty((T, C), dtype=torch.float32, device=dev)
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device=dev)
    out = torch.empty((T, HQ, D), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    names = KERNELS_SELECT if args.select else KERNELS

    main_bufs = {"q": q_in, "k": k_in, "v": v_in, "ids": ids, "out": out}
    # Score and attention both depend only on prep, so without selection they
    # run side by side and the step ends when both have; with selection the
    # chain is serial.  Neither kernel's CTAs fit on an SM beside the other's,
    # so they split the SMs: the score, on a high-priority stream and launched
    # first, takes `score_ctas` SMs (its persistent CTAs are placed before any
    # attention CTA), and the attention's CTAs fill the others.  A score CTA
    # turns out more scores per SM-second on a share of the GPU than on all of
    # it, where the SMs contend for DRAM writes.  With score_ctas = 0 the
    # attention goes first and the score's full grid fills its tail.
    sc = args.score_ctas
    side = torch.cuda.Stream(dev, priority=-1) if sc > 0 else torch.cuda.Stream(dev)
    ev_prep, ev_side = torch.cuda.Event(), torch.cuda.Event()

    def timed(ev, name, st, fn):
        if ev and name in ev:
            ev[name][0].record(st)
        fn()
        if ev and name in ev:
            ev[name][1].record(st)

    def step(ev=None, b=main_bufs, serial=False, kernel_events=True):
        if ev and not kernel_events:
            ev = {"step": ev["step"]}
        if ev:
            ev["step"][0].record(stream)
        timed(ev, "prep", stream,
              lambda: qsa_prep(b["q"], b["k"], b["v"], norm_w, pos0, kq, vq, ksc, vsc, q16, qbar_out=ws))
        if args.select or serial:
            timed(ev, "score", stream,
                  lambda: qsa_score(None, kq, ksc, pos0, scores, ws, workspace_holds_qbar=True))
            if args.select:
                timed(ev, "select", stream, lambda: qsa_select(scores, pos0, b["ids"]))
            timed(ev, "attn", stream, lambda: qsa_attn(q16, kq, vq, ksc, vsc, b["ids"], b["out"]))
        else:
            ev_prep.record(stream)
            side.wait_event(ev_prep)
            run_score = lambda: timed(ev, "score", side, lambda: qsa_score(
                None, kq, ksc, pos0, scores, ws, stream=side, workspace_holds_qbar=True, max_ctas=sc))
            if sc > 0:
                run_score()
            timed(ev, "attn", stream, lambda: qsa_attn(q16, kq, vq, ksc, vsc, b["ids"], b["out"]))
            if sc == 0:
                run_score()
            ev_side.record(side)
            stream.wait_event(ev_side)
        if ev:
            ev["step"][1].record(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()

    K = args.steps
    # The timed region: step events only.  Events between the kernels would
    # serialise them: the attention and the score launch as programmatic
    # dependents of prep and start while its last CTAs finish.
    evs = [{"step": (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))} for _ in range(K)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    wall0 = time.perf_counter()
    for k in range(K):
        flush.zero_()  # L2 flush between steps, outside the step's events
        step(evs[k], kernel_events=False)
    barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_ms = [evs[k]["step"][0].elapsed_time(evs[k]["step"][1]) for k in range(K)]
    ms = max_over_ranks(sum(step_ms) / K, dev)

    # Each kernel's duration in the same overlapped schedule, from a second
    # live pass with events around every kernel on the stream it runs on.
    evk = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for n in names + ("step",)} for _ in range(K)]
    for k in range(K):
        flush.zero_()
        step(evk[k])
    torch.cuda.synchronize()
    per = {n: [evk[k][n][0].elapsed_time(evk[k][n][1]) for k in range(K)] for n in names}
    kernel_pass_step_ms = sum(evk[k]["step"][0].elapsed_time(evk[k]["step"][1]) for k in range(K)) / K

    # Each kernel's own launch time, from a short pass with the kernels run
    # one after another (after the timed region; the overlapped score's event
    # window also spans its wait for SMs).
    KC = min(K, 50)
    evc = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for n in names + ("step",)} for _ in range(KC)]
    for k in range(KC):
        flush.zero_()
        step(evc[k], serial=True)
    torch.cuda.synchronize()
    own = {n: sum(evc[k][n][0].elapsed_time(evc[k][n][1]) for k in range(KC)) / KC for n in names}

    # End to end through the public API, as a serving loop runs it: every
    # step uploads its inputs from pinned host memory, runs the calls and
    # reads its attention output back.  Inputs and outputs are double-buffered
    # so that step k+1's upload and step k's read-back (two copy streams)
    # overlap step k's kernels; the kernels themselves stay on one stream, so
    # the shared K/V cache and scratch buffers are never used concurrently.
    # The timed region spans the first upload to the last read-back.  No L2
    # flush here: every step writes 246 MB of scores, more than L2 holds.
    e2e = None
    if not args.no_e2e:
        h_q, h_k, h_v = (torch.from_numpy(x).pin_memory() for x in (inp.q_in, inp.k_in, inp.v_in))
        h_ids = torch.from_numpy(ids_np).pin_memory()
        h_outs = [torch.empty((T, HQ, D), dtype=torch.float16).pin_memory() for _ in range(2)]
        h_in = (h_q, h_k, h_v) if args.select else (h_q, h_k, h_v, h_ids)  # selected ids are made on the device
        h2d = sum(x.numel() * x.element_size() for x in h_in)
        d2h = h_outs[0].numel() * h_outs[0].element_size()
        bufs = [main_bufs, {"q": torch.empty_like(q_in), "k": torch.empty_like(k_in), "v": torch.empty_like(v_in),
                            "ids": ids if args.select else torch.empty_like(ids), "out": torch.empty_like(out)}]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_up, ev_done, ev_down = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

        def pipeline(nsteps, start=None):
            if start is not None:
                up.wait_event(start)
            for k in range(nsteps + 1):
                if k < nsteps:  # upload step k once step k-2 (same buffers) has finished with them
                    b = bufs[k % 2]
                    with torch.cuda.stream(up):
                        if k >= 2:
                            up.wait_event(ev_done[k % 2])
                        b["q"].copy_(h_q, non_blocking=True)
                        b["k"].copy_(h_k, non_blocking=True)
                        b["v"].copy_(h_v, non_blocking=True)
                        if not args.select:
                            b["ids"].copy_(h_ids, non_blocking=True)
                        ev_up[k % 2].record(up)
                if k >= 1:  # step k-1 on the kernel stream, then its read-back
                    j = k - 1
                    b = bufs[j % 2]
                    stream.wait_event(ev_up[j % 2])
                    if j >= 2:
                        stream.wait_event(ev_down[j % 2])
                    step(b=b)
                    ev_done[j % 2].record(stream)
                    with torch.cuda.stream(down):
                        down.wait_event(ev_done[j % 2])
                        h_outs[j % 2].copy_(b["out"], non_blocking=True)
                        ev_down[j % 2].record(down)
            stream.wait_event(ev_down[(nsteps - 1) % 2])

        pipeline(3)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pipeline(K, start=e0)
        e1.record(stream)
        e1.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, dev)
        e2e = {"value": weak_scaling_value(T, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "schedule": "double-buffered: step k+1 upload and step k read-back overlap step k's kernels"}

    # Roofline of the dominant kernel.
    avg = {n: sum(v) / K for n, v in per.items()}
    # Overlapped, the score's event window also spans its wait for SMs the
    # attention holds; the attention (main stream, the step's critical path)
    # is then the kernel whose own launch time bounds the step.
    dom = max(avg, key=avg.get) if args.select else "attn"
    ab, valid = attn_bytes(ids.cpu().numpy() if args.select else ids_np, T)
    alg = {"attn": ab, "score": score_bytes(T, pos0, C), "prep": prep_bytes(T)}
    if args.select:
        alg["select"] = select_bytes(T, pos0)
    peak, peak_src = peaks()
    achieved = alg[dom] / (avg[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic_record(dom), "kernel": dom, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": alg[dom], "avg_launch_ms": avg[dom]}
    # The attention's gathers come from an L2-resident cache: its binding
    # roofline is L2 bandwidth.  lts bytes per launch (ncu) over the launch
    # time, against the L2 rate measured live for the same access pattern
    # (128-byte rows by id); a device copy's rate is given beside it.
    l2copy = l2_copy_gbs(dev)
    l2gather = l2_gather_gbs(dev)
    l2peak = l2gather if l2gather is not None else l2copy
    lts = traffic_l2_record(dom)
    roof["l2"] = {"peak_gbs": l2peak,
                  "peak_source": ("measured live: 128-byte rows gathered by id from an 8.2 MB L2-resident table, "
                                  "row and id bytes" if l2gather is not None else
                                  "measured live: 32 MiB device copy, L2-resident (gather probe not built)"),
                  "copy_gbs": l2copy, "lts_bytes_per_launch": lts,
                  "achieved_gbs": None if lts is None else lts / (avg[dom] / 1e3) / 1e9,
                  "frac": None if lts is None else lts / (avg[dom] / 1e3) / 1e9 / l2peak,
                  "logical_frac": alg[dom] / (avg[dom] / 1e3) / 1e9 / l2peak}
    kernels = {n: {"avg_ms": avg[n], "own_ms": own[n], "algorithmic_bytes": alg[n],
                   "achieved_gbs": alg[n] / (own[n] / 1e3) / 1e9} for n in names}
    kernels["score"]["pairs"] = score_pairs(T, pos0)
    if not args.select:
        kernels["score"]["overlapped_with"] = "attn (second stream; avg_ms includes waiting for SMs)"
    # The score's tensor-core work as issued (three fp16 128x128x128 products
    # per tile over the head-summed queries), and the bytes it moves; the
    # kernel is bound by its fp32 score writes, not by the tensor pipe.
    tc, tc_src = bf16_peak()
    ex = score_flops_executed(T, pos0) / (own["score"] / 1e3) / 1e12
    kernels["score"].update(tensor_tflops_executed=ex, frac_of_f16_peak_executed=ex / tc, f16_peak_source=tc_src,
                            frac_of_hbm_peak=kernels["score"]["achieved_gbs"] / peaks()[0])
    kernels["attn"]["valid_cells"] = valid
    roof["kernel_pass_step_ms"] = kernel_pass_step_ms
    return {"ms": ms, "wall_s": wall, "e2e": e2e, "clocks": clocks, "roofline": roof, "kernels": kernels,
            "launches_per_step": 4 if args.select else 3}  # prep, score, (select,) attention


def score_tiles(ntok, pos0, tm=128, tn=128):
    """128 x 128 (cell, token) tiles the score kernel runs: per 128-token
    tile, every cell tile up to its last token's causal bound."""
    tiles = 0
    for t0 in range(0, ntok, tn):
        tiles += (pos0 + min(ntok - 1, t0 + tn - 1)) // tm + 1
    return tiles


def score_flops_executed(ntok, pos0):
    """Tensor-core flops the score kernel issues: three 128x128x128 fp16
    products (hi*hi, hi*lo, lo*hi) per tile."""
    return score_tiles(ntok, pos0) * 3 * 2 * 128 ** 3


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


def _device_times(stream, fn, n, flush=None):
    """Device time of each of n calls of fn on `stream` (ms), L2 flushed
    before each call when `flush` is given (outside the call's events).
    Without a flush the calls run back to back: a GPU-side sleep queued
    first lets the host enqueue every call before the first one starts, so
    no host launch gap falls between a call's events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    if flush is None:
        torch.cuda._sleep(int(2e9 * 50e-6 * n))  # about 50 us of GPU time per call queued behind it
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sorted(a.elapsed_time(b) for a, b in evs)


def run_configs(dev, n):
    """Every workload the method is specified on, timed in the same run:
    the two decode windows (fused and split attention, L2 cold and warm),
    the short and long prompt attention, the score sweep, the selection over
    the long-context scores, the attention at the pages' own shape, and prep
    with and without the key rotation."""
    import numpy as np
    import torch

    from sparse_selected_attention_gb300 import qsa_attn, qsa_prep, qsa_score, qsa_score_workspace_bytes, qsa_select
    from sparse_selected_attention_gb300 import workloads as wl

    def to(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    hbm, hbm_src = peaks()
    tc, tc_src = bf16_peak()
    med = lambda t: t[len(t) // 2]
    out = {"peaks": {"hbm_gbs": hbm, "hbm_source": hbm_src, "f16_tflops": tc,
                     "f16_source": tc_src + " (fp16 and bf16 run at the same dense rate)"},
           "calls_per_point": n}

    def attn_case(w):
        cache = wl.make_cache(w.cells, seed=w.seed)
        kq, vq, ksc, vsc = (to(x) for x in (cache.kq, cache.vq, cache.ksc, cache.vsc))
        q = to(wl.queries_f16(w.ntok, seed=w.seed))
        ids_np = w.make_ids()
        ids = to(ids_np)
        o = torch.empty((w.ntok, HQ, D), dtype=torch.float16, device=dev)
        part = torch.empty((w.ntok, w.width // 64, HQ, D + 2), dtype=torch.float32, device=dev)
        fused = lambda: qsa_attn(q, kq, vq, ksc, vsc, ids, o)
        split = lambda: qsa_attn(q, kq, vq, ksc, vsc, ids, o, part=part)
        ab, valid = attn_bytes(ids_np, w.ntok)
        return fused, split, ab, valid

    for key, w in (("0_tiny_decode", wl.TINY_DECODE), ("1_mtp_decode", wl.MTP_DECODE)):
        fused, split, ab, valid = attn_case(w)
        rec = {"workload": w.name, "valid_cells": valid, "algorithmic_bytes": ab}
        for pname, fn in (("fused", fused), ("split", split)):
            for _ in range(5):
                fn()
            cold = med(_device_times(stream, fn, n, flush))
            warm = med(_device_times(stream, fn, n))
            rec[pname] = {"us_cold_l2": 1e3 * cold, "us_warm_l2": 1e3 * warm,
                          "tokens_per_s_cold_l2": w.ntok / (cold / 1e3)}
        out[key] = rec
    for key, w in (("2_prompt_short", wl.PROMPT_SHORT), ("3_prompt_long", wl.PROMPT_LONG)):
        fused, _, ab, valid = attn_case(w)
        for _ in range(3):
            fused()
        t = _device_times(stream, fused, n, flush)
        ms = sum(t) / len(t)
        out[key] = {"workload": w.name, "us": 1e3 * ms, "tokens_per_s": w.ntok / (ms / 1e3), "valid_cells": valid,
                    "algorithmic_bytes": ab, "logical_gbs": ab / (ms / 1e3) / 1e9,
                    "frac_of_hbm_peak": ab / (ms / 1e3) / 1e9 / hbm}
    sweep = []
    T = wl.SCORE_NTOK
    for pos0 in wl.SCORE_POS0:
        C = pos0 + T
        cache = wl.make_cache(C, seed=5)
        kq, ksc = to(cache.kq), to(cache.ksc)
        q = to(wl.queries_f32(T, seed=5))
        sc = torch.empty((T, C), dtype=torch.float32, device=dev)
        ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device=dev)
        fn = lambda: qsa_score(q, kq, ksc, pos0, sc, ws)
        for _ in range(3):
            fn()
        t = _device_times(stream, fn, n, flush)
        ms = sum(t) / len(t)
        pairs = score_pairs(T, pos0)
        # bytes: the fp32 queries read by the head-sum pass and its hi/lo rows
        # written, then the score kernel's own bytes
        nb = T * HQ * D * 4 + (-(-T // 64) * 64) * (2 * D * 2 + 4) + score_bytes(T, pos0, C)
        ex = score_flops_executed(T, pos0)
        sweep.append({"pos0": pos0, "cells": C, "pairs": pairs, "us": 1e3 * ms, "tokens_per_s": T / (ms / 1e3),
                      "algorithmic_bytes": nb, "gbs": nb / (ms / 1e3) / 1e9,
                      "frac_of_hbm_peak": nb / (ms / 1e3) / 1e9 / hbm,
                      "tensor_tflops_executed": ex / (ms / 1e3) / 1e12,
                      "frac_of_f16_peak_executed": ex / (ms / 1e3) / 1e12 / tc,
                      "tflops_head_summed_method": 2 * D * pairs / (ms / 1e3) / 1e12})
        del sc
    out["4_score_sweep"] = sweep

    # The selection over the long-context scores (fp32 queries N(0,1) against
    # the workload's key cache), then the attention at the pages' own shape.
    w = wl.PROMPT_LONG
    T, pos0, C = w.ntok, w.pos0, w.cells
    cache = wl.make_cache(C, seed=5)
    kq, ksc = to(cache.kq), to(cache.ksc)
    sc = torch.empty((T, C), dtype=torch.float32, device=dev)
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device=dev)
    qsa_score(to(wl.queries_f32(T, seed=5)), kq, ksc, pos0, sc, ws)
    ids = torch.empty((T, WIDTH), dtype=torch.int32, device=dev)
    fn = lambda: qsa_select(sc, pos0, ids)
    for _ in range(3):
        fn()
    t = _device_times(stream, fn, n, flush)
    ms = sum(t) / len(t)
    nb = select_bytes(T, pos0)
    out["5_selection"] = {"workload": f"qsa_select over the scores of T={T}, pos0={pos0} (budget {WIDTH}: 64 sink + "
                                      "256 local + current + best free cells)",
                          "us": 1e3 * ms, "tokens_per_s": T / (ms / 1e3), "algorithmic_bytes": nb,
                          "gbs": nb / (ms / 1e3) / 1e9, "frac_of_hbm_peak": nb / (ms / 1e3) / 1e9 / hbm}
    del sc, ws, ids
    hq, hkv, d, grp = wl.PAGES_Q_HEADS, wl.PAGES_KV_HEADS, wl.PAGES_HEAD_DIM, wl.PAGES_GROUP
    cache = wl.make_cache(C, seed=wl.PAGES_SEED, head_dim=d, group=grp, kv_heads=hkv)
    kq, vq, ksc, vsc = (to(x) for x in (cache.kq, cache.vq, cache.ksc, cache.vsc))
    q = to(wl.queries_f16(T, seed=wl.PAGES_SEED, heads=hq, head_dim=d))
    ids_np = wl.even_ids(T, pos0, WIDTH)
    ids = to(ids_np)
    o = torch.empty((T, hq, d), dtype=torch.float16, device=dev)
    fn = lambda: qsa_attn(q, kq, vq, ksc, vsc, ids, o, wl.PAGES_SCALE)
    for _ in range(3):
        fn()
    t = _device_times(stream, fn, max(n // 4, 10), flush)
    ms = sum(t) / len(t)
    ab, valid = attn_bytes(ids_np, T, hkv=hkv, hq=hq, d=d)
    out["6_pages_shape"] = {"workload": f"attention at the pages' shape: {hkv} KV heads x {hq} query heads, "
                                        f"head_dim {d}, per-{grp} scales, T={T}, pos0={pos0}, {WIDTH} evenly spaced ids",
                            "us": 1e3 * ms, "tokens_per_s": T / (ms / 1e3), "valid_cells": valid,
                            "algorithmic_bytes": ab, "logical_gbs": ab / (ms / 1e3) / 1e9,
                            "frac_of_hbm_peak": ab / (ms / 1e3) / 1e9 / hbm}

    # Prep on the long-context tokens, with and without the key rotation.
    inp = wl.prep_inputs(T, seed=5)
    qi, ki, vi, nw = (to(x) for x in (inp.q_in, inp.k_in, inp.v_in, inp.norm_w))
    cache = wl.make_cache(C, seed=5)
    kq, vq, ksc, vsc = (to(x) for x in (cache.kq, cache.vq, cache.ksc, cache.vsc))
    q16 = torch.empty((T, HQ, D), dtype=torch.float16, device=dev)
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device=dev)
    rec = {"workload": f"qsa_prep of T={T} tokens at pos0={pos0} (12 query rows, one K and one V row each; "
                       "the score's head sum written too)", "algorithmic_bytes": prep_bytes(T)}
    for name, rk in (("plain", False), ("rope_k", True)):
        fn = lambda: qsa_prep(qi, ki, vi, nw, pos0, kq, vq, ksc, vsc, q16, rope_k=rk, qbar_out=ws)
        for _ in range(3):
            fn()
        t = _device_times(stream, fn, n, flush)
        ms = sum(t) / len(t)
        rec[name] = {"us": 1e3 * ms, "gbs": prep_bytes(T) / (ms / 1e3) / 1e9,
                     "frac_of_hbm_peak": prep_bytes(T) / (ms / 1e3) / 1e9 / hbm}
    out["7_prep"] = rec
    return out


def run_pages(args, rank, world, local_rank):
    """The attention alone at the pages' shape: 2 KV heads x 12 query heads,
    head_dim 256, per-64 scales, softmax scale 1/16, on the same tokens and
    evenly spaced ids as the default step; L2 flushed between launches."""
    import numpy as np
    import torch

    from sparse_selected_attention_gb300 import qsa_attn
    from sparse_selected_attention_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    T, pos0 = args.ntok, args.pos0
    hq, hkv, d, grp = wl.PAGES_Q_HEADS, wl.PAGES_KV_HEADS, wl.PAGES_HEAD_DIM, wl.PAGES_GROUP
    cache = wl.make_cache(pos0 + T, seed=wl.PAGES_SEED + rank, head_dim=d, group=grp, kv_heads=hkv)
    ids_np = wl.even_ids(T, pos0, WIDTH)

    def to(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    kq, vq, ksc, vsc = to(cache.kq), to(cache.vq), to(cache.ksc), to(cache.vsc)
    q = to(wl.queries_f16(T, seed=wl.PAGES_SEED + rank, heads=hq, head_dim=d))
    ids = to(ids_np)
    out = torch.empty((T, hq, d), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        qsa_attn(q, kq, vq, ksc, vsc, ids, out, wl.PAGES_SCALE)
    torch.cuda.synchronize()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for k in range(K):
        flush.zero_()
        evs[k][0].record(stream)
        qsa_attn(q, kq, vq, ksc, vsc, ids, out, wl.PAGES_SCALE)
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / K, dev)
    ab, valid = attn_bytes(ids_np, T, hkv=hkv, hq=hq, d=d)
    peak, peak_src = peaks()
    achieved = ab / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": None, "kernel": "attn (pages' shape)", "peak_source": peak_src,
            "algorithmic_bytes_per_launch": ab, "avg_launch_ms": ms}
    return {"ms": ms, "clocks": clocks, "roofline": roof, "valid_cells": valid}


def run_decode(args, rank, world, local_rank):
    """Per-call device time of qsa_attn on the two decode windows, L2
    flushed before each call; median over the calls."""
    import numpy as np
    import torch

    from sparse_selected_attention_gb300 import qsa_attn
    from sparse_selected_attention_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for name, w in (("tiny", wl.TINY_DECODE), ("mtp", wl.MTP_DECODE)):
        cache = wl.make_cache(w.cells, seed=w.seed + rank)

        def to(x):
            return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

        kq, vq, ksc, vsc = to(cache.kq), to(cache.vq), to(cache.ksc), to(cache.vsc)
        q = to(wl.queries_f16(w.ntok, seed=w.seed + rank))
        ids_np = w.make_ids()
        ids = to(ids_np)
        out = torch.empty((w.ntok, HQ, D), dtype=torch.float16, device=dev)
        for _ in range(args.warmup):
            qsa_attn(q, kq, vq, ksc, vsc, ids, out)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for k in range(args.steps):
            flush.zero_()
            evs[k][0].record(stream)
            qsa_attn(q, kq, vq, ksc, vsc, ids, out)
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) for a, b in evs)
        ab, valid = attn_bytes(ids_np, w.ntok)
        res[name] = {"workload": w.name, "us_median": 1e3 * t[len(t) // 2], "us_mean": 1e3 * sum(t) / len(t),
                     "tokens_per_s": w.ntok / (t[len(t) // 2] / 1e3), "valid_cells": valid,
                     "algorithmic_bytes": ab}
    res["clocks"] = sampler.stop()
    return res


def run_score_sweep(args, rank, world, local_rank):
    """qsa_score from fp32 queries N(0,1) [T, 12, 128] (its own head-sum pass
    plus the score kernel) at each pos0 of the sweep; L2 flushed before each
    call; mean device time per call."""
    import numpy as np
    import torch

    from sparse_selected_attention_gb300 import qsa_score, qsa_score_workspace_bytes
    from sparse_selected_attention_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peak, peak_src = peaks()
    T = args.ntok
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    out = []
    for pos0 in wl.SCORE_POS0:
        C = pos0 + T
        cache = wl.make_cache(C, seed=5 + rank)

        def to(x):
            return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

        kq, ksc = to(cache.kq), to(cache.ksc)
        q = to(wl.queries_f32(T, seed=5 + rank))
        scores = torch.empty((T, C), dtype=torch.float32, device=dev)
        ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            qsa_score(q, kq, ksc, pos0, scores, ws)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for k in range(args.steps):
            flush.zero_()
            evs[k][0].record(stream)
            qsa_score(q, kq, ksc, pos0, scores, ws)
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
        pairs = score_pairs(T, pos0)
        # bytes: fp32 queries read by the head-sum pass and its fp16 hi/lo rows,
        # then the score kernel's bytes
        nb = T * HQ * D * 4 + 2 * (-(-T // 64) * 64) * 2 * D * 2 + score_bytes(T, pos0, C)
        out.append({"pos0": pos0, "cells": C, "pairs": pairs, "us": 1e3 * ms,
                    "gbs": nb / (ms / 1e3) / 1e9, "frac_hbm": nb / (ms / 1e3) / 1e9 / peak,
                    "tflops_algorithmic_12_heads": 2 * HQ * D * pairs / (ms / 1e3) / 1e12,
                    "tflops_executed_head_sum_hi_lo": 2 * 2 * D * pairs / (ms / 1e3) / 1e12})
    return {"sweep": out, "clocks": sampler.stop(), "peak": peak, "peak_source": peak_src}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    config = {"workload": WORKLOAD_SELECT if args.select else WORKLOAD, "ntok": args.ntok, "pos0": args.pos0, "cache_cells": args.pos0 + args.ntok,
              "width": WIDTH, "heads": "12 query / 1 KV", "head_dim": D,
              "l2": "flushed between steps (256 MiB write), flush outside the step events",
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        # The oracle on every host core; each step is a bounded sample of the
        # workload's token rows, sized so that the whole run takes about two
        # and a half minutes at most.
        pool = OraclePool(os.cpu_count() or 1)
        try:
            n, dt = pool.run(pool.rows(pool.cores), pool.cores)
            budget = min(5.0, 150.0 / max(1, args.steps + args.warmup))
            nrows = int(max(pool.cores, min(NTOK, budget * n / dt)))
            for w in range(args.warmup):
                pool.run(pool.rows(nrows, offset=w), pool.cores)
            walls = [pool.run(pool.rows(nrows, offset=args.warmup + k), pool.cores)[1] for k in range(args.steps)]
        finally:
            pool.close()
        ms = 1e3 * sum(walls) / len(walls)
        value = nrows / (ms / 1e3)
        config["sample"] = (f"each step: {nrows} of the {NTOK} token rows, evenly spaced (offset by the step), "
                            f"on {pool.cores} single-threaded oracle processes")
        cb = {"value": value, "unit": UNIT, "cores": pool.cores, "kind": "oracle", "sample": config["sample"]}
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": cb,
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.pages_shape:
        res = run_pages(args, rank, world, local_rank)
        if rank == 0:
            config["workload"] = ("attention alone at the pages' shape: T=%d query tokens at pos0=%d, 2 KV heads x "
                                  "12 query heads, head_dim 256, fp16 per-64 scales, softmax scale 1/16, int8 K/V "
                                  "cache of %d cells, %d evenly spaced causal ids per token"
                                  % (args.ntok, args.pos0, args.pos0 + args.ntok, WIDTH))
            config["heads"] = "24 query / 2 KV"
            config["head_dim"] = 256
            line = {"metric": METRIC, "value": weak_scaling_value(args.ntok, world, res["ms"]), "unit": UNIT,
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                    "data": "synthetic", "config": config, "roofline": res["roofline"], "clocks": res["clocks"],
                    "gpu_launches": args.steps, "valid_cells": res["valid_cells"]}
            print(json.dumps(line), flush=True)
        return
    if args.score_sweep:
        res = run_score_sweep(args, rank, world, local_rank)
        if rank == 0:
            last = res["sweep"][-1]
            config["workload"] = ("score pass sweep: fp32 queries N(0,1) [%d, 12, 128] against the int8 key cache, "
                                  "pos0 in (0, 2048, 8192, 30000), every causal cell" % args.ntok)
            config["l2"] = "flushed before every call (256 MiB write), outside the call's events"
            line = {"metric": "score pass throughput (query tokens/s) at pos0=30000; the sweep in 'sweep'",
                    "value": args.ntok / (last["us"] / 1e6), "unit": "tokens/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": last["us"] / 1e3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                    "data": "synthetic", "config": config, "sweep": res["sweep"],
                    "roofline": {"bound": "hbm", "achieved": last["gbs"], "peak": res["peak"], "unit": "GB/s",
                                 "frac": last["frac_hbm"], "traffic": None, "kernel": "score (pos0=30000)",
                                 "peak_source": res["peak_source"]},
                    "clocks": res["clocks"], "gpu_launches": 2 * args.steps * len(res["sweep"])}
            print(json.dumps(line), flush=True)
        return
    if args.decode:
        res = run_decode(args, rank, world, local_rank)
        if rank == 0:
            config["workload"] = res["mtp"]["workload"] + "; also " + res["tiny"]["workload"]
            config.update(ntok=8, pos0=30000, cache_cells=30008, width=384,
                          l2="flushed before every call (256 MiB write), outside the call's events")
            line = {"metric": "decode attention latency (device time per qsa_attn call)",
                    "value": res["mtp"]["us_median"], "unit": "us", "n_gpus": world, "steps": args.steps,
                    "warmup": args.warmup, "ms_per_step": res["mtp"]["us_median"] / 1e3,
                    "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                    "data": "synthetic", "config": config, "decode": {k: res[k] for k in ("mtp", "tiny")},
                    "clocks": res["clocks"], "gpu_launches": 2 * args.steps}
            print(json.dumps(line), flush=True)
        return
    res = run_ours(args, rank, world, local_rank)
    cfg = None
    if not args.no_configs and args.ntok == NTOK and args.pos0 == POS0:
        import torch
        cfg = run_configs(torch.device("cuda", local_rank), max(20, min(args.steps, 200)))
    if rank != 0:
        return
    cb = None
    if not args.no_cpu_baseline:
        cb = cpu_baseline(args.cpu_sample_seconds)
    line = {"metric": METRIC, "value": weak_scaling_value(args.ntok, world, res["ms"]), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "precision": "int8 K/V codes with fp16 scales; fp16 tensor-core operands, fp32 accumulation; "
                         "fp32 prep and scores; fp16 attention output",
            "data": "synthetic", "config": config, "roofline": res["roofline"], "cpu_baseline": cb,
            "e2e": res["e2e"], "clocks": res["clocks"], "gpu_launches": res["launches_per_step"] * args.steps,
            "kernels": res["kernels"], "configs": cfg}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
