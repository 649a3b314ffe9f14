#!/usr/bin/env python3
"""Benchmark of physically sparse QSA decode on GB300.

Workload: the long-context decode batch -- 8 independent queries, each with
262,144 visible tokens (65,536 complete four-token groups), budget 512
groups, indexer 8 heads x 64, GQA attention 16 query / 2 KV heads x 128, all
values N(0,1), K/V in a wrapped ring buffer (slot = (t + 131,072) mod
262,144).  One step = one pass of the whole hot path over the batch: group
scoring, set choice + chronological emission, slot resolution + compact
gather, online-softmax attention -- one qsa_decode call (three launches:
scoring, selection, fused gather + attention), bracketed by CUDA events.
Per-kernel durations come from a second pass through qsa_decode_profiled,
which records an event before each of the three launches and after the last.

Timing: W untimed warm-up steps, then K timed steps.  Before each timed step
L2 is flushed (a 256 MiB buffer written, then another 256 MiB read), outside
the events; the step time is the device time between the events around its
three launches.  Under torchrun every rank runs its own batch (weak scaling,
no collective on the data path) and the slowest rank's time counts.

Prints one JSON line.  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QSA decode queries/sec at 262,144 visible tokens; achieved HBM GB/s vs peak"
UNIT = "queries/s"
WORKLOAD = "long_262144"
FLUSH_BYTES = 256 << 20
PROFILE = os.path.join(ROOT, "profiles", "score_groups_long_262144.md")
SCORE_SRC = os.path.join(ROOT, "top_group_sparse_gb300", "csrc", "score.cu")
ATTEND_PROFILE = os.path.join(ROOT, "profiles", "attend_long_262144.md")
ATTEND_SRC = os.path.join(ROOT, "top_group_sparse_gb300", "csrc", "attend.cu")
ATTEND_BATCHED_PROFILE = os.path.join(ROOT, "profiles", "attend_batched_65537.md")
SHARED_PROFILE = os.path.join(ROOT, "profiles", "score_shared_chunked_prefill_100000.md")
SCORE_BATCHED_PROFILE = os.path.join(ROOT, "profiles", "score_groups_batched_65537.md")
SHARED_SRC = os.path.join(ROOT, "top_group_sparse_gb300", "csrc", "score_shared.cu")


def config_dict(w):
    return {
        "workload": WORKLOAD,
        "batch_per_gpu": int(w.batch),
        "visible_tokens": int(w.visible[0]),
        "budget_groups": int(w.budget),
        "indexer": f"{w.idx_heads} heads x {w.idx_dim}",
        "attention": f"{w.q_heads} q / {w.kv_heads} kv heads x {w.head_dim}",
        "slot_map": "ring buffer wrapped once: slot = (t + 131072) mod 262144",
        "values": "N(0,1) float32, seeded",
        "l2": "flushed before every timed step (256 MiB written, then 256 MiB read)",
    }


def algorithmic_bytes(w):
    """Bytes the method must move per step: the whole path (raw index keys,
    selected K and V rows, their slot-map entries, indexer and attention
    queries, output) and the scorer's own share (raw keys + indexer query;
    the scores it writes are an intermediate, as is any scratch)."""
    per_q, scorer = [], 0
    for b in range(w.batch):
        T = int(w.visible[b])
        G = T // 4
        Wb = 4 * min(G, w.budget) + T % 4
        per_q.append(T * w.idx_dim * 4 + Wb * w.kv_heads * w.head_dim * 4 * 2 + Wb * 4 +
                     w.idx_heads * w.idx_dim * 4 + 2 * w.q_heads * w.head_dim * 4)
        scorer += T * w.idx_dim * 4 + w.idx_heads * w.idx_dim * 4
    return sum(per_q), scorer


def attend_bytes(w):
    """Algorithmic bytes of the fused gather + attention launch: the selected
    K and V rows and their slot-map entries, the attention queries and the
    output."""
    total = 0
    for b in range(w.batch):
        T = int(w.visible[b])
        Wb = 4 * min(T // 4, w.budget) + T % 4
        total += Wb * (w.kv_heads * w.head_dim * 4 * 2 + 4) + 2 * w.q_heads * w.head_dim * 4
    return total


def attend_fma(w):
    """Multiply-adds of the attention: every selected row, every query head,
    q.k and p.v over the head width."""
    rows = sum(4 * min(int(T) // 4, w.budget) + int(T) % 4 for T in w.visible)
    return rows * w.q_heads * w.head_dim * 2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def ffma_peak(stream):
    """Binary32 FFMA rate of this GPU from the library's probe
    (qsa_probe_ffma): best of 5 event-timed launches after 2 warm-ups."""
    import torch
    from top_group_sparse_gb300 import qsa
    bps, iters = 4, 256
    sink = torch.zeros(1 << 14, dtype=torch.float32, device="cuda")
    best = float("inf")
    n_fma = 0
    for r in range(7):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n_fma = qsa.qsa_probe_ffma(bps, iters, sink, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if r >= 2:
            best = min(best, e0.elapsed_time(e1) * 1e-3)
    return {"tflops": 2 * n_fma / best / 1e12,
            "how": f"qsa_probe_ffma, {bps} x 256 threads per SM, 8 chains x {16 * iters} FMAs per thread, "
                   "best of 5 launches"}


def profile_traffic(profile=PROFILE, src=SCORE_SRC):
    """Per-launch DRAM bytes of a kernel at the benchmark's batch from its
    committed ncu summary (`traffic_bytes_per_launch`), or None if the summary
    is missing or was taken on a different source of the kernel (its
    `<file>_sha256` line)."""
    if not os.path.exists(profile):
        return None
    text = open(profile).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    key = os.path.basename(src).replace(".", "_") + "_sha256"
    h = re.search(key + r":\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return int(m.group(1)) if cur == h.group(1) else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle, as it stands, on the host cores (rank 0 only)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from top_group_sparse_gb300 import workloads as wl
    w = wl.long_262144(batch=args.batch)
    n_thr = oracle.threads(os.cpu_count() or 1)  # every host core (1 if built without OpenMP)
    t0 = time.perf_counter()
    oracle.decode(w, queries=[0])
    per_query = time.perf_counter() - t0
    budget_s = 150.0
    per_step = max(1, min(w.batch, int(budget_s / max(args.steps + args.warmup, 1) / per_query)))
    queries = list(range(per_step))
    for _ in range(args.warmup):
        oracle.decode(w, queries=queries)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(w, queries=queries)
    dt = time.perf_counter() - t0
    value = args.steps * per_step / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_thr, "kind": "oracle",
                         "sample": f"{per_step} of the {w.batch} queries of the batch per step, "
                                   f"plain C oracle on {n_thr} host threads (OpenMP over queries, "
                                   f"groups and heads; results identical to one thread)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

class Timer:
    """Device timing of one path on one stream: before each call L2 is
    flushed (FLUSH_BYTES written, then FLUSH_BYTES read, outside the events),
    then the call is bracketed by CUDA events recorded on that stream; the
    events are created before timing and the launches queue behind a short
    device-side sleep, so host launch overhead is not timed."""

    def __init__(self, device, stream):
        import torch
        self.torch = torch
        self.stream = stream
        self.flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.zeros(1, dtype=torch.float32, device=device)

    def flush(self):
        self.flush_w.zero_()
        self.torch.sum(self.flush_r, dim=0, out=self.sink[0])

    def events(self, n, per):
        torch = self.torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(per)] for _ in range(n)]
        for ev in evs:
            for e in ev:
                e.record(self.stream)
        torch.cuda.synchronize()
        return evs

    def warm(self, fn, n):
        for _ in range(n):
            self.flush()
            fn(self.stream)
        self.torch.cuda.synchronize()

    def run(self, fn, n):
        """Per-call device times (ms) of n calls of fn(stream)."""
        evs = self.events(n, 2)
        self.torch.cuda._sleep(20_000_000)  # let the launches queue ahead of the device
        for ev in evs:
            self.flush()
            ev[0].record(self.stream)
            fn(self.stream)
            ev[1].record(self.stream)
        self.torch.cuda.synchronize()
        return np.array([e[0].elapsed_time(e[1]) for e in evs])

    def stages(self, db, n):
        """Per-launch times (ms: scorer, selection, gather + attention) of n
        qsa_decode_profiled calls (events between the three launches; this
        form gives up the overlap of launch latencies, so its sum is a little
        above the plain step)."""
        evs = self.events(n, 4)
        self.torch.cuda._sleep(20_000_000)
        for ev in evs:
            self.flush()
            db.decode_profiled(ev, self.stream)
        self.torch.cuda.synchronize()
        return np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs])


def hbm_roofline(kernel, nbytes, ms, peak, peak_src, traffic=None, note=""):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
            "frac": gbs / peak, "traffic": traffic, "us_per_launch": ms * 1e3, "bytes_per_launch": int(nbytes),
            "note": (note + "; " if note else "") + f"peak = {peak_src} HBM copy bandwidth"}


def time_oracle(w, queries, n_threads, min_thread_s=10.0, max_s=12.0):
    """The CPU oracle, as it stands, on n_threads host threads over the given
    queries: passes repeat until about min_thread_s of host-thread time (at
    least 4 passes, at most ~max_s of wall time)."""
    import oracle
    n = oracle.threads(n_threads)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.decode(w, queries=queries)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= 4 and (el * n >= min_thread_s or el >= max_s):
            break
    dt = time.perf_counter() - t0
    return {"value": reps * len(queries) / dt, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{reps} pass(es) over {len(queries)} of the {w.batch} queries of the {w.name} "
                      f"workload, plain C oracle on {n} host thread(s), {dt:.1f} s"}


def oracle_pair(w, queries):
    """The oracle on every host core (OpenMP over queries, groups and heads:
    results identical to one thread) and on one thread."""
    return time_oracle(w, queries, os.cpu_count() or 1), time_oracle(w, queries, 1)


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    if args.gpus != ws and ws > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {ws}")
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    from top_group_sparse_gb300 import build, qsa
    from top_group_sparse_gb300 import workloads as wl
    from top_group_sparse_gb300.sharding import max_over_ranks
    if local == 0:  # one build per node: the ranks share the in-tree library
        build.build()
    barrier()
    qsa.load()

    w = wl.long_262144(seed=4 + 1000 * rank, batch=args.batch)
    db = qsa.DeviceBatch(w, device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    dev = db.out.device
    tm = Timer(dev, stream)
    peak, peak_src = measured_peaks()
    solo = ws == 1 and not args.no_cpu_baseline  # the oracle timings run at N=1 only

    # quick parity sample before timing: query 0's row against the oracle
    db.decode()
    st, flags = db.check_errors()
    if st != 0:
        raise SystemExit(f"device error word {flags:#x}")
    parity = None
    if rank == 0 and not args.no_parity:
        import oracle
        ref = oracle.decode(w, queries=[0])
        n = int(ref["n_ids"][0])
        ids_ok = int(db.n_ids[0]) == n and db.ids[0, :n].cpu().numpy().tobytes() == ref["ids"][0, :n].tobytes()
        slots = w.slot_map[w.slot_offset[0] + ref["ids"][0, :n]]
        err = float(np.abs(db.out[0].cpu().numpy() - ref["out"][0]).max() / np.abs(w.v_cache[slots]).max())
        parity = {"query": 0, "ids_bit_exact": bool(ids_ok), "attn_err_rel_max_v": err}
        if not ids_ok or err > 1e-5:
            raise SystemExit(f"parity check failed: {parity}")

    def step(s):  # one qsa_decode call: the whole path over the batch
        db.decode(s)

    tm.warm(step, args.warmup)
    K = args.steps
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        step_ms = tm.run(step, K)
        barrier()
        loop_wall = time.perf_counter() - t0
    st, flags = db.check_errors()
    if st != 0:
        raise SystemExit(f"device error word {flags:#x} after the timed loop")
    total_ms = max_over_ranks(float(step_ms.sum()), dev)
    ms_per_step = total_ms / K
    value = ws * w.batch * K / (total_ms / 1e3)

    # per-kernel durations: the same steps through qsa_decode_profiled
    stage_mean = tm.stages(db, max(1, min(K, 500))).mean(axis=0)

    # ---- the incremental form: the scorer reads a pooled-key cache -------------
    # A decode step of this form appends the group its new token completes (one
    # per query here: the most a step can add) and runs qsa_decode_pooled.  The
    # cache itself (G pooled keys per query) is built once, before timing.
    db.make_pooled_cache()
    db.pool_all()
    G_all = (w.visible // 4).astype(np.int32)
    gb_t = torch.from_numpy(np.maximum(G_all - 1, 0)).to(dev)
    ge_t = torch.from_numpy(G_all).to(dev)

    def inc_step(s):
        qsa.qsa_pool_groups(db.dims, db.inputs, gb_t, ge_t, 1, db.pooled, db.pool_offset, db.ws, s)
        db.decode_pooled(s)

    tm.warm(inc_step, args.warmup)
    K4 = max(1, min(K, 500))
    inc_ms = max_over_ranks(float(tm.run(inc_step, K4).sum()), dev)
    st, flags = db.check_errors()
    if st != 0:
        raise SystemExit(f"device error word {flags:#x} in the incremental loop")
    inc_value = ws * w.batch * K4 / (inc_ms / 1e3)
    del db.pooled

    # ---- end to end through qsa_decode with host buffers -----------------------
    # Every step copies its own inputs (indexer queries, attention queries,
    # visible lengths, history offsets: one pinned buffer) in, runs qsa_decode,
    # whose last kernel stores the step's ID rows, counts and outputs into
    # another pinned buffer, and the host waits for that step's completion
    # event before it reads them.  Two steps are in flight, as in a serving
    # loop: step k+1's inputs are copied in on a copy stream (into its own
    # device buffer) while step k's kernels run, and the host waits for step
    # k while step k+1 is already queued.  K/V caches and index-key history
    # stay resident.
    K2 = max(1, min(K, args.e2e_steps))
    slot_bufs = [(db.step_in, db.inputs), db.step_slot()]
    host_bufs = [db.step_host_buffers() for _ in slot_bufs]
    h2d = host_bufs[0][0].numel() * host_bufs[0][0].element_size()
    d2h = host_bufs[0][1].numel() * host_bufs[0][1].element_size()
    copy_stream = torch.cuda.Stream()
    ev_copied = [torch.cuda.Event() for _ in slot_bufs]
    ev_done = [torch.cuda.Event() for _ in slot_bufs]
    for e in ev_done:
        e.record(stream)
    outs = [db.host_outputs(h_out) for _, h_out in host_bufs]

    def launch(k):
        i = k % len(slot_bufs)
        buf, inp = slot_bufs[i]
        h_in, _ = host_bufs[i]
        copy_stream.wait_event(ev_done[i])  # the kernels that last read this buffer are done
        with torch.cuda.stream(copy_stream):
            buf.copy_(h_in, non_blocking=True)
        ev_copied[i].record(copy_stream)
        stream.wait_event(ev_copied[i])
        hi, hn, ho = outs[i]
        qsa.qsa_decode(db.dims, inp, hi, hn, ho, db.ws, stream)
        ev_done[i].record(stream)

    def e2e_run(n):
        launch(0)
        for k in range(1, n):
            launch(k)
            ev_done[(k - 1) % len(slot_bufs)].synchronize()  # step k-1's results are on the host
        ev_done[(n - 1) % len(slot_bufs)].synchronize()

    e2e_run(6)
    first = outs[0][2].clone()
    barrier()
    t0 = time.perf_counter()
    e2e_run(K2)
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    e2e_value = ws * w.batch * K2 / e2e_s
    e2e_mode = "two steps in flight (inputs copied on a copy stream while the previous step runs), eager launches"
    if not (torch.equal(outs[0][2], first) and torch.equal(outs[1][2], first)):
        raise SystemExit("end-to-end outputs differ from step to step")
    torch.cuda.synchronize()

    # ---- rooflines of the benchmark workload -------------------------------------
    path_bytes, scorer_bytes = algorithmic_bytes(w)
    path_gbs = path_bytes / (ms_per_step * 1e-3) / 1e9
    G_q = int(w.visible[0]) // 4
    inc_bytes = path_bytes - w.batch * (int(w.visible[0]) - G_q) * w.idx_dim * 4 + w.batch * 5 * w.idx_dim * 4
    roof = hbm_roofline("score_groups", scorer_bytes, stage_mean[0], peak, peak_src,
                        profile_traffic() if args.batch == 8 else None,
                        f"algorithmic bytes {scorer_bytes} per launch (raw index keys + indexer queries; "
                        "the scores written are an intermediate)")
    roof_attend = hbm_roofline("attend_kernel (fused slot resolution, K/V gather and online softmax)",
                               attend_bytes(w), stage_mean[2], peak, peak_src,
                               profile_traffic(ATTEND_PROFILE, ATTEND_SRC) if args.batch == 8 else None,
                               "selected K/V rows + slot entries + queries + outputs per launch; the time is "
                               "the gather + attention stage of qsa_decode_profiled, its launch gap included")

    # ---- the batched decode: 32 queries x 65,537 visible tokens ------------------
    batched = None
    if not args.no_batched:
        w3 = wl.batched_65537(batch=args.batched_queries)
        d3 = qsa.DeviceBatch(w3, device=f"cuda:{local}")

        def step3(s):
            d3.decode(s)

        tm.warm(step3, args.warmup)
        K3 = max(1, min(K, 300))
        ms3 = max_over_ranks(float(tm.run(step3, K3).sum()), dev) / K3
        st3 = tm.stages(d3, max(1, min(K3, 200))).mean(axis=0)
        st, flags = d3.check_errors()
        if st != 0:
            raise SystemExit(f"device error word {flags:#x} in the batched loop")
        p3, s3 = algorithmic_bytes(w3)
        batched = {
            "workload": "batched_65537", "queries_per_step": w3.batch, "visible_tokens": int(w3.visible[0]),
            "value": ws * w3.batch / (ms3 * 1e-3), "unit": UNIT, "ms_per_step": ms3, "steps": K3,
            "roofline": hbm_roofline("score_groups", s3, st3[0], peak, peak_src,
                                     profile_traffic(SCORE_BATCHED_PROFILE) if w3.batch == 32 else None,
                                     f"algorithmic bytes {s3} per launch (raw index keys + indexer queries)"),
            "roofline_attend": hbm_roofline("attend_kernel", attend_bytes(w3), st3[2], peak, peak_src,
                                            profile_traffic(ATTEND_BATCHED_PROFILE, ATTEND_SRC)
                                            if w3.batch == 32 else None,
                                            "selected K/V rows + slot entries + queries + outputs"),
            "path_hbm": {"achieved_gbs": p3 / (ms3 * 1e-3) / 1e9, "frac_of_measured": p3 / (ms3 * 1e-3) / 1e9 / peak,
                         "frac_of_8tbs": p3 / (ms3 * 1e-3) / 1e9 / 8000.0, "algorithmic_bytes_per_step": p3},
            "stages_us": {n: float(v * 1e3) for n, v in zip(("score", "select", "gather_attend"), st3)},
            "note": "32 independent histories of 65,537 tokens (16,384 groups + 1 tail token each), 16-token "
                    "pages in a random permutation; one qsa_decode call per step, L2 flushed before each step"}
        if solo and rank == 0:
            batched["cpu_baseline"], batched["cpu_baseline_1thread"] = oracle_pair(w3, list(range(w3.batch)))
        del d3, w3

    # ---- chunked prefill: 256 queries over one history, shared vs per query -----
    chunk = None
    if not args.no_chunked:
        wc = wl.chunked_prefill_100000()
        dc = qsa.DeviceBatch(wc, device=f"cuda:{local}")

        def time_path(fn, n=50):  # ms per launch, the slowest rank's
            tm.warm(fn, 3)
            return max_over_ranks(float(tm.run(fn, n).mean()), dev)

        ms_shared = time_path(dc.decode_shared)
        ms_single = time_path(dc.decode)
        ms_scorer_shared = time_path(dc.score_shared)
        ms_scorer_single = time_path(dc.score)
        stc = tm.stages(dc, 30).mean(axis=0)
        st, flags = dc.check_errors()
        if st != 0:
            raise SystemExit(f"device error word {flags:#x} in the chunked-prefill loop")
        # This workload is FFMA-bound (one key history, 256 queries): its
        # roofline denominator is the FFMA rate measured here by the library's
        # probe, beside the HBM one.
        ffma = ffma_peak(stream)
        Gs = wc.visible // 4
        fma_score = int(np.sum(Gs.astype(np.int64)) * wc.idx_heads * wc.idx_dim)
        fma_attend = attend_fma(wc)
        key_bytes = int(wc.visible.max()) * wc.idx_dim * 4  # the shared history, streamed once

        def alu_roofline(kernel, ms, traffic=None):
            tf = 2 * fma_score / (ms * 1e-3) / 1e12
            return {"kernel": kernel, "bound": "alu", "achieved": tf, "peak": ffma["tflops"], "unit": "TFLOP/s",
                    "frac": tf / ffma["tflops"], "traffic": traffic, "us_per_launch": ms * 1e3,
                    "fma_per_launch": fma_score, "peak_source": "measured in this run: " + ffma["how"],
                    "hbm_frac": key_bytes / (ms * 1e-3) / 1e9 / peak}

        cpu_c = None
        if solo and rank == 0:
            cpu_c = oracle_pair(wc, list(range(wc.batch)))
        shared = {"value": ws * wc.batch / (ms_shared * 1e-3), "unit": UNIT, "ms_per_step": ms_shared,
                  "roofline": alu_roofline("score_shared_kernel (qsa_score_groups_shared)", ms_scorer_shared,
                                           profile_traffic(SHARED_PROFILE, SHARED_SRC)),
                  "step_fma": fma_score + fma_attend,
                  "step_frac": 2 * (fma_score + fma_attend) / (ms_shared * 1e-3) / 1e12 / ffma["tflops"]}
        per_query = {"value": ws * wc.batch / (ms_single * 1e-3), "unit": UNIT, "ms_per_step": ms_single,
                     "roofline": alu_roofline("score_groups_kernel (qsa_score_groups; each query streams "
                                              "its own keys, mostly from L2)", ms_scorer_single),
                     "roofline_attend": hbm_roofline("attend_kernel", attend_bytes(wc), stc[2], peak, peak_src,
                                                     None, "selected K/V rows (many shared between queries, so "
                                                     "read from L2) + slot entries + queries + outputs"),
                     "stages_us": {n: float(v * 1e3) for n, v in zip(("score", "select", "gather_attend"), stc)}}
        if cpu_c is not None:
            for form in (shared, per_query):
                form["cpu_baseline"], form["cpu_baseline_1thread"] = cpu_c
        chunk = {"workload": "chunked_prefill_100000", "queries_per_step": wc.batch,
                 "shared": shared, "per_query": per_query,
                 "note": "256 queries at positions 100,000..100,255 of one history: qsa_decode_shared "
                         "(each pooled tile scored for every query) vs qsa_decode (each query streams "
                         "its own keys); outputs bit-identical (tests); L2 flushed before each step"}
        del dc, wc

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    cpu = cpu_1t = None
    if solo:
        cpu, cpu_1t = oracle_pair(w, list(range(w.batch)))

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(w),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "launch": e2e_mode,
                "note": "qsa_decode per step; the step's queries, visible lengths and history offsets copied in "
                        "from a pinned host buffer, ID rows, counts and outputs stored into another pinned buffer "
                        "by the last kernel, the host waiting for each step's completion event before reading "
                        "them; two steps in flight (double-buffered inputs); K/V cache and index-key history "
                        "resident in HBM"},
        "gpu_launches": 3 * K,
        "roofline": roof,
        "roofline_attend": roof_attend,
        "path_hbm": {"achieved_gbs": path_gbs, "frac_of_measured": path_gbs / peak,
                     "frac_of_8tbs": path_gbs / 8000.0, "algorithmic_bytes_per_step": path_bytes},
        "incremental": {"value": inc_value, "unit": UNIT, "ms_per_step": inc_ms / K4, "steps": K4,
                        "algorithmic_bytes_per_step": int(inc_bytes),
                        "note": "same workload and timing, scorer reading the pooled-key cache "
                                "(G*d_I*4 bytes per query instead of T*d_I*4): one qsa_pool_groups "
                                "append of one group per query + qsa_decode_pooled per step; rows and "
                                "outputs bit-identical to the full-raw path (tests)"},
        "batched_65537": batched,
        "chunked_prefill": chunk,
        "stages_us": {n: float(v * 1e3) for n, v in zip(("score", "select", "gather_attend"), stage_mean)},
        "loop_wall_s": loop_wall,
        "parity_sample": parity,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["cpu_baseline_1thread"] = cpu_1t
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--batch", type=int, default=8,
                    help="queries per GPU (8 = the benchmark workload; smaller only for profiling)")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chunked", action="store_true", help="skip the chunked-prefill side measurement")
    ap.add_argument("--no-batched", action="store_true", help="skip the 32 x 65,537 batched-decode measurement")
    ap.add_argument("--batched-queries", type=int, default=32,
                    help="queries of the batched-decode measurement (32: the workload; fewer for small profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
