"""Decode-step benchmark of the CSA2 hot path on GB300.

One step = one decode token for every sequence of the workload through its
layer schedule (Full / Reindex / Reuse layers: FP4 write of the new token,
indexer scan + pool + Top-K, Reindex, sparse attention for every layer),
captured once as a CUDA graph and replayed.  Metric: decode queries/s
(sequences x steps / time); achieved HBM GB/s of the algorithmic bytes
against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 128k|1m|1m-fp4|128k-fp4|mix|tiny]
                  [--impl ours|reference]

N > 1 (torchrun): every rank runs its own replica of the workload (no data-
path collective), the timed region is bracketed by barriers, the max over
ranks is reported and `value` counts the queries of all ranks.
`--impl reference` times the CPU oracle (the reference arm of this build) on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode queries/s at 128K and 1M ctx; achieved HBM GB/s vs roofline"
ENTRY_B = 416            # FP4 codes 256 + E4M3 scales 32 + bf16 rope 128
IDXK_B = 128             # E4M3 indexer-K row
L2_BYTES = 129 * 1024 * 1024


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes (per sequence; see the design notes for the derivation)
# ---------------------------------------------------------------------------
def attn_layer_bytes(wl):
    """One sequence's attention layer: its Top-K entries, window, indices, and
    the queries and outputs of its q_len query tokens."""
    H, K, W, Q = wl.heads, wl.topk, wl.swa, wl.q_len
    return (K * ENTRY_B + W * 576 * 2 + Q * H * 576 * 2 + Q * H * 513 * 4 + K * 4)


def idx_row_bytes(wl):
    """Bytes of one indexer-K row: E4M3 128, fp32 4 x Di, FP4 64 + 8."""
    return {"fp8": wl.idx_dim, "fp32": 4 * wl.idx_dim, "fp4": 72}[wl.idx_k_dtype]


def idx_qw_bytes(wl):
    """Indexer query (bf16 for E4M3 / FP4 keys, fp32 otherwise) and weights."""
    return wl.idx_heads * wl.idx_dim * (4 if wl.idx_k_dtype == "fp32" else 2) + wl.idx_heads * 4


def step_bytes(wl):
    """Algorithmic HBM bytes of one decode step over the whole batch."""
    tot = 0
    idx_row, q_w = idx_row_bytes(wl), idx_qw_bytes(wl)
    for n in wl.ctx_lens:
        pool_pos = min(wl.pool_blocks * 8, n)
        for m in wl.schedule:
            tot += attn_layer_bytes(wl)
            if m == "F":
                tot += idx_row * n + q_w + wl.pool_blocks * 4 + wl.topk * 4 + 1024 + ENTRY_B
                if wl.idx_k_dtype == "fp4":
                    tot += 2 * wl.idx_dim + 72                 # the new token's indexer-key write
            elif m == "Ri":
                tot += idx_row * pool_pos + wl.pool_blocks * 4 + q_w + wl.topk * 4
    return tot


def cache_bytes(wl):
    """Bytes of the device-resident cache a step reads from: main-KV planes
    (416 B per row) and indexer keys of every sequence's context."""
    return sum(wl.ctx_lens) * (ENTRY_B + idx_row_bytes(wl))


def full_call_bytes(wl):
    idx_row, q_w = idx_row_bytes(wl), idx_qw_bytes(wl)
    return sum(idx_row * n + q_w + wl.pool_blocks * 4 + wl.topk * 4 for n in wl.ctx_lens)


def src_hash(name):
    """Hash of a kernel source's code: comments, blank lines and trailing blanks are
    left out, so that only a change of the code itself drops the stored traffic."""
    p = os.path.join(ROOT, "compressed_sparse_attention_fp4_gb300", "csrc", name)
    with open(p, encoding="utf-8") as f:
        lines = [ln.split("//", 1)[0].rstrip() for ln in f]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha1(code.encode()).hexdigest()[:12]


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while it is
    open.  The GPU is selected by its UUID (a CUDA ordinal can name another
    physical GPU when CUDA_VISIBLE_DEVICES remaps them)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.rows = []
        # raw samples go to a temporary file (removed on exit); the summary
        # goes into the JSON line
        self.path = os.path.join(tempfile.gettempdir(), f"csa2_clocks_{os.getpid()}.csv")

    def __enter__(self):
        if not self.uuid:
            return self
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.uuid}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass

    def summary(self):
        if not self.uuid or self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "gpu": self.uuid}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows), "gpu": self.uuid}


def gpu_uuid(dev) -> str | None:
    """nvidia-smi id ("GPU-<uuid>") of a torch CUDA device, if torch reports it."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_query(wl, b, kv, layers):
    """One query (sequence b) through the schedule in the CPU oracle."""
    from oracle import schedule
    from oracle import codec as oc
    f64 = lambda x: (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    from oracle import indexer_fp4 as ofp4
    fp4q = lambda x: ofp4.dequantize(*ofp4.quantize(x))                # FP4 keys: the oracle's own write
    if wl.idx_k_dtype == "fp8":
        keys = oc.e4m3_decode(kv["idx_k"])
    elif wl.idx_k_dtype == "fp4":
        keys = fp4q(f64(kv["idx_k"]))
    else:
        keys = kv["idx_k"].astype(np.float64)
    codes, scales = oc.quantize_rows(f64(kv["latent"][-1:]))          # FP4 write of the new token
    lat = np.zeros((kv["latent"].shape[0], 512))
    rope = f64(kv["rope"])
    L = []
    for li in layers:
        L.append({"q": f64(li["q"]), "swa": f64(li["swa"]), "swa_len": li["swa_len"],
                  "idx_q": (f64(li["idx_q"]) if wl.idx_k_dtype == "fp8" else fp4q(f64(li["idx_q"]))
                            if wl.idx_k_dtype == "fp4" else li["idx_q"].astype(np.float64)),
                  "idx_w": li["idx_w"].astype(np.float64)})

    class LazyLatent:
        """Dequantizes (oracle codec) only the rows attention reads."""
        def __getitem__(self, idx):
            idx = np.asarray(idx)
            c, s = oc.quantize_rows(f64(kv["latent"][idx]))
            return oc.dequantize_rows(c, s)
    return schedule.run_sequence(wl.schedule, keys, LazyLatent(), rope, L, wl.pool_blocks,
                                 wl.topk, wl.scale)


def arm_config(wl, world):
    """The workload description both arms print."""
    return {"workload": f"decode-{wl.name}", "batch": wl.batch, "q_len": wl.q_len,
            "ctx": wl.ctx_lens[0] if len(set(wl.ctx_lens)) == 1 else "mixed",
            "schedule": "".join(m[0] if m != "Ri" else "I" for m in wl.schedule),
            "l2": "flushed before every timed step (2x L2 write)",
            "parallelism": f"replicas x{world}"}


def cpu_baseline(wl, budget_s=20.0, max_queries=16):
    from compressed_sparse_attention_fp4_gb300 import synth
    cores = len(os.sched_getaffinity(0))
    done, t_cpu = 0, 0.0
    b = 0
    while done < max_queries and t_cpu < budget_s:
        kv = synth.sequence_kv_parallel(wl, b % wl.batch)
        layers = [synth.layer_inputs(wl, b % wl.batch, l) for l in range(len(wl.schedule))]
        t0 = time.perf_counter()
        oracle_query(wl, b % wl.batch, kv, layers)
        t_cpu += time.perf_counter() - t0
        done += 1
        b += 1
    qps = done / t_cpu
    return {"value": qps, "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} queries (sequences 0..{done - 1} of workload '{wl.name}', "
                      f"full schedule of {len(wl.schedule)} layers each), fp64 numpy oracle, "
                      f"{t_cpu:.1f} s of CPU time"}


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: every rank runs its own copy of the step)
# ---------------------------------------------------------------------------
def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest per-rank value (the slowest replica sets the job time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_queries_per_s(world: int, batch: int, t_step_ms: float) -> float:
    """Queries of all ranks per second: each rank decodes `batch` sequences."""
    return world * batch / (t_step_ms * 1e-3)


# ---------------------------------------------------------------------------
# per-kernel algorithmic bytes (one launch, whole batch) and in-graph timing
# ---------------------------------------------------------------------------
def kernel_bytes(wl, name):
    """Algorithmic HBM bytes of one launch of a library kernel on workload wl
    (None for the latency-bound selection kernels)."""
    idx_row = idx_row_bytes(wl)
    if name in ("indexer_scan_tc", "indexer_scan_fp4", "indexer_scan_cuda_core"):
        return sum(idx_row * n for n in wl.ctx_lens)
    if name in ("reindex_score_tc", "reindex_score_fp4", "reindex_score_cuda_core"):
        return sum(idx_row * min(wl.pool_blocks * 8, n) + wl.pool_blocks * 4 for n in wl.ctx_lens)
    if name in ("attn_cluster_tc", "attn_seq_tc", "attn_partial_tc"):
        return wl.batch * attn_layer_bytes(wl)
    if name == "fp4_quantize":
        return wl.batch * (1024 + 288)
    if name == "fp4_idx_quantize":
        return wl.batch * (2 * wl.idx_dim + 72)
    return None


def time_graph(g, flush, reps, stream):
    """Mean device time (ms) of `reps` replays of graph g, the L2 flushed
    before each (events on the launching stream, around the replay only)."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def graph_attribution(sb, flush, reps=60):
    """Where the graph-replayed step's time goes: the step's first j library
    calls are captured as their own graph (j = 1 .. all) and timed like the
    step; call j's share is t_j - t_{j-1}.  The shares add up to the whole
    step's time and keep the overlap of consecutive kernels inside a graph."""
    import torch
    from compressed_sparse_attention_fp4_gb300.step import GraphedStep, step_calls
    labels = [lab for lab, _ in step_calls(sb)]
    st = torch.cuda.current_stream()
    t_prev, rows = 0.0, []
    for j in range(1, len(labels) + 1):
        g = GraphedStep(sb, warmup=1, ncalls=j)
        t = time_graph(g, flush, reps, st)
        rows.append({"call": labels[j - 1], "us": 1000.0 * (t - t_prev)})
        t_prev = t
        del g
    by_kind = {}
    for r in rows:
        k = r["call"].split("@")[0]
        by_kind.setdefault(k, []).append(r["us"])
    return {"calls": rows, "step_us": 1000.0 * t_prev,
            "per_kind_us": {k: {"calls": len(v), "total": float(np.sum(v)), "mean": float(np.mean(v))}
                            for k, v in by_kind.items()}}


def roofline_table(wl, kern, steps_launches, peak, peak_kind):
    """One entry per library kernel: launches per step, mean event-timed
    duration, algorithmic bytes per launch, achieved GB/s and fraction of peak."""
    tab = {}
    for name, (n, ms) in kern.items():
        avg_us = 1000.0 * ms / n
        byt = kernel_bytes(wl, name)
        e = {"launches_per_step": steps_launches.get(name, 0), "avg_us": avg_us,
             "us_per_step": avg_us * steps_launches.get(name, 0)}
        if byt is None:
            e["bound"] = "latency"
        else:
            gbs = byt / (avg_us * 1e-6) / 1e9
            e.update(bound="hbm", bytes_per_launch=byt, achieved_gbs=gbs, frac=gbs / peak,
                     peak=peak, peak_source=peak_kind)
        tab[name] = e
    return tab


# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# per unit of work, keyed by (kernel, hash of its source file when captured);
# null once the kernel's source changes.  Units: indexed positions for the
# scans, sequence-layers for the attention.
NOMINAL_HBM_GBS = 8000.0      # nominal HBM bandwidth (~8 TB/s; the measured copy peak is the roofline)

TRAFFIC_UNITS = {
    # decode-128k capture (8 x 131,072 = 1,048,576 positions): 134,323,456 B read + 3,971,328 B written
    ("indexer_scan_tc", "34b2a05f427c"): (134323456 + 3971328) / 1048576,
    # decode-128k Reindex capture (8 x 16,384 pool positions): 16,943,104 B read, 0 written
    ("reindex_score_tc", "34b2a05f427c"): 16943104 / 131072,
    # decode-1m-fp4 capture (1,048,576 positions): 75,582,720 B read + 2,287,360 B written
    ("indexer_scan_fp4", "07bb9e54dbfe"): (75582720 + 2287360) / 1048576,
    # decode-128k capture (8 sequence-layers): 3,957,504 B read, 0 written (outputs stay in L2)
    ("attn_cluster_tc", "764442a6e89c"): 3957504 / 8,
}


def traffic_of(wl, name):
    files = {"indexer_scan_tc": "scan.cu", "reindex_score_tc": "scan.cu", "indexer_scan_fp4": "scan_fp4.cu",
             "reindex_score_fp4": "scan_fp4.cu", "attn_cluster_tc": "attention.cu", "attn_seq_tc": "attention.cu",
             "attn_partial_tc": "attention.cu"}
    if name not in files:
        return None
    per_unit = TRAFFIC_UNITS.get((name, src_hash(files[name])))
    if per_unit is None:
        return None
    if name in ("indexer_scan_tc", "indexer_scan_fp4"):
        return per_unit * sum(wl.ctx_lens)
    if name in ("reindex_score_tc", "reindex_score_fp4"):
        return per_unit * sum(min(wl.pool_blocks * 8, n) for n in wl.ctx_lens)
    return per_unit * wl.batch


def measure_workload(wl, args, dev, world, flush, with_e2e):
    """Times one decode workload: graph-replayed step (the headline), per-kernel
    event timing (eager), in-graph attribution and, optionally, the end-to-end
    serving loop through the public API with host buffers."""
    import torch
    from compressed_sparse_attention_fp4_gb300 import csa2, workload
    from compressed_sparse_attention_fp4_gb300.step import GraphedStep, run_step

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    sb = workload.build(wl, device=dev)
    g = GraphedStep(sb, warmup=2)
    st = torch.cuda.current_stream()
    # ---- device-resident timing: graph replay, L2 flushed before each step --
    for _ in range(args.warmup):
        flush.fill_(1)
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_uuid(dev)) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(st)
            g.replay()
            ev[i][1].record(st)
        torch.cuda.synchronize()
    barrier()
    times = np.array([a.elapsed_time(b) for a, b in ev])          # ms
    t_step = max_over_ranks(float(times.mean()), world, dev)
    qps = job_queries_per_s(world, wl.batch * wl.q_len, t_step)
    status = csa2.get_device_status(sb.ws)

    # ---- kernels of one step and their durations (eager, the library's own
    #      event records on the launching stream; the flush and the whole step
    #      are enqueued before any wait, so each pair times GPU work only) -----
    csa2.profile_enable(True)
    torch.cuda.synchronize()
    run_step(sb)
    torch.cuda.synchronize()
    per_step = {k: n for k, (n, _) in csa2.profile_read().items()}
    csa2.profile_enable(False)
    csa2.profile_enable(True)
    n_prof = 5
    for _ in range(n_prof):
        flush.fill_(3)
        run_step(sb)
    torch.cuda.synchronize()
    kern = csa2.profile_read()
    csa2.profile_enable(False)
    kern_us = {k: 1000.0 * ms / n for k, (n, ms) in kern.items()}
    attribution = graph_attribution(sb, flush, args.attribution_reps) if args.attribution_reps > 0 else None

    res = {"wl": wl, "sb": sb, "graph": g, "t_step": t_step, "qps": qps, "status": status,
           "clocks": clk.summary(), "per_step": per_step, "kern": kern, "kern_us": kern_us,
           "attribution": attribution, "launches": sum(per_step.values()) * args.steps,
           "step_ms_spread": [float(np.percentile(times, 5)), float(np.median(times)),
                              float(np.percentile(times, 95))]}
    if with_e2e:
        res.update(e2e_legs(sb, args, dev, world, flush, wl))
    return res


def e2e_legs(sb, args, dev, world, flush, wl):
    """End to end through the public API with host buffers.

    Per-step inputs: every layer's query and indexer query / weights, the new
    token's latent (the FP4 append) and the newest SWA row of every layer (the
    window is a device-resident cache, like the main KV: one row per layer and
    sequence arrives per step, into its last slot).  The step's result: every
    layer's output, lse and Top-K indices.  As in a serving loop, two device
    sets of inputs and results alternate: step i (set i % 2) computes while a
    copy stream uploads step i + 1's inputs and reads back step i - 1's
    results.  Every copy is inside the timed region.  The step itself is the
    library's captured step graph of its set (`GraphedStep`, the way a serving
    loop replays a decode step); `e2e_eager` makes the same run with one eager
    library call per layer step instead.  As for the device-timed value, a
    2x-L2 write on the compute stream precedes every step (inside the timed
    region); `e2e_l2_not_flushed` repeats the graph run without it, as a
    serving loop runs (the inputs are larger than L2: every step's scan
    streams the whole indexer-key cache)."""
    import torch
    from compressed_sparse_attention_fp4_gb300.step import GraphedStep, run_step

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    pin = lambda t: t.cpu().pin_memory()
    names_in = ("q", "idx_q", "idx_w", "new_latent")
    names_out = ("out", "lse", "topk")
    h_in = {k: pin(getattr(sb, k)) for k in names_in}
    h_in["swa_row"] = pin(sb.swa[:, :, -1, :].contiguous())       # [L, B, 576]
    devs = [{k: getattr(sb, k) for k in names_in + ("swa",) + names_out}]
    devs.append({k: v.clone() for k, v in devs[0].items()})
    h_out = [{k: torch.empty_like(getattr(sb, k), device="cpu").pin_memory() for k in names_out}
             for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    comp = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # set s: inputs uploaded
    ev_done = [torch.cuda.Event() for _ in range(2)]    # set s: step computed
    ev_out = [torch.cuda.Event() for _ in range(2)]     # set s: results read back

    def upload(s_):
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(ev_done[s_])                 # the set's last step read its inputs
            for k in names_in:
                devs[s_][k].copy_(h_in[k], non_blocking=True)
            devs[s_]["swa"][:, :, -1, :].copy_(h_in["swa_row"], non_blocking=True)
            ev_in[s_].record(copy_s)

    graphs = []
    for s_ in range(2):
        for k, v in devs[s_].items():
            setattr(sb, k, v)
        graphs.append(GraphedStep(sb, warmup=1))

    def compute(s_, graphed, flush_l2):
        comp.wait_event(ev_in[s_])
        comp.wait_event(ev_out[s_])                        # the set's last results were read back
        if flush_l2:
            flush.fill_(5)
        if graphed:
            graphs[s_].replay()
        else:
            for k, v in devs[s_].items():
                setattr(sb, k, v)
            run_step(sb, stream=comp)
        ev_done[s_].record(comp)

    def download(s_):
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(ev_done[s_])
            for k in names_out:
                h_out[s_][k].copy_(devs[s_][k], non_blocking=True)
            ev_out[s_].record(copy_s)

    def run_pipelined(n, graphed, flush_l2):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload((i + 1) % 2)
            compute(i % 2, graphed, flush_l2)
            download(i % 2)

    def e2e_rate(graphed, flush_l2):
        run_pipelined(args.warmup, graphed, flush_l2)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        run_pipelined(args.steps, graphed, flush_l2)
        torch.cuda.synchronize()
        elapsed = max_over_ranks(time.perf_counter() - t0, world, dev)   # the slowest rank
        return world * wl.batch * wl.q_len * args.steps / elapsed

    e2e_qps = e2e_rate(True, True)
    e2e_warm_qps = e2e_rate(True, False)
    e2e_eager_qps = e2e_rate(False, True)
    for k, v in devs[0].items():
        setattr(sb, k, v)
    cache = cache_bytes(wl)
    return {"e2e": {"value": e2e_qps, "unit": "queries/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "l2": "a 2x-L2 write before every step, inside the timed region (as for value)"},
            "e2e_l2_not_flushed": {
                "value": e2e_warm_qps, "unit": "queries/s",
                "l2": (f"no flush, as in a serving loop; the inputs are larger than L2 (every step's scan "
                       f"streams {idx_row_bytes(wl) * sum(wl.ctx_lens) / 1e6:.0f} MB of indexer keys of a "
                       f"{cache / 1e6:.0f} MB cache)")},
            "e2e_eager": {"value": e2e_eager_qps, "unit": "queries/s",
                          "l2": "a 2x-L2 write before every step, inside the timed region"}}


def summarise(res, peak, peak_kind):
    """The measured figures of one workload as JSON-ready values."""
    wl = res["wl"]
    sbytes = step_bytes(wl)
    t = res["t_step"]
    tab = roofline_table(wl, res["kern"], res["per_step"], peak, peak_kind)
    for name, e in tab.items():
        if "bytes_per_launch" in e:
            e["traffic"] = traffic_of(wl, name)
    # the roofline line names the kernel with the largest share of the step's
    # kernel time (event-timed launches x launches per step)
    dom = max((n for n in tab if "bytes_per_launch" in tab[n]), key=lambda n: tab[n]["us_per_step"])
    d = tab[dom]
    roof = {"bound": "hbm", "kernel": dom, "achieved": d["achieved_gbs"], "peak": peak, "unit": "GB/s",
            "frac": d["frac"], "frac_of_nominal": d["achieved_gbs"] / NOMINAL_HBM_GBS,
            "peak_source": peak_kind, "bytes_per_launch": d["bytes_per_launch"],
            "avg_launch_us": d["avg_us"], "traffic": d.get("traffic")}
    return {
        "value": res["qps"], "ms_per_step": t,
        "ms_per_step_p5_p50_p95": res["step_ms_spread"],
        "algorithmic_bytes_per_step": sbytes,
        "step_gbs": sbytes / (t * 1e-3) / 1e9,
        "step_frac_of_peak": sbytes / (t * 1e-3) / 1e9 / peak,
        "step_frac_of_nominal_hbm": sbytes / (t * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "kernel_us": res["kern_us"],
        "roofline": roof,
        "roofline_kernels": tab,
        "graph_attribution": res["attribution"],
        "device_status": res["status"],
    }


def codec_rates(dev, reps=20):
    """FP4 write and read of the 1,048,576 x 512 codec slab: GB/s of the
    algorithmic bytes (1 KiB of bf16 in, 288 B of codes and scales out per row
    for the write; the reverse for the read), CUDA events around each launch,
    inputs larger than L2."""
    import torch
    from compressed_sparse_attention_fp4_gb300 import csa2, synth
    n = 1 << 20
    x = torch.from_numpy(synth.codec_slab(n=n).view(np.int16)).to(dev).view(torch.bfloat16)
    codes = torch.empty((n, 256), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, 32), dtype=torch.uint8, device=dev)
    y = torch.empty((n, 512), dtype=torch.bfloat16, device=dev)
    st = torch.cuda.current_stream()
    out = {}
    for name, fn in (("quantize", lambda: csa2.fp4_kv_quantize(x, codes, scales)),
                     ("dequantize", lambda: csa2.fp4_kv_dequantize(codes, scales, y))):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            ev[i][0].record(st)
            fn()
            ev[i][1].record(st)
        torch.cuda.synchronize()
        us = 1000.0 * float(np.mean([a.elapsed_time(b) for a, b in ev]))
        byt = n * (1024 + 288)
        out[name] = {"avg_us": us, "bytes_per_launch": byt, "achieved_gbs": byt / (us * 1e-6) / 1e9}
    return out


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attribution-reps", type=int, default=60,
                    help="replays per prefix graph of the in-graph time attribution (0: none)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 1M-context and codec workloads measured beside the headline")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from compressed_sparse_attention_fp4_gb300 import synth
    wl = synth.workload(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return
        # a bounded run: at most 2 untimed and 8 timed queries (or 60 s of
        # timed CPU work), whatever --steps / --warmup ask for
        n_warm, n_steps = min(args.warmup, 2), min(args.steps, 8)
        steps_t = []
        cb = None
        for s in range(n_warm + n_steps):
            r = cpu_baseline(wl, budget_s=8.0, max_queries=1)
            if s >= n_warm:
                steps_t.append(1.0 / r["value"])
                cb = r
                if sum(steps_t) > 60.0:
                    break
        ms = 1000.0 * float(np.mean(steps_t))
        val = 1.0 / float(np.mean(steps_t))
        cb["value"] = val
        cfg = arm_config(wl, world)
        cfg["sample"] = (f"1 query per step (the CPU oracle on the host cores), "
                         f"{len(steps_t)} timed steps")
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "queries/s",
                "n_gpus": world, "steps": len(steps_t), "warmup": n_warm, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded; shapes and value recipes of the workload)",
                "config": cfg,
                "cpu_baseline": cb,
                "e2e": {"value": val, "unit": "queries/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    peak, peak_kind = peaks()

    res = measure_workload(wl, args, dev, world, flush, with_e2e=True)
    summ = summarise(res, peak, peak_kind)
    line = {
        "metric": METRIC, "value": res["qps"], "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["t_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; shapes and value recipes of the workload)",
        "config": arm_config(wl, world),
        "roofline": summ["roofline"],
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "e2e": res["e2e"],
        "e2e_l2_not_flushed": res["e2e_l2_not_flushed"],
        "e2e_eager": res["e2e_eager"],
    }
    for k in ("ms_per_step_p5_p50_p95", "algorithmic_bytes_per_step", "step_gbs", "step_frac_of_peak",
              "step_frac_of_nominal_hbm",
              "kernel_us", "roofline_kernels", "graph_attribution", "device_status"):
        line[k] = summ[k]
    if not args.no_extra and world == 1 and wl.name == "128k":
        # the other context the metric names, and the FP4 codec slab, in the
        # same run (each its own graph-timed workload)
        del res
        torch.cuda.empty_cache()
        wl1 = synth.workload("1m")
        r1 = measure_workload(wl1, args, dev, world, flush, with_e2e=False)
        s1 = summarise(r1, peak, peak_kind)
        s1["config"] = arm_config(wl1, world)
        s1["clocks"] = r1["clocks"]
        del r1
        torch.cuda.empty_cache()
        wl4 = synth.workload("1m-fp4")
        r4 = measure_workload(wl4, args, dev, world, flush, with_e2e=False)
        s4 = summarise(r4, peak, peak_kind)
        s4["config"] = arm_config(wl4, world)
        s4["clocks"] = r4["clocks"]
        del r4
        torch.cuda.empty_cache()
        wlq = synth.workload("128k-q4")
        rq = measure_workload(wlq, args, dev, world, flush, with_e2e=False)
        sq = summarise(rq, peak, peak_kind)
        sq["config"] = arm_config(wlq, world)
        sq["clocks"] = rq["clocks"]
        sq["unit"] = "query tokens/s (4 per sequence and step)"
        del rq
        torch.cuda.empty_cache()
        line["workloads"] = {"decode-1m": s1, "decode-1m-fp4": s4, "decode-128k-q4": sq,
                             "codec-1m-rows": codec_rates(dev)}
    if rank == 0 and not args.no_cpu_baseline and wl.q_len == 1:
        line["cpu_baseline"] = cpu_baseline(wl)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
