"""Decode-step benchmark of the CSA2 hot path on GB300.

One step = one decode token for every sequence of the workload through its
layer schedule (Full / Reindex / Reuse layers: FP4 write of the new token,
indexer scan + pool + Top-K, Reindex, sparse attention for every layer),
captured once as a CUDA graph and replayed.  Metric: decode queries/s
(sequences x steps / time); achieved HBM GB/s of the algorithmic bytes
against the measured peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 128k|1m|mix|tiny]
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
    H, K, W = wl.heads, wl.topk, wl.swa
    return (K * ENTRY_B + W * 576 * 2 + H * 576 * 2 + H * 513 * 4 + K * 4)


def step_bytes(wl):
    """Algorithmic HBM bytes of one decode step over the whole batch."""
    tot = 0
    idx_row = wl.idx_dim * (1 if wl.idx_k_dtype == "fp8" else 4)
    q_w = wl.idx_heads * wl.idx_dim * (2 if wl.idx_k_dtype == "fp8" else 4) + wl.idx_heads * 4
    for n in wl.ctx_lens:
        pool_pos = min(wl.pool_blocks * 8, n)
        for m in wl.schedule:
            tot += attn_layer_bytes(wl)
            if m == "F":
                tot += idx_row * n + q_w + wl.pool_blocks * 4 + wl.topk * 4 + 1024 + ENTRY_B
            elif m == "Ri":
                tot += idx_row * pool_pos + wl.pool_blocks * 4 + q_w + wl.topk * 4
    return tot


def full_call_bytes(wl):
    idx_row = wl.idx_dim * (1 if wl.idx_k_dtype == "fp8" else 4)
    q_w = wl.idx_heads * wl.idx_dim * 2 + wl.idx_heads * 4
    return sum(idx_row * n + q_w + wl.pool_blocks * 4 + wl.topk * 4 for n in wl.ctx_lens)


# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of the scan kernel per indexed position, keyed by the hash of the scan source
# it was captured on (null once the kernel changes).  Captured on decode-128k
# (1,048,576 positions); the traffic grows in proportion to the positions.
TRAFFIC = {"035146e3c735": (134321664 + 3892224) / 1048576}


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
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.idx = gpu_index
        self.proc = None
        # raw samples go to a temporary file; the summary goes into the JSON line
        self.path = os.path.join(tempfile.gettempdir(), f"csa2_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_query(wl, b, kv, layers):
    """One query (sequence b) through the schedule in the CPU oracle."""
    from oracle import schedule
    from oracle import codec as oc
    f64 = lambda x: (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    keys = oc.e4m3_decode(kv["idx_k"]) if wl.idx_k_dtype == "fp8" else kv["idx_k"].astype(np.float64)
    codes, scales = oc.quantize_rows(f64(kv["latent"][-1:]))          # FP4 write of the new token
    lat = np.zeros((kv["latent"].shape[0], 512))
    rope = f64(kv["rope"])
    L = []
    for li in layers:
        L.append({"q": f64(li["q"]), "swa": f64(li["swa"]), "swa_len": li["swa_len"],
                  "idx_q": f64(li["idx_q"]) if wl.idx_k_dtype == "fp8" else li["idx_q"].astype(np.float64),
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
    return {"workload": f"decode-{wl.name}", "batch": wl.batch,
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
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from compressed_sparse_attention_fp4_gb300 import synth
    wl = synth.workload(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return
        steps_t = []
        cb = None
        for s in range(args.warmup + args.steps):
            r = cpu_baseline(wl, budget_s=8.0, max_queries=1)
            if s >= args.warmup:
                steps_t.append(1.0 / r["value"])
                cb = r
        ms = 1000.0 * float(np.mean(steps_t))
        val = 1.0 / float(np.mean(steps_t))
        cb["value"] = val
        cfg = arm_config(wl, world)
        cfg["sample"] = "1 query per step (the CPU oracle on the host cores)"
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "queries/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
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

    from compressed_sparse_attention_fp4_gb300 import csa2, workload
    from compressed_sparse_attention_fp4_gb300.step import GraphedStep, run_step

    sb = workload.build(wl, device=dev)
    g = GraphedStep(sb, warmup=2)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- device-resident timing: graph replay, L2 flushed before each step --
    for _ in range(args.warmup):
        flush.fill_(1)
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
    barrier()
    times = np.array([a.elapsed_time(b) for a, b in ev])          # ms
    t_step = max_over_ranks(float(times.mean()), world, dev)
    qps = job_queries_per_s(world, wl.batch, t_step)
    status = csa2.get_device_status(sb.ws)
    # kernel launches of one step, as the library's launch records count them
    # (one eager step; the graph replays the same launches)
    csa2.profile_enable(True)
    torch.cuda.synchronize()
    run_step(sb)
    torch.cuda.synchronize()
    launches = sum(n for n, _ in csa2.profile_read().values()) * args.steps
    csa2.profile_enable(False)

    # ---- per-call breakdown (eager, events on the launching stream) ---------
    # The library's kernel timing brackets each of its launches with events
    # on the same stream, giving per-kernel durations for the roofline.
    st = torch.cuda.current_stream()
    per = {"F_index": [], "Ri_index": [], "attn": []}
    csa2.profile_enable(True)
    n_prof_steps = 3
    for _ in range(n_prof_steps):
        # the flush and the whole step are enqueued before any wait, so the
        # GPU runs them back to back and each event pair times GPU work only
        # (not the host's enqueue of the next call)
        torch.cuda.synchronize()
        flush.fill_(3)
        cur = None
        marks = []
        for l, m in enumerate(sb.schedule):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(st)
            if m == "F":
                csa2.indexer_full_topk(sb.dims, sb.batch, sb.idx_k, sb.page_table, sb.ctx_len,
                                       sb.idx_q[l], sb.idx_w[l], sb.pool, sb.pool_len, sb.topk[l], sb.ws)
                cur = l
            elif m == "Ri":
                csa2.indexer_reindex_topk(sb.dims, sb.batch, sb.idx_k, sb.page_table, sb.ctx_len,
                                          sb.idx_q[l], sb.idx_w[l], sb.pool, sb.pool_len, sb.topk[l], sb.ws)
                cur = l
            e1.record(st)
            csa2.csa2_sparse_attn_decode(sb.dims, sb.batch, 2, sb.q[l], sb.kv_codes, sb.kv_scales,
                                         sb.kv_rope, sb.page_table, sb.ctx_len, sb.topk[cur], sb.swa[l],
                                         sb.swa_len[l], sb.scale, sb.out[l], sb.lse[l], sb.ws)
            e2.record(st)
            marks.append((m, e0, e1, e2))
        torch.cuda.synchronize()
        for m, e0, e1, e2 in marks:
            if m == "F":
                per["F_index"].append(e0.elapsed_time(e1))
            elif m == "Ri":
                per["Ri_index"].append(e0.elapsed_time(e1))
            per["attn"].append(e1.elapsed_time(e2))
    per_ms = {k: float(np.median(v)) for k, v in per.items() if v}
    kern = csa2.profile_read()
    csa2.profile_enable(False)
    kern_us = {k: 1000.0 * ms / n for k, (n, ms) in kern.items()}

    # ---- end to end through the public API with host buffers --------------
    # Per-step inputs: every layer's query and indexer query / weights, the
    # new token's latent (the FP4 append) and the newest SWA row of every
    # layer (the window is a device-resident cache, like the main KV: one
    # row per layer and sequence arrives per step, into its last slot).  The
    # step's result: every layer's output, lse and Top-K indices.  As in a
    # serving loop, two device sets of inputs and results alternate: step i
    # (set i % 2) computes while a copy stream uploads step i + 1's inputs and
    # reads back step i - 1's results.  Every copy is inside the timed region;
    # the L2 is flushed on the compute stream before every step.  The step
    # itself is the library's captured step graph of its set (`GraphedStep`,
    # the way a serving loop replays a decode step); `e2e_eager` makes the
    # same run with one eager library call per layer step instead.
    pin = lambda t: t.cpu().pin_memory()
    names_in = ("q", "idx_q", "idx_w", "new_latent")
    names_out = ("out", "lse", "topk")
    h_in = {k: pin(getattr(sb, k)) for k in names_in}
    h_in["swa_row"] = pin(sb.swa[:, :, -1, :].contiguous())       # [L, B, 576]
    dev = [{k: getattr(sb, k) for k in names_in + ("swa",) + names_out}]
    dev.append({k: v.clone() for k, v in dev[0].items()})
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
                dev[s_][k].copy_(h_in[k], non_blocking=True)
            dev[s_]["swa"][:, :, -1, :].copy_(h_in["swa_row"], non_blocking=True)
            ev_in[s_].record(copy_s)

    graphs = []
    for s_ in range(2):
        for k, v in dev[s_].items():
            setattr(sb, k, v)
        graphs.append(GraphedStep(sb, warmup=1))

    def compute(s_, graphed):
        comp.wait_event(ev_in[s_])
        comp.wait_event(ev_out[s_])                        # the set's last results were read back
        flush.fill_(5)
        if graphed:
            graphs[s_].replay()
        else:
            for k, v in dev[s_].items():
                setattr(sb, k, v)
            run_step(sb, stream=comp)
        ev_done[s_].record(comp)

    def download(s_):
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(ev_done[s_])
            for k in names_out:
                h_out[s_][k].copy_(dev[s_][k], non_blocking=True)
            ev_out[s_].record(copy_s)

    def run_pipelined(n, graphed):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload((i + 1) % 2)
            compute(i % 2, graphed)
            download(i % 2)

    def e2e_rate(graphed):
        run_pipelined(args.warmup, graphed)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        run_pipelined(args.steps, graphed)
        torch.cuda.synchronize()
        elapsed = max_over_ranks(time.perf_counter() - t0, world, dev)   # the slowest rank
        return world * wl.batch * args.steps / elapsed

    e2e_qps = e2e_rate(True)
    e2e_eager_qps = e2e_rate(False)
    for k, v in dev[0].items():
        setattr(sb, k, v)

    # ---- roofline of the dominant kernel: the Full-layer indexer scan ---------
    peak, peak_kind = peaks()
    scan_name = "indexer_scan_tc" if "indexer_scan_tc" in kern_us else "indexer_scan_cuda_core"
    scan_bytes = sum(wl.idx_dim * (1 if wl.idx_k_dtype == "fp8" else 4) * n for n in wl.ctx_lens)
    achieved = scan_bytes / (kern_us[scan_name] * 1e-6) / 1e9
    th = src_hash("scan.cu")
    per_pos = TRAFFIC.get(th) if wl.idx_k_dtype == "fp8" else None
    traffic = per_pos * sum(wl.ctx_lens) if per_pos is not None else None
    fb = full_call_bytes(wl)
    sbytes = step_bytes(wl)
    line = {
        "metric": METRIC, "value": qps, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; shapes and value recipes of the workload)",
        "config": arm_config(wl, world),
        "step_gbs": sbytes / (t_step * 1e-3) / 1e9,
        "step_frac_of_peak": sbytes / (t_step * 1e-3) / 1e9 / peak,
        "algorithmic_bytes_per_step": sbytes,
        "per_call_ms": per_ms,
        "kernel_us": kern_us,
        "full_indexer_call_gbs": fb / (per_ms["F_index"] * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": scan_name,
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "bytes_per_launch": scan_bytes, "traffic": traffic},
        "clocks": clk.summary(),
        "gpu_launches": launches,
        "device_status": status,
        "e2e_eager": {"value": e2e_eager_qps, "unit": "queries/s"},
        "e2e": {"value": e2e_qps, "unit": "queries/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
