"""Benchmark of one compressed-sparse-attention layer step on GB300.

A step is one pass of the whole layer path over one batch: compress the new token(s) (main c4a /
c128a cache, indexer cache, SWA insert), indexer scores, top-k, sparse attention with the fused
inverse RoPE.  Default workload: the c4a decode batch (32 requests x 65,536-token context, 64
heads, d = 512, indexer 8 x 128 fp8, top-k 512, SWA 128).  Metric: query tokens per second per
layer (one query per request per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Timing: CUDA graphs of the step replayed over 4 resident cache copies (distinct layers), so that
each step's working set was evicted from L2 by the three steps before it; CUDA events on the
launching stream, one pair per graph replay inside the timed region (the median and spread of
those repetitions are reported beside the whole region's mean); max over ranks.  Multi-GPU:
independent replicas (weak scaling), no collective on the data path; ``--gpus N`` without a
launcher starts the N ranks itself under torch.distributed.run.  ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from compressed_sparse_attention_c4a_gb300 import synth  # noqa: E402

METRIC = "c4a DSA decode query-tokens/s per layer"
UNIT = "query-tokens/s"
COPIES = 4
KERNEL_SOURCES = {"index_kernel": "index_scores.cu", "attn_kernel": "attention.cu", "topk_kernel": "topk.cu",
                  "compress_kernel": "compress.cu"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default="c4a_decode_batch", choices=sorted(synth.case_specs()))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU work of the oracle sample")
    ap.add_argument("--copies", type=int, default=COPIES,
                    help="resident cache copies the steps rotate over (fewer for small profiling captures)")
    return ap.parse_args()


def rank_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def relaunch_ranks(args):
    """``--gpus N`` (N > 1) outside a launcher: start N ranks of this script under torch.distributed.run on
    127.0.0.1 and return its exit status.  The GPU arm needs N visible GPUs and fails loudly otherwise."""
    if args.impl == "gb300":
        have = torch.cuda.device_count()
        if have < args.gpus:
            raise SystemExit(f"bench.py --gpus {args.gpus}: only {have} CUDA device(s) visible")
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


# ---------------------------------------------------------------------------------------------
# algorithmic work of a step
# ---------------------------------------------------------------------------------------------
def n_entries(T, kind):
    w, s = synth.WINDOW[kind]
    return 0 if T < w else (T - w) // s + 1


def algorithmic_bytes(spec):
    """Bytes a step must move at minimum: indexer keys (+scale) of every visible entry (e4m3: d + 4 B, e2m1:
    d/2 + 4 B), the gathered top-k (or all visible) rows and the window rows of every query (bf16: 1024 B,
    fp8: 516 B)."""
    row_main = 1024 if spec.main_dtype == "bf16" else 516
    row_swa = 1024 if spec.swa_dtype == "bf16" else 516
    idx_row = (spec.idx_dim // 2 if spec.idx_dtype == "fp4" else spec.idx_dim) + 4
    idx = att = 0
    for r in range(spec.batch):
        T = spec.cached[r] + spec.new[r]
        ms = [T - 1] if spec.queries == "last" else list(range(spec.cached[r], T))
        for m in ms:
            nv = n_entries(m + 1, spec.kind)
            if spec.idx_heads:
                idx += nv * idx_row
                att += min(spec.topk, nv) * row_main
            else:
                att += nv * row_main
            att += min(spec.window, m + 1) * row_swa
    return idx, att


def index_flops(spec):
    """Indexer flops: 2 * heads * dim per visible entry per query (the e4m3 dot products)."""
    f = 0
    for r in range(spec.batch):
        T = spec.cached[r] + spec.new[r]
        ms = [T - 1] if spec.queries == "last" else list(range(spec.cached[r], T))
        for m in ms:
            f += 2 * spec.idx_heads * spec.idx_dim * n_entries(m + 1, spec.kind)
    return f


def attention_flops(spec):
    """QK^T and PV flops over every key a query attends (2 * 2 * d per key and head)."""
    f = 0
    for r in range(spec.batch):
        T = spec.cached[r] + spec.new[r]
        ms = [T - 1] if spec.queries == "last" else list(range(spec.cached[r], T))
        for m in ms:
            nv = n_entries(m + 1, spec.kind)
            keys = (min(spec.topk, nv) if spec.idx_heads else nv) + min(spec.window, m + 1)
            f += 4 * spec.dim * spec.heads * keys
    return f


def queries_per_step(spec):
    return spec.batch if spec.queries == "last" else sum(spec.new)


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------------------
def peaks():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def kernel_source_digest(kernel):
    """sha256 (16 hex digits) of a kernel's source file followed by the headers every kernel includes, so that a
    change in shared device code also marks the kernel's ncu summary as stale."""
    csrc = os.path.join(ROOT, "compressed_sparse_attention_c4a_gb300", "csrc")
    h = hashlib.sha256()
    for name in (KERNEL_SOURCES[kernel], "common.cuh", "topk_cluster.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """dram bytes per launch from the committed ncu summary, or None if absent or the kernel changed."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    digest = kernel_source_digest(kernel)
    txt = open(path).read()
    got_hash = got_bytes = None
    for line in txt.splitlines():
        if line.startswith("source_sha256_16:"):
            got_hash = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            got_bytes = float(line.split(":", 1)[1].strip())
    return got_bytes if got_hash == digest else None


def run_gpu(args, rank, world, local_rank):
    from compressed_sparse_attention_c4a_gb300 import build as _build
    _build.build()
    from compressed_sparse_attention_c4a_gb300 import dsa
    from compressed_sparse_attention_c4a_gb300.step import LayerStep

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    spec = synth.case_specs()[args.workload]
    copies = []
    for c in range(args.copies):
        s = synth.CaseSpec(**{**spec.__dict__, "seed": spec.seed + 100 * c + 10000 * rank})
        copies.append(LayerStep(synth.make_case(s, dev)))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    q_step = queries_per_step(spec)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up (eager; also loads the kernels) then graphs: S steps rotate over the copies
    with torch.cuda.stream(stream):
        for i in range(max(3, min(args.warmup, 50))):
            copies[i % args.copies].run()
    torch.cuda.synchronize()
    # a step that reports a device error (an expired bounded wait costs up to 2 s per launch) is not timed
    warm_status = max(int(c.status.item()) for c in copies)
    if warm_status:
        raise SystemExit(f"device status {warm_status} ({dsa.dsa_status_string(warm_status)}) after the warm-up "
                         f"steps: not timing a failing step")
    per_graph = args.copies * max(1, min(25, args.steps // (args.copies * 20)))  # >= 20 repetitions when steps allow
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=stream):
        for i in range(per_graph):
            copies[i % args.copies].run()
    # same steps with events around the indexer, top-k and attention launches (kernel durations)
    def timing_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None

    ev = {n: [(timing_event(), timing_event()) for _ in range(per_graph)] for n in ("index", "topk", "attend")}
    g_timed = None
    if ev["index"][0][0] is not None:
        g_timed = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_timed, stream=stream):
            for i in range(per_graph):
                st = copies[i % args.copies]
                st.compress()
                if st.has_index:
                    ev["index"][i][0].record(stream)
                    st.index()
                    ev["index"][i][1].record(stream)
                    if not st.fused_select:
                        ev["topk"][i][0].record(stream)
                        st.select()
                        ev["topk"][i][1].record(stream)
                ev["attend"][i][0].record(stream)
                st.select_attend() if st.fused_select else st.attend()
                ev["attend"][i][1].record(stream)
    reps = max(1, math.ceil(args.steps / per_graph))
    steps = reps * per_graph
    warm_reps = max(1, math.ceil(max(3, args.warmup) / per_graph))
    with torch.cuda.stream(stream):       # replay() launches on the current stream
        for _ in range(warm_reps):
            g_plain.replay()
    barrier()
    # one event per replay boundary inside the timed region: `reps` repetitions of `per_graph` steps each
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        marks[0].record(stream)
        for i in range(reps):
            g_plain.replay()
            marks[i + 1].record(stream)
        barrier()
    ms_total = marks[0].elapsed_time(marks[-1])
    rep_ms = sorted(marks[i].elapsed_time(marks[i + 1]) / per_graph for i in range(reps))
    rep_stats = {"reps": reps, "steps_per_rep": per_graph, "median_ms_per_step": round(statistics.median(rep_ms), 6),
                 "min_ms_per_step": round(rep_ms[0], 6), "max_ms_per_step": round(rep_ms[-1], 6)}
    # kernel durations: event nodes around each launch inside the step graph (its own timed region);
    # where event nodes are unavailable, a graph of back-to-back launches of that stage alone
    fused = copies[0].fused_select  # the top-k runs inside the attention call (one kernel when the plan allows)
    stages = (["index", "attend"] if fused else ["index", "topk", "attend"]) if copies[0].has_index else ["attend"]
    k_ms, timing = {}, "event nodes around each launch in the step graph"
    k_launches = 0
    try:
        if g_timed is None:
            raise RuntimeError("no external events")
        samples = {n: [] for n in stages}
        for _ in range(max(1, math.ceil(100 / per_graph))):   # >= 100 launches of each timed kernel
            with torch.cuda.stream(stream):
                g_timed.replay()
            torch.cuda.synchronize()
            for n in stages:
                samples[n] += [a.elapsed_time(b) for a, b in ev[n]]
        k_ms = {n: statistics.median(samples[n]) for n in stages}
        k_launches = len(samples[stages[0]])
        timing = (f"median over {k_launches} launches; event nodes around each launch in a step graph (which "
                  f"also removes that launch's programmatic-launch overlap with its neighbours)")
    except RuntimeError:
        timing = "graph of back-to-back launches of the stage alone"
        for n in stages:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(per_graph):
                    st = copies[i % args.copies]
                    {"index": st.index, "topk": st.select,
                     "attend": st.select_attend if fused else st.attend}[n]()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g.replay()
                a.record(stream)
                for _ in range(4):
                    g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            k_ms[n] = a.elapsed_time(b) / (4 * per_graph)
            k_launches = 4 * per_graph
    status = max(int(c.status.item()) for c in copies)

    # e2e: host (pinned) inputs -> device, step, output -> host, all inside the timed region
    e2e = run_e2e(copies, stream, spec, args, barrier)

    ms_step, e2e_ms = max_over_ranks([ms_total / steps, e2e["ms_step"]], dev)
    value = q_step * world / (ms_step / 1e3)
    idx_bytes, att_bytes = algorithmic_bytes(spec)
    hbm, tfl, src = peaks()
    kern = {}
    if "index" in k_ms:
        kern["index_kernel"] = {"ms": k_ms["index"], "bytes": idx_bytes, "gbs": idx_bytes / (k_ms["index"] * 1e6),
                                "tflops": index_flops(spec) / (k_ms["index"] * 1e9)}
        if not fused:
            kern["topk_kernel"] = {"ms": k_ms["topk"], "counted": bool(copies[0].fused_topk)}
    # fused: the attention kernel also reads every query row's scores (4 B each) for its top-k phase
    a_bytes = att_bytes + (4 * sum(int(n) for n in copies[0].n_visible.tolist()) if fused else 0)
    kern["attn_kernel"] = {"ms": k_ms["attend"], "bytes": a_bytes, "gbs": a_bytes / (k_ms["attend"] * 1e6),
                           "tflops": attention_flops(spec) / (k_ms["attend"] * 1e9)}
    if fused:
        kern["attn_kernel"]["fused_topk"] = True
        kern["attn_kernel"]["kernels_per_call"] = copies[0].select_attend_kernels
    dominant = max((n for n in kern if "bytes" in kern[n]), key=lambda n: kern[n]["ms"])
    if spec.queries == "last":  # decode: every stage streams keys once
        roof = {"kernel": dominant, "bound": "hbm", "achieved": round(kern[dominant]["gbs"], 1),
                "peak": hbm, "unit": "GB/s", "frac": round(kern[dominant]["gbs"] / hbm, 4),
                "traffic": ncu_traffic(dominant, args.workload), "peak_source": f"{src} hbm_gbs (burst copy)",
                "bytes_per_launch": kern[dominant]["bytes"]}
    elif dominant == "index_kernel":  # prefill indexer: an e4m3 contraction (keys shared by a query group)
        peak8 = 2 * tfl
        roof = {"kernel": dominant, "bound": "tensor", "achieved": round(kern[dominant]["tflops"], 1), "peak": peak8,
                "unit": "TFLOP/s", "frac": round(kern[dominant]["tflops"] / peak8, 4),
                "traffic": ncu_traffic(dominant, args.workload),
                "peak_source": f"{src} bf16_tflops (burst) x 2, the nominal e4m3 / bf16 dense ratio"}
    else:
        roof = {"kernel": dominant, "bound": "tensor", "achieved": round(kern[dominant]["tflops"], 1), "peak": tfl,
                "unit": "TFLOP/s", "frac": round(kern[dominant]["tflops"] / tfl, 4),
                "traffic": ncu_traffic(dominant, args.workload), "peak_source": f"{src} bf16_tflops (burst)"}
    # the attention's other bound beside the headline one: dense c128a decode streams 128 flop per byte, so
    # both its HBM fraction and its bf16 tensor fraction are reported
    a = kern["attn_kernel"]
    roof_other = {"kernel": "attn_kernel",
                  "hbm": {"achieved": round(a["gbs"], 1), "peak": hbm, "unit": "GB/s", "frac": round(a["gbs"] / hbm, 4)},
                  "tensor": {"achieved": round(a["tflops"], 1), "peak": tfl, "unit": "TFLOP/s",
                             "frac": round(a["tflops"] / tfl, 4), "peak_source": f"{src} bf16_tflops (burst)"}}
    launches_per_step = copies[0].launches_per_step()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warm_reps * per_graph, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16" if spec.main_dtype == "bf16" else "e4m3 (token-wise scale, codes to bf16 on the tensor cores)")
        + " attention" + ((" + e2m1 indexer keys, e4m3 queries" if spec.idx_dtype == "fp4" else " + e4m3 indexer")
                          if spec.idx_heads else "") + " (fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) caches, queries and tokens; no weights)",
        "config": workload_config(args.workload, spec, world, args.copies),
        "step_bytes": idx_bytes + att_bytes, "step_gbs": round((idx_bytes + att_bytes) / (ms_step * 1e6), 1),
        "kernels": {n: {k: round(v, 6) for k, v in d.items()} for n, d in kern.items()}, "kernel_timing": timing,
        "roofline": roof, "attention_roofline": roof_other, "timing": rep_stats, "kernel_launches_timed": k_launches,
        "gpu_launches": launches_per_step * steps, "device_status": status,
        "e2e": {"value": round(q_step * world / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e_ms, 6)},
        "clocks": clk.summary(),
    }
    return line, copies


def workload_config(name, spec, world, copies=COPIES):
    """The `config` object of both arms' JSON lines."""
    return {"workload": name, "kind": spec.kind, "batch": spec.batch,
            "context": sorted(set(c + n for c, n in zip(spec.cached, spec.new)))[:4],
            "new_tokens_per_request": max(spec.new), "heads": spec.heads, "dim": spec.dim,
            "indexer": (f"{spec.idx_heads}x{spec.idx_dim} " + ("e2m1" if spec.idx_dtype == "fp4" else "e4m3"))
                       if spec.idx_heads else None,
            "topk": spec.topk or None, "window": spec.window, "kv": spec.main_dtype,
            "l2": f"inputs larger than L2: {copies} resident cache copies rotate, each step's working set is "
                  f"evicted by the other copies", "parallelism": f"replicas x{world}"}


def max_over_ranks(values, device):
    """Element-wise max of per-rank floats over the default process group (identity on one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def run_e2e(copies, stream, spec, args, barrier):
    """Per step: pinned host inputs -> device, the step, output -> pinned host, as a serving loop pipelines
    them: one CUDA graph of `rounds` passes over the resident layers, the inputs of step s + len(copies) copied
    in (on an H2D stream) once step s, which used the same device buffers, is done, and each output copied out
    (on a D2H stream) while the next steps compute; a step starts once its inputs are in and its output buffer's
    previous contents are out.  Every byte still moves inside the timed region."""
    names = ["x_new", "z_new", "q", "q_pos", "start_pos"]
    if spec.idx_heads:
        names += ["xi_new", "zi_new", "q8", "q_scale", "w"]
    hosts = []
    for st in copies:
        hosts.append({n: st.case[n].cpu().pin_memory() for n in names})
    outs = [torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True) for st in copies]
    h2d = sum(t.numel() * t.element_size() for t in hosts[0].values())
    d2h = outs[0].numel() * outs[0].element_size()
    nc = len(copies)
    rounds = max(1, min(8, args.steps // (4 * nc)))
    n = nc * rounds  # steps per graph
    graph = torch.cuda.CUDAGraph()
    h2d_stream = torch.cuda.Stream(device=stream.device)
    d2h_stream = torch.cuda.Stream(device=stream.device)

    def copy_in(s):
        i = s % nc
        with torch.cuda.stream(h2d_stream):
            for nm in names:
                copies[i].case[nm].copy_(hosts[i][nm], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(h2d_stream)
        return ev

    with torch.cuda.graph(graph, stream=stream):
        h2d_stream.wait_stream(stream)  # fork
        d2h_stream.wait_stream(stream)
        ev_in = {s: copy_in(s) for s in range(min(nc, n))}
        ev_out = {}
        for s in range(n):
            i = s % nc
            stream.wait_event(ev_in[s])
            if s >= nc:
                stream.wait_event(ev_out[s - nc])  # this layer's previous output has left its buffer
            copies[i].run()
            done = torch.cuda.Event()
            done.record(stream)
            d2h_stream.wait_event(done)
            with torch.cuda.stream(d2h_stream):
                outs[i].copy_(copies[i].out, non_blocking=True)
            ev_out[s] = torch.cuda.Event()
            ev_out[s].record(d2h_stream)
            if s + nc < n:
                h2d_stream.wait_event(done)  # step s has read this layer's inputs
                ev_in[s + nc] = copy_in(s + nc)
        stream.wait_stream(h2d_stream)  # join
        stream.wait_stream(d2h_stream)
    reps = max(1, min(200, args.steps // n))
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
    barrier()
    return {"ms_step": t0.elapsed_time(t1) / (reps * n), "h2d": h2d, "d2h": d2h}


# ---------------------------------------------------------------------------------------------
# the oracle (CPU) arm
# ---------------------------------------------------------------------------------------------
def oracle_sample(spec, case, n_requests, rows_per_request=None):
    """Run the oracle's whole step for the first n_requests requests of a case; returns (seconds, queries)."""
    import numpy as np
    from oracle import layer as OL, compress as OC

    def np64(t):
        t = t.detach().cpu()
        return t.to(torch.float64).numpy() if t.is_floating_point() else t.numpy()

    epb = case["epb"]
    t0 = time.perf_counter()

    def pool(data, scale, rows_per_block, fmt=None):
        d = data.detach().cpu()
        if fmt == "fp4":
            return OL.Pool(rows_per_block, OL.FP4, d.numpy().copy(), np64(scale))
        if d.dtype == torch.bfloat16:
            return OL.Pool(rows_per_block, OL.BF16, d.view(torch.int16).numpy().view(np.uint16).copy())
        return OL.Pool(rows_per_block, OL.FP8, d.numpy().copy(), np64(scale))

    main = pool(case["main_data"], case["main_scale"], epb)
    swa = pool(case["swa_data"], case["swa_scale"], 256)
    copy_s = time.perf_counter() - t0
    cu, start = np64(case["cu_new"]), np64(case["start_pos"])
    bt_main, bt_swa = np64(case["bt_main"]), np64(case["bt_swa"])
    q_pos, q_req = np64(case["q_pos"]), np64(case["q_req"])
    rows = [q for q in range(case["nq"]) if q_req[q] < n_requests]
    if rows_per_request is not None:
        keep = []
        for r in range(n_requests):
            rr = [q for q in rows if q_req[q] == r]
            keep += rr[:rows_per_request]
        rows = keep
    xs = np64(case["x_new"])
    zs = np64(case["z_new"])
    sx, sz = np64(case["state_x"]), np64(case["state_z"])
    t0 = time.perf_counter()
    states = [OC.RollingState(spec.kind, spec.dim, sx[r], sz[r]) for r in range(n_requests)]
    OL.compress(spec.kind, start[:n_requests], [xs[cu[r]:cu[r + 1]] for r in range(n_requests)],
                [zs[cu[r]:cu[r + 1]] for r in range(n_requests)], states, spec.rope_dim, main, bt_main, swa, bt_swa)
    topk = None
    if spec.idx_heads:
        idx = pool(case["idx_data"], case["idx_scale"], 64, spec.idx_dtype)
        if spec.index_compress:
            xi, zi = np64(case["xi_new"]), np64(case["zi_new"])
            sxi, szi = np64(case["state_xi"]), np64(case["state_zi"])
            st2 = [OC.RollingState(spec.kind, spec.idx_dim, sxi[r], szi[r]) for r in range(n_requests)]
            OL.compress(spec.kind, start[:n_requests], [xi[cu[r]:cu[r + 1]] for r in range(n_requests)],
                        [zi[cu[r]:cu[r + 1]] for r in range(n_requests)], st2, min(spec.rope_dim, spec.idx_dim), idx,
                        np64(case["bt_idx"]))
        scores, nvis = OL.index_scores(case["q8"].cpu().numpy(), np64(case["q_scale"]), np64(case["w"]), q_pos, q_req,
                                       idx, np64(case["bt_idx"]), rows=rows)
        topk = np.full((case["nq"], spec.topk), -1, dtype=np.int64)
        for q in rows:
            topk[q] = OL.topk(scores[q], nvis[q], spec.topk)
    OL.sparse_attn(np64(case["q"]), q_pos, q_req, spec.kind, topk, main, bt_main, swa, bt_swa, spec.window,
                   1.0 / math.sqrt(512.0), spec.rope_dim, rows=rows)
    return time.perf_counter() - t0, len(rows), copy_s


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def one_thread_baseline(workload, n_requests):
    """The oracle sample of the first n requests in a child process whose BLAS / OpenMP pools have one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; from compressed_sparse_attention_c4a_gb300 import synth; "
            "spec = synth.case_specs()[%r]; case = synth.make_case(spec, 'cpu'); "
            "rows = None if spec.queries == 'last' else 2; t, q, _ = bench.oracle_sample(spec, case, %d, rows); "
            "print(json.dumps({'t': t, 'q': q}))") % (ROOT, workload, n_requests)
    try:
        res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        r = json.loads(res.stdout.strip().splitlines()[-1])
        return {"value": round(r["q"] / r["t"], 3), "unit": UNIT, "cores": 1, "seconds": round(r["t"], 2),
                "sample": f"the same oracle step for {r['q']} query tokens, one thread"}
    except (OSError, subprocess.SubprocessError, ValueError, IndexError, KeyError):
        return None


def cpu_baseline(spec, case, seconds, workload=None):
    """Time the oracle on a bounded sample (about `seconds` of CPU work) of the workload, on every host core
    the process may use and (in a child process) on one thread."""
    per_req_rows = None if spec.queries == "last" else 2
    t1, q1, _ = oracle_sample(spec, case, 1, per_req_rows)
    n = max(1, min(spec.batch, int(seconds / max(t1, 1e-3))))
    if n > 1:
        t, q, _ = oracle_sample(spec, case, n, per_req_rows)
    else:
        t, q = t1, q1
    what = (f"oracle step (compress, index, top-k, attention) for {n} of {spec.batch} requests"
            if spec.queries == "last" else f"oracle step for {q} of {queries_per_step(spec)} query tokens")
    out = {"value": round(q / t, 3), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": what,
           "seconds": round(t, 2), "cpu_model": cpu_model()}
    if workload is not None:
        out["one_thread"] = one_thread_baseline(workload, max(1, min(n, 4)))
    return out


def run_reference(args, rank, world):
    spec = synth.case_specs()[args.workload]
    if rank != 0:
        return None
    case = synth.make_case(spec, "cpu")
    per_req_rows = None if spec.queries == "last" else 2
    t1, q1, _ = oracle_sample(spec, case, 1, per_req_rows)
    n = max(1, min(spec.batch, int(max(2.0, args.cpu_seconds / 4) / max(t1, 1e-3))))
    times, qs = [], 0
    for _ in range(max(1, args.warmup if args.warmup < 2 else 1)):
        oracle_sample(spec, case, n, per_req_rows)
    steps = max(1, min(args.steps, 3))
    for _ in range(steps):
        t, q, _ = oracle_sample(spec, case, n, per_req_rows)
        times.append(t)
        qs = q
    ms = statistics.mean(times) * 1e3
    value = qs / (ms / 1e3)
    sample = f"each step: the oracle's whole layer step for {qs} of {queries_per_step(spec)} query tokens"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": 1, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": workload_config(args.workload, spec, world),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_ranks(args))
    rank, world, local_rank = rank_env()
    if world != args.gpus:
        raise SystemExit(f"bench.py --gpus {args.gpus} under a launcher of {world} rank(s)")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line, copies = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(copies[0].spec, copies[0].case, args.cpu_seconds, args.workload)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
