"""Benchmark of one tree-verify step (visibility -> RoPE(q) -> RoPE(k into cache) -> attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: B=32 sequences, H=64 heads, q_len=33 draft-tree nodes (chain/random
mix), ragged prefixes U{4096..8192}, d_latent=512, d_rope=64, bf16 latent cache in
shuffled 64-token pages (synthetic, seeded).  Prints one JSON line.

The step's pre-attention part is one fused launch (tv_verify_prologue: visibility, RoPE of
the queries, RoPE of the draft keys into the cache, append of the draft latent rows);
--separate runs tv_build_visibility and two tv_rope_neox calls instead.

Metric: algorithmic attention TFLOP/s of the whole step (visible (row, key) pairs only,
2*(2*d_latent + d_rope) flops per pair and head), with HBM GB/s and the roofline
fraction of the attention kernel beside it.  Inputs are resident in HBM when the timed
region starts; between steps a 256 MB buffer is written so that every step starts with
a cold L2; each step is timed with CUDA events on the launching stream.  The timed steps
replay CUDA graphs captured once from the step's calls, so the same kernels run with the
same arguments without the host's per-call work: the whole step as one graph (its time is
the step time; the attention call's preparation may overlap the prologue), and the calls
before attention and the attention call as two graphs (the attention call's own time, the
roofline's denominator).  --eager times the plain calls instead.  The end-to-end figure
(host buffers: every step copies all of its inputs, the KV cache included, in from pinned
host memory and its results out, inside the timed region) uses the plain calls, pipelined
by HostStepPipeline over two device buffer sets so that a step's upload overlaps the
previous step's compute and download; the same steps one after another are reported
beside it.

--impl reference times the float64 CPU oracle (the repository's own reference
implementation of the same step) on a bounded sample of the workload per step.
With --gpus N > 1 every rank runs an independent replica of the workload (the step has
no cross-GPU exchange); value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["source"] = "fallback"
    return d


def work_of(inp: dict):
    """Algorithmic flops and bytes of the attention call (visible pairs only)."""
    B, H, Q, DL, DR = inp["B"], inp["H"], inp["Q"], inp["DL"], inp["DR"]
    es = 2 if inp["kv_dtype"] == "bf16" else 4
    P = inp["prefix_len"].astype(np.int64)
    tree_pairs = 0
    for b in range(B):
        dep = np.zeros(Q, np.int64)
        for i in range(1, Q):
            dep[i] = dep[inp["parent"][b, i]] + 1
        tree_pairs += int((dep + 1).sum())
    pairs = int((P * Q).sum()) + tree_pairs
    flops = 2.0 * (2 * DL + DR) * pairs * H
    kv_rows = int((P + Q).sum())
    byts = (kv_rows * (DL + DR) * es + B * Q * H * (DL + DR) * es + B * Q * H * (DL + 1) * 4
            + B * Q * (4 + 8) + B * 4)
    return flops, byts, pairs


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


KERNEL_FILES = {"attn_tc": "k_attn_tc.cu", "attn_simt": "k_attn_simt.cu"}


def kernel_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of the attention kernel from the committed ncu summary, when
    it was taken on the current source of that kernel's file (hash match); else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}:{workload}")
    if not ent or ent.get("source_sha") != source_sha(KERNEL_FILES[kernel]):
        return None
    return ent


def source_sha(filename: str | None = None):
    """sha256 prefix of one kernel source file (or of every csrc file)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_tree_04_gb300", "csrc")
    names = [filename] if filename else sorted(os.listdir(csrc))
    for fn in names:
        if fn.endswith((".cu", ".h")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def max_over_ranks(values, pg, device):
    """Each entry's largest value over all ranks (a job's step time is its slowest rank's).
    pg is torch.distributed (initialised) or None for a single process."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _subset(inp, seqs):
    sub = dict(inp)
    sub["B"] = len(seqs)
    sub["parent"] = inp["parent"][seqs]
    sub["prefix_len"] = inp["prefix_len"][seqs]
    return sub


def cpu_baseline(inp, seqs, nthreads=0):
    """One oracle step (visibility, RoPE of the queries, RoPE of the tree keys written into
    the cache, attention) on sequences ``seqs``, each call timed.  Returns (seconds,
    flops, bytes, threads used, per-call seconds)."""
    import oracle
    oracle.build()
    threads = nthreads if nthreads > 0 else (os.cpu_count() or 1)
    oracle.set_threads(threads)
    P = inp["prefix_len"]
    t = {}
    t0 = time.perf_counter()
    vis, depth, anc = oracle.visibility(inp["parent"])
    t["visibility"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    q_pe_rot = oracle.rope_neox(inp["q_pe"][seqs], P[seqs], depth[seqs], inp["rope_base"],
                                out_bf16=inp["q_dtype"] == "bf16")
    t["rope_q"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    kpe_rot = oracle.rope_neox(inp["kpe_tree"][:, :, None, :], P, depth, inp["rope_base"],
                               out_bf16=inp["kv_dtype"] == "bf16")[:, :, 0, :]
    k_pe_cache = oracle.scatter_tree_kpe(kpe_rot, inp["k_pe"], P, inp.get("page_table"),
                                         inp["page_size"], inp["kv_stride_b"])
    t["rope_k"] = time.perf_counter() - t0
    q_full = np.zeros_like(inp["q_pe"])
    q_full[seqs] = q_pe_rot
    t0 = time.perf_counter()
    oracle.verify_attn(inp["q_latent"], q_full, inp["c_kv"], k_pe_cache, P, vis, inp["scale"],
                       inp.get("page_table"), inp["page_size"], inp["kv_stride_b"], seqs=seqs,
                       nthreads=threads)
    t["attention"] = time.perf_counter() - t0
    dt = sum(t.values())
    fl, by, _ = work_of(_subset(inp, seqs))
    return dt, fl, by, oracle.max_threads(), t


def run_reference(args, inp, rank, world):
    from speculative_decoding_tree_04_gb300 import synth
    if rank != 0:
        return
    seqs = synth.sample_sequences(inp, args.ref_seqs)
    for _ in range(args.warmup):          # untimed warm-up steps on the same sample
        cpu_baseline(inp, seqs)
    times = []
    fl = by = 0
    threads = 1
    per = {}
    for _ in range(args.steps):
        dt, fl, by, threads, per = cpu_baseline(inp, seqs)
        times.append(dt)
    t = float(np.mean(times))
    val = fl / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "sample": f"{len(seqs)} of {inp['B']} sequences"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"sequences {list(map(int, seqs))} of {args.workload}",
                         "per_call_s": {k: round(v, 4) for k, v in per.items()}},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "tree-verify attn TFLOP/s and HBM GB/s per GB300, % of binding roofline"


def relaunch_ranks(n):
    """``--gpus N`` without a launcher: start N ranks of this same command through
    torch.distributed.run (one process per GPU, rendezvous on 127.0.0.1) and return its
    exit code."""
    import socket
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        port = sck.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def roofline_of(path, tv, flops, byts, ams, peaks, clk, kernel_tag, workload, dev):
    import torch
    attn_tflops = flops / (ams * 1e-3) / 1e12
    attn_gbs = byts / (ams * 1e-3) / 1e9
    if path == tv.PATH_TCGEN05:
        roof = {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_tflops"],
                "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS bf16_tflops)"}
    else:
        props = torch.cuda.get_device_properties(dev)
        mhz = (clk or {}).get("sm_max_mhz", 2070.0)
        alu = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": attn_tflops, "peak": alu, "unit": "TFLOP/s",
                "frac": attn_tflops / alu,
                "peak_source": f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 x {mhz} MHz"}
    trf = kernel_traffic(kernel_tag, workload)
    roof["traffic"] = None if trf is None else trf["dram_bytes_per_launch"]
    roof["algorithmic_bytes"] = byts
    roof["hbm_gbs_achieved"] = attn_gbs
    roof["hbm_frac"] = attn_gbs / peaks["hbm_gbs"]
    roof["kernel_ms"] = ams
    return roof


def time_steps(step, steps, warmup, eager, flush, dev, barrier, cold=True):
    """Time `steps` verify steps (CUDA events on the launching stream) after `warmup`
    untimed ones.  cold: write the L2-sized flush buffer before every step (outside the
    events).  Returns (mean step ms, mean attention-call ms, graphs)."""
    import torch
    stream = torch.cuda.current_stream(dev)
    graphs = None if eager else step.capture_graphs()
    for _ in range(warmup):
        if graphs is None:
            step.run()
        else:
            graphs[0].replay()
            graphs[1].replay()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for k in range(steps):
        if cold:
            flush.add_(1.0)
        s0, a0, a1, s1 = ev[k]
        s0.record(stream)
        if graphs is None:
            step.pre()
        else:
            graphs[0].replay()
        a0.record(stream)
        if graphs is None:
            step.attention()
        else:
            graphs[1].replay()
        a1.record(stream)
        s1.record(stream)
    barrier()
    ms = float(np.sum([s0.elapsed_time(s1) for s0, _, _, s1 in ev])) / steps
    ams = float(np.sum([a0.elapsed_time(a1) for _, a0, a1, _ in ev])) / steps
    if graphs is not None:
        # The step itself: both parts in one graph, one launch per step (the two-graph
        # replays above give the attention call's own time).
        g_step = step.capture_step_graph()
        for _ in range(warmup):
            g_step.replay()
        barrier()
        ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for k in range(steps):
            if cold:
                flush.add_(1.0)
            ev1[k][0].record(stream)
            g_step.replay()
            ev1[k][1].record(stream)
        barrier()
        ms = float(np.sum([s0.elapsed_time(s1) for s0, s1 in ev1])) / steps
        graphs = (graphs[0], graphs[1], g_step)
    return ms, ams, graphs


def time_tree_build(args, inp, dev, barrier, pg):
    """Time tv_build_tree (the best-first draft tree of the workload's size: budget q_len - 1,
    16 depths x 8 candidates per sequence) replayed from a CUDA graph; the work is a chain of
    budget warp-wide argmax rounds per sequence, so the figure is a latency."""
    import torch
    from speculative_decoding_tree_04_gb300 import synth, tv
    B, budget = inp["B"], inp["Q"] - 1
    d = synth.generate_draft(B, 16, 8, seed=inp.get("seed", 1000) + 17)
    lp = torch.from_numpy(d["logprobs"]).to(dev)
    tk = torch.from_numpy(d["cand_tokens"]).to(dev)
    root = torch.from_numpy(d["root"]).to(dev)
    par = torch.empty((B, budget + 1), dtype=torch.int32, device=dev)
    tks = torch.empty_like(par)
    tv.build_tree(lp, tk, budget, par, tks, root=root)        # first call outside capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g):
            tv.build_tree(lp, tk, budget, par, tks, root=root)
    torch.cuda.current_stream(dev).wait_stream(s)
    for _ in range(args.warmup):
        g.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    barrier()
    us = e0.elapsed_time(e1) / args.steps * 1e3
    (us,) = max_over_ranks([us], pg, dev)
    return {"workload": f"{B} sequences, budget {budget}, 16 depths x 8 candidates",
            "tree_build_us": us, "nodes_per_s": B * budget / (us * 1e-6),
            "bound": "latency (a chain of budget argmax rounds per sequence)"}


def time_post_verify(args, inp, dev, flush, barrier, peaks, pg):
    """Time tv_tree_accept (argmax of every node's logits + the greedy walk) and
    tv_compact_kv on the workload's trees with a 163840-token float32 vocabulary: HBM-bound
    (the logits are read once)."""
    import torch
    from speculative_decoding_tree_04_gb300 import synth, tv
    from speculative_decoding_tree_04_gb300.step import VerifyStep
    B, Q = inp["B"], inp["Q"]
    acc = synth.generate_accept(inp, ties=False)
    logits = torch.from_numpy(acc["logits"]).to(dev)
    del acc["logits"]
    parent = torch.from_numpy(inp["parent"]).to(dev)
    tokens = torch.from_numpy(acc["tokens"]).to(dev)
    a = torch.zeros(B, dtype=torch.int32, device=dev)
    path = torch.zeros((B, Q), dtype=torch.int32, device=dev)
    emit = torch.zeros((B, Q), dtype=torch.int32, device=dev)
    newp = torch.zeros(B, dtype=torch.int32, device=dev)
    step = VerifyStep(inp, device=dev)
    step.run()
    cache = tv.make_cache(step.page_table, inp["page_size"], inp["kv_stride_b"],
                          min(step.c_kv.shape[0], step.k_pe.shape[0]))
    ws = torch.empty(tv.accept_workspace_size(B, Q, acc["vocab"]), dtype=torch.uint8, device=dev)

    def once():
        tv.tree_accept(logits, parent, tokens, a, path, emit, workspace=ws)

    def compact():
        tv.compact_kv(step.c_kv, step.k_pe, cache, step.prefix_len, path, a, newp)

    for _ in range(args.warmup):
        once()
        compact()
    barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.add_(1.0)
        ev[k][0].record()
        once()
        ev[k][1].record()
        compact()
        ev[k][2].record()
    barrier()
    acc_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    cmp_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    acc_ms, cmp_ms = max_over_ranks([acc_ms, cmp_ms], pg, dev)
    nbytes = logits.numel() * logits.element_size()
    gbs = nbytes / (acc_ms * 1e-3) / 1e9
    moved = int(a.sum().item())
    res = {"workload": f"{args.workload} trees, {acc['vocab']}-token float32 logits "
                       f"({nbytes / 1e6:.0f} MB), accepted nodes moved in the paged cache",
           "accept_ms": acc_ms, "compact_ms": cmp_ms, "ms": acc_ms + cmp_ms,
           "accepted_tokens": moved,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                        "peak_source": peaks["source"] + " copy bandwidth (MEASURED_PEAKS hbm_gbs)",
                        "algorithmic_bytes": nbytes, "traffic": None},
           "launches_per_step": 3}
    del logits, step
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="cfg5_bf16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 SIMT, 2 tcgen05")
    ap.add_argument("--ref-seqs", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate", action="store_true",
                    help="run visibility and both RoPE calls as separate launches instead of "
                         "the fused prologue")
    ap.add_argument("--eager", action="store_true",
                    help="time the plain calls instead of replaying CUDA graphs of them")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (smaller profiler captures)")
    ap.add_argument("--also", default=None,
                    help="comma-separated further workloads timed the same way and reported "
                         "under 'configs' (default: cfg4_bf16 and prefill_bf16 beside cfg5_bf16)")
    ap.add_argument("--quick", action="store_true",
                    help="device-timed steps only (no end-to-end pass, no CPU baseline); "
                         "used for profiler runs")
    ap.add_argument("--parts", action="store_true",
                    help="with --quick: also time the tree build and the accept + compaction "
                         "calls (profiler runs of those kernels)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_ranks(args.gpus))
    if world != args.gpus:
        raise SystemExit(f"bench: --gpus {args.gpus} but WORLD_SIZE={world}")

    from speculative_decoding_tree_04_gb300 import synth

    inp = synth.generate(args.workload, **({"B": args.batch} if args.batch > 0 else {}))
    if args.impl == "reference":
        run_reference(args, inp, rank, world)
        return

    import torch
    from speculative_decoding_tree_04_gb300 import build as tvbuild
    from speculative_decoding_tree_04_gb300 import tv
    from speculative_decoding_tree_04_gb300.step import HostStepPipeline, VerifyStep, _dev_float

    tvbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    step = VerifyStep(inp, device=dev, path=args.path, fused=not args.separate)
    path = step.chosen_path()
    flops, byts, pairs = work_of(inp)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    # The timed steps replay CUDA graphs of the step's calls (captured once; the same
    # kernels and arguments as the plain calls, without the host's per-call work): the whole
    # step as one graph for the step time, and the calls before attention and the attention
    # call as two graphs for the attention call's own time.  --eager asks for the plain
    # calls instead.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_wall0 = time.perf_counter()
    ms, ams, graphs = time_steps(step, args.steps, args.warmup, args.eager, flush, dev, barrier)
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    ms, ams = max_over_ranks([ms, ams], pg, dev)

    if args.quick:
        parts = {}
        if args.parts:
            parts["tree_build"] = time_tree_build(args, inp, dev, barrier, pg)
            parts["post_verify"] = time_post_verify(args, inp, dev, flush, barrier,
                                                    load_peaks(), pg)
        if rank == 0:
            print(json.dumps({"quick": True, "workload": args.workload, "ms_per_step": ms,
                              "attn_ms": ams, "attn_tflops": flops / (ams * 1e-3) / 1e12,
                              "launch": "eager" if graphs is None else "graphs",
                              "path": ["auto", "simt", "tcgen05"][path], **parts}), flush=True)
        if pg is not None:
            pg.destroy_process_group()
        return

    # warm L2: the same steps without the flush between them (reported beside the cold)
    _, ams_warm, _ = time_steps(step, args.steps, 1, args.eager, flush, dev, barrier, cold=False)
    (ams_warm,) = max_over_ranks([ams_warm], pg, dev)

    # ---- end to end through the public calls, host buffers in pinned memory ----------
    # Every step copies all of its inputs (the whole KV cache included) from pinned host
    # memory and its out and lse back.  Timed twice: one step after another on one stream,
    # and through HostStepPipeline (two device buffer sets; a step's upload overlaps the
    # previous step's compute and download), which is the reported value.
    host = {k: _dev_float(inp, k, dev, pin=True) for k in
            ("q_latent", "q_pe", "kpe_tree", "ckv_tree", "c_kv", "k_pe")}
    host["parent"] = torch.from_numpy(inp["parent"]).pin_memory()
    host["prefix_len"] = torch.from_numpy(inp["prefix_len"]).pin_memory()
    if inp["page_table"] is not None:
        host["page_table"] = torch.from_numpy(inp["page_table"]).pin_memory()
    outs_h = [(torch.empty(step.out.shape, dtype=torch.float32).pin_memory(),
               torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = outs_h[0][0].numel() * 4 + outs_h[0][1].numel() * 4
    dst = {"q_latent": step.q_latent, "q_pe": step.q_pe_raw, "kpe_tree": step.kpe_tree,
           "ckv_tree": step.ckv_tree, "c_kv": step.c_kv, "k_pe": step.k_pe,
           "parent": step.parent, "prefix_len": step.prefix_len, "page_table": step.page_table}

    def e2e_serial(n):
        for _ in range(n):
            for k, t in host.items():
                dst[k].copy_(t, non_blocking=True)
            step.run()
            outs_h[0][0].copy_(step.out, non_blocking=True)
            outs_h[0][1].copy_(step.lse, non_blocking=True)

    pipe = HostStepPipeline(inp, device=dev, path=args.path, fused=not args.separate)

    def e2e_piped(n):
        for i in range(n):
            pipe.submit(host, *outs_h[i % 2])
        pipe.wait_on(stream)

    def e2e_time(fn):
        fn(2)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(args.e2e_steps)
        e1.record(stream)
        barrier()
        t = e0.elapsed_time(e1) / args.e2e_steps
        (t,) = max_over_ranks([t], pg, dev)
        return t

    e2e_serial_ms = e2e_time(e2e_serial)
    e2e_ms = e2e_time(e2e_piped)
    torch.cuda.synchronize(dev)
    del pipe
    launches = step.launches_per_step() * args.steps
    del step, host, outs_h, graphs
    torch.cuda.empty_cache()

    # ---- further workloads, the same protocol (reported under "configs") ------------
    also = args.also
    if also is None:
        also = "cfg4_bf16,prefill_bf16" if args.workload == "cfg5_bf16" and args.batch == 0 else ""
    peaks = load_peaks()
    configs = {}
    for name in [w for w in also.split(",") if w]:
        inp2 = synth.generate(name)
        st2 = VerifyStep(inp2, device=dev, path=args.path, fused=not args.separate)
        p2 = st2.chosen_path()
        fl2, by2, _ = work_of(inp2)
        ms2, ams2, _ = time_steps(st2, args.steps, args.warmup, args.eager, flush, dev, barrier)
        _, ams2w, _ = time_steps(st2, args.steps, 1, args.eager, flush, dev, barrier, cold=False)
        ms2, ams2, ams2w = max_over_ranks([ms2, ams2, ams2w], pg, dev)
        tag2 = "attn_tc" if p2 == tv.PATH_TCGEN05 else "attn_simt"
        configs[name] = {
            "ms_per_step": ms2, "attn_ms": ams2, "attn_ms_warm_l2": ams2w,
            "value": fl2 / (ms2 * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
            "path": ["auto", "simt", "tcgen05"][p2], "launches_per_step": st2.launches_per_step(),
            "roofline": roofline_of(p2, tv, fl2, by2, ams2, peaks, clk, tag2, name, dev),
            "source_sha": source_sha(KERNEL_FILES[tag2]),
        }
        del st2
        torch.cuda.empty_cache()

    # ---- post-verify: greedy tree acceptance + KV compaction on the same trees -------
    post = pre_tree = None
    if args.workload in ("cfg5_bf16", "cfg4_bf16") and args.batch == 0:
        post = time_post_verify(args, inp, dev, flush, barrier, peaks, pg)
        pre_tree = time_tree_build(args, inp, dev, barrier, pg)

    if rank != 0:
        pg.destroy_process_group() if pg is not None else None
        return

    tflops = flops / (ms * 1e-3) / 1e12 * world
    attn_gbs = byts / (ams * 1e-3) / 1e9
    kernel_tag = "attn_tc" if path == tv.PATH_TCGEN05 else "attn_simt"
    roof = roofline_of(path, tv, flops, byts, ams, peaks, clk, kernel_tag, args.workload, dev)

    cpu = None
    if not args.no_cpu_baseline:
        seqs = synth.sample_sequences(inp, args.ref_seqs)
        dt, fl, by, thr, per = cpu_baseline(inp, seqs)
        one = seqs[:1]
        dt1, fl1, _, thr1, per1 = cpu_baseline(inp, one, nthreads=1)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"full step (visibility, RoPE, attention) of sequences "
                         f"{list(map(int, seqs))} of {args.workload}, {dt:.1f} s",
               "per_call_s": {k: round(v, 4) for k, v in per.items()},
               "single_thread": {"value": fl1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": thr1,
                                 "sample": f"sequence {int(one[0])} of {args.workload}, "
                                           f"{dt1:.1f} s",
                                 "per_call_s": {k: round(v, 4) for k, v in per1.items()}}}

    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if inp["kv_dtype"] == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": args.workload, "B": inp["B"], "H": inp["H"], "q_len": inp["Q"],
                   "d_latent": inp["DL"], "d_rope": inp["DR"],
                   "prefix_len": f"U{{4096..8192}} drawn, mean {float(inp['prefix_len'].mean()):.0f}"
                   if args.workload == "cfg5_bf16" else f"mean {float(inp['prefix_len'].mean()):.0f}",
                   "paged": inp["page_table"] is not None, "path": ["auto", "simt", "tcgen05"][path],
                   "l2": "256 MB buffer written between steps (cold L2); per-step CUDA events",
                   "launch": ("eager calls" if args.eager else
                              "the step as one CUDA graph, captured once (attention call timed "
                              "alone from its own graph)")
                   + ("; visibility + RoPE + cache append as one fused prologue launch"
                      if not args.separate else "; visibility and RoPE as separate launches"),
                   "e2e_launch": "eager calls, pipelined over two buffer sets (e2e.launch)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "hbm_gbs": attn_gbs,
        "attn_ms": ams,
        "attn_ms_warm_l2": ams_warm,
        "roofline": roof,
        "configs": configs,
        "tree_build": pre_tree,
        "post_verify": post,
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "launch": "HostStepPipeline: two device buffer sets, upload / compute / "
                          "download on three streams, each step's copies overlapping its "
                          "neighbours' work",
                "serial": {"value": flops / (e2e_serial_ms * 1e-3) / 1e12 * world,
                           "ms_per_step": e2e_serial_ms,
                           "launch": "upload, step, download one after another on one stream"}},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed": t_wall,
        "cpu_baseline": cpu,
        "source_sha": source_sha(KERNEL_FILES[kernel_tag]),
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
