#!/usr/bin/env python3
"""Benchmark of the ECHO per-layer decode hot path on GB300.

One step = one decode step of every layer for the whole batch: per layer, E4M3
query quantisation, FP8 indexer scores of every context token, early fetch
above the predicted threshold (with recall), exact top-k with the EMA
threshold, and the GPU-cache step (free -> allocate -> recall from the pinned
host pool); the layers run in order (layer l+1 after layer l's rows are in its
cache), all captured as one CUDA graph per step.

Default workload (DeepSeek-V3.2-shaped decode): 32 requests x 131072 context
tokens, 4 layers with independent keys, host pools and caches, 64 index heads
x 128, E4M3 keys with fp32 scales, 5% hot tokens (+2 before quantising),
k = 2048, 8192 GPU slots per request and layer, 576-dim bf16 KV rows in pinned
host pools (19.3 GB), AR(0.9) query drift, predictor on.  --workload picks
another decode workload of workloads.WORKLOADS.

Prints ONE JSON line (rank 0).  Timing: W warm-up graph replays, then K timed
steps, each bracketed by CUDA events on the launching stream, with a 256 MB
write flushing L2 before every timed step (outside the events); the step's
2.2 GB of keys are larger than L2 as well.  Under torchrun each rank runs an
independent replica (its own requests): barrier, max over ranks, value =
total steps of all ranks / slowest time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode steps/s (indexer+top-k+recall per layer) & GB/s vs HBM/PCIe roofline"
UNIT = "steps/s"
SCORE_BYTES_PER_TOKEN = 132      # algorithmic: 128 E4M3 key bytes + the 4-byte fp32 scale
FLUSH_BYTES = 256 << 20          # > 129 MB L2
FALLBACK_HBM_GBS = 6800.0
DECODE_WORKLOADS = ("v32", "batch", "tiny", "skewed", "layers")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--prime", type=int, default=8,
                   help="decode steps run from the empty cache before the warm-up (the step part): they stand "
                        "in for the prefill, which leaves the cache holding the prompt's selected tokens, so "
                        "that warm-up and timed steps are steady-state decode steps")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="v32", choices=DECODE_WORKLOADS,
                   help="decode workload of the step (default: the DeepSeek-V3.2-shaped one)")
    p.add_argument("--cpu-budget-s", type=float, default=15.0,
                   help="seconds of oracle work for the CPU baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--groups", type=int, default=None,
                   help="request groups of the decode step (default: the layer's choice)")
    p.add_argument("--lookup-in", choices=["topk", "cache-step"], default="topk",
                   help="where the selected tokens' slots are looked up (top-k's slices or the cache step)")
    p.add_argument("--e2e-first", action="store_true",
                   help="time the end-to-end pass before the device-resident one")
    p.add_argument("--early-cap", type=int, default=-1,
                   help="early-fetch cap per request and layer (-1: only the free slots cap it)")
    p.add_argument("--hold-early", action="store_true",
                   help="the held-slot variant of the cache step (the late recall need not wait for the early copy)")
    p.add_argument("--part", choices=["step", "mla", "append", "layers", "pool", "prefill", "kernels"], default="step",
                   help="step: the decode step (default); mla: the sparse MLA attention over the selected "
                        "slots alone, at the batch workload's batch, k and GPU slots; append: the append of one "
                        "new token per request (key, host-pool row, cache slot) at the batch workload; layers: "
                        "a 4-layer step on layer-correlated inputs, threshold predictor against the "
                        "cross-layer early fetch; pool: the decode step with one cache pool shared by the "
                        "batch (B x C slots, and 260000) against per-request slot ranges; prefill: the "
                        "chunked prefill of a 102400-token prompt in 2048-row blocks; kernels: the score and "
                        "top-k kernels alone on one layer of 32 requests x 131072 tokens")
    p.add_argument("--first-share", type=float, default=None,
                   help="share of the requests in the first of two groups (default: the layer's choice)")
    return p.parse_args(argv)


def workload_config(w):
    lens = w.lengths
    if len(set(lens)) == 1:
        toks = f"{lens[0]} tokens"
    else:
        toks = f"{min(lens)}-{max(lens)} tokens (sum {sum(lens)})"
    desc = (f"{w.name}: {w.B} requests x {toks}, {w.L} layer{'s' if w.L > 1 else ''} (independent keys, host pools "
            f"and caches), 64x128 index heads, E4M3 keys + fp32 scales, k={w.k}, {w.C} GPU slots/request/layer, "
            f"576-dim bf16 host KV rows, "
            + (f"{round(100 * w.hot_frac)}% hot tokens (+{w.hot_offset:g} before quantising), " if w.hot_frac else "")
            + ("queries redrawn every 8 steps" if w.drift == "redraw8" else "AR(0.9) query drift")
            + f", EMA predictor {'on' if w.predictor else 'off'}")
    return {"workload": desc, "requests": w.B, "tokens_per_request": lens[0] if len(set(lens)) == 1 else list(lens),
            "layers": w.L, "k": w.k, "gpu_slots_per_request_per_layer": w.C, "predictor": w.predictor,
            "alpha": 0.5, "l2": "inputs larger than L2 (keys of a step) and flushed by a 256 MB write before "
                                "every timed step", "cuda_graph": "one graph per step (all layers)"}


# ----------------------------------------------------------------------------- multi-rank plumbing
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def combine_over_ranks(elapsed_s: float, steps: int, world: int, reduce_max) -> tuple[float, float]:
    """Whole-job throughput of independent replicas: every rank ran `steps` steps;
    the job took as long as the slowest rank.  reduce_max(x) returns the max over ranks."""
    slowest = reduce_max(elapsed_s)
    return world * steps / slowest, slowest


# ----------------------------------------------------------------------------- peaks, clocks, profile
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def score_kernel_traffic(profile: str):
    """DRAM bytes per launch of the score kernel from a committed ncu summary,
    or None when the kernel source changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", profile)
    src = os.path.join(ROOT, "sparse_attention_kv_echo_gb300", "csrc", "echo_scores.cu")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return int(m_tr.group(1))
    except OSError:
        pass
    return None


def vmstat(keys=("pgmigrate_success", "compact_migrate_scanned", "compact_stall", "thp_fault_fallback",
                  "thp_collapse_alloc_failed")) -> dict:
    """The host kernel's page-migration and compaction counters (/proc/vmstat; {} when unreadable):
    the GPU's reads of page-locked host memory slow down while the kernel moves pages."""
    out = {}
    try:
        with open("/proc/vmstat") as f:
            for line in f:
                k, v = line.split()
                if k in keys:
                    out[k] = int(v)
    except (OSError, ValueError):
        pass
    return out


def vm_delta(a: dict, b: dict) -> dict:
    return {k: b[k] - a[k] for k in a if k in b}


class ClockSampler:
    """nvidia-smi sampling of the GPU's clocks and throttle reasons while running."""

    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.bus_id and not parts[0].lower().endswith(self.bus_id[-12:]):
                    continue
                rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return None
        mhz = [float(r[1].split()[0]) for r in rows if r[1].split()[0].replace(".", "").isdigit()]
        mx = [float(r[2].split()[0]) for r in rows if r[2].split()[0].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                 r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle (CPU) leg
def sample_requests(w) -> int:
    """Requests of the bounded oracle sample: one per host core, at most 8."""
    return max(1, min(w.B, len(os.sched_getaffinity(0)), 8))


def oracle_inputs(w, R, q_all, keys=None, wts=None, hosts=None, device="cpu"):
    """numpy inputs of the oracle for the first R requests of every layer: tok_off, and per layer
    (k8, ks, w, host rows as bytes); q [S, L, R, 64, 128].  keys / wts / hosts: the full tensors
    already drawn (sliced here), else the sample is drawn on `device` (the same draws)."""
    import numpy as np
    import torch
    from sparse_attention_kv_echo_gb300 import workloads as wl
    off = wl.tok_offsets(w.lengths[:R])
    n = int(off[-1])
    per = []
    for l in range(w.L):
        if keys is not None:
            k8, ks = keys[l][0][:n], keys[l][1][:n]
        else:
            k8, ks = wl.make_keys(w, l, device=device, requests=range(R))
        wt = (wts[l] if wts is not None else wl.make_weights(w, l, device=device))[:R]
        if hosts is not None:
            host = hosts[l][:n]
        else:
            rows = n if n % 65536 == 0 else None
            host = wl.make_host_pool(w, l, device=device, rows=rows)[:n]
        per.append((k8.cpu().numpy(), ks.cpu().numpy(), wt.cpu().numpy(),
                    host.contiguous().view(torch.uint8).numpy().reshape(n, -1)))
    q = q_all[:, :, :R].cpu().numpy()
    return off, per, np.ascontiguousarray(q)


def oracle_steps(w, R, inputs, max_steps: int, budget_s: float, warmup: int = 0):
    """The CPU oracle's decode steps over the first R requests of every layer (state carried
    from step to step, layers in order).  Returns (timed steps, seconds, threads)."""
    import numpy as np
    import oracle
    oracle.build()
    off, per, q = inputs
    threads = max(1, min(R, len(os.sched_getaffinity(0))))
    n = int(off[-1])
    state = []
    for l in range(w.L):
        row = per[l][3].shape[1]
        state.append(dict(theta=np.full(R, np.inf, np.float32), t2s=np.full(n, -1, np.int32),
                          s2t=np.full(R * w.C, -1, np.int32), dev=np.zeros((R * w.C, row), np.uint8)))

    def one(t):
        for l in range(w.L):
            k8, ks, wt, host = per[l]
            st = state[l]
            oracle.decode_step(off, q[t % len(q), l], wt, k8, ks, w.k, 0.5, w.predictor, -1, st["theta"], w.C,
                               st["t2s"], st["s2t"], host, st["dev"], nthreads=threads)

    for t in range(warmup):
        one(t)
    t0 = time.perf_counter()
    done = 0
    while done < max_steps:
        one(warmup + done)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0, threads


def sample_share(w, R) -> float:
    """The sample's share of the workload's work (its share of the context tokens)."""
    return sum(w.lengths[:R]) / max(1, sum(w.lengths))


# ----------------------------------------------------------------------------- our arm
def park(stream):
    """Holds the GPU (~10 ms spin kernel, before the first timed event) while the host
    enqueues the timed steps, so no step's events time a pause of the Python loop."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(20_000_000)


def h2d_probes(dev):
    """Host-to-device rates over the host link: the copy engine (pinned cudaMemcpyAsync) and
    zero-copy 16-byte loads (an elementwise kernel reading pinned memory through its device
    alias and writing HBM), best of 5 each over 256 MB."""
    import torch
    from sparse_attention_kv_echo_gb300 import _lib as L
    nb = 256 << 20
    hbuf = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
    hbuf.fill_(1)
    dbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
    alias = L.host_alias_tensor(hbuf.view(torch.int32), dev)
    dst = dbuf.view(torch.int32)
    out = {}
    for name, op in (("copy_engine", lambda: dbuf.copy_(hbuf, non_blocking=True)),
                     ("zero_copy_16B", lambda: torch.bitwise_or(alias, 0, out=dst))):
        rates = []
        for i in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            op()
            b.record()
            torch.cuda.synchronize()
            if i:
                rates.append(nb / (a.elapsed_time(b) / 1e3) / 1e9)
        out[name] = round(max(rates), 1)
    del alias
    return out


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from sparse_attention_kv_echo_gb300 import DecodeLayer, DecodeStack
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(dev))
    L.load(build_if_missing=True)

    w = wl.WORKLOADS[args.workload]
    if rank:
        w = wl.scaled(w, w.name, seed=rank)                 # each replica serves its own requests
    off = wl.tok_offsets(w.lengths)
    P = max(0, args.prime)
    S = max(1, min(w.steps, P + args.warmup + args.steps))   # distinct queries: the step sequence never wraps
    keys = [wl.make_keys(w, l, device=dev) for l in range(w.L)]
    wts = [wl.make_weights(w, l, device=dev) for l in range(w.L)]
    hosts = [wl.make_host_pool(w, l, device=dev, pin=True) for l in range(w.L)]
    qsrc = [wl.QueryStream(w, l, device=dev) for l in range(w.L)]
    q_all = torch.stack([torch.stack([qs.next() for _ in range(S)]) for qs in qsrc], dim=1)   # [S, L, B, 64, 128]
    kw = {} if args.first_share is None else {"first_share": args.first_share}
    kw["resolved"] = args.lookup_in == "topk"
    kw["hold_early"] = bool(args.hold_early)
    kw["early_cap"] = int(args.early_cap)
    lays = [DecodeLayer(off, keys[l][0], keys[l][1], w.k, w.C, hosts[l], predictor=w.predictor, device=dev,
                        groups=args.groups, **kw) for l in range(w.L)]
    stack = DecodeStack(lays)
    main = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    nl = w.L

    def reset():
        torch.cuda.synchronize()
        for lay in lays:
            lay.reset()
        torch.cuda.synchronize()

    with torch.cuda.stream(main):
        for l, lay in enumerate(lays):
            lay.w_in.copy_(wts[l])
        stack.step([q_all[0, l] for l in range(nl)], [lay.w_in for lay in lays], stream=main)   # eager, untimed
    reset()
    # one graph per step of the query sequence: each layer's quantiser reads that step's query in HBM
    graphs = []
    for i in range(S):
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi, stream=main):
            stack.step([q_all[i, l] for l in range(nl)], [lay.w_in for lay in lays], stream=main)
        graphs.append(gi)
    torch.cuda.synchronize()
    for i in range(S):  # untimed: every graph launched once (its first launch uploads it)
        with torch.cuda.stream(main):
            graphs[i].replay()
    reset()

    props = torch.cuda.get_device_properties(local)
    try:
        bus = f"{int(props.pci_domain_id):08x}:{int(props.pci_bus_id):02x}:{int(props.pci_device_id):02x}.0"
    except Exception:
        bus = None

    def reduce_max(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def timed(replay, at_start=None):
        """P priming and W warm-up steps, then K timed steps (events around each, L2 flushed before
        each); at_start() runs after the warm-up, just before the timed steps."""
        for t in range(P + args.warmup):
            with torch.cuda.stream(main):
                replay(t)
        torch.cuda.synchronize()
        if at_start is not None:
            at_start()
        if world > 1:
            dist.barrier()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        park(main)
        for i in range(args.steps):
            with torch.cuda.stream(main):
                flush.zero_()
                starts[i].record(main)
                replay(P + args.warmup + i)
                ends[i].record(main)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    def device_pass():
        reset()
        # timed region: graph replays, inputs resident in HBM
        stats0 = []      # the layers' counters as the timed steps start
        sampler = ClockSampler(bus)
        sampler.start()
        vm0 = vmstat()
        step_ms = timed(lambda t: graphs[t % S].replay(), at_start=lambda: stats0.extend(lay.stats.clone() for lay in lays))
        vm_timed = vm_delta(vm0, vmstat())
        clocks = sampler.stop()
        elapsed_s = sum(step_ms) / 1e3
        status = 0
        for lay in lays:
            status |= int(lay.status.item())
        stats = sum((lay.stats - s0).cpu().numpy().astype(np.int64) for lay, s0 in zip(lays, stats0))
        boundary_max = max(int(lay.stats[L.STAT_BOUNDARY_MAX].item()) for lay in lays)
        value, slowest = combine_over_ranks(elapsed_s, args.steps, world, reduce_max)

        return dict(step_ms=step_ms, clocks=clocks, vm_timed=vm_timed, elapsed_s=elapsed_s, status=status,
                    stats=stats, boundary_max=boundary_max, value=value, slowest=slowest)

    def e2e_pass():
        # end to end through the public API with host buffers
        # one graph per step: each layer's quantiser reads the step's queries from pinned memory, each
        # layer's slots and k-th scores are written to pinned memory (DecodeStack.capture_host_step)
        q_host = q_all.cpu().pin_memory()
        w_host = torch.stack(wts).cpu().pin_memory()
        slot_host = torch.empty((nl,) + tuple(lays[0].sel_slot.shape), dtype=torch.int32).pin_memory()
        kth_host = torch.empty((nl,) + tuple(lays[0].kth.shape), dtype=torch.float32).pin_memory()
        host_graphs = [stack.capture_host_step(q_host[i], w_host, slot_host, kth_host, stream=main) for i in range(S)]
        for i in range(S):
            with torch.cuda.stream(main):
                host_graphs[i].replay()
        reset()
        vm1 = vmstat()
        e2e_ms = timed(lambda t: host_graphs[t % S].replay())
        vm_e2e = vm_delta(vm1, vmstat())
        e2e_value, _ = combine_over_ranks(sum(e2e_ms) / 1e3, args.steps, world, reduce_max)
        h2d_bytes = q_host[0].numel() * 4 + w_host.numel() * 4
        d2h_bytes = slot_host.numel() * 4 + kth_host.numel() * 4
        del host_graphs
        return dict(e2e_ms=e2e_ms, e2e_value=e2e_value, vm_e2e=vm_e2e, h2d_bytes=h2d_bytes, d2h_bytes=d2h_bytes)

    # ---------------- the two timed passes (the end-to-end one first with --e2e-first)
    if args.e2e_first:
        r_e2e = e2e_pass()
        r_dev = device_pass()
    else:
        r_dev = device_pass()
        r_e2e = e2e_pass()
    step_ms, clocks, vm_timed, elapsed_s, status = (r_dev[k] for k in ("step_ms", "clocks", "vm_timed", "elapsed_s", "status"))
    stats, boundary_max, value, slowest = (r_dev[k] for k in ("stats", "boundary_max", "value", "slowest"))
    e2e_ms, e2e_value, vm_e2e, h2d_bytes, d2h_bytes = (r_e2e[k] for k in ("e2e_ms", "e2e_value", "vm_e2e", "h2d_bytes", "d2h_bytes"))


    # ---------------- per-call pass on layer 0: each call timed alone with events (L2 flushed)
    lay = lays[0]
    reps = max(4, min(args.steps, 16))
    names = ("quantize", "scores", "topk", "cache_step")
    kt = {n: [] for n in names}
    recall_ms, recall_rows, early_ms, early_rows = [], [], [], []
    side = lay.side
    above_all = torch.zeros(max(L.above_words(lay.B, lay.n_tokens), 1), dtype=torch.int32, device=dev)
    fb0 = int(lay.stats[L.STAT_TOPK_FALLBACK].item())
    cm0 = int(lay.stats[L.STAT_CAND_MISS].item())
    for r in range(reps + 2):
        t = (P + args.warmup + args.steps + r) % S
        with torch.cuda.stream(main):
            # park the GPU while the host enqueues everything, so the events time
            # GPU work only and not the host's launch latency between calls
            torch.cuda._sleep(4_000_000)
            flush.zero_()
            ev = {k: torch.cuda.Event(enable_timing=True)
                  for k in ("q0", "q1", "s1", "e1", "t0", "t1", "c1", "r1")}
            ev["q0"].record(main)
            L.quantize_q(q_all[t, 0], lay.w_in, lay.q8, lay.qscale, lay.wfold, lay.status, hist=lay.hist,
                         stream=main, cand_cnt=None if lay.cands is None else lay.cands.cnt)
            ev["q1"].record(main)
            L.index_scores(lay.tok_off, lay.n_tokens, lay.q8, lay.wfold, lay.k8, lay.ks, lay.scores, lay.theta,
                           lay.hist, lay.status, above=above_all, cache=lay.cache, stream=main, cands=lay.cands)
            ev["s1"].record(main)
            side.wait_stream(main)
            # as in the step: early rows on `main`, top-k and the tables on `side`
            L.early_fetch(lay.tok_off, lay.n_tokens, above_all, lay.early_cap, lay.cache, lay.status, stream=main)
            ev["e1"].record(main)
            ev["t0"].record(side)
            if lay.resolved:
                lay._select(lay.tok_off, 0, lay.B, lay.cands, side, cache=lay.cache, above=above_all,
                            early_cap=lay.early_cap)
                ev["t1"].record(side)
                L.cache_step_resolved(lay.tok_off, lay.n_tokens, lay.sel_idx, lay.cache, lay.sel_slot, lay.status,
                                      stream=side, copy_stream=main)
            else:
                lay._select(lay.tok_off, 0, lay.B, lay.cands, side)
                ev["t1"].record(side)
                L.cache_step(lay.tok_off, lay.n_tokens, lay.sel_idx, lay.cache, lay.sel_slot, lay.status,
                             stream=side, copy_stream=main, above=above_all, early_cap=lay.early_cap)
            ev["c1"].record(side)       # cache-step kernel done; the late recall runs on `main` after it
            ev["r1"].record(main)
        torch.cuda.synchronize()
        if r < 2:                       # the first calls follow a jump in the query sequence
            continue
        kt["quantize"].append(ev["q0"].elapsed_time(ev["q1"]))
        kt["scores"].append(ev["q1"].elapsed_time(ev["s1"]))
        kt["topk"].append(ev["t0"].elapsed_time(ev["t1"]))
        kt["cache_step"].append(ev["t1"].elapsed_time(ev["c1"]))
        early_ms.append(ev["s1"].elapsed_time(ev["e1"]))
        early_rows.append(int(lay.cache.early_cnt.sum().item()))
        recall_ms.append(max(0.0, ev["c1"].elapsed_time(ev["r1"])))
        recall_rows.append(int(lay.cache.miss_cnt.sum().item()))
    pass_fallbacks = int(lay.stats[L.STAT_TOPK_FALLBACK].item()) - fb0
    pass_cand_miss = int(lay.stats[L.STAT_CAND_MISS].item()) - cm0
    status |= int(lay.status.item())
    kern_us = {n: 1e3 * statistics.mean(v) for n, v in kt.items()}
    t_score = statistics.mean(kt["scores"]) / 1e3
    t_topk = statistics.mean(kt["topk"]) / 1e3
    tokens_layer = w.total_tokens
    score_bytes = SCORE_BYTES_PER_TOKEN * tokens_layer
    peak, peak_kind = measured_peaks()
    achieved = score_bytes / t_score / 1e9
    traffic = score_kernel_traffic(f"score_kernel_{w.name}.txt")
    scoring_topk_gbs = score_bytes / (t_score + t_topk) / 1e9
    step_s = slowest / args.steps
    step_scoring_gbs = score_bytes * nl / step_s / 1e9
    probes = h2d_probes(dev)
    link_peak = max(probes.values())
    # the early fetch alone (per-call pass): its rows over its duration
    early_alone_gbs = (sum(early_rows) * lay.cache.row_bytes) / (sum(early_ms) / 1e3) / 1e9
    # the host link in the step: every row the timed steps moved (early fetches and late misses,
    # all layers) over the timed time -- a lower bound of the two copy kernels' combined rate,
    # since the link also idles while a layer's first group is scored
    link_bytes = float(stats[L.STAT_EARLY] + stats[L.STAT_MISSES]) * lay.cache.row_bytes
    link_gbs = link_bytes / elapsed_s / 1e9

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * slowest / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 MMA, fp32 accumulate/epilogue, int32 tables",
        "data": "synthetic (seeded; shapes of the evaluation workloads)",
        "config": dict(workload_config(w), request_groups=len(lays[0].groups),
                       state=f"cache primed by {P} decode steps from empty (untimed, before the warm-up)",
                       slot_lookup="top-k" if lays[0].resolved else "cache step",
                       early_slots="held through the miss placement" if lays[0].hold_early else "free for misses",
                       early_cap=lays[0].early_cap),
        "roofline": {"kernel": "score_kernel (echo_index_scores), one layer of the batch per launch",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"hbm_gbs, {peak_kind} (burst copy)", "algorithmic_bytes": score_bytes,
                     "bytes_per_token": SCORE_BYTES_PER_TOKEN, "launch_us": round(1e6 * t_score, 2)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes},
        "gpu_launches": stack.kernel_launches_per_step() * args.steps,
        "clocks": clocks,
        "status": status,
        "detail": {"kernel_us_layer0": {k: round(v, 2) for k, v in kern_us.items()},
                   "late_recall_us_after_cache_step": round(1e3 * statistics.mean(recall_ms), 2),
                   "early_fetch_us": round(1e3 * statistics.mean(early_ms), 2),
                   "early_rows_per_layer_kernel_pass": round(statistics.mean(early_rows), 1),
                   "scoring_topk_gbs": round(scoring_topk_gbs, 1),
                   "scoring_topk_frac_of_8tbs": round(scoring_topk_gbs / 8000.0, 4),
                   "scoring_topk_frac_of_measured": round(scoring_topk_gbs / peak, 4),
                   "step_scoring_gbs": round(step_scoring_gbs, 1),
                   "step_scoring_frac_of_8tbs": round(step_scoring_gbs / 8000.0, 4),
                   "misses_per_step": round(float(stats[L.STAT_MISSES]) / args.steps, 1),
                   "early_per_step": round(float(stats[L.STAT_EARLY]) / args.steps, 1),
                   "early_used_per_step": round(float(stats[L.STAT_EARLY_USED]) / args.steps, 1),
                   "topk_boundary_bin_max": boundary_max,
                   "topk_boundary_fallbacks_timed": int(stats[L.STAT_TOPK_FALLBACK]),
                   "topk_boundary_fallbacks_kernel_pass": pass_fallbacks,
                   "topk_candidate_lists": lay.cands is not None,
                   "topk_list_misses_timed": int(stats[L.STAT_CAND_MISS]),
                   "topk_list_misses_kernel_pass": pass_cand_miss,
                   "recall_rows_per_layer_kernel_pass": round(statistics.mean(recall_rows), 1),
                   "early_fetch_alone_gbs": round(early_alone_gbs, 1),
                   "host_link_gbs_in_step": round(link_gbs, 1), "h2d_probes_gbs": probes,
                   "recall_frac_of_h2d": round(link_gbs / link_peak, 4) if link_peak else None,
                   "host_pool_huge_page_share": [round(wl.huge_page_share(h), 3) for h in hosts],
                   "step_ms": [round(x, 3) for x in step_ms],
                   "host_vmstat_during_timed": vm_timed, "host_vmstat_during_e2e": vm_e2e,
                   "step_ms_min": round(min(step_ms), 4), "step_ms_median": round(statistics.median(step_ms), 4),
                   "e2e_ms_median": round(statistics.median(e2e_ms), 4)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        R = sample_requests(w)
        inputs = oracle_inputs(w, R, q_all, keys=keys, wts=wts, hosts=hosts)
        n, secs, threads = oracle_steps(w, R, inputs, max_steps=args.steps, budget_s=args.cpu_budget_s)
        share = sample_share(w, R)
        result["cpu_baseline"] = {
            "value": round(n * share / secs, 5), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {R} of {w.B} requests x all {w.L} layers, {n} decode steps from a fresh cache "
                      f"(fp64 scores, stable-sort top-k, map/set cache), {secs:.1f} s on {threads} threads; "
                      f"value = steps/s of the sample x its share of the tokens ({share:.4f})"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ----------------------------------------------------------------------------- reference arm (the oracle)
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from sparse_attention_kv_echo_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    gen = "cuda" if torch.cuda.is_available() else "cpu"   # same draws as our arm when a GPU is present
    R = sample_requests(w)
    S = max(1, min(w.steps, args.warmup + args.steps))
    qsrc = [wl.QueryStream(w, l, device=gen) for l in range(w.L)]
    q_all = torch.stack([torch.stack([qs.next() for _ in range(S)]) for qs in qsrc], dim=1)
    inputs = oracle_inputs(w, R, q_all, device=gen)
    n, secs, threads = oracle_steps(w, R, inputs, max_steps=args.steps, budget_s=float("inf"), warmup=args.warmup)
    share = sample_share(w, R)
    value = n * share / secs
    sample = (f"{n} timed decode steps (after {args.warmup} untimed) of the first {R} of {w.B} requests x all "
              f"{w.L} layers on the CPU oracle, {threads} threads; value = steps/s of the sample x its share of "
              f"the tokens ({share:.4f})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / max(n, 1) / share, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp64 scores, fp32 selection", "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------- consumer alone
MLA_METRIC = "sparse MLA decode attention over the selected slots: requests/s (128 heads, k selected rows)"


def run_mla(args):
    """The sparse MLA decode attention alone: 8 requests, k = 2048 selected slots
    each (distinct, random) out of 4096 GPU slots of 576-dim bf16 rows, 128 heads."""
    import numpy as np
    import torch
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["batch"]
    B, k, C = w.B, w.k, w.C
    g = torch.Generator(device=dev).manual_seed(11 + rank)
    q = torch.randn((B, L.MLA_HEADS, L.MLA_DQK), generator=g, device=dev).to(torch.bfloat16)
    kv = torch.randn((B * C, L.MLA_DQK), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(11 + rank)
    sel = torch.from_numpy(np.stack([rng.permutation(C)[:k] for _ in range(B)]).astype(np.int32)).to(dev)
    out = torch.empty((B, L.MLA_HEADS, L.MLA_DV), dtype=torch.float32, device=dev)
    lse = torch.empty((B, L.MLA_HEADS), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    main = torch.cuda.Stream()
    scale = 1.0 / math.sqrt(192.0)

    def call():
        L.mla_decode(q, sel, kv, C, scale, out, lse, st, stream=main)

    for _ in range(args.warmup):
        with torch.cuda.stream(main):
            flush.zero_()
            call()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    park(main)
    for i in range(args.steps):
        with torch.cuda.stream(main):
            flush.zero_()
            starts[i].record(main)
            call()
            ends[i].record(main)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    t = statistics.mean(ms) / 1e3
    flops = 2.0 * L.MLA_HEADS * B * k * (L.MLA_DQK + L.MLA_DV)
    nbytes = B * k * L.MLA_DQK * 2 + q.numel() * 2 + out.numel() * 4 + lse.numel() * 4
    peak, kind = measured_peaks()
    print(json.dumps({
        "metric": MLA_METRIC, "value": round(B / t, 1), "unit": "requests/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t, 5), "higher_is_better": True,
        "dtype": "bf16 MMA, fp32 accumulate/softmax", "data": "synthetic (seeded)",
        "config": {"workload": f"{B} requests x {k} selected of {C} GPU slots, 576-dim bf16 rows, 128 heads",
                   "l2": "flushed by a 256 MB write before every timed call"},
        "roofline": {"kernel": "mla_split_kernel", "bound": "hbm",
                     "achieved": round(nbytes / t / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(nbytes / t / 1e9 / peak, 4), "algorithmic_bytes": nbytes,
                     "peak_source": f"hbm_gbs, {kind}"},
        "tflops": round(flops / t / 1e12, 2), "us_min": round(1e3 * min(ms), 2), "status": int(st.item()),
    }), flush=True)


KERNELS_METRIC = "indexer score and exact top-k alone, one layer: GB/s of the score kernel against HBM"


def run_kernels(args):
    """The score kernel and the top-k kernel alone on one layer of the DeepSeek-V3.2-shaped
    workload (32 requests x 131072 tokens, k = 2048, 5% hot keys): 554 MB of keys and scales
    per launch, so the launch's start-up and tail weigh little next to the read.  Predictor
    on (theta from the previous call's top-k, so the histogram is shifted), and the score call
    of the decode step: the layer's GPU cache (8192 slots per request) filters the above-
    threshold marks, so the kernel reads 136 B per token (128 key bytes, the fp32 scale, the
    4-byte slot entry) of which 132 are the method's.  L2 flushed before each call; the top-k
    reads the scores the score kernel just wrote (L2-resident)."""
    import torch
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["v32"]
    if rank:
        w = wl.scaled(w, w.name, seed=rank)
    B, n = w.B, w.total_tokens
    tok_off = torch.from_numpy(wl.tok_offsets(w.lengths)).to(dev)
    k8, ks = wl.make_keys(w, 0, device=dev)
    wt = wl.make_weights(w, 0, device=dev)
    qsrc = wl.QueryStream(w, 0, device=dev)
    f32 = {"dtype": torch.float32, "device": dev}
    i32 = {"dtype": torch.int32, "device": dev}
    q8 = torch.zeros((B, L.HEADS, L.DIM), dtype=torch.uint8, device=dev)
    qscale, wfold = torch.zeros((B, L.HEADS), **f32), torch.zeros((B, L.HEADS), **f32)
    hist, scores = torch.zeros((B, 256), **i32), torch.zeros(n, **f32)
    theta, kth = torch.full((B,), math.inf, **f32), torch.zeros(B, **f32)
    sel = torch.full((B, w.k), -1, **i32)
    status, stats = torch.zeros(1, **i32), torch.zeros(L.STATS_N, **i32)
    cands = L.Cands(B, device=dev)
    # the scores read only the cache's tables here: a one-row host pool stands in for the rows
    cache = L.LayerCache(B, n, w.C, torch.empty((1, wl.KV_DIM), dtype=torch.bfloat16).pin_memory(), device=dev)
    above = torch.zeros(max(L.above_words(B, n), 1), **i32)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    main = torch.cuda.Stream()
    qs = [qsrc.next() for _ in range(args.warmup + args.steps)]
    s_ms, t_ms = [], []
    for i, q in enumerate(qs):
        with torch.cuda.stream(main):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            L.quantize_q(q, wt, q8, qscale, wfold, status, hist=hist, stream=main, cand_cnt=cands.cnt)
            flush.zero_()
            ev[0].record(main)
            L.index_scores(tok_off, n, q8, wfold, k8, ks, scores, theta, hist, status, above=above, cache=cache,
                           stream=main, cands=cands)
            ev[1].record(main)
            ev[2].record(main)
            L.topk_select_cands(tok_off, n, scores, w.k, hist, theta, 0.5, cands, sel, kth, status, stats=stats,
                                stream=main)
            ev[3].record(main)
        torch.cuda.synchronize()
        if i >= args.warmup:
            s_ms.append(ev[0].elapsed_time(ev[1]))
            t_ms.append(ev[2].elapsed_time(ev[3]))
    ts, tt = statistics.mean(s_ms) / 1e3, statistics.mean(t_ms) / 1e3
    score_bytes = 132 * n
    peak, kind = measured_peaks()
    gbs = score_bytes / ts / 1e9
    both = (score_bytes + 4 * n) / (ts + tt) / 1e9
    print(json.dumps({
        "metric": KERNELS_METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * (ts + tt), 4),
        "higher_is_better": True, "dtype": "fp8-e4m3 MMA, fp32 accumulate, fp32 selection",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{B} requests x {w.lengths[0]} tokens, 1 layer, k={w.k}, 5% hot keys",
                   "l2": "flushed by a 256 MB write before every score call"},
        "roofline": {"kernel": "score_kernel (echo_index_scores)", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "algorithmic_bytes": score_bytes, "bytes_per_token": 132, "peak_source": f"hbm_gbs, {kind}",
                     "traffic": score_kernel_traffic(f"score_kernel_{w.name}.txt")},
        "score_us": round(1e6 * ts, 2), "topk_us": round(1e6 * tt, 2),
        "scoring_topk_gbs": round(both, 1), "scoring_topk_frac_of_8tbs": round(both / 8000.0, 4),
        "scoring_topk_frac_of_measured": round(both / peak, 4),
        "topk_boundary_fallbacks": int(stats[L.STAT_TOPK_FALLBACK].item()),
        "topk_list_misses": int(stats[L.STAT_CAND_MISS].item()),
        "list_entries_last_call": [int(x) for x in cands.cnt.cpu().tolist()[:4]], "status": int(status.item()),
    }), flush=True)


APPEND_METRIC = "appends/s: one new token per request (E4M3 key + scale, host-pool row, cache slot)"


def run_append(args):
    """echo_append_tokens alone: 8 requests of 32768 tokens in regions with room for every timed
    call, 4096 GPU slots each with free slots, 576-dim bf16 rows into the pinned host pool."""
    import numpy as np
    import torch
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["batch"]
    B, C, n0 = w.B, w.C, w.lengths[0]
    room = args.warmup + args.steps
    off = torch.arange(B + 1, dtype=torch.int64, device=dev) * (n0 + room)
    end = off[:-1] + n0
    n = int(off[-1].item())
    k8 = torch.zeros((n, L.DIM), dtype=torch.uint8, device=dev)
    ks = torch.zeros(n, dtype=torch.float32, device=dev)
    host = torch.empty((n, 576), dtype=torch.bfloat16).pin_memory()
    cache = L.LayerCache(B, n, C, host, device=dev)
    g = torch.Generator(device=dev).manual_seed(13 + rank)
    k_new = torch.randn((room, B, L.DIM), generator=g, device=dev)
    kv_new = torch.randn((room, B, 576), generator=g, device=dev).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    main = torch.cuda.Stream()
    for i in range(args.warmup):
        with torch.cuda.stream(main):
            flush.zero_()
            L.append_tokens(off, end, n, k_new[i], kv_new[i], k8, ks, cache, st, stream=main)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    park(main)
    for i in range(args.steps):
        with torch.cuda.stream(main):
            flush.zero_()
            starts[i].record(main)
            L.append_tokens(off, end, n, k_new[args.warmup + i], kv_new[args.warmup + i], k8, ks, cache, st,
                            stream=main)
            ends[i].record(main)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(end, off[:-1] + n0 + room)
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    t = statistics.mean(ms) / 1e3
    # per appended token: key in (512 B) and codes + scale out (132 B), row in (1152 B) and out to the
    # cache (1152 B) and over the host link (1152 B), ~12 B of tables
    per_tok = 512 + 132 + 1152 * 3 + 12
    print(json.dumps({
        "metric": APPEND_METRIC, "value": round(B / t, 1), "unit": "appends/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t, 5), "higher_is_better": True,
        "dtype": "fp32 key -> E4M3, bf16 rows", "data": "synthetic (seeded)",
        "config": {"workload": f"{B} requests x {n0} tokens (+{room} rows of room), {C} GPU slots each",
                   "l2": "flushed by a 256 MB write before every timed call"},
        "roofline": {"kernel": "append_kernel", "bound": "latency", "achieved_us": round(1e6 * t, 2),
                     "bytes_per_call": B * per_tok, "gbs": round(B * per_tok / t / 1e9, 2)},
        "us_min": round(1e3 * min(ms), 2), "status": int(st.item()),
    }), flush=True)


LAYERS_METRIC = "decode steps/s, 4 layers (indexer+top-k+recall each), cross-layer early fetch"


def run_layers(args):
    """A 4-layer decode step (8 requests x 32768 tokens per layer, k = 2048, 4096 slots per request
    and layer; keys and queries correlated 0.9 from layer to layer) as one CUDA graph, timed with
    the threshold predictor on every layer and with layers 1-3 seeded from the layer before."""
    import numpy as np
    import torch
    from sparse_attention_kv_echo_gb300 import DecodeLayer, DecodeStack
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["layers"]
    off = wl.tok_offsets(w.lengths)
    keys = [wl.make_keys(w, l, device=dev) for l in range(w.L)]
    wts = [wl.make_weights(w, l, device=dev) for l in range(w.L)]
    hosts = [wl.make_host_pool(w, l, device=dev, pin=True) for l in range(w.L)]
    S = 16
    qsrc = [wl.QueryStream(w, l, device=dev) for l in range(w.L)]
    q_all = [torch.stack([qsrc[l].next() for _ in range(S)]) for l in range(w.L)]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    main = torch.cuda.Stream()
    # the rest of a transformer layer between two indexers, emulated by a spin of ~40 us (the page's
    # 40-80 us window between an early layer's indexing and a later layer's attention)
    gap_cycles = 80000

    def spin(stream):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(gap_cycles)

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        a.record(main)
        spin(main)
        b.record(main)
    torch.cuda.synchronize()
    gap_us = 1e3 * a.elapsed_time(b)

    out = {}
    for mode, gap in (("threshold", False), ("cross", False), ("threshold_gap", True), ("cross_gap", True)):
        cross = mode.startswith("cross")
        lays = [DecodeLayer(off, keys[l][0], keys[l][1], w.k, w.C, hosts[l], cross_layer=cross and l > 0, device=dev)
                for l in range(w.L)]
        stack = DecodeStack(lays, cross_layer=cross)
        with torch.cuda.stream(main):
            for l, lay in enumerate(lays):
                lay.w_in.copy_(wts[l])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            stack.step([lay.q_in for lay in lays], [lay.w_in for lay in lays], stream=main,
                       between=spin if gap else None)
        torch.cuda.synchronize()
        for lay in lays:
            lay.reset()

        def load_q(t):
            for l, lay in enumerate(lays):
                lay.q_in.copy_(q_all[l][t % S])

        for t in range(args.warmup):
            with torch.cuda.stream(main):
                load_q(t)
                g.replay()
        torch.cuda.synchronize()
        stats0 = [lay.stats.clone() for lay in lays]
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        park(main)
        for i in range(args.steps):
            with torch.cuda.stream(main):
                load_q(args.warmup + i)
                flush.zero_()
                starts[i].record(main)
                g.replay()
                ends[i].record(main)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        st = [(lay.stats - s0).cpu().numpy().astype(np.int64) for lay, s0 in zip(lays, stats0)]
        out[mode] = dict(
            steps_s=round(args.steps / (sum(ms) / 1e3), 1), ms_per_step=round(statistics.mean(ms), 4),
            early_per_layer=[round(float(x[L.STAT_EARLY]) / args.steps, 1) for x in st],
            early_used_per_layer=[round(float(x[L.STAT_EARLY_USED]) / args.steps, 1) for x in st],
            late_misses_per_layer=[round(float(x[L.STAT_MISSES]) / args.steps, 1) for x in st],
            status=int(sum(int(lay.status.item()) for lay in lays)), launches=stack.kernel_launches_per_step())
        del g, stack, lays
        torch.cuda.synchronize()
    print(json.dumps({
        "metric": LAYERS_METRIC, "value": out["cross"]["steps_s"], "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": out["cross"]["ms_per_step"],
        "higher_is_better": True, "dtype": "fp8-e4m3 MMA, fp32 accumulate, int32 tables",
        "data": "synthetic (seeded; layers correlated 0.9)",
        "config": {"workload": f"{w.B} requests x {w.lengths[0]} tokens x {w.L} layers, k={w.k}, "
                               f"{w.C} GPU slots/request/layer, keys and queries correlated 0.9 layer to layer",
                   "l2": "flushed by a 256 MB write before every timed step", "cuda_graph": True},
        "threshold": out["threshold"], "cross_layer": out["cross"],
        "with_layer_gap": {"gap": f"{gap_us:.1f} us spin between layers ({gap_cycles} cycles)",
                           "threshold": out["threshold_gap"], "cross_layer": out["cross_gap"]},
    }), flush=True)


POOL_METRIC = "decode steps/s (indexer+top-k+recall per layer), one cache pool shared by the batch"


def run_pool(args):
    """The decode step of the batch workload (8 x 32768 tokens, k = 2048) with its cache as one pool
    shared by the requests -- 8 x 4096 slots (the per-request capacity in total) and the decode
    server's 260000 -- against the per-request slot ranges (4096 each), each as one CUDA graph per
    query, L2 flushed before every timed step."""
    import numpy as np
    import torch
    from sparse_attention_kv_echo_gb300 import DecodeLayer
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["batch"]
    off = wl.tok_offsets(w.lengths)
    k8, ks = wl.make_keys(w, 0, device=dev)
    wt = wl.make_weights(w, 0, device=dev)
    host = wl.make_host_pool(w, 0, device=dev, pin=True)
    S = 16
    qsrc = wl.QueryStream(w, 0, device=dev)
    q_all = torch.stack([qsrc.next() for _ in range(S)])
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    main = torch.cuda.Stream()
    out = {}
    for name, pool, lazy in (("per_request", 0, False), ("pool_32768", w.B * w.C, False), ("pool_260000", 260000, False),
                             ("per_request_lazy", 0, True), ("pool_260000_lazy", 260000, True)):
        lay = DecodeLayer(off, k8, ks, w.k, w.C, host, pool_slots=pool, groups=1 if pool else None, lazy=lazy,
                          device=dev)
        with torch.cuda.stream(main):
            lay.w_in.copy_(wt)
        torch.cuda.synchronize()
        graphs = []
        for i in range(S):
            gi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gi, stream=main):
                lay.step(q_all[i], stream=main)
            graphs.append(gi)
        torch.cuda.synchronize()
        lay.reset()
        for i in range(max(S, args.warmup)):
            with torch.cuda.stream(main):
                graphs[i % S].replay()
        torch.cuda.synchronize()
        stats0 = lay.stats.clone()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        park(main)
        for i in range(args.steps):
            with torch.cuda.stream(main):
                flush.zero_()
                starts[i].record(main)
                graphs[i % S].replay()
                ends[i].record(main)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        st = (lay.stats - stats0).cpu().numpy().astype(np.int64)
        out[name] = dict(steps_s=round(args.steps / (sum(ms) / 1e3), 1), ms_per_step=round(statistics.mean(ms), 4),
                         early_per_step=round(float(st[L.STAT_EARLY]) / args.steps, 1),
                         late_misses_per_step=round(float(st[L.STAT_MISSES]) / args.steps, 1),
                         revived_per_step=round(float(st[L.STAT_REVIVED]) / args.steps, 1),
                         status=int(lay.status.item()), launches=lay.kernel_launches_per_step())
        del graphs, lay
        torch.cuda.synchronize()
    print(json.dumps({
        "metric": POOL_METRIC, "value": out["pool_32768"]["steps_s"], "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": out["pool_32768"]["ms_per_step"],
        "higher_is_better": True, "dtype": "fp8-e4m3 MMA, fp32 accumulate, int32 tables", "data": "synthetic (seeded)",
        "config": dict(workload_config(w), l2="flushed by a 256 MB write before every timed step"),
        "per_request_slots": out["per_request"], "pool_32768": out["pool_32768"], "pool_260000": out["pool_260000"],
        "lazy_reuse": {"per_request_slots": out["per_request_lazy"], "pool_260000": out["pool_260000_lazy"]},
    }), flush=True)


PREFILL_METRIC = "chunked prefill, prompt tokens/s (scores, per-row one-round histogram top-k, union, recall)"


def run_prefill(args):
    """The chunked prefill of one 102400-token prompt: 50 blocks of 2048 query rows, k = 2048 per
    row, a 260000-slot cache; one timed step = the whole prompt (every block enqueued, block i's
    recall on the copy stream under block i+1's scores), from a fresh cache and threshold."""
    import torch
    from sparse_attention_kv_echo_gb300 import _lib as L
    from sparse_attention_kv_echo_gb300 import workloads as wl
    from sparse_attention_kv_echo_gb300.prefill import PrefillRunner

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    L.load(build_if_missing=True)
    w = wl.WORKLOADS["prefill"]
    k8, ks = wl.make_keys(w, 0, device=dev)
    host = wl.make_host_pool(w, 0, device=dev, pin=True)
    pr = PrefillRunner(k8, ks, w.k, w.C, host, w.prefill_block)
    nb = pr.blocks()
    qs = [wl.make_prefill_queries(w, i, device=dev) for i in range(nb)]
    main = torch.cuda.Stream()

    def prompt():
        with torch.cuda.stream(main):
            pr.cache.reset()
            pr.theta.fill_(math.inf)
            for i in range(nb):
                pr.block(i, qs[i][0], qs[i][1], stream=main)
            pr.wait_recall(main)

    for _ in range(max(1, args.warmup)):
        prompt()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(main):
            a.record(main)
        prompt()
        with torch.cuda.stream(main):
            b.record(main)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    t = statistics.mean(ms) / 1e3
    n = w.total_tokens
    # scoring work of the prompt: every row p sees p + 1 keys, 64 heads x 128 dims (2 FLOP per MAC)
    flops = 2.0 * 64 * 128 * n * (n + 1) / 2

    # the score kernel alone: every block's echo_prefill_scores between events (its quantised
    # queries made beforehand), L2 flushed before each; summed over the prompt's blocks
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    R0 = w.prefill_block
    q8 = torch.empty((R0, 64, 128), dtype=torch.uint8, device=dev)
    qsc = torch.empty((R0, 64), dtype=torch.float32, device=dev)
    wf = torch.empty((R0, 64), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    score_ms = []
    for rep in range(max(1, args.steps)):
        tot = 0.0
        for i in range(nb):
            row0, R = i * R0, qs[i][0].shape[0]
            with torch.cuda.stream(main):
                L.quantize_q(qs[i][0], qs[i][1], q8[:R], qsc[:R], wf[:R], st, hist=pr.hist[:R], stream=main)
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(main)
                L.prefill_scores(R, row0, n, q8[:R], wf[:R], k8, ks, pr.scores, pr.W, pr.theta, pr.hist, st,
                                 stream=main)
                b.record(main)
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        score_ms.append(tot)
    t_sc = statistics.mean(score_ms) / 1e3
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            fp8_peak = 2.0 * float(json.load(f)["bf16_tflops"])   # measured bf16 x the nominal fp8/bf16 ratio
        kind = "measured bf16 x 2 (nominal fp8 / bf16)"
    except Exception:
        fp8_peak, kind = 2.0 * 1900.0, "fallback bf16 x 2"
    tf = flops / t / 1e12
    tf_sc = flops / t_sc / 1e12
    print(json.dumps({
        "metric": PREFILL_METRIC, "value": round(n / t, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t, 3), "higher_is_better": True,
        "dtype": "fp8-e4m3 MMA, fp32 accumulate, int32 tables", "data": "synthetic (seeded)",
        "config": {"workload": f"1 prompt x {n} tokens, {w.prefill_block}-row blocks ({nb}), k={w.k} per row, "
                               f"{w.C} GPU slots", "step": "the whole prompt"},
        "roofline": {"kernel": "prefill_score_kernel (echo_prefill_scores), every block of the prompt",
                     "bound": "tensor", "achieved": round(tf_sc, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(tf_sc / fp8_peak, 4), "algorithmic_flops": flops, "peak_source": kind,
                     "kernel_ms_per_prompt": round(1e3 * t_sc, 3)},
        "whole_prompt": {"achieved_tflops": round(tf, 1), "frac": round(tf / fp8_peak, 4),
                         "note": "the prompt's scoring FLOPs over the whole step (scores, top-k, union, cache "
                                 "step, recall)"},
        "status": int(pr.status.item()) | int(st.item()), "ms_min": round(min(ms), 3),
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.part == "prefill":
        run_prefill(args)
    elif args.part == "kernels":
        run_kernels(args)
    elif args.part == "pool":
        run_pool(args)
    elif args.part == "layers":
        run_layers(args)
    elif args.part == "append":
        run_append(args)
    elif args.part == "mla":
        run_mla(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
