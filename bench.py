"""Benchmark: verified tree nodes/s for one GDN layer's verify + commit round.

One step = one round of the whole hot path over one batch, through the C ABI on
one CUDA stream: the round's topology, the closed-form verification and the
factorised commit of the accepted paths.  Where it applies (bf16 trees of up to
64 nodes) a round is one bole_commit_verify launch -- the previous round's
commit applied to each head's state as the verification loads it, then this
round's verification from the committed state (one state read per round; each
input copy's first round, in the warm-up, is a plain verification); elsewhere
bole_tree_verify (forming the topology itself where it can, else after
bole_pack_forest) then bole_commit.  --no-fuse times verify + commit as two
launches.  Inputs are seeded synthetic workloads (see
gated_deltanet_verification_gb300/inputs.py); the headline workload is the
ragged budgeted batch (64 requests x 32 heads, trees of 8..64 nodes selected
greedily under a 2048-node budget, depth <= 12, dk = dv = 128, bf16 q/k/v,
fp32 state) -- the largest workload on one GPU -- and the batched packed
forest (16 requests x 32 heads, 32-node trees of depth <= 8) is measured in
the same run and reported under "configs" with its own roofline, per-kernel
times, e2e and oracle baseline.

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier and
torch.cuda.synchronize(), CUDA events on the launching stream; the timed
steps replay one CUDA graph per input copy (so the GPU, not the Python issue
cost, is measured).  Inputs rotate over enough independent copies that the
bytes touched between two uses of the same copy exceed 3x the L2 cache, so
every step streams from HBM.  The committed state of a copy becomes that
copy's next S_pre, as in a serving loop.  Per-kernel durations come from a
separate pass: per call kind (the fused round, and bole_tree_verify and
bole_commit on their own), a graph of that call on every input copy, replayed
between events.  The JSON line also carries the roofline of the
dominant kernel, the end-to-end throughput from pinned host buffers (e2e),
the oracle on the host cores (cpu_baseline), the clocks seen, and the rows
beyond the round (cross-layer commit, stage 1, device-side selection).

--impl reference runs the CPU oracle (fp64, all host cores) on the same
workload: the slow reference arm, not a target.
Multi-GPU (torchrun): requests are independent, so every rank runs its own
batch (seeded by rank) with no collective on the data path ("weak" scaling);
rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("verified tree nodes/sec (GDN verify+commit, 1×GB300); "
          "achieved HBM GB/s vs peak")
L2_BYTES = 129 * 1024 * 1024
MAX_SETS = 64  # input copies at most; smaller workloads flush L2 before each step
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="bole", choices=["bole", "reference"])
    p.add_argument("--config", type=int, default=3,
                   help="workload of the headline line (default: the ragged budgeted batch, "
                        "the largest single-GPU workload)")
    p.add_argument("--extra-configs", default="2",
                   help="comma-separated workloads measured in the same run and reported "
                        "under 'configs' (each with its own roofline, kernels, e2e and "
                        "cpu_baseline); empty for none")
    p.add_argument("--shape", default="chain", help="tree shape for config 4")
    p.add_argument("--force-simt", action="store_true", help="use the FP32 CUDA-core kernels")
    p.add_argument("--one-tile-per-head", action="store_true",
                   help="trees of up to 32 nodes: force one CTA per (request, head)")
    p.add_argument("--io-dtype", default=None, choices=[None, "bf16", "f32"],
                   help="the workload's q/k/v (and O) dtype: f32 draws the same values at full "
                        "float32 precision (tensor-core value tiles for trees of up to 32 "
                        "nodes; commit on the CUDA cores)")
    p.add_argument("--no-fuse", action="store_true",
                   help="run each round as verify -> commit even where the previous round's "
                        "commit can be fused into the verification (bole_commit_verify)")
    p.add_argument("--pack-round", action="store_true",
                   help="run the round as pack -> verify -> commit even where the "
                        "verification can form the topology itself")
    p.add_argument("--value-tiles", action="store_true",
                   help="trees of up to 32 nodes: force the value-tiled kernel (two CTAs "
                        "per head)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--conv-width", type=int, default=4,
                   help="width of the stage-1 causal convolution measurement (0 skips it)")
    p.add_argument("--no-selection", action="store_true",
                   help="skip the device-side selection measurement")
    p.add_argument("--layers", type=int, default=8,
                   help="layers of the unified cross-layer commit measurement (0 skips it)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--kernel-steps", type=int, default=200,
                   help="steps of the separate per-kernel timing pass")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# algorithmic traffic and work (per launch)
# ---------------------------------------------------------------------------

def path_lengths(batch):
    L = np.zeros(batch.B, dtype=np.int64)
    for b in range(batch.B):
        a = int(batch.accepted[b])
        o = batch.offsets[b]
        n = 0
        while a >= 0:
            n += 1
            a = int(batch.parent[o + a])
        L[b] = n
    return L


def algorithmic(batch, inline_topology=False):
    """Bytes each kernel must move at least once, and tensor flops of verify.
    With the topology formed in the verification there is no pack launch and
    the verification reads the parent links instead of pack's outputs."""
    B, H, dk, dv, N = batch.B, batch.H, batch.dk, batch.dv, batch.N
    s_in = 2 if batch.dtype == "bf16" else 4
    topo_pack = 0 if inline_topology else 4 * (B + 1) + 4 * N + 4 * N + 16 * N + 4 * B
    topo_verify = 4 * (B + 1) + (4 * N if inline_topology else 4 * N + 20 * N + 4 * B)
    verify = (B * H * dk * dv * 4 + N * H * (2 * dk + dv) * s_in + 8 * N * H
              + N * H * dv * (s_in + 4) + 4 * N * H + topo_verify)
    L = path_lengths(batch)
    committed = int(np.sum(L > 0))
    commit = (2 * committed * H * dk * dv * 4 + int(np.sum(L)) * H * (dk * s_in + 4 * dv + 4)
              + 4 * (B + 1) + 4 * B + 4 * int(np.sum(L)))
    sizes = np.diff(batch.offsets)
    depths = batch.node_depths()
    flops = 0
    for b in range(B):
        T = int(sizes[b])
        if T == 0:
            continue
        d = int(depths[batch.offsets[b]:batch.offsets[b + 1]].max())
        flops += H * (4 * T * dk * dv + 4 * T * T * dk + 2 * d * T * T * dv + 2 * T * T * dv)
    flops += int(np.sum(L)) * H * 2 * dk * dv
    return {"pack": topo_pack, "verify": verify, "commit": commit, "verify_flops": flops}


# source file of each tensor-core kernel (a recorded DRAM figure is only
# reported while that file is unchanged)
KERNEL_SOURCES = {"tc_verify_kernel": "tc_verify.cu", "tc_commit_kernel": "tc_verify.cu",
                  "tc_commit_verify": "tc_verify.cu",
                  "tc_big_fused_kernel": "tc_big.cu", "tc_vtile_kernel": "tc_vtile.cu"}


def workload_key(config: int, shape: str, io_dtype: str = "bf16") -> str:
    key = f"{config}{shape}" if config == 4 else str(config)
    return key if io_dtype == "bf16" or config == 0 else key + io_dtype


def recorded_traffic(kernels, workload: str):
    """DRAM bytes of one call (the sum over its kernels' launches) from the
    committed ncu summary profiles/traffic.txt, or None when a kernel's source
    changed since the capture (or a kernel has no capture).  Lines:
    `source <file> <sha256>` and `<kernel> <workload> <bytes>`."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    csrc = os.path.join(ROOT, "gated_deltanet_verification_gb300", "csrc")
    if not kernels:
        return None
    try:
        lines = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
        shas = {ln[1]: ln[2] for ln in lines if len(ln) == 3 and ln[0] == "source"}
        got = {ln[0]: int(ln[2]) for ln in lines
               if len(ln) == 3 and ln[0] != "source" and ln[1] == workload}
        for k in kernels:
            f = KERNEL_SOURCES[k]
            sha = hashlib.sha256(open(os.path.join(csrc, f), "rb").read()).hexdigest()
            if shas.get(f) != sha or k not in got:
                return None
        return sum(got[k] for k in kernels)
    except Exception:
        return None


def rank_seed(config: int, rank: int) -> int:
    """Each rank verifies its own batch of the same shape (weak scaling)."""
    return 1000 + config + 7919 * rank


def max_over_ranks(value: float, device) -> float:
    """Slowest rank's value (the job's wall time); identity on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(nodes_per_rank: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job nodes/s: every rank's nodes over the slowest rank's time."""
    return nodes_per_rank * steps * world / (elapsed_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def run_oracle_sample(batch, target_s: float):
    """Time the oracle's verify + commit over whole repetitions of the batch
    until about target_s seconds have passed; returns nodes/s and details."""
    import oracle
    oracle.load()
    threads = oracle.default_threads()
    prep = oracle.Prepared(batch, nthreads=threads)  # converted once, as in the reference arm
    units = batch.B * batch.H
    reps, t0 = 0, time.perf_counter()
    while True:
        prep.verify(0, units)
        prep.commit(0, units)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s or reps >= 1000:
            break
    return reps * batch.N / el, el, reps, threads


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from gated_deltanet_verification_gb300 import build

    build.build()
    head = measure_config(args, args.config, world, rank, local_rank, dev, args.steps)
    extras = {}
    for c in [int(x) for x in args.extra_configs.split(",") if x.strip()]:
        if c == args.config:
            continue
        extras[str(c)] = measure_config(args, c, world, rank, local_rank, dev, args.steps)
    stream = torch.cuda.current_stream()
    layers = run_layers(args, head["_batch"], head["_flags"], stream) if args.layers > 0 else None
    stage1 = run_stage1(args, head["_batch"], stream) if args.conv_width > 0 else None
    selection = run_selection(stream) if not args.no_selection else None

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    out = {k: v for k, v in head.items() if not k.startswith("_")}
    launches = head["_launches"]
    if extras:
        out["configs"] = {k: {kk: vv for kk, vv in v.items() if not kk.startswith("_")
                              and kk not in ("metric", "n_gpus", "higher_is_better", "scaling",
                                             "vs_baseline", "data")}
                          for k, v in extras.items()}
        launches += sum(v["_launches"] for v in extras.values())
    out.update({"commit_layers": layers, "stage1": stage1, "selection": selection,
                "gpu_launches": launches})
    print(json.dumps(out))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def measure_config(args, cfg, world, rank, local_rank, dev, steps):
    """One workload: warm-up, K timed graph-replayed steps (clocks sampled),
    per-kernel durations, roofline, e2e and the oracle baseline.  Returns the
    fields of the JSON line (keys starting with '_' are internal)."""
    import torch
    import torch.distributed as dist
    from gated_deltanet_verification_gb300 import bole, device, inputs

    flags = (bole.FLAG_FORCE_SIMT if args.force_simt else 0) | \
        (bole.FLAG_ONE_TILE_PER_HEAD if args.one_tile_per_head else 0) | \
        (bole.FLAG_VALUE_TILES if args.value_tiles else 0) | \
        getattr(args, "verify_flags", 0)
    seed = rank_seed(cfg, rank)
    if cfg == 0:  # the float32 toy; its values are kept as drawn
        batch = inputs.config_batch(cfg, seed=seed, shape=args.shape)
        if args.io_dtype:
            batch.dtype = args.io_dtype
    else:  # f32: the same draws at full float32 precision
        batch = inputs.config_batch(cfg, seed=seed, shape=args.shape, dtype=args.io_dtype)
    probe_db = device.to_device(batch, device=dev)
    # the topology step inside the verification where the kernels allow it
    inline = (not args.pack_round) and device.inline_topology_supported(probe_db, flags)
    # the previous round's commit fused into each verification (one state read
    # per round instead of two), where bole_commit_verify applies
    fz = (inline and not args.no_fuse and not args.value_tiles
          and device.commit_verify_supported(probe_db, flags))
    del probe_db
    if inline:
        flags |= bole.FLAG_INLINE_TOPOLOGY
    alg = algorithmic(batch, inline)
    # fused: the verification's and the commit's bytes less one read of the state
    alg["commit_verify"] = (alg["verify"] + alg["commit"]
                            - batch.B * batch.H * batch.dk * batch.dv * 4)
    step_bytes = (alg["commit_verify"] if fz
                  else alg["pack"] + alg["verify"] + alg["commit"])
    # L2 hygiene: rotate over enough input copies that > 3x L2 is touched
    # between reuses; a workload too small for that (more than MAX_SETS
    # copies) keeps two copies and writes a buffer of twice the L2 before
    # every timed step instead, each step then timed on its own.
    need = max(2, int(np.ceil(3 * L2_BYTES / step_bytes)) + 1)
    flush_mode = need > MAX_SETS
    n_sets = 2 if flush_mode else need
    flush_buf = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
                 if flush_mode else None)

    sets = []
    for _ in range(n_sets):
        db = device.to_device(batch, device=dev)
        rb = device.alloc_round(db, flags)
        sets.append((db, rb))
    stream = torch.cuda.current_stream()
    tc_dims = not args.force_simt and batch.dk == 128 and batch.dv == 128
    tc_shape = tc_dims and batch.dtype == "bf16"
    # value-tiled kernel: fp32 inputs always; bf16 forced, or by default while
    # the heads leave the one-CTA kernel (two CTAs per SM) short of one wave
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    vtile = (tc_dims and batch.max_T <= 32 and batch.max_depth < 16
             and not args.one_tile_per_head
             and (batch.dtype == "f32" or args.value_tiles or batch.B * batch.H < 2 * sms))
    fused = tc_shape and batch.max_T <= 64 and batch.max_depth < 16   # single-CTA kernel
    big = tc_shape and not fused and batch.max_T <= 128              # fused large-tree kernel
    tc_used = fused or big or vtile
    # pack (unless the verification forms the topology), verify (one tensor-core
    # kernel, or the CUDA-core producer + solve), commit
    launches_per_step = 1 if fz else (0 if inline else 1) + (1 if tc_used else 2) + 1
    # Step j of a period: input copy j % n_sets; with the fused round the copies
    # alternate their U / logP pair, parity (j // n_sets) % 2, so a period is
    # two passes over the copies and every copy is back at parity 0 after it.
    period = 2 * n_sets if fz else n_sets

    def one_round(j, cs):
        db, rb = sets[j % n_sets]
        if fz:
            device.commit_verify_round(db, rb, (j // n_sets) % 2, cs)
        else:
            device.run_round(db, rb, flags, cs)

    if fz:  # the first round of each copy: a plain verification (its factors
        for db, rb in sets:  # are what the first fused round commits)
            device.alloc_alt(db, rb)
            device.verify(db, rb, flags, stream)
    warm = -(-args.warmup // period) * period if fz else args.warmup
    for i in range(warm):
        one_round(i, stream)
    torch.cuda.synchronize()
    for _, rb in sets:
        bole.check_status(rb.status, "warm-up")

    # The steps are replayed from CUDA graphs, so the timed region measures
    # the GPU work, not the Python and ctypes cost of issuing the launches
    # (the end-to-end number below keeps that cost): one graph holds a round
    # on every input copy in turn (replayed while whole passes remain), one
    # graph per copy serves the rest and the flushed steps.
    graphs = []
    for j in range(period):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one_round(j, torch.cuda.current_stream())
        graphs.append(g)
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all):
        for j in range(period):
            one_round(j, torch.cuda.current_stream())
    for j in range(period):
        graphs[j].replay()
    g_all.replay()
    torch.cuda.synchronize()
    for _, rb in sets:
        bole.check_status(rb.status, "graph warm-up")

    # ---- timed region: K steps, events only at its ends ----
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if flush_mode:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush_buf.fill_(float(i & 1))
            evs[i][0].record(stream)
            graphs[i % period].replay()
            evs[i][1].record(stream)
    else:
        start.record(stream)
        for _ in range(steps // period):
            g_all.replay()
        for j in range(steps % period):
            graphs[j].replay()
        end.record(stream)
    for j in range(steps % period, period if steps % period else 0):
        graphs[j].replay()  # untimed: every copy back at parity 0
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    for _, rb in sets:
        bole.check_status(rb.status, "timed steps")
    elapsed_ms = (sum(a.elapsed_time(b) for a, b in evs) if flush_mode
                  else start.elapsed_time(end))

    # ---- separate pass: per-kernel durations.  One graph per call kind runs
    #      that call once on every input copy, back to back and without launch
    #      overlap (the copies keep the L2 cold between reuses); events bracket
    #      each replay ----
    ks = max(1, min(args.kernel_steps, steps))
    per_kernel = {"pack": [], "verify": [], "commit": []}
    if fz:  # the fused kernel: whole periods (both parities on every copy)
        per_kernel["commit_verify"] = []
        if flush_mode:
            reps = -(-max(1, ks) // period) * period
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(reps)]
            for r, (a, b) in enumerate(pairs):
                flush_buf.fill_(0.0)
                a.record(stream)
                graphs[r % period].replay()
                b.record(stream)
            torch.cuda.synchronize()
            per_kernel["commit_verify"].append(sum(a.elapsed_time(b) for a, b in pairs) / reps)
        else:
            reps = max(1, ks // period)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g_all.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            per_kernel["commit_verify"].append(e0.elapsed_time(e1) / (reps * period))
    cflags = flags & ~bole.FLAG_INLINE_TOPOLOGY
    calls = {"pack": lambda db, rb, cs: device.pack(db, rb, cs),
             "verify": lambda db, rb, cs: device.verify(db, rb, flags, cs),
             "commit": lambda db, rb, cs: device.commit(db, rb, cflags, cs)}
    if inline:
        del calls["pack"]
        per_kernel["pack"].append(0.0)
    for name, call in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for db, rb in (sets[:1] if flush_mode else sets):
                call(db, rb, cs)
        g.replay()
        torch.cuda.synchronize()
        if flush_mode:  # one call per flushed replay, each timed on its own
            reps = max(1, ks)
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(reps)]
            for a, b in pairs:
                flush_buf.fill_(0.0)
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            per_kernel[name].append(sum(a.elapsed_time(b) for a, b in pairs) / reps)
            continue
        reps = max(1, ks // n_sets)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        per_kernel[name].append(e0.elapsed_time(e1) / (reps * n_sets))
    for _, rb in sets:
        bole.check_status(rb.status, "per-kernel pass")
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    e2e = None if args.no_e2e else run_e2e(args, batch, sets, flags, stream, world, fz)
    res = {"_batch": batch, "_flags": flags & ~bole.FLAG_INLINE_TOPOLOGY,
           "_launches": launches_per_step * steps}
    if rank != 0:
        return res

    hbm, tflops, peak_kind = measured_peaks()
    ms_step = elapsed_ms / steps
    value = job_throughput(batch.N, steps, world, elapsed_ms)
    avg = {k: float(np.mean(v)) for k, v in per_kernel.items()}
    kern_rf = {}
    for k in ("pack", "verify", "commit") + (("commit_verify",) if fz else ()):
        if k == "pack" and inline:
            kern_rf[k] = {"ms": 0.0, "alg_bytes": 0, "note": "formed inside the verification"}
            continue
        gbs = alg[k] / (avg[k] * 1e-3) / 1e9 if avg[k] > 0 else 0.0
        kern_rf[k] = {"ms": round(avg[k], 5), "alg_bytes": int(alg[k]),
                      "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4)}
    dominant = "commit_verify" if fz else max(("verify", "commit"), key=lambda k: avg[k])
    step_gbs = step_bytes / (ms_step * 1e-3) / 1e9
    verify_kernels = (["tc_vtile_kernel"] if vtile else ["tc_verify_kernel"] if fused
                      else ["tc_big_fused_kernel"] if big else [])
    commit_kernels = ["tc_commit_kernel"] if tc_dims else []
    traffic = (recorded_traffic(["tc_commit_verify"] if fz else
                                verify_kernels if dominant == "verify" else commit_kernels,
                                workload_key(cfg, args.shape, batch.dtype)) if tc_used else None)
    roofline = {"bound": "hbm", "kernel": dominant,
                "achieved": kern_rf[dominant]["achieved_gbs"], "peak": hbm, "unit": "GB/s",
                "frac": kern_rf[dominant]["frac"], "traffic": traffic, "peak_source": peak_kind,
                "step_achieved_gbs": round(step_gbs, 1), "step_frac": round(step_gbs / hbm, 4),
                "verify_plus_commit_frac": round(
                    (alg["verify"] + alg["commit"]) / ((avg["verify"] + avg["commit"]) * 1e-3)
                    / 1e9 / hbm, 4)}

    cpu = None
    if not args.no_cpu_baseline:
        v, el, reps, thr = run_oracle_sample(batch, args.cpu_seconds)
        cpu = {"value": round(v, 1), "unit": "nodes/s", "cores": thr, "kind": "oracle",
               "sample": f"{reps} full repetition(s) of the workload's verify + commit "
                         f"({batch.N} nodes x {batch.H} heads each), {el:.1f} s"}

    res.update({
        "metric": METRIC, "value": round(value, 1), "unit": "nodes/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16x2+tf32 (f32 acc)" if tc_shape and tc_used
                  else "f32 as bf16x3 (6 products) + tf32x2 (f32 acc)" if tc_used else "f32"),
        "io_dtype": batch.dtype,
        "data": "synthetic",
        "config": {"workload": inputs.CONFIG_NAMES[cfg]
                   + (f" [{args.shape}]" if cfg == 4 else ""),
                   "config_index": cfg, "B": batch.B, "H": batch.H, "dk": batch.dk,
                   "dv": batch.dv, "nodes": batch.N, "max_depth": batch.max_depth,
                   "seed": seed,
                   "kernels": ("tcgen05 (one CTA per head), the previous round's commit "
                               "inside" if fz
                               else "tcgen05 value-tiled (two CTAs per head)" if vtile
                               else "tcgen05 (one CTA per head)" if fused
                               else "tcgen05 fused large-tree kernel" if big else "cuda-core"),
                   "round": ("one launch: the previous round's commit, then this round's "
                             "verify (topology inside) from the committed state "
                             "(bole_commit_verify)" if fz
                             else "verify (topology inside) -> commit" if inline
                             else "pack -> verify -> commit"),
                   "l2": (f"L2 flushed before every timed step (a {2 * L2_BYTES >> 20} MiB "
                          f"write outside the events; the inputs would need {need} copies)"
                          if flush_mode else
                          f"inputs rotate over {n_sets} copies (> 3x L2 between reuses)"),
                   "launch": ("CUDA graph replay: one graph per step, each step between its "
                              "own events" if flush_mode else
                              f"CUDA graph replay: one graph of {n_sets} rounds (one per input "
                              "copy), replayed while whole passes remain, then one graph per "
                              "remaining round"),
                   "kernel_timing": (f"separate pass: per call kind, one call per flushed "
                                     f"replay, {max(1, ks)} replays each between events"
                                     if flush_mode else
                                     f"separate pass: per call kind, a graph of one call on each "
                                     f"of the {n_sets} input copies, replayed "
                                     f"{max(1, ks // n_sets)}x between events")},
        "roofline": roofline, "kernels": kern_rf, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clock_info,
    })
    return res


def run_selection(stream):
    """Device-side proposal selection + forest build on drafts shaped like the
    ragged budgeted batch: 64 requests, 64..256 drafted candidates each (edge
    probabilities Dirichlet(1) over 1..4 children, depth <= 12), per-request
    caps U[8, 64], a budget of 2048 nodes.  Three small kernels, bound by
    latency rather than bandwidth; timed from a CUDA graph."""
    import torch
    from gated_deltanet_verification_gb300 import bole, inputs

    d = inputs.draft_candidates(2024, 64, 64, 256, 12)
    budget = 2048
    dev = torch.device("cuda", torch.cuda.current_device())

    def t(a, dt=torch.int32):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)

    p, co, cp, caps = t(d.p, torch.float32), t(d.cand_offsets), t(d.cand_parent), t(d.caps)
    off = torch.empty(d.B + 1, dtype=torch.int32, device=dev)
    par = torch.empty(budget, dtype=torch.int32, device=dev)
    src = torch.empty(budget, dtype=torch.int32, device=dev)
    rho = torch.empty(d.M, dtype=torch.float32, device=dev)
    ws = torch.empty(bole.lib().bole_select_workspace_size(d.B), dtype=torch.uint8, device=dev)
    st = bole.new_status(dev)

    def run():
        bole.select_forest(p, co, cp, budget, caps=caps, offsets=off, parent=par, src=src,
                           rho=rho, workspace=ws, status=st)

    run()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    g.replay()
    reps = 200
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    bole.check_status(st, "selection")
    ms = e0.elapsed_time(e1) / reps
    return {"requests": d.B, "candidates": d.M, "budget": budget,
            "nodes": int(off[-1].item()), "ms": round(ms, 5),
            "candidates_per_s": round(d.M / (ms * 1e-3), 1), "bound": "latency",
            "launches": 3}


def stage1_bytes(batch, W: int):
    """Algorithmic bytes of bole_conv_gates and bole_conv_commit per launch."""
    B, H, dk, dv, N = batch.B, batch.H, batch.dk, batch.dv, batch.N
    s_in = 2 if batch.dtype == "bf16" else 4
    C = H * (2 * dk + dv)
    topo = 4 * (B + 1) + 4 * N
    gates = (2 * N * C * s_in + B * (W - 1) * C * s_in + C * W * 4 + C * 4 + 16 * N * H
             + topo)
    L = path_lengths(batch)
    commit = int(np.sum(np.minimum(L, W - 1))) * C * s_in + 2 * int(np.sum(L > 0)) * (W - 1) * C \
        * s_in + topo + 4 * B
    return gates, commit


def run_stage1(args, batch, stream):
    """Stage 1 on this workload: bole_conv_gates (tree-parallel causal
    convolution of width W, SiLU, q/k normalisation, gates) and
    bole_conv_commit, each timed over input copies that rotate through more
    than 3x L2, from a CUDA graph of one launch per copy."""
    import torch
    from gated_deltanet_verification_gb300 import bole, inputs

    W = args.conv_width
    s = inputs.stage1_inputs(batch, W=W, seed=77)
    dev = torch.device("cuda", torch.cuda.current_device())
    dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    gb, cb = stage1_bytes(batch, W)
    n = max(2, int(np.ceil(3 * L2_BYTES / gb)) + 1)

    def t(a, d):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=d)

    offsets, parent = t(batch.offsets, torch.int32), t(batch.parent, torch.int32)
    accepted = t(batch.accepted, torch.int32)
    w, bias = t(s.conv_w, torch.float32), t(s.conv_b, torch.float32)
    ga, gbt = t(s.a, torch.float32), t(s.b, torch.float32)
    copies = [(t(s.x, dt), t(s.conv_state, dt)) for _ in range(n)]
    outs = [(torch.empty((batch.N, batch.H, batch.dk), dtype=dt, device=dev),
             torch.empty((batch.N, batch.H, batch.dk), dtype=dt, device=dev),
             torch.empty((batch.N, batch.H, batch.dv), dtype=dt, device=dev),
             torch.empty((batch.N, batch.H), dtype=torch.float32, device=dev),
             torch.empty((batch.N, batch.H), dtype=torch.float32, device=dev)) for _ in range(n)]
    st = bole.new_status(dev)

    def gates_all():
        for (x, cs), (q, k, v, g, bt) in zip(copies, outs):
            bole.conv_gates(x, cs, w, bias, ga, gbt, offsets, parent, batch.H, batch.dk,
                            batch.dv, max(batch.max_T, 1), q=q, k=k, v=v, gamma=g, beta=bt,
                            status=st)

    def commit_all():
        for x, cs in copies:
            bole.conv_commit(cs, x, offsets, parent, accepted, status=st)

    hbm, _, _ = measured_peaks()
    out = {"W": W, "copies": n}
    for name, fn, nbytes in (("conv_gates", gates_all, gb), ("conv_commit", commit_all, cb)):
        fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        reps = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * n)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "alg_bytes": int(nbytes), "achieved_gbs": round(gbs, 1),
                     "frac": round(gbs / hbm, 4)}
    bole.check_status(st, "stage 1")
    return out


def run_layers(args, batch, flags, stream):
    """Unified cross-layer commit on this workload: `args.layers` GDN layers
    (each its own S_pre and operands, one shared forest) verified into
    contiguous [layers, ...] factor buffers, then committed by ONE
    bole_commit_layers launch -- timed against the same layers committed by
    one bole_commit launch each.  Both in the default [dk, dv] state layout
    and in the slot layout [dv, dk] (BOLE_FLAG_STATE_VK).  The states of all
    layers (layers x B x H x 64 KB) exceed L2 for the batched workloads; each
    timing replays a CUDA graph of the launch(es)."""
    import torch
    from gated_deltanet_verification_gb300 import bole, inputs

    L = args.layers
    lbs = inputs.layer_batches(batch, L, seed=4242)
    dev = torch.device("cuda", torch.cuda.current_device())
    dt = torch.bfloat16 if batch.dtype == "bf16" else torch.float32

    def t(a, d):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=d)

    offsets, parent = t(batch.offsets, torch.int32), t(batch.parent, torch.int32)
    accepted = t(batch.accepted, torch.int32)
    depth, anc, req, st = bole.pack_forest(offsets, parent, batch.max_depth)
    k_all = torch.stack([t(lb.k, dt) for lb in lbs])
    U_all = torch.empty((L, batch.N, batch.H, batch.dv), dtype=torch.float32, device=dev)
    lp_all = torch.empty((L, batch.N, batch.H), dtype=torch.float32, device=dev)
    alg = 0
    for lb in lbs:
        alg += algorithmic(lb)["commit"]
    out = {"layers": L, "alg_bytes": int(alg)}
    hbm, _, _ = measured_peaks()
    for layout in ("kv", "vk"):
        f = flags | (bole.FLAG_STATE_VK if layout == "vk" else 0)
        S_all = torch.stack([t(lb.S_pre if layout == "kv" else lb.S_pre.transpose(0, 1, 3, 2),
                               torch.float32) for lb in lbs])
        for li, lb in enumerate(lbs):
            bole.tree_verify(S_all[li], t(lb.q, dt), k_all[li], t(lb.v, dt),
                             t(lb.gamma, torch.float32), t(lb.beta, torch.float32), offsets,
                             parent, depth, anc, req, max(batch.max_T, 1), batch.max_depth,
                             U=U_all[li], logP=lp_all[li], status=st, flags=f)
        torch.cuda.synchronize()
        bole.check_status(st, "layered verify")

        def one_launch():
            bole.commit_layers(S_all, k_all, U_all, lp_all, offsets, parent, accepted,
                               status=st, flags=f)

        def per_layer():
            for li in range(L):
                bole.commit(S_all[li], k_all[li], U_all[li], lp_all[li], offsets, parent,
                            accepted, status=st, flags=f)

        res = {}
        for name, fn in (("one_launch", one_launch), ("per_layer", per_layer)):
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            reps = 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res[name] = e0.elapsed_time(e1) / reps
        bole.check_status(st, "layered commit")
        gbs = alg / (res["one_launch"] * 1e-3) / 1e9
        out[layout] = {"ms_one_launch": round(res["one_launch"], 5),
                       "ms_per_layer_launches": round(res["per_layer"], 5),
                       "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4)}
    return out


def run_e2e(args, batch, sets, flags, stream, world, fz=False):
    """Same metric through the public API with host buffers: per step the
    round's inputs (tree, q/k/v, gates, accepted) are copied from pinned host
    memory, the round runs, and O and the status word are copied back to
    pinned host memory.  The state slots stay resident in HBM (they are the
    persistent per-request state the commit updates in place).

    The serving form: each input copy's per-round tensors are views of one
    packed device buffer, filled by ONE host-to-device copy per step from a
    packed pinned buffer on a copy stream; rounds run on the compute stream
    and the copy of step i+1 overlaps the round of step i (events order each
    copy after the round that last used its buffer, and each round after its
    copy).  The plain form -- eight copies, the round and the two copies back,
    all on one stream -- is reported beside it."""
    import torch
    from gated_deltanet_verification_gb300 import bole, device

    names = ["offsets", "parent", "q", "k", "v", "gamma", "beta", "accepted"]
    db0, rb0 = sets[0]
    # packed layout: every field 256-byte aligned
    layout, off = [], 0
    for n in names:
        t = getattr(db0, n)
        nbytes = t.numel() * t.element_size()
        layout.append((n, off, t.dtype, tuple(t.shape), nbytes))
        off = (off + nbytes + 255) // 256 * 256
    total = off
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n, o, dt, shape, nb in layout:
        host[o:o + nb].copy_(getattr(db0, n).cpu().contiguous().view(-1).view(torch.uint8))
    packs = []
    for db, _ in sets:
        buf = torch.empty(total, dtype=torch.uint8, device=db.q.device)
        for n, o, dt, shape, nb in layout:
            view = buf[o:o + nb].view(dt).view(shape)
            view.copy_(getattr(db, n))
            setattr(db, n, view)
        packs.append(buf)
    par = [0] * len(sets)  # fused rounds: each copy's U / logP parity

    def round_(k, db, rb, cs):
        if fz:
            device.commit_verify_round(db, rb, par[k], cs)
            par[k] ^= 1
        else:
            device.run_round(db, rb, flags, cs)

    O_host = torch.empty_like(rb0.O, device="cpu").pin_memory()
    st_host = torch.empty_like(rb0.status, device="cpu").pin_memory()
    h2d = total
    d2h = O_host.numel() * O_host.element_size() + st_host.numel() * st_host.element_size()
    n_sets = len(sets)

    def timed(run, steps, side=None):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        if side is not None:  # work on a side stream starts inside the timed region too
            side.wait_event(start)
        for i in range(steps):
            run(i)
        end.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(start.elapsed_time(end), "cuda")

    # plain form: one stream, the packed copy included in line
    def plain(i):
        db, rb = sets[i % n_sets]
        packs[i % n_sets].copy_(host, non_blocking=True)
        round_(i % n_sets, db, rb, torch.cuda.current_stream())
        O_host.copy_(rb.O, non_blocking=True)
        st_host.copy_(rb.status, non_blocking=True)

    for i in range(args.warmup):
        plain(i)
    plain_steps = min(args.steps, 2000)
    ms_plain = timed(plain, plain_steps)

    # serving form: copy stream + compute stream, one packed copy per step
    copy_stream = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(n_sets)]
    free = [torch.cuda.Event() for _ in range(n_sets)]
    for e in free:
        e.record(stream)

    def pipelined(i):
        k = i % n_sets
        db, rb = sets[k]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[k])
            packs[k].copy_(host, non_blocking=True)
            ready[k].record(copy_stream)
        stream.wait_event(ready[k])
        round_(k, db, rb, stream)
        O_host.copy_(rb.O, non_blocking=True)
        st_host.copy_(rb.status, non_blocking=True)
        free[k].record(stream)

    for i in range(args.warmup):
        pipelined(i)
    torch.cuda.synchronize()
    ms = timed(pipelined, args.steps, side=copy_stream)
    for _, rb in sets:
        bole.check_status(rb.status, "e2e steps")
    return {"value": round(job_throughput(batch.N, args.steps, world, ms), 1), "unit": "nodes/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / args.steps, 5),
            "mode": "per step: one pinned-host -> device copy of the round's packed inputs on a "
                    "copy stream (overlapping the previous round), the round (" +
                    ("the previous round's commit and this round's verify in one launch" if fz
                     else "verify with the topology step inside, commit"
                     if flags & bole.FLAG_INLINE_TOPOLOGY
                     else "pack, verify, commit") + "), O and status back to pinned host memory",
            "plain": {"value": round(job_throughput(batch.N, plain_steps, world, ms_plain), 1),
                      "ms_per_step": round(ms_plain / plain_steps, 5),
                      "mode": "the same copies and calls, all on one stream"}}


def reference_arm(args, world, rank):
    """The CPU oracle timed on the host cores, same workload and metric.  Each
    step runs the oracle's verify + commit over a rotating slice of the
    (request, head) units, sized so the whole run stays within about a minute;
    nodes/s counts node-heads processed divided by the head count."""
    if rank != 0:
        return 0
    from gated_deltanet_verification_gb300 import inputs
    batch = inputs.config_batch(args.config, shape=args.shape)
    import oracle
    oracle.load()
    thr = oracle.default_threads()
    units = batch.B * batch.H
    sizes = np.diff(batch.offsets)
    prep = oracle.Prepared(batch, nthreads=thr)  # converted once, outside the timed steps

    def run(u0, u1):
        prep.verify(u0, u1)
        prep.commit(u0, u1)
        return int(sum(sizes[u // batch.H] for u in range(u0, u1)))

    probe_units = min(units, max(1, 4 * thr))
    run(0, probe_units)  # first touch of the converted arrays
    t0 = time.perf_counter()
    run(0, probe_units)
    t_unit = (time.perf_counter() - t0) / probe_units
    budget_s = 60.0
    # at least one unit per host thread per step (else the cores idle), at most
    # the whole batch, else what keeps the timed steps near the budget
    per_step = int(max(min(units, thr),
                       min(units, budget_s / max(1, args.steps) / max(t_unit, 1e-9))))
    for w in range(max(0, min(args.warmup, 2))):
        run(0, per_step)
    node_heads, u0 = 0, 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        u1 = min(units, u0 + per_step)
        node_heads += run(u0, u1)
        u0 = 0 if u1 >= units else u1
    el = time.perf_counter() - t0
    value = node_heads / batch.H / el
    sample = (f"{per_step} of {units} (request, head) units per step, rotating; "
              f"{node_heads} node-heads in {el:.1f} s")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "nodes/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": inputs.CONFIG_NAMES[args.config]
                   + (f" [{args.shape}]" if args.config == 4 else ""),
                   "config_index": args.config, "B": batch.B, "H": batch.H, "dk": batch.dk,
                   "dv": batch.dv, "nodes": batch.N},
        "cpu_baseline": {"value": round(value, 1), "unit": "nodes/s", "cores": thr,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "nodes/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
