#!/usr/bin/env python
"""Benchmark of the full Barnes-Hut step on one GB300 (per rank).

A step is one bh_compute: bounding cube -> Morton keys -> radix sort +
reorder -> octree build -> centre of mass -> warp-cooperative walk -> results
in caller order, over the whole workload already resident in HBM, with the
library's defaults (a repeated identical call replays its captured CUDA
graph).  A second loop launches the same step kernel by kernel with
per-stage events for the stage breakdown (``eager_ms_per_step``).  The
default workload is the 1,000,000-particle lattice (100^3, spacing 0.01,
masses 1e-6, eps 5e-3, theta 0.5) in shuffled order (permutation seed 1).

metric: useful interactions per second over the full step, where "useful" is
the per-target Barnes-Hut interaction count (accepted cells + particle
pairs) of the same tree and theta, counted on the GPU outside the timed
region.  The group walk evaluates a superset of those terms; the roofline
object reports the executed terms as fp32 FLOP/s (20 flops per term).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

With N > 1 (launched by torch.distributed.run) the ranks split one problem
(--split targets, the default): every rank builds the whole tree from the
replicated sources, walks its contiguous share of the Morton-ordered target
groups, and an all-reduce of zero-filled result buffers gives every rank all
rows in caller order, inside each timed step; value is the problem's useful
interactions divided by the slowest rank's time ("scaling": "strong").
--split replicas runs a whole replica per rank instead ("weak").

The default run also times the 5,000,000-particle galaxy pair (reported
under "also"); --also names other workloads, or none.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FLOPS_PER_TERM = 20
# fp32 peak from unit counts and clock: 152 SMs x 128 FP32 lanes x 2 flop
# (FMA) x 2070 MHz (maximum SM clock).
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0
# Up to this many keys the radix sort is one kernel (all passes in one block).
ONE_BLOCK_SORT_MAX = 4096
# Up to this many 63-bit keys the sort tries the bucket path (256 top-digit
# buckets of at most 4608 keys each).
BUCKET_SORT_MAX = 256 * 4608


def kernels_per_step(order: str, n: int, m: int | None, sms: int = 152,
                     scheduled: bool = True) -> int:
    """Our kernels per step (63-bit source keys, 30-bit target keys): per
    particle set (n sources, and m separate targets unless m is None) bbox,
    keys and the order (order_kernels; or the tree order's histogram, top
    levels, insert, node count, count and place kernels); then build
    count/scan/write/tile prefix, centre of mass and children factors, the
    group schedule (on a repeated call with more walk groups than 16 per SM)
    and walk."""
    def per_set(rows: int, key_bits: int) -> int:
        if order != "radix":
            return 2 + 6
        return 2 + order_kernels(rows, key_bits)
    targets = n if m is None else m
    groups = -(-targets // walk_group(targets))
    sched = 2 if scheduled and groups > 16 * sms else 0     # class counts, placement
    return per_set(n, 63) + (0 if m is None else per_set(m, 30)) + 7 + sched


def order_kernels(rows: int, key_bits: int) -> int:
    """Kernels of the radix order (sort + gather) of one particle set: one
    kernel up to ONE_BLOCK_SORT_MAX keys, else one pass per 8 key bits,
    preceded for 63-bit keys by the top-digit pass and the bucket sort while
    the 256 top-digit buckets can all fit (rows <= BUCKET_SORT_MAX; the digit
    passes and the gather then return at once if the bucket sort ran),
    + gather."""
    if rows <= ONE_BLOCK_SORT_MAX:
        return 2
    passes = (key_bits + 7) // 8
    bucket = 2 if key_bits == 63 and rows <= BUCKET_SORT_MAX else 0
    return bucket + passes + 1


# DRAM bytes per walk launch from the committed ncu capture of the same
# kernel (profiles/); None until a capture of the current kernel exists.
WALK_TRAFFIC_BYTES = 29.84e6    # walk_ws_kernel<2,vote> on lattice1m_shuffled, from that capture
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="default lattice1m_shuffled (surface2e20 with --stochastic)")
    ap.add_argument("--theta", type=float, default=None,
                    help="override the workload's opening angle")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--also", default=None,
                    help="comma-separated workloads timed after the headline one and "
                         "reported under 'also' (default galaxy5m with the default "
                         "workload, else none)")
    ap.add_argument("--split", choices=["targets", "replicas"], default="targets",
                    help="N > 1: split one problem's target groups over the ranks "
                         "(default), or run a whole replica per rank")
    ap.add_argument("--cpu-sample", type=int, default=4096,
                    help="targets the CPU oracle walks per baseline step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--direct", action="store_true",
                    help="time the brute-force kernel (bh_direct) on the workload instead")
    ap.add_argument("--integrate", action="store_true",
                    help="time leapfrog simulation steps (bh_leapfrog) instead")
    ap.add_argument("--dt", type=float, default=1e-4)
    ap.add_argument("--stochastic", action="store_true",
                    help="time the stochastic Barnes-Hut estimator (default workload "
                         "surface2e20) beside the deterministic walk")
    ap.add_argument("--neighbors", action="store_true",
                    help="time the SPH neighbour search (bh_neighbors with lists) on "
                         "a Plummer sphere with density-based smoothing lengths")
    ap.add_argument("--nb-n", type=int, default=1 << 20)
    ap.add_argument("--samples", type=int, default=1)
    ap.add_argument("--strata-level", type=int, default=2)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--fused-walk", action="store_true",
                    help="one warp per group both traverses and evaluates (BH_OPT_PIPELINE 0) "
                         "instead of the default producer/consumer warp pairs")
    ap.add_argument("--order", choices=["radix", "tree"], default="radix",
                    help="spatial sort: radix sort (default) or the tree-topology order "
                         "of an insertion-built tree (BH_ORDER_TREE)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed helpers (host logic; exercised by a gloo test on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (the one leg allowed to run oracle/)
# ---------------------------------------------------------------------------
def cpu_oracle_step(src, tgt, G, eps, theta, sample: int, leaf_cap: int = 16,
                    with_measured: bool = False):
    """One oracle step on a bounded sample: the whole build over all sources,
    then the per-target walk of `sample` targets; the walk time is scaled to
    all targets.  Returns (seconds for a full step, useful terms per step),
    and with `with_measured` also the seconds the sampled step took."""
    import numpy as np
    import oracle as O
    import workloads as W
    t0 = time.perf_counter()
    o = O.OracleBH(src, theta=theta, G=G, eps=eps, leaf_cap=leaf_cap)
    t1 = time.perf_counter()
    m = src.shape[0] if tgt is None else tgt.shape[0]
    idx = W.error_sample(m, sample, seed=5)
    _, terms = o.bh(tgt, idx=idx)
    t2 = time.perf_counter()
    scale = m / idx.shape[0]
    full = (t1 - t0) + (t2 - t1) * scale
    if with_measured:
        return full, float(terms.mean()) * m, t2 - t0
    return full, float(terms.mean()) * m


def cpu_oracle_stages(src, tgt, G, eps, theta, sample: int = 4096,
                      direct_sample: int = 256, leaf_cap: int = 16) -> dict:
    """The oracle's stages timed one by one (seconds for the whole problem):
    bounding cube + Morton keys, stable sort + reorder, octree build, centre
    of mass, the per-target walk of `sample` targets and the fp64 direct sum
    of `direct_sample` targets, both scaled to all targets (the direct sum is
    an extrapolation)."""
    import numpy as np
    import oracle as O
    import workloads as W
    t = [time.perf_counter()]
    cube = O.bbox(src)
    k = O.keys(src, cube, 21)
    t.append(time.perf_counter())
    perm = O.sort(k)
    sk = k[perm]
    spm = np.ascontiguousarray(src[perm])
    t.append(time.perf_counter())
    tree = O.build_tree(sk, 21, leaf_cap)
    t.append(time.perf_counter())
    O.com(spm, sk, tree, cube, 21)
    t.append(time.perf_counter())
    o = O.OracleBH(src, theta=theta, G=G, eps=eps, leaf_cap=leaf_cap)
    m = src.shape[0] if tgt is None else tgt.shape[0]
    idx = W.error_sample(m, sample, seed=5)
    t.append(time.perf_counter())
    o.bh(tgt, idx=idx)
    t.append(time.perf_counter())
    didx = idx[:min(direct_sample, idx.shape[0])]
    o.direct(tgt, idx=didx)
    t.append(time.perf_counter())
    st = {"bbox_keys": t[1] - t[0], "sort_reorder": t[2] - t[1], "build": t[3] - t[2],
          "com": t[4] - t[3], "walk": (t[6] - t[5]) * m / idx.shape[0],
          "direct_extrapolated": (t[7] - t[6]) * m / didx.shape[0]}
    st["step"] = st["bbox_keys"] + st["sort_reorder"] + st["build"] + st["com"] + st["walk"]
    return {k: round(v, 4) for k, v in st.items()}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, on this workload."""
    if rank != 0:
        return 0
    import oracle as O
    import workloads as W
    src, tgt, G, eps, theta = W.make(args.workload)
    theta = args.theta if args.theta is not None else theta
    for _ in range(args.warmup):
        cpu_oracle_step(src, tgt, G, eps, theta, args.cpu_sample)
    secs, measured, useful = [], [], 0.0
    for _ in range(args.steps):
        s, useful, t = cpu_oracle_step(src, tgt, G, eps, theta, args.cpu_sample,
                                       with_measured=True)
        secs.append(s)
        measured.append(t)
    # the rate is the whole problem's (the sampled walk scaled to every
    # target); ms_per_step is what each timed step took on the host
    full_ms = 1e3 * statistics.mean(secs)
    ms = 1e3 * statistics.mean(measured)
    value = useful / (full_ms / 1e3)
    m = src.shape[0] if tgt is None else tgt.shape[0]
    sample = (f"build over all {src.shape[0]} sources + per-target walk of "
              f"{min(args.cpu_sample, m)} sampled targets per step (ms_per_step); "
              f"value = the whole problem's useful terms over that step with the walk "
              f"time scaled to {m} targets (ms_per_step_full_extrapolated)")
    line = {
        "impl": "reference", "metric": "useful_interactions_per_s", "value": value,
        "unit": "interactions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_full_extrapolated": full_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, src, tgt, theta, eps, args.order,
                                  args.fused_walk),
        "cpu_baseline": {"value": value, "unit": "interactions/s", "cores": O.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "interactions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def measured_fp32_tflops(ctx, stream, iters: int = 1 << 16, reps: int = 5) -> dict:
    """Measured fp32 peak: the library's FMA-chain probe (bh_fp32_probe), in
    scalar and packed (fma.rn.f32x2) form, 3 untimed launches then the best
    of `reps`, each timed with CUDA events on the launching stream."""
    import torch
    import barnes_hut_body_gb300 as B
    out = {}
    for name, packed in (("scalar", False), ("packed", True)):
        for _ in range(3):
            flops = B.bh_fp32_probe(ctx, packed, iters, stream.cuda_stream)
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            B.bh_fp32_probe(ctx, packed, iters, stream.cuda_stream)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        out[name] = flops / (best / 1e3) / 1e12
    return out


def measured_hbm_gbs() -> float:
    """HBM copy bandwidth measured on this GPU pool (generated file),
    else the fallback figure for a GB300."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return 6800.0


def stage_bytes(n: int, m: int, nodes: int, self_mode: bool, order: str = "radix") -> dict:
    """Algorithmic DRAM bytes of each build-side stage for one step (63-bit
    keys, 8 radix passes): what the stage must read and write at least --
    bbox 16 B per particle; keys 16 in + 8 out; a radix pass 24 B per
    element; reorder 36; build 8 B per key + 32 B per node; centre of mass
    16 B per particle + 32 B per node.  The tree order's "sort" is the
    insertion tree: keys read, and per row at least one 4-byte child slot
    written and its count and offset settled (12 bytes); its "reorder" reads
    keys and rows and writes the sorted key, index and row (8 + 16 in,
    8 + 4 + 16 out)."""
    sort = 8 * 24 * n if order == "radix" else 8 * n + 12 * n
    reorder = 4 * n + 16 * n + 16 * n if order == "radix" else 24 * n + 28 * n
    b = {
        "bbox": 16 * n,
        "keys": 16 * n + 8 * n,
        "sort": sort,
        "reorder": reorder,
        "build": 8 * n + 32 * nodes,
        "com": 16 * n + 32 * nodes,
    }
    if not self_mode:
        tsort = 8 * 24 * m + 36 * m if order == "radix" else 20 * m + 52 * m
        b["targets"] = 16 * m + 24 * m + tsort
    return b


def kernel_bytes(n: int, m: int, nodes: int) -> dict:
    """Bytes the build and centre-of-mass kernels move by their design: the
    build reads the keys in its count and write passes and writes 25 B of
    topology per node; the centre of mass reads the particles, 33 B of
    topology per node and writes a 32-byte record and 4 more per node."""
    return {"build": 2 * 8 * n + 25 * nodes, "com": 16 * n + 69 * nodes}


def walk_group(m: int) -> int:
    """The library's default group size for m targets (BH_OPT_GROUP 0): 64,
    or 32 when m fills fewer groups of 64 than 16 per SM."""
    sms = 152
    try:
        import torch
        if torch.cuda.is_available():
            sms = torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 32 if (m + 63) // 64 < 16 * sms else 64


def workload_config(name, src, tgt, theta, eps, order="radix", fused=False, shards=1):
    m = int(src.shape[0] if tgt is None else tgt.shape[0])
    extra = {} if shards == 1 else {
        "parallelism": f"targets split over {shards} ranks: sources replicated, each rank "
                       "builds the whole tree and walks 1/N of the target groups; rows "
                       "combined by an all-reduce of zero-filled buffers"}
    return {"workload": name, "n_sources": int(src.shape[0]), **extra,
            "n_targets": m,
            "theta": theta, "eps": eps, "opening": f"warp vote, groups of {walk_group(m)}",
            "walk": "fused" if fused else "producer/consumer warp pairs",
            "leaf_cap": 16, "key_bits": 63, "order": order,
            **({} if tgt is None else {"target_key_bits": 30}),
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def shard_groups(ngroups: int, shards: int, shard: int) -> tuple[int, int]:
    """The walk groups [G s / S, G (s + 1) / S) that shard s of S walks
    (integer division; the library's BH_OPT_SHARDS rule)."""
    return ngroups * shard // shards, ngroups * (shard + 1) // shards


def gather_rows(out, world: int) -> None:
    """Give every rank all result rows, in caller order.  Each rank's buffer
    holds the rows of the groups its shard walked and +0.0 in every other
    row, so a sum over ranks reproduces each row exactly (x + 0 = x in IEEE
    arithmetic, whatever order the collective adds in)."""
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(out, op=dist.ReduceOp.SUM)


def gpu_stage_medians(stage_times: list[dict]) -> dict:
    """Per-stage medians (ms) of the GPU stage times of the timed steps
    (bh_get_stage_times, one dict per step)."""
    return {k: statistics.median(s[k] for s in stage_times) for k in stage_times[0]}


def stage_hbm(stages_ms: dict, nbytes: dict, peak_gbs: float) -> dict:
    gbs = {k: nbytes[k] / (stages_ms[k] * 1e-3) / 1e9
           for k in nbytes if stages_ms.get(k, 0) > 0}
    return {"unit": "GB/s", "peak": peak_gbs,
            "achieved": {k: round(v, 1) for k, v in gbs.items()},
            "frac": {k: round(v / peak_gbs, 3) for k, v in gbs.items()}}


def measure_workload(name, args, device, rank, local_rank, world, split: bool,
                     e2e_steps: int):
    """Time one workload: the headline loop (library defaults, so a
    repeated call replays its captured graph), the per-stage loop, and the
    end-to-end loop from pinned host memory.  With split (N > 1) every rank
    builds the whole tree from the replicated sources, walks its shard of the
    target groups into a zeroed buffer, and the rows are combined over the
    ranks (gather_rows) inside every timed step."""
    import torch

    import barnes_hut_body_gb300 as B
    import workloads as W

    src, tgt, G, eps, theta = W.make(name)
    theta = args.theta if args.theta is not None else theta
    m = src.shape[0] if tgt is None else tgt.shape[0]
    d_src = torch.from_numpy(src).to(device)
    d_tgt = None if tgt is None else torch.from_numpy(tgt).to(device)
    d_out = torch.zeros((m, 4), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    order = B.BH_ORDER_TREE if args.order == "tree" else B.BH_ORDER_RADIX
    opts = dict(theta=theta, G=G, eps=eps, device=local_rank, timing=1, order=order,
                pipeline=0 if args.fused_walk else 1)
    if split:
        opts.update(shards=world, shard=rank)
    bh = B.BarnesHut(**opts)

    def step(out=d_out, s_in=d_src, t_in=d_tgt):
        if split:
            out.zero_()
        bh.compute(s_in, t_in, out)
        if split:
            gather_rows(out, world)

    for _ in range(max(args.warmup, 3)):
        step()
    if bh.status() != 0:
        raise RuntimeError(f"warm-up failed: {B.bh_last_error(bh.ctx)}")
    useful = B.bh_count_interactions(bh.ctx)          # all targets, every shard
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]

    # breakdown: the step with per-stage CUDA events (launched kernel by
    # kernel, since events cannot be recorded inside the captured graph)
    stage_list, executed = [], []
    barrier(world, device)
    torch.cuda.synchronize(device)
    for k in range(args.steps):
        flush.fill_(float(k))                    # evict L2 (untimed)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
        stage_list.append(B.bh_get_stage_times(bh.ctx))   # waits for the step
        executed.append(B.bh_get_counters(bh.ctx)[0])
    torch.cuda.synchronize(device)
    if bh.status() != 0:
        raise RuntimeError(f"timed steps failed: {B.bh_last_error(bh.ctx)}")
    eager_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, device)

    # headline: the library's defaults (no stage events)
    B.bh_set_option(bh.ctx, B.BH_OPT_TIMING, 0)
    for _ in range(3):
        step()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    barrier(world, device)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.start()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(float(k))
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    barrier(world, device)
    clocks = sampler.stop() if sampler else None
    if bh.status() != 0:
        raise RuntimeError(f"timed steps failed: {B.bh_last_error(bh.ctx)}")
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, device)
    # one problem split over the ranks: its useful terms; replicas: the sum
    total_useful = useful if split else sum_over_ranks(useful, world, device)

    # end to end from pinned host memory, with the library's defaults
    h_src = torch.from_numpy(src).pin_memory()
    h_tgt = None if tgt is None else torch.from_numpy(tgt).pin_memory()
    h_out = torch.empty((m, 4), dtype=torch.float32).pin_memory()

    def e2e_step():
        if not split:
            B.bh_compute_host(bh.ctx, h_src, h_tgt, h_out, stream.cuda_stream)
            return
        d_src.copy_(h_src, non_blocking=True)
        if h_tgt is not None:
            d_tgt.copy_(h_tgt, non_blocking=True)
        step()
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):                   # the second identical call captures the graph
        e2e_step()
    barrier(world, device)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_ms = max_over_ranks(1e3 * (time.perf_counter() - t0) / e2e_steps, world, device)
    h2d = 16 * (src.shape[0] + (0 if tgt is None else tgt.shape[0]))

    stages = gpu_stage_medians(stage_list)
    walk_ms = stages["traverse"]
    nodes = int(B.bh_debug_export(bh.ctx, B.BH_EXPORT_NODE_COUNT)[0])
    hbm_peak = measured_hbm_gbs()
    exec_terms = statistics.median(executed)
    props = torch.cuda.get_device_properties(device)
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
    achieved = exec_terms * FLOPS_PER_TERM / (walk_ms / 1e3) / 1e12
    traffic = WALK_TRAFFIC_BYTES if (not args.fused_walk and args.order == "radix"
                                     and name == "lattice1m_shuffled" and not split) else None
    res = {
        "ms_per_step": ms, "eager_ms_per_step": eager_ms,
        "stage_ms": {k: round(v, 4) for k, v in stages.items()},
        "useful_per_step": useful, "executed_per_step": exec_terms, "nodes": nodes,
        "value": total_useful / (ms / 1e3),
        "stage_hbm": stage_hbm(stages, stage_bytes(src.shape[0], m, nodes, tgt is None,
                                                   args.order), hbm_peak),
        "stage_hbm_kernel_bytes": stage_hbm(stages, kernel_bytes(src.shape[0], m, nodes),
                                            hbm_peak),
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "kernel": "walk_kernel<2,vote>" if args.fused_walk
                               else "walk_ws_kernel<2,vote>",
                     "peak_note": "fp32 FMA: SMs x 128 lanes x 2 x 2070 MHz"},
        "e2e": {"value": total_useful / (e2e_ms / 1e3), "unit": "interactions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 16 * m,
                "ms_per_step": e2e_ms},
        "gpu_launches": kernels_per_step(args.order, src.shape[0],
                                         None if tgt is None else tgt.shape[0],
                                         props.multi_processor_count,
                                         scheduled=not split) * args.steps,
        "clocks": clocks, "wall_s_timed": wall,
        "config": workload_config(name, src, tgt, theta, eps, args.order, args.fused_walk,
                                  shards=world if split else 1),
    }
    return res, bh, stream, (src, tgt, G, eps, theta)


def run_ours(args, rank, local_rank, world):
    import torch

    import barnes_hut_body_gb300 as B

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    split = world > 1 and args.split == "targets"
    res, bh, stream, (src, tgt, G, eps, theta) = measure_workload(
        args.workload, args, device, rank, local_rank, world, split, args.e2e_steps)
    probe = measured_fp32_tflops(bh.ctx, stream)
    bh.close()
    peak_meas = max(probe.values())
    res["roofline"].update(peak_measured=peak_meas,
                           frac_measured=res["roofline"]["achieved"] / peak_meas,
                           probe_tflops=probe)
    also = {}
    for name in [a for a in args.also.split(",") if a and a != "none" and a != args.workload]:
        r, b2, _, _ = measure_workload(name, args, device, rank, local_rank, world, split,
                                       min(args.e2e_steps, 3))
        b2.close()
        r["roofline"].update(frac_measured=r["roofline"]["achieved"] / peak_meas)
        also[name] = {k: r[k] for k in ("config", "ms_per_step", "eager_ms_per_step", "value",
                                        "stage_ms", "useful_per_step", "executed_per_step",
                                        "nodes", "stage_hbm", "roofline", "e2e", "clocks",
                                        "gpu_launches")}

    if rank == 0:
        m = src.shape[0] if tgt is None else tgt.shape[0]
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            import oracle as O
            s, u = cpu_oracle_step(src, tgt, G, eps, theta, args.cpu_sample)
            cores = O.num_threads()
            cpu_stages = cpu_oracle_stages(src, tgt, G, eps, theta, args.cpu_sample)
            O.set_threads(1)
            cpu_stages1 = cpu_oracle_stages(src, tgt, G, eps, theta, args.cpu_sample)
            O.set_threads(cores)
            cpu = {"value": u / s, "unit": "interactions/s", "cores": cores,
                   "kind": "oracle",
                   "sample": f"build over all {src.shape[0]} sources + per-target walk of "
                             f"{min(args.cpu_sample, m)} sampled targets, walk time scaled to {m}",
                   "stages_s": cpu_stages,
                   "one_core": {"value": u / cpu_stages1["step"], "cores": 1,
                                "stages_s": cpu_stages1},
                   "stages_note": "each stage timed alone over the whole problem; walk of "
                                  f"{min(args.cpu_sample, m)} and fp64 direct sum of "
                                  f"{min(256, m)} sampled targets, scaled to {m} "
                                  "(direct: extrapolated)"}
        line = {
            "metric": "useful_interactions_per_s", "value": res["value"],
            "unit": "interactions/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "strong" if split else "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": res["config"],
            **{k: res[k] for k in ("eager_ms_per_step", "stage_ms", "useful_per_step",
                                   "executed_per_step", "nodes", "stage_hbm",
                                   "stage_hbm_kernel_bytes", "roofline", "e2e",
                                   "gpu_launches", "clocks", "wall_s_timed")},
            "stage_bytes_note": "stage_hbm: the algorithmic bytes per unit (bbox 16/particle, "
                                "keys 24, sort 24 per pass and element, reorder 36, build "
                                "8/key + 32/node, CoM 16/particle + 32/node); "
                                "stage_hbm_kernel_bytes: what the build and CoM kernels "
                                "read and write by design (keys read twice + 25/node; "
                                "16/particle + 69/node)",
        }
        if also:
            line["also"] = also
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    return 0


def run_direct(args, rank, local_rank, world):
    """Brute-force kernel on the workload: pairs/s and its fp32 roofline."""
    import torch

    import barnes_hut_body_gb300 as B
    import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    src, tgt, G, eps, theta = W.make(args.workload)
    theta = args.theta if args.theta is not None else theta
    n = src.shape[0]
    m = n if tgt is None else tgt.shape[0]
    pairs = n * (n - 1) if tgt is None else n * m
    d_src = torch.from_numpy(src).to(device)
    d_tgt = None if tgt is None else torch.from_numpy(tgt).to(device)
    d_out = torch.empty((m, 4), dtype=torch.float32, device=device)
    bh = B.BarnesHut(theta=theta, G=G, eps=eps, device=local_rank)
    for _ in range(max(args.warmup, 3)):
        bh.direct(d_src, d_tgt, d_out)
    if bh.status() != 0:
        raise RuntimeError(B.bh_last_error(bh.ctx))
    stream = torch.cuda.current_stream(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world, device)
    torch.cuda.synchronize(device)
    for k in range(args.steps):
        ev[k][0].record(stream)
        bh.direct(d_src, d_tgt, d_out)
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, device)
    props = torch.cuda.get_device_properties(device)
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
    achieved = pairs * FLOPS_PER_TERM / (ms / 1e3) / 1e12
    probe = measured_fp32_tflops(bh.ctx, stream)
    peak_meas = max(probe.values())
    if rank == 0:
        print(json.dumps({
            "metric": "direct_pairs_per_s", "value": sum_over_ranks(pairs, world, device) / (ms / 1e3),
            "unit": "pairs/s", "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "n_sources": n, "n_targets": m, "eps": eps,
                       "kernel": "direct (fp32 tiles, fp64 across tiles)"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "peak_note": "fp32 FMA: SMs x 128 lanes x 2 x 2070 MHz",
                         "peak_measured": peak_meas, "frac_measured": achieved / peak_meas,
                         "probe_tflops": probe},
            "gpu_launches": 2 * args.steps}), flush=True)
    bh.close()
    return 0


def run_integrate(args, rank, local_rank, world):
    """Leapfrog simulation steps: kick + drift, tree gravity, kick."""
    import numpy as np
    import torch

    import barnes_hut_body_gb300 as B
    import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    src, tgt, G, eps, theta = W.make(args.workload)
    theta = args.theta if args.theta is not None else theta
    if tgt is not None:
        raise SystemExit("--integrate needs a self-gravity workload")
    n = src.shape[0]
    d_pm = torch.from_numpy(src).to(device)
    d_v = torch.zeros((n, 4), dtype=torch.float32, device=device)
    d_a = torch.zeros((n, 4), dtype=torch.float32, device=device)
    bh = B.BarnesHut(theta=theta, G=G, eps=eps, device=local_rank)
    B.bh_leapfrog(bh.ctx, d_pm, d_v, d_a, args.dt, max(args.warmup, 3))
    if bh.status() != 0:
        raise RuntimeError(B.bh_last_error(bh.ctx))
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    e0.record(stream)
    B.bh_leapfrog(bh.ctx, d_pm, d_v, d_a, args.dt, args.steps, acc_valid=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    useful = B.bh_count_interactions(bh.ctx)
    if rank == 0:
        print(json.dumps({
            "metric": "leapfrog_steps_per_s", "value": world * 1e3 / ms, "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "useful_interactions_per_s": sum_over_ranks(useful, world, device) / (ms / 1e3),
            "config": dict(workload_config(args.workload, src, tgt, theta, eps), dt=args.dt,
                           step="kick+drift, tree gravity, kick",
                           l2="not flushed: one bh_leapfrog call advances all timed steps "
                              "(the particles move, so every step rebuilds the tree)")}),
              flush=True)
    bh.close()
    return 0


def run_stochastic(args, rank, local_rank, world):
    """Stochastic Barnes-Hut steps (page "Stochastic Barnes-Hut Approximation
    for Fast Summation on the GPU") timed beside the deterministic walk on the
    same workload, with the potential's absolute error against the direct sum
    on sampled targets (the page's table reports mean / median / max absolute
    error of the potential and the time)."""
    import numpy as np
    import torch

    import barnes_hut_body_gb300 as B
    import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    src, tgt, G, eps, theta = W.make(args.workload)
    theta = args.theta if args.theta is not None else theta
    n = src.shape[0]
    m = n if tgt is None else tgt.shape[0]
    d_src = torch.from_numpy(src).to(device)
    d_tgt = None if tgt is None else torch.from_numpy(tgt).to(device)
    d_out = torch.empty((m, 4), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    rows = W.error_sample(m, 4096, seed=7)
    d_rows = torch.from_numpy(rows).to(device)
    ref = B.BarnesHut(theta=theta, G=G, eps=eps, device=local_rank)
    exact = ref.direct(d_src, d_src[d_rows] if d_tgt is None else d_tgt[d_rows])
    exact = exact.cpu().numpy().astype(np.float64)
    ref.close()
    stream = torch.cuda.current_stream(device)

    def timed(bh):
        for _ in range(max(args.warmup, 3)):
            bh.compute(d_src, d_tgt, d_out)
        if bh.status() != 0:
            raise RuntimeError(B.bh_last_error(bh.ctx))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(world, device)
        torch.cuda.synchronize(device)
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            bh.compute(d_src, d_tgt, d_out)
            ev[k][1].record(stream)
        torch.cuda.synchronize(device)
        ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, device)
        executed, _ = B.bh_get_counters(bh.ctx)
        got = d_out.index_select(0, d_rows).cpu().numpy().astype(np.float64)
        e = np.abs(got[:, 3] - exact[:, 3])
        return ms, executed, dict(mean=float(e.mean()), median=float(np.median(e)),
                                  max=float(e.max()))

    sto = B.BarnesHut(theta=theta, G=G, eps=eps, device=local_rank,
                      estimator=B.BH_EST_STOCHASTIC, samples=args.samples,
                      strata_level=args.strata_level, seed=args.seed)
    ms_s, ex_s, err_s = timed(sto)
    sto.close()
    det = B.BarnesHut(theta=theta, G=G, eps=eps, device=local_rank)
    ms_d, ex_d, err_d = timed(det)
    det.close()
    props = torch.cuda.get_device_properties(device)
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": "stochastic_queries_per_s",
            "value": sum_over_ranks(m, world, device) / (ms_s / 1e3), "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms_s, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(args.workload, src, tgt, theta, eps),
                           estimator="stochastic", samples=args.samples,
                           strata_level=args.strata_level, seed=args.seed,
                           l2="flushed (256 MiB write) before every step"),
            "evaluations_per_query": ex_s / m,
            "pot_abs_error": err_s,
            "roofline": {"bound": "alu", "achieved": ex_s * FLOPS_PER_TERM / (ms_s / 1e3) / 1e12,
                         "peak": peak, "unit": "TFLOP/s",
                         "frac": ex_s * FLOPS_PER_TERM / (ms_s / 1e3) / 1e12 / peak,
                         "traffic": None, "note": "whole step, evaluations x 20 flop"},
            "deterministic": {"theta": theta, "ms_per_step": ms_d,
                              "evaluations_per_query": ex_d / m, "pot_abs_error": err_d},
            "error_sample": "4096 targets (PCG64 seed 7) against the direct-sum kernel",
            # per step: bbox, keys and the order of the sources (63-bit keys)
            # and of separate targets (30-bit keys), 4 build passes, centre of
            # mass and children factors, strata, stochastic walk
            "gpu_launches": (2 + order_kernels(n, 63) + 6 + 2 +
                             (0 if tgt is None else 2 + order_kernels(m, 30)))
                            * args.steps}), flush=True)
    return 0


def run_neighbors(args, rank, local_rank, world):
    """SPH neighbour search: the whole bh_neighbors call (tree build, counting
    walk, scan, list walk) on resident inputs."""
    import ctypes
    import numpy as np
    import torch

    import barnes_hut_body_gb300 as B
    import workloads as W

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    n = args.nb_n
    pm, h = W.sph_plummer(n, seed=4)
    d_pm = torch.from_numpy(pm).to(device)
    d_h = torch.from_numpy(h).to(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    bh = B.BarnesHut(device=local_rank)
    counts, offs, lst = B.bh_neighbors(bh.ctx, d_pm, d_h, 2.0, B.BH_NB_SYMMETRIC)
    total = int(offs[n].item())
    L = B.lib()
    stream = torch.cuda.current_stream(device)
    st = ctypes.c_void_p(stream.cuda_stream)

    def call(with_list=True):
        rc = L.bh_neighbors(bh.ctx, d_pm.data_ptr(), d_h.data_ptr(), n, 2.0, B.BH_NB_SYMMETRIC,
                            counts.data_ptr(), offs.data_ptr(),
                            lst.data_ptr() if with_list else None,
                            total if with_list else 0, st)
        if rc != 0:
            raise RuntimeError(B.bh_last_error(bh.ctx))

    for _ in range(max(args.warmup, 3)):
        call()
    if bh.status() != 0:
        raise RuntimeError(B.bh_last_error(bh.ctx))

    def timed(with_list):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(world, device)
        torch.cuda.synchronize(device)
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            call(with_list)
            ev[k][1].record(stream)
        torch.cuda.synchronize(device)
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world, device)

    ms_count = timed(False)
    tests, _ = B.bh_get_counters(bh.ctx)
    ms = timed(True)
    if bh.status() != 0:
        raise RuntimeError(B.bh_last_error(bh.ctx))
    c = counts.cpu().numpy()
    if rank == 0:
        print(json.dumps({
            "metric": "neighbour_pairs_per_s",
            "value": sum_over_ranks(total, world, device) / (ms / 1e3), "unit": "pairs/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"sph_plummer n={n} (a 0.1, h from the analytic density, "
                                   "64 neighbours within 2h on average)",
                       "kappa": 2.0, "mode": "symmetric",
                       "l2": "flushed (256 MiB write) before every step"},
            "ms_counts_and_offsets_only": ms_count,
            "pairs": total, "neighbours_per_particle": {"mean": float(c.mean()),
                                                        "max": int(c.max())},
            "pair_tests": tests, "tests_per_pair": tests / max(total, 1),
            # per call: bbox, keys, the order (top-digit pass, bucket sort, 8
            # digit passes, gather), 4 build passes, h gather, node boxes,
            # counting walk, 3 scan kernels, list walk
            "gpu_launches": (2 + order_kernels(n, 63) + 4 + 7) * args.steps}),
          flush=True)
    bh.close()
    return 0


def main():
    args = parse()
    default_workload = args.workload is None
    if args.workload is None:
        args.workload = "surface2e20" if args.stochastic else "lattice1m_shuffled"
    if args.also is None:
        args.also = "galaxy5m" if default_workload else "none"
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.direct:
        return run_direct(args, rank, local_rank, world)
    if args.integrate:
        return run_integrate(args, rank, local_rank, world)
    if args.stochastic:
        return run_stochastic(args, rank, local_rank, world)
    if args.neighbors:
        return run_neighbors(args, rank, local_rank, world)
    return run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    sys.exit(main())
