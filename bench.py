#!/usr/bin/env python3
"""Throughput of the graph-based 3pCF path on GB300, printed as one JSON line.

One step = the whole hot path on one synthetic catalogue already resident in
device memory: cell sort, neighbour graph (count + fill), 3pCF merge-walk
count with its histogram. The default workload is the BAO-scale 3pCF
(2,000,000 Neyman-Scott points in an open 2000 h^-1 Mpc box, r_max 150,
30 bins, ~6.7e9 directed edges). The parity-4pCF path is timed the same way
on its own workload and reported in the "parity_4pcf" object; the six-bin
4pCF, the internal 2pCF and the weighted (signed int16 weights, exact)
2pCF / 3pCF / six-bin 4pCF counts are timed beside it ("fourpcf6", "twopcf",
"weighted"), and so is the 3pCF count on a graph kept in pinned host
memory in row windows ("windowed"), all outside the headline step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (oracle/, plain C) on a bounded
random sample of the workload's hubs, each with its full row found by brute
force over all points, as the "cpu_baseline" object of the default line does.
Under torchrun every rank counts its own realisation of the workload (weak
scaling, no collective on the data path); with --strong the ranks split one
catalogue's hubs into ranges of equal work and sum their histograms. Rank 0
prints the line.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from cosmology_point_correlation_gb300 import catalogues, configs  # noqa: E402

METRIC = "3pCF triangles/s and edges/s on 1 GB300; achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
BYTES_PER_EDGE = 5                      # int32 neighbour id + uint8 bin
PROFILE_COUNTERS = os.path.join(ROOT, "profiles", "k_count3m_bao_3pcf.json")
PARITY_COUNTERS = os.path.join(ROOT, "profiles", "k_count4_small_parity_4pcf.json")
KERNEL_SOURCES = [os.path.join(ROOT, "cosmology_point_correlation_gb300", "csrc", f)
                  for f in ("gs_count3.cu", "gs_internal.cuh")]
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--strong", action="store_true",
                   help="under torchrun: all ranks count one catalogue, each a hub range balanced on the "
                        "merge-walk work, and the histograms are summed over ranks (strong scaling)")
    p.add_argument("--workload", default="bao_3pcf", choices=sorted(configs.ALL))
    p.add_argument("--parity-workload", default="parity_4pcf")
    p.add_argument("--scale", type=float, default=1.0,
                   help="fraction of the workload's points, box shrunk to keep the density")
    p.add_argument("--no-parity", action="store_true")
    p.add_argument("--only-parity", action="store_true",
                   help="time only the parity-4pCF path and print its own line")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-windowed", action="store_true",
                   help="skip the out-of-core (row window) 3pCF timings")
    p.add_argument("--windowed-workload", default="large_3pcf")
    p.add_argument("--no-weighted", action="store_true",
                   help="skip the weighted 2pCF / 3pCF / six-bin 4pCF timings")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ------------------------------------------------------------------ workloads

def catalogue(w: configs.Workload, scale: float, rank: int):
    """(xyz, box_lu, description) of one realisation; rank r uses seed + 1000 r."""
    n = max(1, int(round(w.n * scale)))
    box_mpc = w.box_mpc * (n / w.n) ** (1.0 / 3.0)
    seed = w.seed + 1000 * rank
    if w.process == "uniform":
        xyz = catalogues.uniform(n, box_mpc, seed)
    else:
        xyz = catalogues.neyman_scott(n, box_mpc, max(1, int(round(w.ns["n_parents"] * n / w.n))),
                                      w.ns["mu"], w.ns["sigma"], seed)
    desc = {"workload": w.name, "n": n, "box_mpc": round(box_mpc, 3), "periodic": w.periodic,
            "r_max_mpc": w.r_max_mpc, "nbins": w.nbins, "process": w.process, "seed": seed}
    if w.ns:
        desc["neyman_scott"] = w.ns
    return xyz, catalogues.box_lattice(box_mpc), desc


L2_BYTES = 129e6                        # GB300 L2 (a constant, so both arms state the same)


def l2_note(desc: dict) -> str:
    """How the timed steps relate to L2, from the catalogue's size alone (the
    uniform-density edge estimate; clustering only adds edges)."""
    n, box, r = desc["n"], desc["box_mpc"], desc["r_max_mpc"]
    csr = BYTES_PER_EDGE * n * n * (4.0 / 3.0) * math.pi * r ** 3 / box ** 3
    if csr > L2_BYTES:
        return (f"inputs larger than L2: the graph (about {csr / 1e9:.0f} GB of CSR at the mean density) is "
                "rebuilt and re-read every step; no flush needed")
    return (f"the graph (about {csr / 1e6:.0f} MB of CSR) fits in L2: each step rebuilds it and the count "
            "reads it from L2")


# ------------------------------------------------------------------ CPU oracle (baseline only)

SAMPLE_SEED = 4242
CPU_TARGET_S = 12.0


def oracle_hub_sample(xyz, box_lu, w, n_hubs):
    """The oracle on a seeded random sample of hubs of the full catalogue: each
    hub's row by brute force over all points, then every pair of its
    neighbours tested for the closing side (no graph). Returns (triangles
    incident to the hubs, hubs, seconds, threads)."""
    import oracle
    oracle.build()
    hubs = np.random.default_rng(SAMPLE_SEED).choice(len(xyz), size=min(n_hubs, len(xyz)), replace=False)
    t0 = time.perf_counter()
    h = oracle.count_3pcf_hubs(xyz, box_lu, int(w.periodic), w.edges_lu, hubs)
    dt = time.perf_counter() - t0
    return int(h.sum()), len(hubs), dt, oracle.threads()


def oracle_sample_size(xyz, box_lu, w):
    """Hubs for about CPU_TARGET_S seconds of oracle work, from two shorter runs
    (the first sizes a run of about a tenth of the target, which sizes the sample)."""
    import oracle
    k = 2 * oracle.threads()
    for target in (CPU_TARGET_S / 10, CPU_TARGET_S):
        _, nh, dt, _ = oracle_hub_sample(xyz, box_lu, w, k)
        k = int(max(k, min(len(xyz), nh * target / max(dt, 1e-3))))
    return k


def oracle_line(xyz, box_lu, w, n_hubs, runs=1):
    """cpu_baseline object: the oracle's rate over the hub sample, as
    full-catalogue triangles per second (every triangle is incident to three
    hubs, so the sample's incident triangles / 3 per second is the rate at
    which the oracle would produce the full histogram)."""
    times, inc, cores = [], 0, 1
    for _ in range(runs):
        inc, nh, dt, cores = oracle_hub_sample(xyz, box_lu, w, n_hubs)
        times.append(dt)
    sec = statistics.mean(times)
    sample = (f"{nh} hubs drawn at random (seed {SAMPLE_SEED}) from the whole {w.name} catalogue of {len(xyz)} "
              f"points; per hub the oracle finds its row by brute force over all points and tests every "
              f"pair of neighbours for the closing side; {inc} hub-incident triangles in {sec:.1f} s; "
              "value = incident triangles / 3 per second")
    return {"value": inc / 3.0 / sec, "unit": "triangles/s", "cores": cores, "kind": "oracle",
            "sample": sample}, sec, times


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    xyz, box_lu, desc = catalogue(w, args.scale, 0)
    desc["l2"] = l2_note(desc)
    k = oracle_sample_size(xyz, box_lu, w)
    for _ in range(args.warmup):
        oracle_hub_sample(xyz, box_lu, w, max(1, k // 8))
    cpu, sec, times = oracle_line(xyz, box_lu, w, k, runs=args.steps)
    value = cpu["value"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "triangles/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": desc, "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "triangles/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu_index)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for r in csv.reader(io.StringIO(f.read())):
                    if len(r) >= 9:
                        rows.append([c.strip() for c in r])
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": reasons, "samples": len(rows)}


def gpu_index_of(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(parts) and parts[local_rank].isdigit():
            return int(parts[local_rank])
    return local_rank


# ------------------------------------------------------------------ peaks / profiles

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_counters(workload: str):
    """ncu counters of the 3pCF count kernel, scaled to one full-size launch,
    from the committed data file; None when they were taken on other kernel
    source or another workload."""
    try:
        with open(PROFILE_COUNTERS) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256") != kernel_source_hash() or d.get("workload") != workload:
        return None
    return d


def parity_roofline(workload: str, cliques: int, count_s: float, dev, sm_mhz: float):
    """The parity count's on-chip ceilings: L1 data-pipe wavefronts and warp
    instructions per clique from the ncu capture of the same kernel source
    (profiles/k_count4_small_parity_4pcf.json), times the clique rate of this
    run, against one wavefront and four instruction issues per SM per cycle."""
    import torch
    try:
        with open(PARITY_COUNTERS) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for p in d.get("sources", []):
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    if d.get("workload") != workload or d.get("kernel_source_sha256") != h.hexdigest() or \
            d.get("cliques_per_launch") != cliques:
        return None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk = sm_mhz * 1e6
    l1_rate = d["l1_wavefronts_per_launch"] / count_s
    return {"bound": "alu", "kernel": "k_count4_small",
            "ceiling": "the L1 / shared-memory data pipe and instruction issue of the clique search",
            "achieved": l1_rate / 1e9, "peak": sms * clk / 1e9, "unit": "G wavefronts/s",
            "frac": l1_rate / (sms * clk),
            "peak_kind": f"derived: {sms} SMs x 1 wavefront per cycle x the sampled SM clock ({sm_mhz:.0f} MHz)",
            "issue_frac": d["warp_inst_per_launch"] / count_s / (sms * 4 * clk),
            "counters": "profiles/k_count4_small_parity_4pcf.json (ncu, kernel source hash checked)"}


# ------------------------------------------------------------------ distributed

def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and not (world == 1 and n_gpus == 1):
        if world == 1:
            raise SystemExit(f"--gpus {n_gpus} needs torchrun with {n_gpus} processes")
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_sum(world, values_max, values_sum):
    """Element-wise max of values_max and sum of values_sum over ranks."""
    if world == 1:
        return values_max, values_sum
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    a = torch.tensor(values_max, dtype=torch.float64, device=dev)
    b = torch.tensor(values_sum, dtype=torch.float64, device=dev)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return a.tolist(), b.tolist()


# ------------------------------------------------------------------ GPU arm

def time_path(coords, box_lu, w, steps, kind, hist_out=None, hub_range=None, reduce=False):
    """Run `steps` passes; returns per-step (step_ms, count_ms, result) lists.
    hub_range: count only these hubs (strong scaling); reduce: sum the
    histogram over the ranks inside the step."""
    import torch
    from cosmology_point_correlation_gb300 import build_graph
    from cosmology_point_correlation_gb300.sharding import reduce_histograms
    stream = torch.cuda.current_stream()
    res = []
    for _ in range(steps):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        g = build_graph(coords, box_lu, w.periodic, w.edges_lu, stream=stream)
        e1.record(stream)
        if kind == "3pcf":
            b, e = hub_range if hub_range else (0, None)
            out = g.count_3pcf(b, e, out=hist_out, stream=stream)
            if reduce:
                reduce_histograms(out)
        else:
            out = g.count_4pcf_parity(out=hist_out, stream=stream)
        e2.record(stream)
        stream.synchronize()
        n_edges = g.n_edges
        g.free()
        res.append((e0.elapsed_time(e2), e1.elapsed_time(e2), e0.elapsed_time(e1), n_edges, out))
    return res


def run_ours(args, w):
    import torch
    from cosmology_point_correlation_gb300 import (as_uint64, build_graph, count_3pcf_from_host,
                                                    kernel_launches)
    rank, world, local = dist_init(args.gpus)
    dev = torch.device("cuda", local)
    # weak scaling: every rank its own realisation; strong: one catalogue, hub
    # ranges balanced on the merge-walk work, histograms summed over ranks
    strong = args.strong and world > 1
    xyz, box_lu, desc = catalogue(w, args.scale, 0 if args.strong else rank)
    coords = torch.from_numpy(xyz).to(dev)
    ncfg = w.nbins * (w.nbins + 1) * (w.nbins + 2) // 6
    hist = torch.empty(ncfg, dtype=torch.int64, device=dev)

    # work statistics of this catalogue's graph (untimed), and the internal
    # 2pCF pass on the same graph (one sweep of the bin bytes)
    with build_graph(coords, box_lu, w.periodic, w.edges_lu) as g:
        st = g.stats()
        walk = g.count3_walk
        hub_range = None
        if strong:
            from cosmology_point_correlation_gb300.sharding import balanced_ranges
            f_h, w_h = (t.cpu().numpy() for t in g.hub_work())
            hub_range = balanced_ranges(f_h, w_h, world)[rank]
        kernel_name = {"map": "k_count3m (byte map, one spoke per warp)",
                       "mapgroup": "k_count3m (byte map, four spokes per warp)",
                       "group": "k_count3 (bitmap, four spokes per warp)",
                       "warp": "k_count3 (bitmap, one spoke per warp)"}.get(walk, walk)
        dd = g.count_2pcf()
        torch.cuda.synchronize()
        t2 = []
        for _ in range(max(args.steps, 3)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.count_2pcf(out=dd)
            e1.record()
            torch.cuda.synchronize()
            t2.append(e0.elapsed_time(e1))
        pairs = int(as_uint64(dd).sum())
        # weighted counts on the same graph: signed int16 weights, exact 128-bit sums
        weighted = None
        if not args.no_weighted:
            wts = torch.from_numpy(np.random.default_rng(w.seed + 17).integers(
                -32767, 32768, size=len(xyz)).astype(np.int16)).to(dev)
            g.set_weights(wts)

            def _timed(fn):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1)

            g.count_3pcf_weighted(0, max(1, len(xyz) // 64))          # warm-up on a hub slice
            g.count_2pcf_weighted()
            t3w = _timed(lambda: g.count_3pcf_weighted())
            t2w = statistics.mean(_timed(lambda: g.count_2pcf_weighted()) for _ in range(3))
            weighted = {"weights": "uniform random int16 in [-32767, 32767]",
                        "threepcf_count_ms": t3w, "twopcf_ms": t2w}
    alg_bytes = BYTES_PER_EDGE * (st["n_edges"] // 2 + st["spoke_walk"])
    peak, peak_kind = hbm_peak()
    t2_ms = statistics.mean(t2)
    twopcf = {"ms": t2_ms, "pairs": pairs, "pairs_per_s": pairs / (t2_ms / 1e3),
              "roofline": {"bound": "hbm", "achieved": st["n_edges"] / (t2_ms / 1e3) / 1e9, "peak": peak,
                           "unit": "GB/s", "frac": st["n_edges"] / (t2_ms / 1e3) / 1e9 / peak,
                           "per_unit": "1 B per directed edge (the bin byte)"}}

    time_path(coords, box_lu, w, args.warmup, "3pcf", hist, hub_range, strong)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = kernel_launches()
    with ClockSampler(gpu_index_of(local)) as clk:
        t_wall0 = time.perf_counter()
        res = time_path(coords, box_lu, w, args.steps, "3pcf", hist, hub_range, strong)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    launches = kernel_launches() - launches0
    clocks = clk.summary()
    if any(r in BAD_REASONS for r in clocks["reasons"]):
        # throttled: measure once more
        launches0 = kernel_launches()
        with ClockSampler(gpu_index_of(local)) as clk:
            res = time_path(coords, box_lu, w, args.steps, "3pcf", hist, hub_range, strong)
            torch.cuda.synchronize()
        launches = kernel_launches() - launches0
        clocks = clk.summary()
        clocks["remeasured"] = True

    step_ms = statistics.mean(r[0] for r in res)
    count_ms = statistics.mean(r[1] for r in res)
    build_ms = statistics.mean(r[2] for r in res)
    n_edges = res[-1][3]
    tris = int(as_uint64(res[-1][4]).sum())
    (step_ms_max, count_ms_max), (tris_all, edges_all) = reduce_max_sum(world, [step_ms, count_ms],
                                                                        [float(tris), float(n_edges)])
    if strong:                      # one catalogue: the reduced histogram is the whole job's
        tris_all, edges_all = float(tris), float(n_edges)

    # end to end: host coordinates in, host histogram out, through the C ABI
    e2e = None
    if not args.no_e2e:
        pinned = torch.from_numpy(xyz).pin_memory()
        out = torch.zeros(ncfg, dtype=torch.int64).pin_memory()
        host_xyz = pinned.numpy()
        host_out = out.numpy().view(np.uint64)
        def e2e_step():
            if not strong:
                count_3pcf_from_host(host_xyz, box_lu, w.periodic, w.edges_lu, out=host_out)
                return
            # strong scaling: host coordinates in, this rank's hub range, the sum
            # over ranks, the host histogram out (the public Python API)
            from cosmology_point_correlation_gb300.sharding import reduce_histograms
            dc = pinned.to(dev, non_blocking=True)
            with build_graph(dc, box_lu, w.periodic, w.edges_lu) as ge:
                h = ge.count_3pcf(*hub_range)
                reduce_histograms(h)
                out.copy_(h)
            torch.cuda.synchronize()

        e2e_step()
        times = []
        for _ in range(max(1, min(args.steps, 2))):
            torch.cuda.synchronize()
            barrier(world)
            t0 = time.perf_counter()
            e2e_step()
            times.append(time.perf_counter() - t0)
        e2e_s = statistics.mean(times)
        [e2e_s_max], _ = reduce_max_sum(world, [e2e_s], [0.0])
        e2e = {"value": tris_all / e2e_s_max, "unit": "triangles/s",
               "h2d_bytes_per_step": int(xyz.nbytes), "d2h_bytes_per_step": int(ncfg * 8),
               "ms_per_step": e2e_s_max * 1e3}

    # parity 4pCF on its own workload
    parity = None
    if not args.no_parity:
        pw = configs.ALL[args.parity_workload]
        pxyz, pbox, pdesc = catalogue(pw, args.scale, rank)
        pcoords = torch.from_numpy(pxyz).to(dev)
        time_path(pcoords, pbox, pw, max(1, args.warmup), "4pcf")
        torch.cuda.synchronize()
        pres = time_path(pcoords, pbox, pw, args.steps, "4pcf")
        p_step = statistics.mean(r[0] for r in pres)
        p_count = statistics.mean(r[1] for r in pres)
        even, odd = pres[-1][4]
        cliques = int(as_uint64(even).sum())
        (p_step, p_count), (cl_all, pe_all) = reduce_max_sum(world, [p_step, p_count],
                                                             [float(cliques), float(pres[-1][3])])
        parity = {"config": pdesc, "ms_per_step": p_step, "count_ms": p_count,
                  "cliques_per_s": cl_all / (p_step / 1e3), "edges_per_s": pe_all / (p_step / 1e3),
                  "cliques": cliques, "odd_sum": int(odd.sum().item()), "n_edges": pres[-1][3],
                  "roofline": (parity_roofline(pw.name, cliques, p_count / 1e3, dev, clocks.get("sm_mhz") or 2070.0)
                               if args.scale == 1.0 else None)}

    # six-edge-bin 4pCF (276 configurations) on the parity catalogue with 4 bins
    fourpcf6 = None
    if not args.no_parity:
        import dataclasses
        pw = configs.ALL[args.parity_workload]
        w6 = dataclasses.replace(pw, name=pw.name + "_4bins", nbins=4)
        xyz6, box6, desc6 = catalogue(w6, args.scale, rank)
        c6 = torch.from_numpy(xyz6).to(dev)
        res6 = []
        for k in range(max(1, args.warmup) + args.steps):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record()
            g6 = build_graph(c6, box6, w6.periodic, w6.edges_lu)
            e1.record()
            ev6, od6 = g6.count_4pcf6()
            e2.record()
            torch.cuda.synchronize()
            if k >= max(1, args.warmup):
                res6.append((e0.elapsed_time(e2), e1.elapsed_time(e2), int(as_uint64(ev6).sum()),
                             int(od6.sum().item())))
            g6.free()
        s6 = statistics.mean(r[0] for r in res6)
        k6 = statistics.mean(r[1] for r in res6)
        fourpcf6 = {"config": desc6, "ms_per_step": s6, "count_ms": k6, "configurations": int(len(ev6)),
                    "tetrahedra": res6[-1][2], "odd_sum": res6[-1][3],
                    "tetrahedra_per_s": res6[-1][2] / (s6 / 1e3)}

    # weighted six-bin 4pCF on the same 4-bin parity catalogue
    if fourpcf6 is not None and weighted is not None:
        with build_graph(c6, box6, w6.periodic, w6.edges_lu) as g6:
            g6.set_weights(torch.from_numpy(np.random.default_rng(w6.seed + 17).integers(
                -32767, 32768, size=len(xyz6)).astype(np.int16)).to(dev))
            g6.count_4pcf6_weighted()
            t6 = []
            for _ in range(max(1, args.steps)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g6.count_4pcf6_weighted()
                e1.record()
                torch.cuda.synchronize()
                t6.append(e0.elapsed_time(e1))
        weighted["fourpcf6_count_ms"] = statistics.mean(t6)

    # out-of-core row windows: the 3pCF count with the edge arrays in pinned
    # host memory, against the device-resident count, on the 2M-point uniform
    # workload (inputs staged per tile inside the timed call)
    windowed = None
    if not args.no_windowed:
        ww = configs.ALL[args.windowed_workload]
        wxyz, wbox, wdesc = catalogue(ww, args.scale, rank)
        wc = torch.from_numpy(wxyz).to(dev)

        def _count_ms(g):
            g.count_3pcf()                                   # warm-up
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                h = g.count_3pcf()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            return statistics.mean(ts), as_uint64(h), ts

        with build_graph(wc, wbox, ww.periodic, ww.edges_lu) as g:
            t_res, h_res, ts_res = _count_ms(g)
            e_all = g.n_edges
            res_walk = g.count3_walk
        rows = []
        for nwin in (2, 4, 8):
            with build_graph(wc, wbox, ww.periodic, ww.edges_lu, window_edges=e_all // nwin + 1) as g:
                t_w, h_w, ts_w = _count_ms(g)
                rows.append({"window_edges": e_all // nwin + 1, "windows": g.windows()[0], "walk": g.count3_walk,
                             "count_ms": t_w, "count_ms_runs": ts_w, "overhead": t_w / t_res - 1.0,
                             "exact": bool(np.array_equal(h_w, h_res))})
        # pinned host -> device copy rate in this process, which bounds the window staging
        hbuf = torch.empty(1 << 28, dtype=torch.int32).pin_memory()
        dbuf = torch.empty(1 << 28, dtype=torch.int32, device=dev)
        dbuf.copy_(hbuf, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dbuf.copy_(hbuf, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        h2d_gbs = hbuf.numel() * 4 / 1e9 / (e0.elapsed_time(e1) / 1e3)
        del hbuf, dbuf
        windowed = {"config": wdesc, "resident_count_ms": t_res, "resident_count_ms_runs": ts_res,
                    "resident_walk": res_walk,
                    "overhead_against": "resident_count_ms (the tiles run the same walk)",
                    "n_edges": e_all, "tiles": rows, "pinned_h2d_gbs": h2d_gbs}

    # CPU oracle on a bounded hub sample of the same catalogue (rank 0 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _, _ = oracle_line(xyz, box_lu, w, oracle_sample_size(xyz, box_lu, w))

    # roofline of the count kernel. The merge-walk re-reads its rows from L2
    # (profiles/), so HBM is not its ceiling. Every probe of a spoke-row entry
    # is two shared-memory loads and every closed triangle a shared-memory add,
    # and the rows come in through L1 as well: the binding unit is the L1 data
    # pipe, one 128-byte wavefront per SM per cycle. Its use per triangle comes
    # from the ncu capture of the same kernel source (scaled by triangles), the
    # time from this run; the atomic, issue, DRAM and walk ceilings are given
    # beside it.
    from cosmology_point_correlation_gb300 import measure_smem_atomics
    count_s = count_ms / 1e3
    n3 = w.nbins ** 3
    probe_cfg = min(n3, 27648) if walk in ("map", "mapgroup") else min(ncfg, 12288)
    atom_rate = measure_smem_atomics(probe_cfg, 0, 20)
    tri_rate = tris / count_s
    prof = profiled_counters(w.name) if args.scale == 1.0 else None
    traffic = prof["dram_bytes_per_full_launch"] if prof else None
    sm_mhz = clocks.get("sm_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    walk_gbs = alg_bytes / count_s / 1e9
    l1_peak = sms * sm_mhz * 1e6                                  # wavefronts per second
    l1_rate = prof["l1_wavefronts_per_full_launch"] / count_s if prof and "l1_wavefronts_per_full_launch" in prof \
        else None
    roofline = {
        "bound": "alu", "kernel": kernel_name,
        "ceiling": ("the L1 / shared-memory data pipe (one 128-byte wavefront per SM per cycle): per spoke-row "
                    "entry two shared-memory loads (segment slot, bin byte), per closed triangle one shared-memory "
                    "add, and the row loads; the rows are re-read from L2, so HBM is not the ceiling"),
        "achieved": l1_rate / 1e9 if l1_rate else None, "peak": l1_peak / 1e9, "unit": "G wavefronts/s",
        "frac": l1_rate / l1_peak if l1_rate else None,
        "per_unit": ("L1 data-pipe wavefronts per closed triangle, from the ncu capture of this kernel source "
                     "(profiles/k_count3m_bao_3pcf.json), times the triangles per second of this run"),
        "peak_kind": f"derived: {sms} SMs x 1 wavefront per cycle x the sampled SM clock ({sm_mhz:.0f} MHz)",
        "wavefronts_per_triangle": (prof["l1_wavefronts_per_full_launch"] / tris) if l1_rate else None,
        "traffic": traffic,
        "dram_gbs": traffic / count_s / 1e9 if traffic else None,
        "dram_frac": traffic / count_s / 1e9 / peak if traffic else None,
        "walk_bytes_per_launch": alg_bytes,
        "walk_gbs_l2": walk_gbs,
        "walk_frac_l2": walk_gbs / peak,
        "walk_note": ("effective merge-walk bandwidth: 5 B per spoke-row entry the intersections read plus 5 B per "
                      "forward edge of hub rows, divided by the count time, against the measured HBM copy peak; "
                      "almost all of it is served from L2, so it is not DRAM traffic"),
        "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "atomic_adds_per_s": tri_rate, "atomic_peak_per_s": atom_rate, "atomic_frac": tri_rate / atom_rate,
        "atomic_peak_kind": (f"measured in this run: gs_measure_smem_atomics, two 512-thread blocks per SM doing "
                             f"only shared-memory atomic adds of 1 into {probe_cfg} random 32-bit counters, 20 of 32 "
                             "lanes active (one add per closed triangle)"),
        "issue_frac": (prof["warp_inst_per_full_launch"] / (count_s * sms * 4 * sm_mhz * 1e6)) if prof else None,
        "lane_adds_per_triangle": (prof["shared_atom_lane_ops_per_full_launch"] / tris) if prof else None,
        "counters": ("profiles/k_count3m_bao_3pcf.json (ncu, kernel source hash checked)" if prof else
                     "none for this kernel source and workload"),
    }

    if rank == 0:
        value = tris_all / (step_ms_max / 1e3)
        desc["l2"] = l2_note(desc)
        line = {"metric": METRIC, "value": value, "unit": "triangles/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True,
                "scaling": "strong" if strong else "weak",
                "vs_baseline": None, "dtype": "int64", "data": "synthetic", "config": desc,
                "edges_per_s": edges_all / (step_ms_max / 1e3),
                "count_edges_per_s": edges_all / 2 / (count_ms_max / 1e3),
                "triangles_per_step": tris_all, "n_edges": n_edges, "build_ms": build_ms,
                "count_ms": count_ms_max, "wall_s_timed": t_wall,
                "graph_stats": st, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clocks, "parity_4pcf": parity,
                "fourpcf6": fourpcf6, "twopcf": twopcf, "weighted": weighted, "windowed": windowed}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_parity_only(args):
    """One JSON line for the parity-4pCF path alone (build + count per step)."""
    import torch
    from cosmology_point_correlation_gb300 import as_uint64, kernel_launches
    rank, world, local = dist_init(args.gpus)
    pw = configs.ALL[args.parity_workload]
    pxyz, pbox, pdesc = catalogue(pw, args.scale, rank)
    pcoords = torch.from_numpy(pxyz).to(torch.device("cuda", local))
    time_path(pcoords, pbox, pw, args.warmup, "4pcf")
    torch.cuda.synchronize()
    barrier(world)
    l0 = kernel_launches()
    pres = time_path(pcoords, pbox, pw, args.steps, "4pcf")
    launches = kernel_launches() - l0
    step = statistics.mean(r[0] for r in pres)
    count = statistics.mean(r[1] for r in pres)
    even, odd = pres[-1][4]
    cliques = int(as_uint64(even).sum())
    (step, count), (cl_all, e_all) = reduce_max_sum(world, [step, count], [float(cliques), float(pres[-1][3])])
    if rank == 0:
        print(json.dumps({"metric": "parity 4pCF (hub, clique) counts/s", "value": cl_all / (step / 1e3),
                          "unit": "cliques/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": step, "count_ms": count, "higher_is_better": True, "scaling": "weak",
                          "dtype": "int64", "data": "synthetic", "config": pdesc,
                          "edges_per_s": e_all / (step / 1e3), "odd_sum": int(odd.sum().item()),
                          "gpu_launches": launches}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    w = configs.ALL[args.workload]
    if args.only_parity and args.impl == "ours":
        run_parity_only(args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
