#!/usr/bin/env python
"""Benchmark of the P-Cloth implicit-integration hot path on GB300.

One "step" is one whole implicit step of the hot path through the C ABI
(pcloth_step): per-step contact merge and assembly of A = M + h^2 sum K,
b = h f; block-Jacobi PCG to |r| <= 1e-6 |b|; state update.  The default
workload is the four-layer folded stack (4 x 455^2 vertices, 1,648,928
triangles, ~82,810 fresh contacts per step, h = 5e-3), the synthetic stand-in
for the pages' largest garment (1.65M triangles).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  The path does not shard: with N > 1 every
rank runs an independent replica of the workload ("replicas only"), the
barrier and the max over ranks of the timed region stay, and `value` counts
the steps of all ranks.  `--impl reference` times the fp64 CPU oracle on the
host cores on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PCG iterations/s + implicit steps/s at 1.65M tris; SpMV GB/s vs HBM peak"
UNIT = "implicit steps/s"
FALLBACK_HBM_GBS = 6800.0
# contact radius of the multi-layer cloths when contacts are found geometrically
FOUND_RADIUS = {"C4": 3e-3, "C5": 2e-3}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default="C5", help="workload C1..C5 (default C5)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-layouts", action="store_true", help="skip the SpMV layout comparison")
    p.add_argument("--contacts", choices=("synthetic", "found"), default="synthetic",
                   help="synthetic: the configuration's seeded contact lists; found: vertex "
                        "pairs closer than the contact radius, found by spatial hashing on "
                        "the GPU every step inside the timed region (multi-layer cloths)")
    p.add_argument("--oracle-iters", type=int, default=8,
                   help="oracle PCG iterations per reference sample step")
    return p.parse_args()


def workload_desc(w):
    return dict(workload="%s: %s" % (w.name, w.description), vertices=w.n_verts,
                triangles=w.triangles, springs=w.n_springs, contacts_per_step=w.max_contacts,
                h=w.h, tol=w.tol, maxit=w.maxit)


def bench_config(w):
    """The `config` of both arms' JSON lines (identical, so that the two
    lines compare): the workload, the parallelism and the L2 statement.  The
    matrix size is the bound from the workload's counts: 28 B per block (24 B
    of packed symmetric values + the column), for the diagonal and both
    directions of every spring and contact."""
    a_mb = 28 * (w.n_verts + 2 * (w.n_springs + w.max_contacts)) / 1e6
    l2 = ("inputs larger than L2: A is about %.0f MB per step vs 129 MB L2" % a_mb if a_mb > 129
          else "A (about %.1f MB) fits in the 129 MB L2: L2-resident, not an HBM-bound case"
          % a_mb)
    return dict(workload_desc(w), parallelism="replicas only (one independent cloth per GPU)",
                l2=l2)


# ------------------------------------------------------------------ peaks --
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


TRAFFIC_FILE = "pcg_loop_folded_stack_C5_traffic.json"
KERNEL_SOURCES = ("spmv_pipe.cuh", "pcg.cu", "async_copy.cuh", "pcloth_internal.cuh")


# the workload the committed capture was taken on: its traffic is reported
# for that workload only (the default folded stack with its synthetic contacts)
TRAFFIC_WORKLOAD = ("C5", "synthetic")


def stored_traffic(kernel_src_digest):
    """DRAM bytes per PCG iteration of the persistent PCG kernel from the
    committed ncu summary, only if it was taken on the current kernel
    source."""
    path = os.path.join(ROOT, "profiles", TRAFFIC_FILE)
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_digest") == kernel_src_digest:
            return float(d["dram_bytes_per_iteration"])
    except Exception:
        pass
    return None


def traffic_per_launch(config, contacts, iterations_per_launch):
    """ncu DRAM bytes of one PCG launch, from the committed capture scaled by
    the launch's iterations: only while the kernel sources are the ones the
    capture was taken on, and only for the workload it was taken on."""
    per_it = stored_traffic(kernel_source_digest())
    if per_it is None or (config, contacts) != TRAFFIC_WORKLOAD:
        return None
    return per_it * iterations_per_launch


def kernel_source_digest():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_linear_solve_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- clocks --
class Clocks:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None,
                    power_w_max=max(power) if power else None,
                    samples=len(sm), reasons=sorted(reasons))


# ------------------------------------------------------------ CPU oracle --
def oracle_sample(w, x, v, contacts, iters):
    """Time the fp64 oracle on one bounded sample of a step: the full assembly
    plus `iters` PCG iterations.  Returns (t_assembly, t_per_iteration)."""
    from oracle import oracle
    t0 = time.perf_counter()
    s = oracle.assemble_workload(w, x, v, contacts)
    t1 = time.perf_counter()
    s.pcg(w.tol, iters)
    t2 = time.perf_counter()
    return t1 - t0, (t2 - t1) / max(iters, 1)


def oracle_step_iterations(config):
    """PCG iterations the oracle needs at each step of its own trajectory,
    from the committed table written by oracle/iteration_table.py (fp64
    oracle runs only); an empty list if the table has none."""
    path = os.path.join(ROOT, "oracle", "iteration_table.json")
    try:
        with open(path) as f:
            return [int(i) for i in json.load(f)[config]["iterations"]]
    except Exception:
        return []


def oracle_whole_step(w, x, v, contacts):
    """Time one whole implicit step of the fp64 oracle (assembly, PCG to the
    workload's tolerance, state update).  Returns (seconds, iterations)."""
    from oracle import oracle
    t0 = time.perf_counter()
    res = oracle.step(w, x, v, contacts)
    return time.perf_counter() - t0, int(res.get("iterations", 0))


# ------------------------------------------------------------- ranks --
def max_over_ranks(x, device):
    """The maximum of a per-rank time over all ranks (x itself on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, seconds):
    """Units all ranks processed per second of the slowest rank."""
    return world * units_per_rank / seconds


# ------------------------------------------------------- SpMV layouts --
def spmv_layouts(cloth, n, dev, reps=50):
    """The plain product out = A in of the last assembled matrix in the two
    layouts: streamed BSR3 (pcloth_spmv) and the pages' block-ELL tables
    (pcloth_spmv_bell), each timed over `reps` launches with CUDA events (A
    is larger than L2, so every launch streams it from HBM)."""
    import torch
    x = torch.randn(n, 3, device=dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(5):
            fn(x, y)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn(x, y)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3   # us per launch

    nnzb = cloth.nnzb()
    algo = 28 * nnzb + 28 * n
    bsr_us = timed(cloth.spmv)
    width = cloth.bell_build()
    bell_us = timed(cloth.spmv_bell)
    peak, _ = hbm_peak()
    return dict(bytes_per_launch=algo,
                bsr3=dict(us=bsr_us, gbs=algo / (bsr_us * 1e-6) / 1e9,
                          frac=algo / (bsr_us * 1e-6) / 1e9 / peak),
                block_ell=dict(us=bell_us, gbs=algo / (bell_us * 1e-6) / 1e9,
                               frac=algo / (bell_us * 1e-6) / 1e9 / peak, width=width,
                               table_slots_per_block=width * n / nnzb),
                timing="CUDA events over %d launches each, same matrix and input" % reps)


# ------------------------------------------------------------------- arms --
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    from sparse_linear_solve_gb300 import pcloth as pc
    from sparse_linear_solve_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.make(args.config)
    K, Wm = args.steps, args.warmup
    found_mode = args.contacts == "found"
    if found_mode:
        # the configuration's contact radius; room for a growing contact set
        radius = FOUND_RADIUS.get(args.config)
        if radius is None:
            raise SystemExit("--contacts found is for the multi-layer cloths (C4, C5)")
        w.max_contacts = 6 * w.n_verts
        args.no_e2e = True
        args.no_cpu_baseline = True
    cloth = pc.PCloth.from_workload(w, device=dev)
    x = torch.from_numpy(w.x0).to(dev)
    v = torch.from_numpy(w.v0).to(dev)
    dv = torch.empty_like(x)
    host_contacts = [w.contacts(t) for t in range(Wm + K)]
    dev_contacts = [pc.to_device_elements(c, dev) for c in host_contacts]
    found_counts = []

    def one_step(t):
        if found_mode:
            c, nf = cloth.find_contacts(x, radius, W.K_CONTACT)
            found_counts.append(nf)
        else:
            c = dev_contacts[t]
        return cloth.step(x, v, c, w.h, w.tol, w.maxit, dv)

    for t in range(Wm):
        one_step(t)
    torch.cuda.synchronize()
    x_start, v_start = x.clone(), v.clone()

    def timed_steps(profile_mode):
        """K steps from the saved state; returns (ms, iterations, codes, profile)."""
        x.copy_(x_start)
        v.copy_(v_start)
        cloth.profile(profile_mode)
        cloth.profile_read(reset=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        its, codes = [], []
        del found_counts[:]
        for t in range(K):
            it, rr, code = one_step(Wm + t)
            its.append(it)
            codes.append(code)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        prof = cloth.profile_read(reset=True)
        cloth.profile(0)
        return e0.elapsed_time(e1), its, codes, prof

    # pass 1: the measured value, no profiling events inside the timed region
    clocks = Clocks(local_rank)
    ms, its, codes, prof_clean = timed_steps(0)
    clk = clocks.stop()
    ms = max_over_ranks(ms, dev)
    # pass 2: the same K steps again with CUDA events around every assembly
    # and every PCG launch on the library's stream, and the PCG kernel's own
    # phase timers
    ms_prof, its_prof, _, prof = timed_steps(2)
    nnzb_seen = [cloth.nnzb()]

    # ---- roofline of the dominant kernel: the persistent PCG -------------
    # Algorithmic bytes per PCG iteration: the matrix once (28 B/block:
    # 24 packed symmetric values + 4 colind; 4 B/row rowptr), p read once and
    # q written (24 B/row), the update phase (q, r read, the symmetric P read
    # 24 B, r, z written: 72 B/row) and the direction phase (p, dv, z read,
    # dv, p written: 60 B/row).  Per launch: that times the iterations, plus
    # the start (b 12, P 24 read; r, z, p, dv written 48) and dv out
    # (12 + 12) = 108 B/row.
    n = w.n_verts
    nnzb = nnzb_seen[-1]
    it_bytes = 28 * nnzb + 160 * n
    spmv_bytes = 28 * nnzb + 28 * n
    vec_bytes = 132 * n
    iters = max(prof["iterations"], 1)
    solves = max(prof["solves"], 1)
    launch_bytes = (iters * it_bytes + solves * 108 * n) / solves
    launch_ms = prof["solve_ms"] / solves
    achieved = launch_bytes / (launch_ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    samples = max(prof["samples"], 1)
    spmv_avg_ms = prof["spmv_ms"] / samples
    vec_avg_ms = prof["update_ms"] / samples

    # ---- end to end through the host-buffer entry point ------------------
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(w.x0.copy()).pin_memory()
        vh = torch.from_numpy(w.v0.copy()).pin_memory()
        hc = []
        for c in host_contacts:
            if c.n:
                hc.append(tuple(torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                                for a in (c.i, c.j, c.k, c.rest)))
            else:
                hc.append(None)
        # the same trajectory as the device-timed leg: same warm-up steps from
        # the same initial state, then the same K steps, so the iteration
        # counts (and so the work) are identical
        e2e_its = []
        for t in range(Wm):
            cloth.step_host(xh, vh, hc[t], w.h, w.tol, w.maxit)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for t in range(K):
            e2e_its.append(cloth.step_host(xh, vh, hc[Wm + t], w.h, w.tol, w.maxit)[0])
        t1 = time.perf_counter()
        e_s = t1 - t0
        e_s = max_over_ranks(e_s, dev)
        nc_mean = sum(c.n for c in host_contacts[Wm:]) / K
        e2e = dict(value=whole_job_rate(world, K, e_s), unit=UNIT,
                   h2d_bytes_per_step=int(2 * 12 * n + 16 * nc_mean),
                   d2h_bytes_per_step=int(2 * 12 * n),
                   pcg_iterations_mean=sum(e2e_its) / K)

    traffic = traffic_per_launch(args.config, args.contacts, iters / solves)
    result = dict(
        metric=METRIC, value=whole_job_rate(world, K, ms * 1e-3), unit=UNIT, n_gpus=world, steps=K,
        warmup=Wm, ms_per_step=ms / K, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="f32 (fp32 storage and arithmetic; PCG dot products reduced as fp32 pairs, double-float)",
        data="synthetic (seeded generator; no garment meshes available)",
        config=bench_config(w),
        pcg_iterations_per_s=whole_job_rate(world, sum(its), ms * 1e-3),
        pcg_iterations_per_s_solve_only=sum(its_prof) / (prof["solve_ms"] * 1e-3),
        pcg_iterations_mean=sum(its) / K,
        assembly_ms=prof["assemble_ms"] / max(prof["assemble_calls"], 1),
        spmv_phase_us=spmv_avg_ms * 1e3,
        spmv_phase_gbs=spmv_bytes / (spmv_avg_ms * 1e-3) / 1e9 if spmv_avg_ms > 0 else None,
        vector_phases_us=vec_avg_ms * 1e3,
        vector_phases_gbs=vec_bytes / (vec_avg_ms * 1e-3) / 1e9 if vec_avg_ms > 0 else None,
        iteration_us=launch_ms * 1e3 / (iters / solves),
        codes=sorted(set(codes)),
        roofline=dict(bound="hbm", kernel="pcg_loop<6> (persistent PCG: streaming SpMV, "
                                          "update and direction phases, grid barriers)",
                      timing="CUDA events on the library stream around each PCG launch (one "
                             "per solve) of a second pass over the same %d steps (%d launches, "
                             "%.1f ms/step with the events)" % (K, prof["solves"], ms_prof / K),
                      achieved=achieved, peak=peak, unit="GB/s", frac=achieved / peak,
                      peak_source=peak_src, bytes_per_launch=launch_bytes,
                      bytes_model="per iteration 28 B/block (24 packed symmetric values + "
                                  "4 colind) + 160 B/row (rowptr 4; SpMV p 12 read, q 12 "
                                  "written; update q r 24 + P 24 read, r z 24 written; "
                                  "direction p dv z 36 read, dv p 24 written); per launch "
                                  "+108 B/row (start and dv out)",
                      traffic=traffic),
        clocks=clk,
        gpu_launches=int(prof_clean["kernel_launches"]),
        e2e=e2e,
    )
    if found_mode:
        result["config"]["contacts"] = ("found every step by spatial hashing inside the timed "
                                        "region: vertex pairs closer than %g m that are not "
                                        "springs, k = %g" % (radius, W.K_CONTACT))
        result["config"]["contacts_per_step"] = sum(found_counts) / max(len(found_counts), 1)
        # the capacity set for found contacts is far above what is found: the
        # L2 statement takes the matrix actually assembled
        a_mb = 28 * nnzb / 1e6
        result["config"]["l2"] = (
            "inputs larger than L2: A is %.0f MB per step vs 129 MB L2" % a_mb if a_mb > 129
            else "A (%.1f MB) fits in the 129 MB L2: L2-resident, not an HBM-bound case" % a_mb)
        result["e2e_note"] = "not measured in this mode (the contacts are found on the device)"
    if not args.no_layouts:
        result["spmv_layouts"] = spmv_layouts(cloth, n, dev)

    # ---- CPU baseline: the oracle on the host cores, one whole step -------
    # the first timed step, from the same state and contacts as the GPU's
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c = host_contacts[Wm]
        step_s, it_o = oracle_whole_step(w, x_start.cpu().numpy(), v_start.cpu().numpy(),
                                         c if c.n else None)
        result["cpu_baseline"] = dict(
            value=1.0 / step_s, unit=UNIT, cores=1, kind="oracle",
            sample="fp64 C++ oracle, one thread: one whole implicit step (assembly, PCG to "
                   "%g, update; %.1f s, measured, not extrapolated) -- the first timed step, "
                   "from the GPU's state and contacts of that step; PCG iterations: oracle %d, "
                   "GPU %d" % (w.tol, step_s, it_o, its[0]),
            iterations=it_o, gpu_iterations=its[0])
    cloth.close()
    return result


def run_reference(args):
    """The fp64 oracle on the host cores, same config, metric and unit.

    A whole oracle step takes tens of seconds, so each step is a bounded
    sample -- the step's full assembly plus a few PCG iterations, timed --
    extrapolated to a whole step with the oracle's own iteration count for
    that step of its trajectory (oracle/iteration_table.json).  The line
    says so: `extrapolated` is true and `ms_per_step` is not wall time."""
    from sparse_linear_solve_gb300 import workloads as W
    w = W.make(args.config)
    K, Wm = args.steps, args.warmup
    table = oracle_step_iterations(args.config)
    mean_it = float(sum(table)) / len(table) if table else float(w.maxit)
    samples, its = [], []
    wall0 = time.perf_counter()
    for t in range(Wm + K):
        c = w.contacts(t)
        iters = args.oracle_iters if t >= Wm else 1
        t_asm, t_it = oracle_sample(w, w.x0, w.v0, c if c.n else None, iters)
        if t >= Wm:
            it_t = table[t] if t < len(table) else mean_it
            its.append(it_t)
            samples.append(t_asm + it_t * t_it)
    wall = time.perf_counter() - wall0
    step_s = sum(samples) / len(samples)
    value = 1.0 / step_s
    src = ("the oracle's own trajectory, steps %d-%d" % (Wm, Wm + K - 1)
           if Wm + K <= len(table) else
           "the oracle's trajectory table (%d steps; its mean past them)" % len(table))
    sample = ("EXTRAPOLATED, not measured whole: fp64 C++ oracle, one thread; per step the "
              "full assembly plus %d PCG iterations timed at the initial state, scaled to "
              "the PCG iterations of that step (%s; mean %.1f); %.1f s of wall time in all"
              % (args.oracle_iters, src, sum(its) / len(its), wall))
    return dict(metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus, steps=K, warmup=Wm,
                ms_per_step=step_s * 1e3, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic",
                config=bench_config(w),
                impl="reference", extrapolated=True, wall_s=wall,
                pcg_iterations_mean=sum(its) / len(its),
                cpu_baseline=dict(kind="oracle", cores=1, sample=sample, value=value, unit=UNIT),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
