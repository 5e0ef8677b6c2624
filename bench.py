"""Benchmark of the DoRA norm + compose hot path on GB300.

One step = the whole path on one module of the 8192-wide rank-384 workload
(out = in = 8192, r = 384, T = 15360 tokens = batch 3 x seq 5120, bf16
activations, fp32 weights): factored norm -> compose forward -> compose
backward, through the C ABI.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the method's plain definition) on
a bounded sample of the same workload, on all the host cores (a process pool
over independent columns and rows).

Multi-GPU: one process per GPU under torchrun; every rank runs an independent
replica on its own seeded inputs (the path has no exchange step), timing is
the max over ranks, and the value is the aggregate over ranks ("weak").
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

# one BLAS thread per process: the single-core baseline runs here, the
# all-core one in a pool of worker processes
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from parameter_efficient_fine_gb300 import workloads as wl  # noqa: E402

METRIC = "fused DoRA compose fwd+bwd HBM GB/s (% of GB300 peak); factored-norm µs/module"
WORKLOAD = "high_rank"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# dram__bytes_read.sum + dram__bytes_write.sum of one compose_bwd_kernel launch
# on this workload with the inputs rotated as below, from one ncu capture of
# that kernel (755,076,352 read: exactly dy, base and lora; 459,657,984
# written of the 503 MB of d_base and d_lora, the rest still dirty in L2 when
# the kernel ends); None whenever the kernel changes, until captured again
COMPOSE_BWD_TRAFFIC_BYTES = 755076352 + 459657984
INPUT_SETS = 3   # input sets rotated over the steps: each is larger than L2


def algorithmic(sh) -> dict:
    """Bytes each kernel must move at minimum (each input read once, each output
    written once) and the norm's algorithmic flops (single pass, no TF32 split)."""
    e = sh.act_bytes
    T, out, inp, r = sh.T, sh.out, sh.inp, sh.r
    return {
        "fwd_bytes": 3 * T * out * e + 4 * out,                # base, lora -> y ; g
        "bwd_bytes": 5 * T * out * e + 3 * 4 * out,            # dy, base, lora -> d_base, d_lora ; g, n, d_mag
        "norm_bytes": 4 * (out * inp + r * inp + out * r + 3 * out),
        "norm_flops": 2 * out * (inp + r) * r + 2 * r * r * inp,     # norm pass + Gram pass
    }


def peaks() -> dict:
    p = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": 1700.0,
         "tf32_tflops": 1700.0 / 2, "source": "fallback"}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        p = {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
             "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "source": "measured"}
        p["tf32_tflops"] = p["bf16_tflops_sustained"] / 2
    except Exception:
        pass
    return p


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank helpers (replicas: no data-path collective, only timing)
# ---------------------------------------------------------------------------
def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of a list of floats over all ranks (identity at N = 1)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_gbs(bytes_per_rank, seconds_max, world):
    """Whole-job throughput of `world` replicas that each moved bytes_per_rank,
    the slowest taking seconds_max."""
    return world * bytes_per_rank / seconds_max / 1e9


# ---------------------------------------------------------------------------
# CPU oracle arm (also the cpu_baseline leg of our own line)
# ---------------------------------------------------------------------------
def oracle_sample(sh, d, tokens: int, rows: int) -> dict:
    """Times the fp64 oracle on a bounded sample: compose fwd + bwd on the first
    `tokens` tokens (all columns), and the dense norm on the first `rows` rows."""
    import oracle
    s = d["s"]
    base = oracle.bf16_bits_to_f64(d["base"][:tokens])
    lora = oracle.bf16_bits_to_f64(d["lora"][:tokens])
    dy = oracle.bf16_bits_to_f64(d["dy"][:tokens])
    t0 = time.perf_counter()
    n, g = oracle.weight_norm(d["W0"][:rows], d["A"], d["B"][:rows], d["m"][:rows], s)
    t1 = time.perf_counter()
    g_full = np.ones(sh.out)
    g_full[:rows] = g
    n_full = np.ones(sh.out)
    n_full[:rows] = n
    y = oracle.compose_fwd(base, lora, g_full, s)
    t2 = time.perf_counter()
    oracle.compose_bwd(dy, base, lora, g_full, n_full, s)
    t3 = time.perf_counter()
    sub = wl.ModuleShape(sh.name, sh.out, sh.inp, sh.r, tokens, sh.act, sh.sigma_B, sh.sigma_m, True, False)
    a = algorithmic(sub)
    del y
    return {"compose_s": (t3 - t1), "norm_s": (t1 - t0), "compose_bytes": a["fwd_bytes"] + a["bwd_bytes"],
            "norm_us_per_module": (t1 - t0) * 1e6 * sh.out / rows, "tokens": tokens, "rows": rows}


def _shm_put(arrays):
    """Copies arrays into shared memory blocks; returns the blocks and their
    (name, shape, dtype) descriptions for the workers."""
    from multiprocessing import shared_memory
    blocks, desc = [], {}
    for k, a in arrays.items():
        a = np.ascontiguousarray(a)
        b = shared_memory.SharedMemory(create=True, size=max(a.nbytes, 1))
        np.ndarray(a.shape, a.dtype, buffer=b.buf)[...] = a
        blocks.append(b)
        desc[k] = (b.name, a.shape, a.dtype.str)
    return blocks, desc


def _oracle_part(task):
    """Worker: the oracle on one slice, from the shared-memory sample.
    kind 'norm': dense norm of rows [lo, hi); kind 'compose': compose fwd + bwd
    of columns [lo, hi) (columns are independent in both)."""
    from multiprocessing import shared_memory
    import oracle
    kind, desc, s, lo, hi = task
    blocks, a = [], {}
    for k, (name, shape, dt) in desc.items():
        b = shared_memory.SharedMemory(name=name)
        blocks.append(b)
        a[k] = np.ndarray(shape, np.dtype(dt), buffer=b.buf)
    if kind == "norm":
        oracle.weight_norm(a["W0"][lo:hi], a["A"], a["B"][lo:hi], a["m"][lo:hi], s)
    else:
        base = oracle.bf16_bits_to_f64(a["base"][:, lo:hi])
        lora = oracle.bf16_bits_to_f64(a["lora"][:, lo:hi])
        dy = oracle.bf16_bits_to_f64(a["dy"][:, lo:hi])
        g = np.ones(hi - lo)
        oracle.compose_fwd(base, lora, g, s)
        oracle.compose_bwd(dy, base, lora, g, g, s)
    a.clear()
    for b in blocks:
        b.close()
    return hi - lo


class ParallelOracle:
    """The oracle as it stands on every host core: a pool of worker processes
    (spawn start method: safe beside a CUDA context), each taking a slice of
    columns (compose) or rows (norm) of a bounded sample held in shared memory."""

    def __init__(self, sh, d, tokens, rows, cores=None):
        import concurrent.futures as cf
        import multiprocessing as mp
        self.sh, self.tokens, self.rows = sh, tokens, rows
        self.cores = cores or os.cpu_count() or 1
        self.blocks, self.desc = _shm_put({
            "base": d["base"][:tokens], "lora": d["lora"][:tokens], "dy": d["dy"][:tokens],
            "W0": d["W0"][:rows], "A": d["A"], "B": d["B"][:rows], "m": d["m"][:rows]})
        self.s = d["s"]
        self.pool = cf.ProcessPoolExecutor(max_workers=self.cores, mp_context=mp.get_context("spawn"))
        self.run()   # start the workers and import numpy / the oracle in each

    def _map(self, kind, n):
        cuts = np.linspace(0, n, self.cores + 1).astype(int)
        tasks = [(kind, self.desc, self.s, int(cuts[i]), int(cuts[i + 1])) for i in range(self.cores)
                 if cuts[i + 1] > cuts[i]]
        t0 = time.perf_counter()
        list(self.pool.map(_oracle_part, tasks))
        return time.perf_counter() - t0

    def run(self) -> dict:
        norm_s = self._map("norm", self.rows)
        compose_s = self._map("compose", self.sh.out)
        sub = wl.ModuleShape(self.sh.name, self.sh.out, self.sh.inp, self.sh.r, self.tokens, self.sh.act,
                             self.sh.sigma_B, self.sh.sigma_m, True, False)
        a = algorithmic(sub)
        return {"compose_s": compose_s, "norm_s": norm_s, "compose_bytes": a["fwd_bytes"] + a["bwd_bytes"],
                "norm_us_per_module": norm_s * 1e6 * self.sh.out / self.rows}

    def close(self):
        self.pool.shutdown()
        for b in self.blocks:
            b.close()
            b.unlink()


def cpu_baseline(sh, d, tokens=4096, rows=1024, budget_s=10.0, max_reps=8) -> dict:
    """The oracle as it stands, repeated on the same bounded sample until about
    `budget_s` seconds of CPU work have been timed: on all host cores (the
    reported value) and on one core."""
    def repeat(fn):
        cb = cs = ns = 0.0
        reps = 0
        t0 = time.perf_counter()
        while reps < max_reps and (reps == 0 or time.perf_counter() - t0 < budget_s):
            r = fn()
            cb += r["compose_bytes"]
            cs += r["compose_s"]
            ns += r["norm_s"]
            reps += 1
        return cb / cs / 1e9, ns / reps * 1e6 * sh.out / rows, reps

    one_gbs, one_norm, one_reps = repeat(lambda: oracle_sample(sh, d, tokens, rows))
    po = ParallelOracle(sh, d, tokens, rows)
    try:
        all_gbs, all_norm, all_reps = repeat(po.run)
    finally:
        po.close()
    return {"value": all_gbs, "unit": "GB/s", "cores": po.cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle on {po.cores} worker processes (one thread each), {all_reps} repetitions: "
                      f"compose fwd+bwd on {tokens} of {sh.T} tokens x {sh.out} columns, split by columns; dense "
                      f"norm on {rows} of {sh.out} rows, split by rows",
            "norm_us_per_module": all_norm,
            "single_core": {"value": one_gbs, "unit": "GB/s", "cores": 1, "norm_us_per_module": one_norm,
                            "repetitions": one_reps}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    sh = wl.shape(WORKLOAD)
    d = wl.make_module(sh, wl.seed_for(WORKLOAD))
    # per-step sample sized so that warm-up + steps stay within about two
    # minutes on all host cores
    n = max(1, args.steps + args.warmup)
    tokens = int(min(4096, max(64, 4096 * 40 // n)))
    rows = int(min(1024, max(32, 1024 * 40 // n)))
    po = ParallelOracle(sh, d, tokens, rows)
    try:
        for _ in range(args.warmup):
            po.run()
        times, vals, norm_us = [], [], []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            r = po.run()
            times.append(time.perf_counter() - t0)
            vals.append(r["compose_bytes"] / r["compose_s"] / 1e9)
            norm_us.append(r["norm_us_per_module"])
    finally:
        po.close()
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: out=in={sh.out}, r={sh.r}, T={sh.T} bf16 activations, fp32 weights",
                   "sample_per_step": f"compose fwd+bwd on {tokens} tokens, dense norm on {rows} rows"},
        "norm_us_per_module": statistics.mean(norm_us),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": po.cores, "kind": "oracle",
                         "sample": f"{tokens} tokens x {sh.out} columns compose fwd+bwd (split by columns); "
                                   f"{rows} norm rows (split by rows); {po.cores} worker processes"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import parameter_efficient_fine_gb300 as dora
    from parameter_efficient_fine_gb300 import build as dbuild

    dbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    sh = wl.shape(WORKLOAD)
    d = wl.make_module(sh, wl.seed_for(WORKLOAD, rank))
    s = d["s"]
    alg = algorithmic(sh)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def bf16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    W0, A, B, m = (f32(d[k]) for k in ("W0", "A", "B", "m"))
    base, lora, dy = (bf16(d[k]) for k in ("base", "lora", "dy"))
    # INPUT_SETS copies of the inputs in separate buffers (each ~1 GB, far
    # above L2), rotated over the steps: no launch reads lines that the
    # previous step left in L2
    sets_in = [(W0, A, B, m, base, lora, dy)]
    for _ in range(INPUT_SETS - 1):
        sets_in.append(tuple(t.clone() for t in sets_in[0]))
    norm = torch.empty(sh.out, device=dev)
    g = torch.empty(sh.out, device=dev)
    y = torch.empty_like(base)
    db = torch.empty_like(base)
    dl = torch.empty_like(base)
    dm = torch.empty(sh.out, device=dev)
    ws_n = torch.empty(dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(dora.dora_compose_bwd_workspace(sh.T, sh.out), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(k, ev=None):
        W0_, A_, B_, m_, base_, lora_, dy_ = sets_in[k % INPUT_SETS]
        if ev is not None:
            ev[0].record(stream)
        dora.dora_norm_factored(W0_, A_, B_, m_, s, norm, g, ws_n, stream)
        if ev is not None:
            ev[1].record(stream)
        dora.dora_compose_fwd(base_, lora_, g, s, y, stream)
        if ev is not None:
            ev[2].record(stream)
        dora.dora_compose_bwd(dy_, base_, lora_, g, norm, s, db, dl, dm, ws_b, stream)
        if ev is not None:
            ev[3].record(stream)

    # the clock sampler starts before the warm-up, so that its start-up (an
    # nvidia-smi process) is not inside the timed region
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    if dora.dora_device_error() != 0:
        raise RuntimeError("a kernel wait gave up during warm-up")

    def barrier():
        if dist is not None:
            dist.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    launches0 = dora.dora_kernel_launches()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(k, evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = dora.dora_kernel_launches() - launches0
    clk = clocks.stop()
    if dora.dora_device_error() != 0:
        raise RuntimeError("a kernel wait gave up during the timed steps")

    total_ms = t_start.elapsed_time(t_end)
    norm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    total_ms, norm_ms, fwd_ms, bwd_ms = max_over_ranks([total_ms, norm_ms, fwd_ms, bwd_ms], dist, dev)

    compose_bytes = alg["fwd_bytes"] + alg["bwd_bytes"]
    value = aggregate_gbs(compose_bytes, (fwd_ms + bwd_ms) * 1e-3, world)
    pk = peaks()

    # ---- end to end through the public API, host buffers, copies timed.
    # Every step uploads all its inputs from pinned host memory and reads all
    # its outputs back.  Three streams and two device buffer sets pipeline the
    # steps: step i+1's uploads overlap step i's compute and downloads.
    e2e = None
    if not args.no_e2e:
        names_in = ("W0", "A", "B", "m", "base", "lora", "dy")
        names_out = ("y", "db", "dl", "dm", "norm", "g")
        set0 = {"W0": W0, "A": A, "B": B, "m": m, "base": base, "lora": lora, "dy": dy,
                "y": y, "db": db, "dl": dl, "dm": dm, "norm": norm, "g": g}
        set1 = {k: torch.empty_like(v) for k, v in set0.items()}
        sets = (set0, set1)
        host_in = {k: set0[k].cpu().pin_memory() for k in names_in}
        host_out = {k: torch.empty(set0[k].shape, dtype=set0[k].dtype, pin_memory=True) for k in names_out}
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())
        s_h2d, s_comp, s_d2h = torch.cuda.Stream(), stream, torch.cuda.Stream()
        ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("up", "comp", "down")}
        started = [False, False]

        def e2e_step(i):
            k = i % 2
            d = sets[k]
            if started[k]:
                s_h2d.wait_event(ev["comp"][k])      # compute of step i-2 is done reading set k
            with torch.cuda.stream(s_h2d):
                for n in names_in:
                    d[n].copy_(host_in[n], non_blocking=True)
            ev["up"][k].record(s_h2d)
            s_comp.wait_event(ev["up"][k])
            if started[k]:
                s_comp.wait_event(ev["down"][k])     # outputs of step i-2 are copied out
            dora.dora_norm_factored(d["W0"], d["A"], d["B"], d["m"], s, d["norm"], d["g"], ws_n, s_comp)
            dora.dora_compose_fwd(d["base"], d["lora"], d["g"], s, d["y"], s_comp)
            dora.dora_compose_bwd(d["dy"], d["base"], d["lora"], d["g"], d["norm"], s, d["db"], d["dl"], d["dm"],
                                  ws_b, s_comp)
            ev["comp"][k].record(s_comp)
            s_d2h.wait_event(ev["comp"][k])
            with torch.cuda.stream(s_d2h):
                for n in names_out:
                    host_out[n].copy_(d[n], non_blocking=True)
            ev["down"][k].record(s_d2h)
            started[k] = True

        e2e_steps = min(args.steps, args.e2e_steps)
        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_h2d)
        for i in range(e2e_steps):
            e2e_step(i)
        b.record(s_d2h)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = a.elapsed_time(b) / e2e_steps
        e2e_ms = max_over_ranks([e2e_ms], dist, dev)[0]
        e2e = {"value": aggregate_gbs(compose_bytes, e2e_ms * 1e-3, world), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
               "pipelining": "upload, compute and download streams, 2 buffer sets: uploads of step i+1 overlap "
                             "compute and downloads of step i (bound by the host link)"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    bwd_gbs = alg["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = alg["fwd_bytes"] / (fwd_ms * 1e-3) / 1e9
    norm_us = norm_ms * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: DoRA module out=in={sh.out}, r={sh.r} (s=32/sqrt(r)), "
                               f"T={sh.T} tokens (batch 3 x seq 5120), bf16 activations, fp32 weights; "
                               "step = factored norm + compose fwd + compose bwd",
                   "l2": f"{INPUT_SETS} input sets in separate buffers (each ~1 GB: W0 268 MB, each activation "
                         "252 MB) rotated over the steps, so no launch reads what the previous step left in L2",
                   "parallelism": "replicas" if world > 1 else "single"},
        "pct_of_hbm_peak": 100.0 * value / world / pk["hbm_gbs"],
        "norm_us_per_module": norm_us,
        "breakdown": {"norm_us": norm_us, "fwd_us": fwd_ms * 1e3, "bwd_us": bwd_ms * 1e3,
                      "fwd_gbs": fwd_gbs, "bwd_gbs": bwd_gbs,
                      "norm_tflops_algorithmic": alg["norm_flops"] / (norm_ms * 1e-3) / 1e12},
        "roofline": {"bound": "hbm", "kernel": "compose_bwd", "achieved": bwd_gbs, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": bwd_gbs / pk["hbm_gbs"],
                     "traffic": COMPOSE_BWD_TRAFFIC_BYTES,
                     "algorithmic_bytes": alg["bwd_bytes"], "peak_source": pk["source"] + " (copy bandwidth)"},
        "roofline_norm": {"bound": "tensor",
                          "kernel": "factored norm (the split of A, then one launch: Gram pieces, reduction of "
                                    "s/2 G and the norm GEMM)",
                          "achieved": 3 * alg["norm_flops"] / (norm_ms * 1e-3) / 1e12,
                          "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                          "frac": 3 * alg["norm_flops"] / (norm_ms * 1e-3) / 1e12 / pk["bf16_tflops_sustained"],
                          "note": "achieved = issued bf16 tensor work (each fp32 product is three bf16 products "
                                  "h_x h_y + l_x h_y + h_x l_y: 3x the algorithmic flops) / norm time; peak = "
                                  "measured sustained bf16 (of " + pk["source"] + "; the norm runs inside a long "
                                  "step)",
                          "algorithmic_tflops": alg["norm_flops"] / (norm_ms * 1e-3) / 1e12,
                          "peak_algorithmic": pk["bf16_tflops"] / 2,
                          "frac_algorithmic": alg["norm_flops"] / (norm_ms * 1e-3) / 1e12 / (pk["bf16_tflops"] / 2),
                          "note_algorithmic": "the method's flops (one pass, fp32 products) against the dense TF32 "
                                              "rate: measured burst bf16 x 1/2 (nominal TF32:bf16 ratio)"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_workloads:
        # the other workloads, timed in the same run after the timed region
        # (inputs drawn on the device; each kernel timed over repeated calls)
        del sets_in
        torch.cuda.empty_cache()
        line["workloads"] = {
            "attn_proj_inference": attn_proj_row(dora, dev, stream),
            "rank_sweep": rank_sweep_rows(dora, dev, stream, wl.RANK_SWEEP),
            "mlp_stack": mlp_stack_row(dora, dev, stream)}
        line["workloads"]["mlp_stack"]["frac_of_hbm"] = (
            line["workloads"]["mlp_stack"]["aggregate_algorithmic_gbs"] / pk["hbm_gbs"])
        line["workloads"]["mlp_stack"]["frac_of_hbm_graph"] = (
            line["workloads"]["mlp_stack"]["aggregate_algorithmic_gbs_graph"] / pk["hbm_gbs"])
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, d)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reports for the other workloads (one JSON line each; not the bench line)
# ---------------------------------------------------------------------------
def _time_ms(fn, reps, stream):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _device_module(sh, seed, dev):
    """Seeded inputs drawn on the device (torch Philox), same distributions as
    parameter_efficient_fine_gb300.workloads: fast enough for 64-module stacks."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    W0 = torch.randn(sh.out, sh.inp, device=dev, generator=gen) / math.sqrt(sh.inp)
    A = torch.randn(sh.r, sh.inp, device=dev, generator=gen) / math.sqrt(sh.inp)
    B = torch.randn(sh.out, sh.r, device=dev, generator=gen) * sh.sigma_B
    m = W0.double().norm(dim=1).float() * (1 + sh.sigma_m * torch.randn(sh.out, device=dev, generator=gen))
    return W0, A, B, m


def rank_sweep_rows(dora, dev, stream, ranks):
    """out = in = 8192, T = 8192 bf16, per rank: norm time (and its host time
    per call), compose GB/s and the norm's whole transient (its workspace)
    against one dense fp32 out x in matrix.  Inputs drawn on the device,
    seeded by position."""
    import torch
    rows = []
    for k, r in enumerate(ranks):
        sh = wl.shape("rank_sweep", r=r)
        W0, A, B, m = _device_module(sh, wl.seed_for("rank_sweep", k), dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed_for("rank_sweep", k) + 7)
        act = [torch.randn(sh.T, sh.out, device=dev, generator=gen).bfloat16() for _ in range(3)]
        act[1] = (act[1].float() * math.sqrt(sh.r) * sh.sigma_B).bfloat16()
        base, lora, dy = act
        norm = torch.empty(sh.out, device=dev)
        g = torch.empty(sh.out, device=dev)
        nbytes = dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        y, db, dl = torch.empty_like(base), torch.empty_like(base), torch.empty_like(base)
        dm = torch.empty(sh.out, device=dev)
        wsb = torch.empty(dora.dora_compose_bwd_workspace(sh.T, sh.out), dtype=torch.uint8, device=dev)
        t_norm = _time_ms(lambda: dora.dora_norm_factored(W0, A, B, m, sh.s, norm, g, ws, stream), 20, stream)
        # host time of one call (the device is kept busy, so the call returns
        # as soon as its launches are queued)
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        for _ in range(20):
            dora.dora_norm_factored(W0, A, B, m, sh.s, norm, g, ws, stream)
        host_us = (time.perf_counter() - h0) / 20 * 1e6
        torch.cuda.synchronize()
        t_fwd = _time_ms(lambda: dora.dora_compose_fwd(base, lora, g, sh.s, y, stream), 20, stream)
        t_bwd = _time_ms(lambda: dora.dora_compose_bwd(dy, base, lora, g, norm, sh.s, db, dl, dm, wsb, stream),
                         20, stream)
        alg = algorithmic(sh)
        dense = sh.out * sh.inp * 4
        rows.append({"r": r, "out": sh.out, "in": sh.inp, "T": sh.T,
                     "norm_us": t_norm * 1e3, "norm_host_us_per_call": host_us,
                     "norm_tflops_algorithmic": alg["norm_flops"] / (t_norm * 1e-3) / 1e12,
                     "fwd_gbs": alg["fwd_bytes"] / (t_fwd * 1e-3) / 1e9,
                     "bwd_gbs": alg["bwd_bytes"] / (t_bwd * 1e-3) / 1e9,
                     "norm_transient_bytes": nbytes, "dense_fp32_matrix_bytes": dense,
                     "dense_over_transient": dense / nbytes,
                     "rank_dependent_theory": sh.out * sh.inp / (sh.out * sh.r + sh.r * sh.r)})
        del W0, A, B, m, act, base, lora, dy, ws, y, db, dl
        torch.cuda.empty_cache()
    return rows


def mlp_stack_row(dora, dev, stream, reps=3):
    """32 gate/up (4096 -> 14336) + 32 down (14336 -> 4096) modules, r = 512,
    T = 16384, training step per module (norm + fwd + bwd), independent seeds,
    back to back: modules/s and aggregate algorithmic GB/s."""
    import torch
    shapes = [wl.shape("mlp_gate_up"), wl.shape("mlp_down")]
    mods = []
    for k in range(wl.MLP_REPEATS):
        for j, sh in enumerate(shapes):
            mods.append((sh, _device_module(sh, wl.seed_for(sh.name, 2 * k + j), dev)))
    bufs = {}
    for sh in shapes:
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed_for(sh.name) + 99)
        act = [torch.randn(sh.T, sh.out, device=dev, generator=gen).bfloat16() for _ in range(3)]
        act[1] = (act[1].float() * math.sqrt(sh.r) * sh.sigma_B).bfloat16()
        bufs[sh.name] = {
            "act": act, "y": torch.empty_like(act[0]), "db": torch.empty_like(act[0]),
            "dl": torch.empty_like(act[0]), "norm": torch.empty(sh.out, device=dev),
            "g": torch.empty(sh.out, device=dev), "dm": torch.empty(sh.out, device=dev),
            "ws": torch.empty(dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8,
                              device=dev),
            "wsb": torch.empty(dora.dora_compose_bwd_workspace(sh.T, sh.out), dtype=torch.uint8, device=dev)}

    def stack():
        st = torch.cuda.current_stream()   # the capture stream while a graph is captured
        for sh, (W0, A, B, m) in mods:
            b = bufs[sh.name]
            base, lora, dy = b["act"]
            dora.dora_norm_factored(W0, A, B, m, sh.s, b["norm"], b["g"], b["ws"], st)
            dora.dora_compose_fwd(base, lora, b["g"], sh.s, b["y"], st)
            dora.dora_compose_bwd(dy, base, lora, b["g"], b["norm"], sh.s, b["db"], b["dl"], b["dm"], b["wsb"], st)

    t = _time_ms(stack, reps, stream)
    total = sum(sum(v for k, v in algorithmic(sh).items() if k.endswith("_bytes")) for sh, _ in mods)
    compose = sum(algorithmic(sh)["fwd_bytes"] + algorithmic(sh)["bwd_bytes"] for sh, _ in mods)
    row = {"modules": len(mods), "ms_per_stack": t, "modules_per_s": len(mods) / (t * 1e-3),
           "us_per_module": t * 1e3 / len(mods), "aggregate_algorithmic_gbs": total / (t * 1e-3) / 1e9,
           "compose_share_of_bytes": compose / total,
           "inputs": "device-drawn (torch Philox), seed per module; activations shared per shape"}
    # the same stack captured once in a CUDA graph (the calls above have set
    # up every plan and tensor map) and replayed: the kernels' own launch
    # overhead without the host's
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        stack()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        stack()
    tg = _time_ms(graph.replay, reps, stream)
    row.update({"ms_per_stack_graph": tg, "modules_per_s_graph": len(mods) / (tg * 1e-3),
                "aggregate_algorithmic_gbs_graph": total / (tg * 1e-3) / 1e9})
    del graph, mods, bufs
    torch.cuda.empty_cache()
    return row


def attn_proj_row(dora, dev, stream, reps=20):
    """The attention-projection module, inference path: out = in = 4096,
    r = 64, T = 8192 bf16; factored norm then compose forward."""
    import torch
    sh = wl.shape("attn_proj")
    W0, A, B, m = _device_module(sh, wl.seed_for("attn_proj"), dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed_for("attn_proj") + 7)
    base = torch.randn(sh.T, sh.out, device=dev, generator=gen).bfloat16()
    lora = (torch.randn(sh.T, sh.out, device=dev, generator=gen) * math.sqrt(sh.r) * sh.sigma_B).bfloat16()
    norm = torch.empty(sh.out, device=dev)
    g = torch.empty(sh.out, device=dev)
    y = torch.empty_like(base)
    ws = torch.empty(dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8, device=dev)
    t_norm = _time_ms(lambda: dora.dora_norm_factored(W0, A, B, m, sh.s, norm, g, ws, stream), reps, stream)
    t_fwd = _time_ms(lambda: dora.dora_compose_fwd(base, lora, g, sh.s, y, stream), reps, stream)

    def step():
        dora.dora_norm_factored(W0, A, B, m, sh.s, norm, g, ws, stream)
        dora.dora_compose_fwd(base, lora, g, sh.s, y, stream)

    t_step = _time_ms(step, reps, stream)
    alg = algorithmic(sh)
    row = {"out": sh.out, "in": sh.inp, "r": sh.r, "T": sh.T, "norm_us": t_norm * 1e3, "fwd_us": t_fwd * 1e3,
           "fwd_gbs": alg["fwd_bytes"] / (t_fwd * 1e-3) / 1e9, "us_per_step": t_step * 1e3,
           "norm_transient_bytes": ws.numel()}
    del W0, A, B, m, base, lora, y, ws
    torch.cuda.empty_cache()
    return row


def run_report(args):
    import torch
    import parameter_efficient_fine_gb300 as dora
    from parameter_efficient_fine_gb300 import build as dbuild

    dbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    if args.report == "rank_sweep":
        for row in rank_sweep_rows(dora, dev, stream, args.ranks or wl.RANK_SWEEP):
            print(json.dumps(dict(report="rank_sweep", **row)), flush=True)
    elif args.report == "bf16_norm":
        # the factored norm with bf16 W0, A, B (the same seeded weights rounded
        # to bf16) at out = in = 8192 over the swept ranks; the row norms of W0
        # are computed once (W0 is frozen) and timed separately
        for k, r in enumerate(sorted(wl.RANK_SWEEP + (384,))):
            if args.ranks and r not in args.ranks:
                continue
            sh = wl.shape("rank_sweep", r=r)
            W0, A, B, m = _device_module(sh, wl.seed_for("rank_sweep", k), dev)
            W0, A, B = W0.bfloat16(), A.bfloat16(), B.bfloat16()
            n0 = torch.empty(sh.out, device=dev)
            norm = torch.empty(sh.out, device=dev)
            g = torch.empty(sh.out, device=dev)
            nbytes = dora.dora_norm_factored_bf16_workspace(sh.out, sh.inp, sh.r)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            t_row = _time_ms(lambda: dora.dora_row_sumsq_bf16(W0, n0, stream), 20, stream)
            t_norm = _time_ms(lambda: dora.dora_norm_factored_bf16(W0, A, B, m, n0, sh.s, norm, g, ws, stream), 20,
                              stream)
            alg = algorithmic(sh)
            w_bytes = sh.out * sh.inp * 2
            print(json.dumps({"report": "bf16_norm", "r": r, "out": sh.out, "in": sh.inp,
                              "norm_us": t_norm * 1e3,
                              "norm_tflops_algorithmic": alg["norm_flops"] / (t_norm * 1e-3) / 1e12,
                              "row_sumsq_us": t_row * 1e3, "row_sumsq_gbs": w_bytes / (t_row * 1e-3) / 1e9,
                              "w0_stream_gbs_in_norm": w_bytes / (t_norm * 1e-3) / 1e9,
                              "norm_transient_bytes": nbytes}), flush=True)
            del W0, A, B, m, ws
            torch.cuda.empty_cache()
    elif args.report == "norm_grad":
        # gradient through the norm (the variant with the norm not detached):
        # dora_norm_factored_bwd beside the forward norm at out = in = 8192 over
        # the swept ranks; algorithmic flops of the products it evaluates
        # (W0 A^T, B G, A A^T for dB; (c B)^T W0, H A, B^T diag(c) B for dA)
        for k, r in enumerate(sorted(wl.RANK_SWEEP + (384,))):
            if args.ranks and r not in args.ranks:
                continue
            sh = wl.shape("rank_sweep", r=r)
            W0, A, B, m = _device_module(sh, wl.seed_for("rank_sweep", k), dev)
            gen = torch.Generator(device=dev)
            gen.manual_seed(wl.seed_for("rank_sweep", k) + 11)
            d_mag = 0.1 * torch.randn(sh.out, device=dev, generator=gen)
            norm = torch.empty(sh.out, device=dev)
            g = torch.empty(sh.out, device=dev)
            ws = torch.empty(dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8, device=dev)
            nbytes = dora.dora_norm_factored_bwd_workspace(sh.out, sh.inp, sh.r)
            wsb = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            dA = torch.empty(sh.r, sh.inp, device=dev)
            dB = torch.empty(sh.out, sh.r, device=dev)
            t_norm = _time_ms(lambda: dora.dora_norm_factored(W0, A, B, m, sh.s, norm, g, ws, stream), 20, stream)
            t_grad = _time_ms(lambda: dora.dora_norm_factored_bwd(W0, A, B, norm, g, d_mag, sh.s, dA, dB, wsb,
                                                                  stream), 20, stream)
            flops = 4 * sh.out * sh.inp * sh.r + 4 * sh.r * sh.r * (sh.out + sh.inp)
            print(json.dumps({"report": "norm_grad", "r": r, "out": sh.out, "in": sh.inp,
                              "norm_us": t_norm * 1e3, "norm_grad_us": t_grad * 1e3,
                              "norm_grad_tflops_algorithmic": flops / (t_grad * 1e-3) / 1e12,
                              "norm_grad_transient_bytes": nbytes,
                              "dense_fp32_matrix_bytes": sh.out * sh.inp * 4}), flush=True)
            del W0, A, B, m, ws, wsb, dA, dB
            torch.cuda.empty_cache()
    elif args.report == "fused":
        # the compose folded into its adjacent products on the high-rank layer
        # (T = 15360, out = in = 8192, r = 384, bf16), beside the unfused path:
        # cuBLAS bf16 products (torch.matmul) writing base / lora, then the
        # library's compose pass
        sh = wl.shape("high_rank")
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed_for("high_rank") + 31)
        T, inp, out, r = sh.T, sh.inp, sh.out, sh.r
        x = torch.randn(T, inp, device=dev, generator=gen).bfloat16()
        W0 = (torch.randn(out, inp, device=dev, generator=gen) / math.sqrt(inp)).bfloat16()
        xa = torch.randn(T, r, device=dev, generator=gen).bfloat16()
        B = torch.randn(out, r, device=dev, generator=gen) * sh.sigma_B
        g = 1 + sh.sigma_m * torch.randn(out, device=dev, generator=gen)
        base = torch.randn(T, out, device=dev, generator=gen).bfloat16()
        y = torch.empty(T, out, device=dev, dtype=torch.bfloat16)
        ws = torch.empty(dora.dora_compose_fused_workspace(out, r), dtype=torch.uint8, device=dev)
        Bs16 = (sh.s * B).bfloat16()
        t_lora = _time_ms(lambda: dora.dora_compose_lora_fwd(base, xa, B, g, sh.s, y, ws, stream), 20, stream)
        t_lin = _time_ms(lambda: dora.dora_linear_fwd(x, W0, xa, B, g, sh.s, y, ws, stream), 10, stream)
        # the lora form for an adapter kept in bf16 (one product, no split)
        B16 = B.bfloat16()
        t_lb = _time_ms(lambda: dora.dora_compose_lora_fwd_bf16(base, xa, B16, g, sh.s, y, stream), 20, stream)

        def unfused_lora_bf16():
            lora = torch.matmul(xa, B16.t())
            dora.dora_compose_fwd(base, lora, g, sh.s, y, stream)

        t_lb_u = _time_ms(unfused_lora_bf16, 20, stream)

        def unfused_lora():
            lora = torch.matmul(xa, Bs16.t())
            dora.dora_compose_fwd(base, lora, g, 1.0, y, stream)

        def unfused_linear():
            b = torch.matmul(x, W0.t())
            lora = torch.matmul(xa, Bs16.t())
            dora.dora_compose_fwd(b, lora, g, 1.0, y, stream)

        t_lora_u = _time_ms(unfused_lora, 20, stream)
        t_lin_u = _time_ms(unfused_linear, 10, stream)
        t_gemm = _time_ms(lambda: torch.matmul(x, W0.t()), 10, stream)
        lora_bytes = 2 * T * out * 2 + T * r * 2 + 2 * out * r * 2      # base, y, xa, the two bf16 halves of s B
        lb_bytes = 2 * T * out * 2 + T * r * 2 + out * r * 2            # base, y, xa, B
        flops = 2 * T * out * (inp + r)
        print(json.dumps({"report": "fused", "T": T, "in": inp, "out": out, "r": r,
                          "lora_form_us": t_lora * 1e3, "lora_form_gbs": lora_bytes / (t_lora * 1e-3) / 1e9,
                          "unfused_lora_matmul_plus_compose_us": t_lora_u * 1e3,
                          "lora_form_bf16_b_us": t_lb * 1e3, "lora_form_bf16_b_gbs": lb_bytes / (t_lb * 1e-3) / 1e9,
                          "unfused_lora_bf16_b_matmul_plus_compose_us": t_lb_u * 1e3,
                          "linear_form_us": t_lin * 1e3,
                          "linear_form_tflops_algorithmic": flops / (t_lin * 1e-3) / 1e12,
                          "unfused_two_matmuls_plus_compose_us": t_lin_u * 1e3,
                          "cublas_base_matmul_us": t_gemm * 1e3,
                          "cublas_base_matmul_tflops": 2 * T * out * inp / (t_gemm * 1e-3) / 1e12}), flush=True)
    elif args.report == "mlp_stack":
        print(json.dumps(dict(report="mlp_stack", **mlp_stack_row(dora, dev, stream))), flush=True)
    elif args.report == "attn_proj":
        print(json.dumps(dict(report="attn_proj", **attn_proj_row(dora, dev, stream))), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the attention-projection, rank-sweep and MLP-stack keys of the bench line")
    ap.add_argument("--report", choices=["rank_sweep", "mlp_stack", "attn_proj", "bf16_norm", "norm_grad", "fused"],
                    default=None,
                    help="extra per-workload report lines instead of the bench line")
    ap.add_argument("--ranks", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="report rank_sweep: these ranks instead of the sweep; bf16_norm / norm_grad: only "
                         "these ranks (comma separated)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    if args.report is not None:
        run_report(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
