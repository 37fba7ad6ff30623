"""Benchmark of the online-softmax hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. attention forward, bf16, B=2 H=16 N=8192 d=128, causal, scale 1/sqrt(128)
     (fa_fwd, the tcgen05 kernel), and
  2. the row online-softmax state of a 4096 x 32768 fp32 array N(0, 9) with the
     special rows (online_softmax_rows).
Inputs are resident in HBM before the timed region; every step re-reads inputs far
larger than the 129 MB L2 (Q, K, V: 201 MB; x: 537 MB), so no L2 flush is needed.

Printed JSON (one line, rank 0):
  value      attention TFLOP/s = 4*B*H*N^2*d/2 / mean attention kernel time (CUDA events
             on the launching stream, max over ranks); ms_attention_median beside it;
  errors     O max / mean abs and LSE max abs error of the bench step's output against
             the fp64 oracle on seeded rows of four heads (the stated gates alongside);
  row_softmax  the row kernel's GB/s = (rows*len*4 + rows*8) / mean kernel time;
  clocks     nvidia-smi samples from a loaded window: the same steps run untimed for
             --load-seconds right before the timed ones, then the timed steps;
  workloads  the other attention configurations (B4 H16 N4096 d64; B1 H8 N32768 d128
             causal, Q std 4), each timed alone on this GPU: mean / median ms, TFLOP/s,
             roofline fraction and oracle errors (not part of the step);
  e2e        the same attention metric through the public Python API with pinned host
             buffers: host->device copy of Q, K, V, the kernel and device->host read of
             O and LSE inside the timed region;
  roofline   the attention kernel against the measured dense bf16 peak; the row kernel
             (inside row_softmax) against the measured HBM copy bandwidth;
  cpu_baseline  the fp64 oracle timed on a bounded sample of the same workload on the
             host cores (rank 0, one GPU only).
``--impl reference`` times the oracle alone (see ``reference_arm``); ``--suite``,
``--backward [B,H,N,d,causal]``, ``--forward B,H,N,d,causal[,splits]``, ``--block-study``
and ``--rows state|softmax``
print per-workload lines instead (the commands the committed profiles were taken with).
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

ATTN = dict(name="attn_bf16_b2h16n8192d128_causal", B=2, H=16, N=8192, d=128, causal=True)
ROWS = dict(name="rows_4096x32768", rows=4096, length=32768)
METRIC = "attn fwd TFLOP/s and % of GB300 bf16 dense peak (1 GPU); row-softmax HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def run_config(world):
    """The workload both arms report (the bench line's ``config``)."""
    return {
        "workload": f"{ATTN['name']} + {ROWS['name']}",
        "attention": {"B": ATTN["B"], "H": ATTN["H"], "N": ATTN["N"], "d": ATTN["d"],
                      "causal": ATTN["causal"], "scale": 1.0 / math.sqrt(ATTN["d"]),
                      "inputs": "Q, K, V i.i.d. N(0,1) rounded to bf16"},
        "rows": {"rows": ROWS["rows"], "len": ROWS["length"],
                 "inputs": "N(0,9) fp32 with all-equal, +1000 and -1e4 special rows"},
        "l2": "inputs larger than L2 (201 MB attention, 537 MB rows); no flush",
        "parallelism": f"replicas x{world} (each GPU runs the full workload)",
    }


def attn_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def row_bytes(rows, length):
    return rows * length * 4.0 + rows * 8.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", 0) or 0),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# Source files each measured kernel is built from (its launch configuration included):
# recorded DRAM traffic stays valid only while these files are unchanged.
KERNEL_FILES = {
    "attn_fwd_tc_kernel": ["attn_tc.cuh", "attn_tc_impl.cuh", "ptx.cuh", "attn_tc_d128.cu",
                           "api.cu"],
    "row_state_block_kernel": ["row_state.cu", "api.cu"],
    "attn_bwd_dkdv_kernel": ["attn_bwd.cuh", "attn_bwd_impl.cuh", "attn_tc.cuh",
                             "attn_tc_impl.cuh", "ptx.cuh", "attn_bwd_d128.cu", "api_bwd.cu"],
    "attn_bwd_dq_kernel": ["attn_bwd.cuh", "attn_bwd_impl.cuh", "attn_tc.cuh",
                           "attn_tc_impl.cuh", "ptx.cuh", "attn_bwd_d128.cu", "api_bwd.cu"],
    # the d = 64 instance of attn_bwd_dkdv_kernel: the one-pass backward
    "attn_bwd_dkdv_kernel_d64": ["attn_bwd.cuh", "attn_bwd_impl.cuh", "attn_tc.cuh",
                                 "attn_tc_impl.cuh", "ptx.cuh", "attn_bwd_d64.cu", "api_bwd.cu"],
}


def kernel_sources_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "online_softmax_07_gb300", "csrc")
    for name in sorted(KERNEL_FILES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel)
    if not ent or ent.get("sources") != kernel_sources_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ ranks
def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (a no-op on one rank): the
    timing rule is the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def rank_env():
    """(world, rank, local_rank) from the launcher's environment (1, 0, 0 if absent)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every `period_ms` while the workload runs; each line is kept with
    its arrival time, so that the summary can be restricted to the window in which the
    GPU was loaded."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []   # (arrival time, line)
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={self.period_ms}", f"--id={self.index}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None):
        """Summary of the samples; with `window` = (t0, t1) (host time) the clock median,
        power and reasons come from the samples that arrived inside it (the loaded
        period), and `samples_under_load` counts them."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0, "samples_under_load": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, power, reasons, total = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                vals = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            total += 1
            if window is not None and not (window[0] <= t <= window[1]):
                continue
            sm.append(vals[0])
            smax.append(vals[1])
            power.append(vals[2])
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": total, "samples_under_load": len(sm)}


# ------------------------------------------------------------------ oracle sample (CPU)
_SHARED = {}


def _attach(spec):
    """Pool initialiser: map the parent's input arrays (shared memory, read only)."""
    from multiprocessing import shared_memory
    for key, (name, shape, dtype) in spec.items():
        shm = shared_memory.SharedMemory(name=name)
        _SHARED[key] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))
    import oracle  # noqa: F401  (import cost outside the timing)


def _arr(key):
    return _SHARED[key][1]


def _oracle_attention_task(args):
    """Query rows `rows` of head (b, h) through the fp64 oracle; returns the
    algorithmic FLOPs of those rows (4 d per visible key) and the seconds taken."""
    import oracle
    b, h, rows, scale, causal = args
    q, k, v = _arr("q")[b, h], _arr("k")[b, h], _arr("v")[b, h]
    t0 = time.perf_counter()
    oracle.attention_forward(q[None, None], k[None, None], v[None, None], scale, causal,
                             rows=rows)
    dt = time.perf_counter() - t0
    n, d = q.shape
    keys = (rows + 1) if causal else np.full(rows.shape, n)
    return 4.0 * d * float(np.sum(keys)), dt


def _oracle_rows_task(args):
    import oracle
    r0, r1 = args
    x = _arr("x")[r0:r1]
    t0 = time.perf_counter()
    oracle.row_state(x)
    return row_bytes(*x.shape), time.perf_counter() - t0


def _noop(_):
    return 0


class OraclePool:
    """A spawn pool over the host cores.  Each worker uses one BLAS thread (so that
    `cores` is the number of workers) and maps the inputs from shared memory."""

    def __init__(self, arrays: dict, workers: int):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.workers = workers
        self.shms = []
        spec = {}
        for key, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            self.shms.append(shm)
            spec[key] = (shm.name, a.shape, a.dtype.str)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(workers, initializer=_attach,
                                                     initargs=(spec,))
        finally:
            for k, val in saved.items():
                if val is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = val
        self.pool.map(_noop, range(workers))   # start-up outside any timing

    def close(self):
        self.pool.terminate()
        self.pool.join()
        for shm in self.shms:
            shm.close()
            shm.unlink()


def attention_sample_tasks(shape, rows_per_task, n_tasks, seed):
    """Tasks of a bounded oracle sample: heads (b, h) in turn, each task with
    `rows_per_task` query rows drawn uniformly (seeded) over the whole sequence."""
    B, H, N, d = shape
    g = np.random.Generator(np.random.PCG64(seed))
    tasks = []
    for i in range(n_tasks):
        b, h = (i // H) % B, i % H
        rows = np.sort(g.choice(N, size=rows_per_task, replace=False))
        tasks.append((b, h, rows, 1.0 / math.sqrt(d), ATTN["causal"]))
    return tasks


def cpu_baseline(q, k, v, x, budget_s=15.0):
    """The oracle as it stands on a bounded sample of the same workload: batches of
    tasks (64 attention query rows of one head each, rows drawn uniformly) for about
    2/3 of the budget, then batches of row states (4 whole rows per task) of the row
    workload for the rest."""
    workers = os.cpu_count() or 1
    op = OraclePool({"q": q, "k": k, "v": v, "x": x}, workers)
    try:
        flops, done, s, t0 = 0.0, 0, 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s * 2 / 3:
            tasks = attention_sample_tasks(q.shape, 64, 2 * workers, seed=4242 + s)
            flops += sum(f for f, _ in op.pool.map(_oracle_attention_task, tasks))
            done += len(tasks)
            s += 1
        att_s = time.perf_counter() - t0
        nrows = x.shape[0]
        nbytes, rdone, i, t0 = 0.0, 0, 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s / 3:
            chunks = [((4 * (i + w)) % nrows, (4 * (i + w)) % nrows + 4) for w in range(workers)]
            nbytes += sum(b for b, _ in op.pool.map(_oracle_rows_task, chunks))
            rdone += 4 * workers
            i += workers
        row_s = time.perf_counter() - t0
    finally:
        op.close()
    return {
        "value": flops / att_s / 1e12, "unit": "TFLOP/s", "cores": workers, "kind": "oracle",
        "sample": (f"{done} tasks x 64 query rows of {ATTN['name']} (rows uniform over the "
                   f"sequence, heads in turn), fp64, {workers} spawn workers x 1 BLAS thread, "
                   f"{att_s:.1f} s wall"),
        "row_softmax": {"value": nbytes / row_s / 1e9, "unit": "GB/s",
                        "sample": f"{rdone} rows of {ROWS['name']}, {row_s:.1f} s wall"},
    }


# ------------------------------------------------------------------ reference arm
def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a bounded sample of
    the workload (one task of 32 attention query rows per worker, plus 2 rows of the
    row-state array per worker), timed with the wall clock."""
    if rank != 0:
        return None
    from online_softmax_07_gb300 import synth
    q, k, v = synth.workload_attention_inputs(ATTN["name"])
    x = synth.row_inputs(64, ROWS["length"], seed=2000)
    workers = os.cpu_count() or 1
    op = OraclePool({"q": q, "k": k, "v": v, "x": x}, workers)
    try:
        flops = secs = 0.0
        for s in range(args.warmup + args.steps):
            tasks = attention_sample_tasks(q.shape, 32, workers, seed=900 + s)
            t0 = time.perf_counter()
            res = op.pool.map(_oracle_attention_task, tasks)
            op.pool.map(_oracle_rows_task, [((2 * i) % 64, (2 * i) % 64 + 2)
                                            for i in range(workers)])
            dt = time.perf_counter() - t0
            if s >= args.warmup:
                flops += sum(r[0] for r in res)
                secs += dt
    finally:
        op.close()
    value = flops / secs / 1e12
    sample = (f"per step {workers} tasks x 32 query rows of {ATTN['name']} plus "
              f"{2 * workers} rows of {ROWS['name']}; fp64 oracle, {workers} spawn workers "
              f"x 1 BLAS thread")
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": workers, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ errors against the oracle
def attention_errors(q, k, v, o, lse, scale, causal, n_heads=4, n_rows=32, seed=7):
    """Max and mean abs error of O and max abs error of LSE against the fp64 oracle on
    the first and last row and `n_rows` seeded rows of `n_heads` heads spread over the
    batch (q, k, v: host arrays holding the values the kernel read; o, lse: device
    results)."""
    import torch

    import oracle
    B, H, N, d = q.shape
    all_heads = [(b, h) for b in range(B) for h in range(H)]
    step = max(1, len(all_heads) // n_heads)
    heads = all_heads[::step][:n_heads]
    errs, lerrs = [], []
    for i, (b, h) in enumerate(heads):
        g = np.random.Generator(np.random.PCG64(seed + i))
        rows = np.unique(np.concatenate([[0, N - 1], g.choice(N, min(n_rows, N), False)]))
        o_ref, lse_ref = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                                  v[b:b + 1, h:h + 1], scale, causal, rows=rows)
        idx = torch.from_numpy(rows).to(o.device)
        errs.append(np.abs(o[b, h].index_select(0, idx).float().cpu().numpy() - o_ref[0, 0]))
        lerrs.append(np.abs(lse[b, h].index_select(0, idx).cpu().numpy() - lse_ref[0, 0]))
    e = np.concatenate([x.ravel() for x in errs])
    le = np.concatenate([x.ravel() for x in lerrs])
    return {"o_max_abs_err": float(e.max()), "o_mean_abs_err": float(e.mean()),
            "lse_max_abs_err": float(le.max()), "rows_checked": int(le.size),
            "gates": {"o_max_abs": 2e-2, "o_mean_abs": 2e-3, "lse_max_abs": 1e-3}}


def extra_workload(name, peaks, stream, reps=20):
    """One more attention workload of the configuration list, measured like the bench
    workload (CUDA events around each of `reps` launches after 3 warm-ups): mean and
    median time, TFLOP/s, fraction of the measured bf16 peak, and oracle errors."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    w = synth.WORKLOADS[name]
    q, k, v = synth.workload_attention_inputs(name)
    B, H, N, d = q.shape
    dev = torch.device("cuda", torch.cuda.current_device())
    tq, tk, tv = (torch.from_numpy(t).to(dev, torch.bfloat16) for t in (q, k, v))
    o = torch.empty_like(tq)
    lse = torch.empty((B, H, N), device=dev)
    scale = 1.0 / math.sqrt(d)
    call = lambda: abi.fa_fwd(tq, tk, tv, o, lse, B, H, N, d, scale, int(w["causal"]), stream)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for e0, e1 in ev:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    if abi.fa_last_device_error() != abi.FA_OK:
        raise RuntimeError(f"device-side error in {name}")
    ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms_mean, ms_med = statistics.mean(ms), statistics.median(ms)
    flops = attn_flops(B, H, N, d, w["causal"])
    tf = flops / (ms_mean * 1e-3) / 1e12
    out = {"ms_mean": ms_mean, "ms_median": ms_med, "TFLOP/s": tf,
           "TFLOP/s_median": flops / (ms_med * 1e-3) / 1e12,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"]},
           "launches": reps}
    out.update(attention_errors(q, k, v, o, lse, scale, w["causal"], n_heads=2))
    del tq, tk, tv, o, lse
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ our arm
def our_arm(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from online_softmax_07_gb300 import abi, attention_forward, synth
    from online_softmax_07_gb300.build import build_library

    build_library()
    abi.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    B, H, N, d, causal = ATTN["B"], ATTN["H"], ATTN["N"], ATTN["d"], ATTN["causal"]
    scale = 1.0 / math.sqrt(d)
    q, k, v = synth.workload_attention_inputs(ATTN["name"])
    x = synth.workload_row_inputs()[0]
    dq, dk, dv = (torch.from_numpy(t).to(dev, torch.bfloat16) for t in (q, k, v))
    do = torch.empty_like(dq)
    dlse = torch.empty((B, H, N), device=dev)
    dx = torch.from_numpy(x).to(dev)
    rows, length = x.shape
    dm = torch.empty(rows, device=dev)
    dl = torch.empty(rows, device=dev)

    for _ in range(args.warmup):
        abi.fa_fwd(dq, dk, dv, do, dlse, B, H, N, d, scale, int(causal), stream)
        abi.online_softmax_rows(dx, dm, dl, rows, length, stream)
    torch.cuda.synchronize()
    if abi.fa_last_device_error() != abi.FA_OK:
        raise RuntimeError("device-side error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)   # let the sampler come up
    # Load window: the same steps, untimed, for at least --load-seconds right before the
    # timed ones, so that the clock record covers the kernels running.
    t_load0 = time.time()
    while time.time() - t_load0 < args.load_seconds:
        for _ in range(20):
            abi.fa_fwd(dq, dk, dv, do, dlse, B, H, N, d, scale, int(causal), stream)
            abi.online_softmax_rows(dx, dm, dl, rows, length, stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        abi.fa_fwd(dq, dk, dv, do, dlse, B, H, N, d, scale, int(causal), stream)
        ev[i][1].record(stream)
        abi.online_softmax_rows(dx, dm, dl, rows, length, stream)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    t_load1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.1)   # the samples of the last loaded moments arrive
    clocks = sampler.stop(window=(t_load0, t_load1 + 0.05))
    clocks["load_window_s"] = t_load1 - t_load0
    if abi.fa_last_device_error() != abi.FA_OK:
        raise RuntimeError("device-side error in the timed region")

    attn_list = [e[0].elapsed_time(e[1]) for e in ev]
    rows_list = [e[1].elapsed_time(e[2]) for e in ev]
    attn_ms, rows_ms = statistics.mean(attn_list), statistics.mean(rows_list)
    attn_med, rows_med = statistics.median(attn_list), statistics.median(rows_list)
    step_ms = t_start.elapsed_time(t_end) / args.steps
    attn_ms, rows_ms, step_ms, attn_med, rows_med = max_over_ranks(
        [attn_ms, rows_ms, step_ms, attn_med, rows_med], dev)
    errors = attention_errors(q, k, v, do, dlse, scale, causal) if rank == 0 else None

    flops = attn_flops(B, H, N, d, causal)
    rbytes = row_bytes(rows, length)
    value = flops * world / (attn_ms * 1e-3) / 1e12
    row_gbs = rbytes * world / (rows_ms * 1e-3) / 1e9
    peaks = load_peaks()
    per_gpu_tflops = flops / (attn_ms * 1e-3) / 1e12
    per_gpu_gbs = rbytes / (rows_ms * 1e-3) / 1e9

    # End to end through the public API with pinned host buffers.
    qh, kh, vh = (torch.from_numpy(t).to(torch.bfloat16).pin_memory() for t in (q, k, v))
    oh = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True)
    lh = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 30))
    for _ in range(3):
        attention_forward(qh, kh, vh, scale, causal, out=oh, lse_out=lh)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        attention_forward(qh, kh, vh, scale, causal, out=oh, lse_out=lh)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks([e2e_s], dev)[0]
    h2d = 3 * qh.numel() * 2
    d2h = oh.numel() * 2 + lh.numel() * 4

    out = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": run_config(world),
        "pct_of_peak": per_gpu_tflops / peaks["bf16_tflops"] * 100.0,
        "ms_attention": attn_ms,
        "ms_attention_median": attn_med,
        "ms_rows": rows_ms,
        "ms_rows_median": rows_med,
        "errors": errors,
        "row_softmax": {
            "value": row_gbs, "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": per_gpu_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": per_gpu_gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("row_state_block_kernel"),
                         "peak_source": peaks["source"]},
        },
        # `peak` is the burst figure.  The timed steps run back to back after a load
        # window, under the board's power cap (see `clocks`), so the fraction of the
        # sustained figure is given beside it.
        "roofline": {"bound": "tensor", "achieved": per_gpu_tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": per_gpu_tflops / peaks["bf16_tflops"],
                     "traffic": recorded_traffic("attn_fwd_tc_kernel"),
                     "peak_source": peaks["source"] + " bf16 burst",
                     "peak_sustained": peaks["bf16_tflops_sustained"] or None,
                     "frac_of_sustained": (per_gpu_tflops / peaks["bf16_tflops_sustained"]
                                           if peaks["bf16_tflops_sustained"] else None)},
        "clocks": clocks,
        "e2e": {"value": flops * world / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "online_softmax_07_gb300.attention_forward(pinned host tensors)"},
        "gpu_launches": 2 * args.steps,
    }
    if rank == 0 and not args.no_workloads:
        # The other attention configurations, each on this GPU alone (not part of the
        # step): B4 H16 N4096 d64 and the long sequence B1 H8 N32768 d128 causal, Q std 4.
        del qh, kh, vh, oh, lh
        out["workloads"] = {n: extra_workload(n, peaks, stream) for n in
                            ("attn_bf16_b4h16n4096d64", "attn_bf16_b1h8n32768d128_causal_qstd4")}
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(q, k, v, x, budget_s=args.cpu_seconds)
    return out


# ------------------------------------------------------------------ per-workload suite
def suite(args):
    """One JSON line per workload (not the bench contract line): the five configurations,
    fp16 inputs, split-KV against the plain kernel on a small-B*H long sequence, and the
    normalised row softmax.  CUDA events around `reps` back-to-back launches after 5
    warm-up launches; inputs larger than L2 except the tiny fp32 case."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    from online_softmax_07_gb300.build import build_library

    build_library()
    abi.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    def timed(fn, reps):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if abi.fa_last_device_error() != abi.FA_OK:
            raise RuntimeError("device-side error")
        return e0.elapsed_time(e1) / reps

    def attn_line(name, q, k, v, causal, dtype, splits=None, label=None):
        B, H, N, d = q.shape
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
        code = {"bf16": abi.FA_BF16, "f16": abi.FA_F16, "f32": abi.FA_F32}[dtype]
        dq, dk, dv = (torch.from_numpy(t).to(dev, tdt) for t in (q, k, v))
        o = torch.empty_like(dq)
        lse = torch.empty((B, H, N), device=dev)
        scale = 1.0 / math.sqrt(d)
        if splits is None:
            fn = lambda: abi.fa_fwd_dt(dq, dk, dv, o, lse, B, H, N, d, scale, int(causal), code,
                                       stream)
        else:
            nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits)
            ws = torch.empty(max(1, nbytes // 4), device=dev)
            fn = lambda: abi.fa_fwd_splitkv(dq, dk, dv, o, lse, B, H, N, d, scale, int(causal),
                                            splits, ws, nbytes, code, stream)
        ms = timed(fn, 20 if N * N * B * H > 1e9 else 200)
        tf = attn_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        line = {"workload": label or name, "dtype": dtype, "ms": ms, "TFLOP/s": tf,
                "pct_of_bf16_peak": 100 * tf / peaks["bf16_tflops"]}
        line.update(attn_errors(q, k, v, o, lse, scale, causal))
        if splits is not None:
            line["splits"] = splits
        print(json.dumps(line), flush=True)

    def attn_errors(q, k, v, o, lse, scale, causal):
        """Errors against the fp64 oracle: every row for small problems, else 32 seeded
        rows (plus the first and last) of each of up to 4 heads."""
        import oracle
        B, H, N, d = q.shape
        errs, lerrs = [], []
        heads = [(b, h) for b in range(B) for h in range(H)][:4]
        for (b, h) in heads:
            rows = np.arange(N) if N * N <= 1 << 24 else np.unique(np.concatenate(
                [[0, N - 1], np.random.Generator(np.random.PCG64(7 + h)).choice(N, 32, False)]))
            o_ref, lse_ref = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                                      v[b:b + 1, h:h + 1], scale, causal, rows=rows)
            idx = torch.from_numpy(rows).to(dev)
            errs.append(np.abs(o[b, h].index_select(0, idx).float().cpu().numpy() - o_ref[0, 0]))
            lerrs.append(np.abs(lse[b, h].index_select(0, idx).cpu().numpy() - lse_ref[0, 0]))
        e = np.concatenate([x.ravel() for x in errs])
        le = np.concatenate([x.ravel() for x in lerrs])
        return {"o_max_abs_err": float(e.max()), "o_mean_abs_err": float(e.mean()),
                "lse_max_abs_err": float(le.max()), "rows_checked": int(le.size)}

    def bwd_line(name, q, k, v, do, causal):
        """fa_bwd after fa_fwd; TFLOP/s counts the five algorithmic products
        (2.5 x the forward's FLOPs; the kernels execute those five at d = 64, one pass with
        the dQ partials, and seven at d = 128, where the dQ pass recomputes S and dP); errors
        against the oracle on 32 seeded query and key rows (plus the first and last) of
        the first and last head."""
        import oracle
        B, H, N, d = q.shape
        tq, tk, tv, tdo = (torch.from_numpy(t).to(dev, torch.bfloat16) for t in (q, k, v, do))
        o = torch.empty_like(tq)
        lse = torch.empty((B, H, N), device=dev)
        scale = 1.0 / math.sqrt(d)
        abi.fa_fwd_dt(tq, tk, tv, o, lse, B, H, N, d, scale, int(causal), abi.FA_BF16, stream)
        nbytes = abi.fa_bwd_workspace_bytes_dt(B, H, N, d, abi.FA_BF16)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        gq, gk, gv = torch.empty_like(tq), torch.empty_like(tq), torch.empty_like(tq)
        fn = lambda: abi.fa_bwd(tq, tk, tv, o, lse, tdo, gq, gk, gv, B, H, N, d, scale,
                                int(causal), ws, nbytes, abi.FA_BF16, stream)
        ms = timed(fn, 20)
        tf = 2.5 * attn_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        rows = np.unique(np.concatenate(
            [[0, N - 1], np.random.Generator(np.random.PCG64(11)).choice(N, 32, False)]))
        rel = {"dQ": [], "dK": [], "dV": []}
        for (b, h) in ((0, 0), (B - 1, H - 1)):
            ref = oracle.attention_backward_rows(q, k, v, do, scale, causal, (b, h), rows, rows)
            idx = torch.from_numpy(rows).to(dev)
            for key, t, r in zip(("dQ", "dK", "dV"), (gq, gk, gv), ref):
                got = t[b, h].index_select(0, idx).float().cpu().numpy()
                rel[key].append(float(np.linalg.norm(got - r) / np.linalg.norm(r)))
        line = {"workload": name.replace("attn_", "attn_bwd_"), "dtype": "bf16", "ms": ms,
                "TFLOP/s": tf, "pct_of_bf16_peak": 100 * tf / peaks["bf16_tflops"],
                "executed_TFLOP/s": tf * (5 if d == 64 else 7) / 5}
        line.update({f"{k}_rel_rms_err": max(v) for k, v in rel.items()})
        print(json.dumps(line), flush=True)

    for name in ("attn_f32_b1h1n128d64", "attn_bf16_b4h16n4096d64",
                 "attn_bf16_b2h16n8192d128_causal", "attn_bf16_b2h16n8191d128_causal",
                 "attn_bf16_b1h8n32768d128_causal_qstd4"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.workload_attention_inputs(name)
        attn_line(name, q, k, v, w["causal"], w["dtype"])
        if name == "attn_bf16_b2h16n8192d128_causal":
            qh, kh, vh = (synth.round_to_f16(t) for t in (q, k, v))
            attn_line(name, qh, kh, vh, True, "f16", label=name.replace("bf16", "f16"))
    # split-KV where the grid is small: B=1 H=1 N=32768 d=128 causal (128 query blocks)
    q, k, v = synth.attention_inputs(1, 1, 32768, 128, seed=96000)
    label = "attn_bf16_b1h1n32768d128_causal"
    attn_line(label, q, k, v, True, "bf16", label=label + " (no split)")
    s_def = abi.fa_fwd_splitkv_default_splits(1, 1, 32768, True)
    attn_line(label, q, k, v, True, "bf16", splits=s_def, label=label + " (split-KV)")
    # and where the grid is smaller still: B=1 H=1 N=16384 (64 query blocks)
    q, k, v = synth.attention_inputs(1, 1, 16384, 128, seed=96100)
    label = "attn_bf16_b1h1n16384d128_causal"
    attn_line(label, q, k, v, True, "bf16", label=label + " (no split)")
    s_def = abi.fa_fwd_splitkv_default_splits(1, 1, 16384, True)
    attn_line(label, q, k, v, True, "bf16", splits=s_def, label=label + " (split-KV)")
    # backward (fa_bwd) on the attention workloads with a seeded dO of the same shape
    for name in ("attn_bf16_b4h16n4096d64", "attn_bf16_b2h16n8192d128_causal",
                 "attn_bf16_b1h8n32768d128_causal_qstd4"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.workload_attention_inputs(name)
        B, H, N, d = q.shape
        do = synth.attention_inputs(B, H, N, d, seed=97000 + d)[0]
        bwd_line(name, q, k, v, do, w["causal"])
    # row state and normalised softmax on the 4096 x 32768 array
    x = torch.from_numpy(synth.workload_row_inputs()[0]).to(dev)
    rows, length = x.shape
    m = torch.empty(rows, device=dev)
    l = torch.empty(rows, device=dev)
    y = torch.empty_like(x)
    ms = timed(lambda: abi.online_softmax_rows(x, m, l, rows, length, stream), 100)
    gbs = row_bytes(rows, length) / (ms * 1e-3) / 1e9
    import oracle
    xs = x[:256].cpu().numpy()
    m_ref, l_ref = oracle.row_state(xs)
    l_rel = float(np.max(np.abs(l[:256].cpu().numpy() - l_ref) / l_ref))
    m_exact = bool(np.all(m[:256].cpu().numpy() == m_ref))
    print(json.dumps({"workload": "rows_4096x32768 state", "ms": ms, "GB/s": gbs,
                      "frac_of_hbm": gbs / peaks["hbm_gbs"], "l_max_rel_err_256_rows": l_rel,
                      "m_exact_256_rows": m_exact}), flush=True)
    ms = timed(lambda: abi.online_softmax_forward(x, y, m, l, rows, length, stream), 100)
    gbs = (2 * rows * length * 4 + rows * 8) / (ms * 1e-3) / 1e9
    print(json.dumps({"workload": "rows_4096x32768 softmax output", "ms": ms, "GB/s": gbs,
                      "frac_of_hbm": gbs / peaks["hbm_gbs"]}), flush=True)


def backward_run(args):
    """The backward alone: by default on the B=2 H=16 N=8192 d=128 causal workload with the
    suite's seeded dO, or on the shape --backward B,H,N,d,causal gives (bf16, Q, K, V, dO
    i.i.d. N(0,1) drawn on the device from fixed seeds): fa_fwd once for O and LSE, then
    --warmup and --steps fa_bwd calls (three launches each: at d = 128 a prep, the dK/dV
    pass and the dQ pass; at d = 64 a prep, the one-pass kernel and the dQ finalize) timed
    with CUDA events.  One JSON line; this is the command the backward's launch lists and ncu
    captures are taken with."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    from online_softmax_07_gb300.build import build_library

    shape = None
    if args.backward != "default":
        try:
            shape = tuple(int(x) for x in args.backward.split(","))
            if len(shape) != 5:
                raise ValueError
        except ValueError:
            raise SystemExit("--backward wants B,H,N,d,causal (five integers)")
    build_library()
    abi.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    if shape is None:
        name = "attn_bf16_b2h16n8192d128_causal"
        causal = int(synth.WORKLOADS[name]["causal"])
        q, k, v = synth.workload_attention_inputs(name)
        B, H, N, d = q.shape
        do = synth.attention_inputs(B, H, N, d, seed=97000 + d)[0]
        tq, tk, tv, tdo = (torch.from_numpy(t).to(dev, torch.bfloat16) for t in (q, k, v, do))
    else:
        B, H, N, d, causal = shape
        name = f"attn_bf16_b{B}h{H}n{N}d{d}" + ("_causal" if causal else "")
        tq, tk, tv, tdo = (synth.device_normal((B, H, N, d), seed=98000 + i, dtype=torch.bfloat16)
                           for i in range(4))
    o = torch.empty_like(tq)
    lse = torch.empty((B, H, N), device=dev)
    scale = 1.0 / math.sqrt(d)
    abi.fa_fwd_dt(tq, tk, tv, o, lse, B, H, N, d, scale, causal, abi.FA_BF16, stream)
    nbytes = abi.fa_bwd_workspace_bytes_dt(B, H, N, d, abi.FA_BF16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    gq, gk, gv = torch.empty_like(tq), torch.empty_like(tq), torch.empty_like(tq)

    def call():
        abi.fa_bwd(tq, tk, tv, o, lse, tdo, gq, gk, gv, B, H, N, d, scale, causal, ws, nbytes,
                   abi.FA_BF16, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    if abi.fa_last_device_error() != abi.FA_OK:
        raise RuntimeError("device-side error")
    ms = e0.elapsed_time(e1) / args.steps
    tf = 2.5 * attn_flops(B, H, N, d, bool(causal)) / (ms * 1e-3) / 1e12
    print(json.dumps({"workload": name.replace("attn_", "attn_bwd_"), "steps": args.steps,
                      "warmup": args.warmup, "ms": ms, "TFLOP/s": tf}), flush=True)


def forward_run(args):
    """The attention forward alone on one shape, --forward B,H,N,d,causal[,splits] (bf16;
    Q, K, V i.i.d. N(0,1) drawn on the device from fixed seeds): --warmup and --steps
    fa_fwd_dt calls (fa_fwd_splitkv with a workspace when splits > 1; splits 0 takes
    fa_fwd_splitkv_default_splits) timed with CUDA events.  One JSON line; this is the
    command that single-shape launch lists and ncu captures of the forward are taken with."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    from online_softmax_07_gb300.build import build_library

    try:
        vals = [int(x) for x in args.forward.split(",")]
        B, H, N, d, causal = vals[:5]
        splits = vals[5] if len(vals) == 6 else 1
        if len(vals) not in (5, 6) or splits < 0:
            raise ValueError
    except ValueError:
        raise SystemExit("--forward wants B,H,N,d,causal[,splits] (integers)")
    build_library()
    abi.load()
    stream = torch.cuda.current_stream()
    q, k, v = (synth.device_normal((B, H, N, d), seed=98000 + i, dtype=torch.bfloat16)
               for i in range(3))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device)
    scale = 1.0 / math.sqrt(d)
    if splits == 0:
        splits = abi.fa_fwd_splitkv_default_splits(B, H, N, causal)
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, N, d, splits) if splits > 1 else 0
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)

    def call():
        if splits > 1:
            abi.fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, splits, ws, nbytes,
                               abi.FA_BF16, stream)
        else:
            abi.fa_fwd_dt(q, k, v, o, lse, B, H, N, d, scale, causal, abi.FA_BF16, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    if abi.fa_last_device_error() != abi.FA_OK:
        raise RuntimeError("device-side error")
    ms = e0.elapsed_time(e1) / args.steps
    name = f"attn_bf16_b{B}h{H}n{N}d{d}" + ("_causal" if causal else "")
    print(json.dumps({"workload": name, "splits": splits, "steps": args.steps,
                      "warmup": args.warmup, "ms": ms,
                      "TFLOP/s": attn_flops(B, H, N, d, bool(causal)) / (ms * 1e-3) / 1e12}),
          flush=True)


def block_study(args):
    """The block-size study: each attention workload (B4 H16 N4096 d64; B2 H16 N8192 d128
    causal; B1 H8 N32768 d128 causal, Q std 4) through fa_fwd_block with 64-, 128- and (at
    d = 64) 192- and 256-key tiles: median and mean of 20 CUDA-event-timed launches after 3 warm-ups,
    TFLOP/s, and the O / LSE errors against the fp64 oracle on 34 seeded rows of four
    heads.  One JSON line per (workload, block)."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    from online_softmax_07_gb300.build import build_library

    build_library()
    abi.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    for name in ("attn_bf16_b4h16n4096d64", "attn_bf16_b2h16n8192d128_causal",
                 "attn_bf16_b1h8n32768d128_causal_qstd4"):
        w = synth.WORKLOADS[name]
        q, k, v = synth.workload_attention_inputs(name)
        B, H, N, d = q.shape
        tq, tk, tv = (torch.from_numpy(t).to(dev, torch.bfloat16) for t in (q, k, v))
        o = torch.empty_like(tq)
        lse = torch.empty((B, H, N), device=dev)
        scale = 1.0 / math.sqrt(d)
        for block_n in ((64, 128, 192, 256) if d == 64 else (64, 128)):
            call = lambda: abi.fa_fwd_block(tq, tk, tv, o, lse, B, H, N, d, scale,
                                            int(w["causal"]), abi.FA_BF16, block_n, stream)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(20)]
            for e0, e1 in ev:
                e0.record(stream)
                call()
                e1.record(stream)
            torch.cuda.synchronize()
            if abi.fa_last_device_error() != abi.FA_OK:
                raise RuntimeError("device-side error")
            ms = [e0.elapsed_time(e1) for e0, e1 in ev]
            med = statistics.median(ms)
            tf = attn_flops(B, H, N, d, w["causal"]) / (med * 1e-3) / 1e12
            line = {"workload": name, "block_n": block_n, "merges_per_row": -(-N // block_n),
                    "ms_median": med, "ms_mean": statistics.mean(ms), "TFLOP/s": tf,
                    "frac_of_bf16_peak": tf / peaks["bf16_tflops"]}
            line.update(attention_errors(q, k, v, o, lse, scale, w["causal"], n_heads=4))
            print(json.dumps(line), flush=True)
        del tq, tk, tv, o, lse
        torch.cuda.empty_cache()


def rows_run(args):
    """The row kernels alone on the 4096 x 32768 fp32 workload (N(0, 9) with the special
    rows): --rows state times online_softmax_rows, --rows softmax online_softmax_forward
    (the normalised output), --warmup and --steps calls with CUDA events.  One JSON line;
    this is the command the row kernels' ncu captures are taken with."""
    import torch

    from online_softmax_07_gb300 import abi, synth
    from online_softmax_07_gb300.build import build_library

    if args.rows not in ("state", "softmax"):
        raise SystemExit("--rows wants state or softmax")
    build_library()
    abi.load()
    stream = torch.cuda.current_stream()
    x = torch.from_numpy(synth.workload_row_inputs()[0]).cuda()
    rows, length = x.shape
    m = torch.empty(rows, device=x.device)
    l = torch.empty(rows, device=x.device)
    y = torch.empty_like(x) if args.rows == "softmax" else None

    def call():
        if y is None:
            abi.online_softmax_rows(x, m, l, rows, length, stream)
        else:
            abi.online_softmax_forward(x, y, m, l, rows, length, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # Algorithmic bytes: x read once (+ y written once for the softmax) and m, l.
    nbytes = rows * length * 4 * (2 if y is not None else 1) + rows * 8
    print(json.dumps({"workload": f"rows_{rows}x{length} {args.rows}", "steps": args.steps,
                      "warmup": args.warmup, "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9}),
          flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the extra attention configurations after the bench step")
    ap.add_argument("--load-seconds", type=float, default=1.0,
                    help="untimed steps run under the clock sampler before the timed ones")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--suite", action="store_true",
                    help="one line per workload instead of the bench line (1 GPU)")
    ap.add_argument("--backward", nargs="?", const="default", metavar="B,H,N,d,causal",
                    help="time fa_bwd alone, on B2 H16 N8192 d128 causal or the shape given "
                         "(1 GPU)")
    ap.add_argument("--forward", metavar="B,H,N,d,causal[,splits]",
                    help="time the bf16 forward alone on one shape, split-KV with splits > 1 "
                         "(0: the library's default count) (1 GPU)")
    ap.add_argument("--block-study", action="store_true",
                    help="time and check the forward with 64-, 128- and 256-key tiles on the "
                         "attention workloads (1 GPU)")
    ap.add_argument("--rows", metavar="state|softmax",
                    help="time a row kernel alone on the 4096 x 32768 workload (1 GPU)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local_rank = rank_env()
    if args.suite:
        suite(args)
        return
    if args.backward:
        backward_run(args)
        return
    if args.forward:
        forward_run(args)
        return
    if args.rows:
        rows_run(args)
        return
    if args.block_study:
        block_study(args)
        return
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    if args.impl == "reference":
        out = reference_arm(args, rank, world)
    else:
        out = our_arm(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
