"""Benchmark of the batched decode sampler (one JSON line on rank 0).

A step is one vt_sample call over one batch of synthetic logits: penalties,
temperature, min-p / top-k / top-p, the seeded Gumbel-max draw, log-probs and
top-n log-probs for every row.  The default workload is B=256 rows of
V=151,936 bf16 logits with mixed per-row strategies (25% greedy, 25% top-k
only, 25% top-p only, 25% top_k=50 + top_p=0.95 + min_p=0.05; T ~ U[0.3, 1.5];
20 top log-probs), the configuration the 70%-of-HBM-peak target is stated on.

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload b256|b32|b64|large|tiny]
                  [--impl reference]
For N > 1 launch with torchrun; each rank samples its own batch (weak scaling,
no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import glob
import json
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from device_token_sampling_gb300 import workloads as W  # noqa: E402

METRIC = "sampled rows/s, full sampling pipeline"
UNIT = "rows/s"
PEAK_FALLBACK_GBS = 6800.0
N_ROTATE = 4  # input buffers rotated between steps (b256: 4 x 77.8 MB > 129 MB L2)


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def make_workload(name: str, rank: int) -> W.Workload:
    if name == "b256":
        return W.b256(seed=3 + 1000 * rank)
    if name == "b32":
        return W.b32(seed=1 + 1000 * rank)
    if name == "b64":
        return W.b64(seed=2 + 1000 * rank)
    if name == "tiny":
        return W.tiny(seed=1000 * rank)
    if name == "large":  # the step logits are made on the device (large_step_device)
        return W.large(seed=4 + 1000 * rank, with_logits=False)
    raise ValueError(name)


def whole_job_rate(local_s: float, rows_per_rank: int, world: int, device) -> tuple:
    """The slowest rank's time (seconds) and the whole job's rows per second:
    every rank samples rows_per_rank rows in its own time; the job takes the
    longest of them."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_s], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    slowest = float(t.item())
    return slowest, rows_per_rank * world / slowest


def algorithmic_bytes_per_row(w: W.Workload) -> np.ndarray:
    """Bytes one row must move at minimum: its logits once, its distinct
    (id, count) history pairs, its parameters and seed (read + write), and its
    outputs (token, log-prob, status, kept boundary, top-n ids and log-probs)."""
    uniq = np.zeros(w.B, np.int64)
    for r in range(w.B):
        ids = np.concatenate([w.prompt_ids[w.prompt_offsets[r]:w.prompt_offsets[r + 1]],
                              w.output_ids[w.output_offsets[r]:w.output_offsets[r + 1]]])
        pen = (w.presence[r] != 0) or (w.frequency[r] != 0) or (w.repetition[r] != 1)
        uniq[r] = len(np.unique(ids)) if pen else 0
    params = 48 + 16
    outputs = 4 + 4 + 4 + 12 + 8 * w.num_logprobs
    return w.V * w.elem_size + 8 * uniq + params + outputs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return PEAK_FALLBACK_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "device_token_sampling_gb300", "csrc", "*"))):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes of one step (all its launches) from the committed ncu summary,
    if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"vt_sample_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_t = re.search(r"dram_bytes_per_step:\s*([0-9]+)", text)
    if not m_h or not m_t or m_h.group(1) != kernel_source_hash():
        return None
    return int(m_t.group(1))


class ClockSampler:
    """Samples the SM clock and clock-event reasons through NVML (read only)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.ok = False
        self.max_mhz = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value & ~0x1
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self):
        if self._t:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        names = [n for b, n in self.REASONS.items() if self.reasons & b]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples), "source": "nvml"}


# --------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of the workload
# --------------------------------------------------------------------------

def time_oracle_rows(w: W.Workload, rows: np.ndarray):
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.sample_workload(w, rows=rows)
    return time.perf_counter() - t0


def time_oracle_rows_threads(w: W.Workload, rows: np.ndarray, nthreads: int):
    """The same rows split over nthreads host threads (rows are independent; the
    oracle's C calls release the interpreter lock, so the threads run at once)."""
    import concurrent.futures as cf

    import oracle
    oracle.build()
    chunks = [c for c in np.array_split(rows, nthreads) if len(c)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        list(ex.map(lambda c: oracle.sample_workload(w, rows=c), chunks))
    return time.perf_counter() - t0


def cpu_baseline(w: W.Workload, budget_rows: int | None = None):
    rows = np.arange(w.B) if budget_rows is None else np.arange(min(w.B, budget_rows))
    dt = time_oracle_rows(w, rows)
    cores = os.cpu_count() or 1
    dt_all = time_oracle_rows_threads(w, rows, cores)
    return {"value": len(rows) / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(rows)} rows of one {w.name} step (every strategy class), "
                      f"single-threaded C++ oracle, {dt:.2f} s",
            "all_cores": {"value": len(rows) / dt_all, "unit": UNIT, "cores": cores,
                          "sample": f"the same rows split over {cores} host threads, "
                                    f"{dt_all:.2f} s"}}


# --------------------------------------------------------------------------
# reference arm
# --------------------------------------------------------------------------

def run_reference(args, w: W.Workload):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # a step of the reference arm is one row of the workload (the oracle is
    # timed as it stands, single-threaded); rows cycle through every class
    import oracle
    oracle.build()
    order = np.arange(w.B)
    if w.logits.shape[0] == 0:  # Large: its step logits are made on the device; here 64
        rows = 64              # host rows of the same distribution stand in
        w.logits = W.pad_rows(W.peaked_rows(np.random.default_rng(1000), rows, w.V), w.V,
                              w.dtype)
        order = np.arange(rows)
    for i in range(args.warmup):
        oracle.sample_workload(w, rows=[int(order[i % len(order)])])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.sample_workload(w, rows=[int(order[(args.warmup + i) % len(order)])])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"one {w.name} row per step, rows cycling through "
                                       "every strategy class, single thread"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w: W.Workload):
    return {"workload": w.name, "B": w.B, "V": w.V, "ld": w.ld,
            "logits_dtype": "f32" if w.dtype == W.DTYPE_F32 else "bf16",
            "num_logprobs": w.num_logprobs,
            "l2": f"{N_ROTATE} rotating input buffers"
                  f" ({N_ROTATE * w.logits_bytes() / 1e6:.0f} MB > 129 MB L2)",
            "parallelism": "row batches per GPU (replicas)"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def host_steps_rate(s, host, V, dt, n, update, stream, steps, rows, world, dev):
    """The end-to-end rate through the public host API, both ways: synchronous
    steps (vt_sample_host) and steps enqueued back to back (vt_sample_host_async,
    each copy-in overlapping the previous step's sampling, then one
    vt_sample_host_wait).  Returns (rate, api, other_rate)."""
    import torch.distributed as dist
    hos = [pinned_outputs(rows, n) for _ in range(2)]
    s.sample_host(host, V, dt, n, update, stream=stream, out=hos[0])
    rates = {}
    for mode in ("async", "sync"):
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        if mode == "async":
            for i in range(steps):
                s.sample_host_async(host, V, dt, n, update, stream=stream, out=hos[i % 2])
            s.sample_host_wait()
        else:
            for i in range(steps):
                s.sample_host(host, V, dt, n, update, stream=stream, out=hos[0])
        _, rates[mode] = whole_job_rate(time.perf_counter() - t0, rows * steps, world, dev)
    best = "async" if rates["async"] >= rates["sync"] else "sync"
    api = {"async": "vt_sample_host_async steps back to back, then vt_sample_host_wait",
           "sync": "vt_sample_host, one synchronous step at a time"}[best]
    return rates[best], api + " (pinned host logits in, pinned host outputs back)", \
        rates["sync" if best == "async" else "async"], hos[0]


def pinned_outputs(B: int, n: int):
    """Host output arrays of one step in pinned memory (asynchronous copies)."""
    import torch
    mk = lambda dt, *sh: torch.empty(*sh, dtype=dt, pin_memory=True).numpy()  # noqa: E731
    return (mk(torch.int32, B), mk(torch.float32, B), mk(torch.int32, B, n),
            mk(torch.float32, B, n))


def large_step_device(step: int, B: int, V: int, dev, rank: int = 0):
    """The Large workload's step logits, made on the device: N(0, 1.5) plus 8
    positions per row raised by U(8, 12), from seed 1000 + step (per rank)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + step + 1_000_000 * rank)
    x = torch.randn(B, V, device=dev, generator=g) * 1.5
    pos = torch.randint(0, V, (B, 8), device=dev, generator=g)
    add = torch.rand(B, 8, device=dev, generator=g) * 4.0 + 8.0
    x.scatter_add_(1, pos, add)
    return x


def run_gpu_decode(args, w: W.Workload):
    """Large: consecutive decode steps, each on its own logits made on the device
    outside the timed region; every step is timed with events on the launching
    stream and the counts grow by the drawn tokens."""
    import torch
    import torch.distributed as dist

    from device_token_sampling_gb300 import sampler as S

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    B, V, n = w.B, w.V, w.num_logprobs
    hist = int(np.max(np.diff(w.prompt_offsets) + np.diff(w.output_offsets)))
    s = S.Sampler(max_batch=B, max_vocab=V, max_logprobs=n,
                  max_history=hist + args.steps + args.warmup + 64, device=local, host_io=True)
    s.reset_workload(w)
    stream = torch.cuda.Stream(device=dev)
    out = (torch.empty(B, dtype=torch.int32, device=dev),
           torch.empty(B, dtype=torch.float32, device=dev),
           torch.empty((B, n), dtype=torch.int32, device=dev),
           torch.empty((B, n), dtype=torch.float32, device=dev))
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            x = large_step_device(10_000 + i, B, V, dev, rank)
            s.sample(x, V=V, num_logprobs=n, update_counts=True, out=out, stream=stream)
    stream.synchronize()
    s.check_device_errors()
    s.reset_workload(w)  # the timed decode starts from the workload's state
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        for t in range(args.steps):
            x = large_step_device(t, B, V, dev, rank)  # outside the timed region
            e0, e1 = evs[t]
            e0.record(stream)
            s.sample(x, V=V, num_logprobs=n, update_counts=True, out=out, stream=stream)
            e1.record(stream)
    stream.synchronize()
    clocks.stop()
    s.check_device_errors()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = sum(step_ms) / 1e3
    max_s, value = whole_job_rate(total_s, B * args.steps, world, dev)
    ms_per_step = max_s * 1e3 / args.steps
    launches = s.last_launches()
    handed = s.last_handover()
    # end to end: the step-0 logits from pinned host memory every step, the
    # steps enqueued back to back (each copy-in overlaps the previous step)
    host = large_step_device(0, B, V, dev, rank).cpu().pin_memory().numpy()
    e2e_steps = max(3, min(args.steps, 20))
    e2e_value, e2e_api, e2e_other, ho = host_steps_rate(s, host, V, W.DTYPE_F32, n, True, stream,
                                                        e2e_steps, B, world, dev)
    if rank == 0:
        peak, peak_kind = load_peaks()
        alg = int(algorithmic_bytes_per_row(w).sum())
        achieved = alg / (ms_per_step * 1e-3) / 1e9
        cfg = workload_config(w)
        cfg["l2"] = "one fresh 1.02 GB batch per step (> 129 MB L2), made on the device"
        cfg["decode_steps"] = args.steps
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                         "peak_source": f"{peak_kind} (hbm_gbs)",
                         "algorithmic_bytes_per_step": alg,
                         "kernel": "vt_sample step (sample_kernel + select_kernel)",
                         "kernel_ms": ms_per_step},
            "step_ms": {"median": float(np.median(step_ms)), "max": float(np.max(step_ms)),
                        "first": float(step_ms[0]), "last": float(step_ms[-1])},
            "rows_handed_to_select_kernel_last_step": handed,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(host.nbytes),
                    "d2h_bytes_per_step": int(sum(a.nbytes for a in ho)), "steps": e2e_steps,
                    "api": e2e_api, "other_mode_value": e2e_other},
            "gpu_launches": launches * args.steps,
            "clocks": clocks.summary(),
            "ns_per_row": 1e6 * ms_per_step / B,
        }
        if world == 1 and not args.no_cpu_baseline:
            hw = W.large(seed=4, with_logits=False)
            hw.logits = host  # the oracle times rows of a real step
            line["cpu_baseline"] = cpu_baseline(hw, budget_rows=args.cpu_rows or 256)
        print(json.dumps(line), flush=True)
    s.close()
    if world > 1:
        dist.destroy_process_group()


def run_gpu(args, w: W.Workload):
    import torch
    import torch.distributed as dist

    from device_token_sampling_gb300 import sampler as S

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    B, V, n = w.B, w.V, w.num_logprobs
    penalised = bool(((w.presence != 0) | (w.frequency != 0) | (w.repetition != 1)).any())
    hist = int(np.max(np.diff(w.prompt_offsets) + np.diff(w.output_offsets))) if B else 0
    max_hist = hist + args.steps + args.warmup + 512 if penalised else 0
    s = S.Sampler(max_batch=B, max_vocab=V, max_logprobs=n, max_history=max_hist, device=local,
                  host_io=True)
    s.set_path(args.path)
    s.reset_workload(w)
    update = penalised
    # device inputs: N_ROTATE distinct batches (inputs larger than L2)
    base = torch.from_numpy(np.ascontiguousarray(w.logits))
    if w.dtype == W.DTYPE_BF16:
        base = base.view(torch.int16)
    bufs = []
    gen = torch.Generator(device=dev)
    for i in range(N_ROTATE):
        x = base.to(dev)
        if i > 0:  # a different batch of the same distribution: permute rows
            gen.manual_seed(1000 * rank + i)
            x = x[torch.randperm(B, device=dev, generator=gen)].contiguous()
        bufs.append(x)
    dt = W.DTYPE_BF16 if w.dtype == W.DTYPE_BF16 else W.DTYPE_F32
    stream = torch.cuda.Stream(device=dev)
    outs = [(torch.empty(B, dtype=torch.int32, device=dev),
             torch.empty(B, dtype=torch.float32, device=dev),
             torch.empty((B, n), dtype=torch.int32, device=dev),
             torch.empty((B, n), dtype=torch.float32, device=dev)) for _ in range(N_ROTATE)]

    def step(i):
        s.sample(bufs[i % N_ROTATE], V=V, num_logprobs=n, update_counts=update,
                 out=outs[i % N_ROTATE], stream=stream, dtype=dt)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()
    s.check_device_errors()
    # capture N_ROTATE steps into one graph (launch overhead out of the timed region)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(N_ROTATE):
            step(i)
    for _ in range(2):
        graph.replay()
    stream.synchronize()
    reps, rem = divmod(args.steps, N_ROTATE)
    clocks = ClockSampler(local)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            graph.replay()
        for i in range(rem):
            step(i)
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    clocks.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    s.check_device_errors()
    handed = s.last_handover()
    launches_per_step = s.last_launches()

    # the two launches of a step timed apart: events on the launching stream
    # before the step, between its launches (recorded by the library) and after
    split = max(3, min(args.steps, 200))
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(split)]
    with torch.cuda.stream(stream):
        for trio in evs:  # create the events
            for e in trio:
                e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i, (ea, em, eb) in enumerate(evs):
            ea.record(stream)
            s.set_phase_event(em)
            step(i)
            eb.record(stream)
    s.set_phase_event(None)
    stream.synchronize()
    s.check_device_errors()
    k1_ms = float(np.mean([ea.elapsed_time(em) for ea, em, _ in evs]))
    k2_ms = float(np.mean([em.elapsed_time(eb) for _, em, eb in evs]))
    max_s, value = whole_job_rate(elapsed_ms / 1e3, B * args.steps, world, dev)
    max_ms = max_s * 1e3
    ms_per_step = max_ms / args.steps

    # end to end through the C ABI with host buffers: H2D of the step's logits
    # from pinned memory, sampling, D2H of the step's outputs, every step; the
    # steps are enqueued back to back (vt_sample_host_async: a step's copy-in
    # overlaps the previous step's sampling) and waited for at the end
    e2e_steps = max(3, min(args.steps, 200))
    host = torch.from_numpy(np.ascontiguousarray(w.logits)).pin_memory().numpy()
    e2e_value, e2e_api, e2e_other, ho = host_steps_rate(s, host, V, dt, n, update, stream,
                                                        e2e_steps, B, world, dev)
    h2d = int(host.nbytes)
    d2h = int(sum(a.nbytes for a in ho))

    if rank == 0:
        peak, peak_kind = load_peaks()
        per_row = algorithmic_bytes_per_row(w)
        alg = int(per_row.sum())
        # A step is one vt_sample: the streaming kernel over every row and the
        # selection kernel over the rows handed to it, on the caller's stream and
        # (bf16 batches with top-p-only rows) a second stream beside it.  The
        # launches overlap, so the roofline is taken over the whole step: the
        # step's algorithmic bytes over its device time.
        kernel = ("vt_sample step (sample_kernel + select_kernel)" if args.path == 1 else
                  "vt_sample step (the six flat kernels + select_kernel)")
        kernel_ms, kbytes = ms_per_step, alg
        traffic = profiled_traffic(w.name) if args.path == 1 else None
        achieved = kbytes / (kernel_ms * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict(workload_config(w),
                           sampling_path="streaming" if args.path == 1 else "flat"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} (hbm_gbs)",
                         "algorithmic_bytes_per_step": kbytes, "kernel": kernel,
                         "kernel_ms": kernel_ms},
            "launch_split_ms": {"to_end_of_main_sample_kernel": k1_ms,
                                "rest_of_step": k2_ms,
                                "rows_handed_to_select_kernel": handed},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "api": e2e_api,
                    "other_mode_value": e2e_other},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
            "ns_per_row": 1e6 * ms_per_step / B,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, budget_rows=args.cpu_rows)
        print(json.dumps(line), flush=True)
    s.close()
    if world > 1:
        dist.destroy_process_group()


SHARD_K = 256  # the records each shard keeps per row


def shard_bounded(w: W.Workload) -> W.Workload:
    """The workload with every sampled row bounded by a top-k of at most
    SHARD_K, the rows the vocabulary-split path takes: top-k rows keep
    min(k, SHARD_K); rows without top-k get top_k = SHARD_K."""
    import copy
    v = copy.copy(w)
    v.top_k = w.top_k.copy()
    greedy = (w.temperature == 0) | (w.top_k == 1) | (w.top_p == 0) | (w.min_p == 1)
    k = v.top_k
    k[~greedy & ((k <= 1) | (k > SHARD_K))] = SHARD_K
    v.name = f"{w.name} bounded to top_k <= {SHARD_K}"
    return v


def run_gpu_sharded(args, w: W.Workload):
    """The vocabulary split over args.shards devices, run one shard after
    another on one GPU: per step, vt_shard_partials over each shard's columns
    (the work one device of a tensor-parallel group does), then vt_shard_merge
    over the stacked records (what every device does after the all-gather)."""
    import torch

    from device_token_sampling_gb300 import sampler as S

    rank, world, local = dist_env()
    if world > 1:
        raise SystemExit("--shards runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    w = shard_bounded(w)
    B, V, n, Sh = w.B, w.V, w.num_logprobs, args.shards
    s = S.Sampler(max_batch=B, max_vocab=V, max_logprobs=n, max_history=0, device=local)
    s.reset_workload(w)
    base = torch.from_numpy(np.ascontiguousarray(w.logits))
    if w.dtype == W.DTYPE_BF16:
        base = base.view(torch.int16)
    bufs = [base.to(dev)]
    gen = torch.Generator(device=dev)
    for i in range(1, N_ROTATE):
        gen.manual_seed(1000 + i)
        bufs.append(bufs[0][torch.randperm(B, device=dev, generator=gen)].contiguous())
    edges = np.linspace(0, V, Sh + 1).astype(int)
    pb = int(s._lib.vt_shard_part_bytes(SHARD_K))
    parts = torch.empty((Sh, B, pb), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, mid=None):
        x = bufs[i % N_ROTATE]
        for sh in range(Sh):
            s.shard_partials(x[:, edges[sh]:edges[sh + 1]], int(edges[sh]), V, SHARD_K,
                             out=parts[sh], stream=stream)
        if mid is not None:
            mid.record(stream)
        return s.shard_merge(parts, V, SHARD_K, n, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()
    s.check_device_errors()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(N_ROTATE):
            step(i)
    graph.replay()
    stream.synchronize()
    reps = max(1, args.steps // N_ROTATE)
    clocks = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    clocks.stop()
    s.check_device_errors()
    steps = reps * N_ROTATE
    ms_per_step = ev0.elapsed_time(ev1) / steps
    # the partials and the merge timed apart (eager steps, events on the stream)
    split = []
    with torch.cuda.stream(stream):
        for i in range(20):
            a, m, b = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record(stream)
            step(i, mid=m)
            b.record(stream)
            split.append((a, m, b))
    stream.synchronize()
    part_ms = float(np.mean([a.elapsed_time(m) for a, m, _ in split[3:]]))
    merge_ms = float(np.mean([m.elapsed_time(b) for _, m, b in split[3:]]))
    # end to end: the step's logits from pinned host memory, the step, the
    # outputs back to pinned host memory, every step
    host = torch.from_numpy(np.ascontiguousarray(w.logits)).pin_memory()
    if w.dtype == W.DTYPE_BF16:
        host = host.view(torch.int16)
    stage = torch.empty_like(bufs[0])
    ho = pinned_outputs(B, n)
    e2e_steps = 50
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            stage.copy_(host, non_blocking=True)
            for sh in range(Sh):
                s.shard_partials(stage[:, edges[sh]:edges[sh + 1]], int(edges[sh]), V, SHARD_K,
                                 out=parts[sh], stream=stream)
            tok, lp, tid, tlp = s.shard_merge(parts, V, SHARD_K, n, stream=stream)
            for dst, src in zip(ho, (tok, lp, tid, tlp)):
                torch.from_numpy(dst).copy_(src, non_blocking=True)
    stream.synchronize()
    e2e_value = B * e2e_steps / (time.perf_counter() - t0)
    peak, peak_kind = load_peaks()
    alg = int(w.V * w.elem_size * B + 2 * Sh * B * pb + B * (16 + 8 * n))
    achieved = alg / (ms_per_step * 1e-3) / 1e9
    cfg = workload_config(w)
    cfg["workload"] = f"b256 (top_k <= {SHARD_K}) with the vocabulary split in {Sh} shards"
    cfg["shards"] = Sh
    cfg["parallelism"] = f"{Sh} vocabulary shards run one after another on one GPU"
    line = {
        "metric": METRIC, "value": B / (ms_per_step * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} (hbm_gbs)", "algorithmic_bytes_per_step": alg,
                     "kernel": "vt_shard_partials x shards + vt_shard_merge",
                     "kernel_ms": ms_per_step},
        "split_ms": {"partials_all_shards": part_ms, "merge": merge_ms},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(host.numel() * host.element_size()),
                "d2h_bytes_per_step": int(sum(a.nbytes for a in ho)), "steps": e2e_steps,
                "api": "pinned host logits copied in, vt_shard_partials per shard, vt_shard_merge, "
                       "outputs copied to pinned host memory, every step"},
        "gpu_launches": (Sh + 1) * steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    s.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000; Large: 100 decode steps)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="b256", choices=W.NAMES)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", type=int, default=1, choices=[1, 2],
                    help="1: the streaming kernel; 2: the flat kernels where they apply")
    ap.add_argument("--shards", type=int, default=0,
                    help="time the vocabulary-split variant with this many shards (one GPU)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 100 if args.workload == "large" else 2000
    rank, world, _ = dist_env()
    w = make_workload(args.workload, rank)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        from device_token_sampling_gb300 import _build
        _build.build()
        if args.shards > 0:
            run_gpu_sharded(args, w)
        elif args.workload == "large":
            run_gpu_decode(args, w)
        else:
            run_gpu(args, w)


if __name__ == "__main__":
    main()
