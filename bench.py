"""Benchmark: packed-THD attention forward on one GB300 (or N weak-scaled replicas).

Default workload: long-context context-parallel query chunks -- 2 documents of
65536 keys, a 4096-row query chunk per document at causal offset k_len - q_len
(bottom-right causal), h_q = h_kv = 16, d = 128, bf16, head-major LSE. One step
is one ``thd_attn_fwd`` over that batch: setup kernel, attention kernel and, on
the tensor-core path, the kernel that merges split key ranges.

Metric: TFLOP/s counted over unmasked score entries, 4 * d * N_visible (QK^T and
PV, multiply-add = 2), summed over sequences and query heads.

``--impl reference`` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed-THD attn fwd TFLOP/s (unmasked FLOPs) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD_DESC = {
    "cp_chunks": "long-context CP chunks: 2 docs x 65536 K rows (131072 K/V tokens), one 4096-row Q chunk "
                 "per doc at q_causal_offset = k_len - q_len (bottom-right causal), h_q=h_kv=16, d=128, "
                 "bf16, packed K/V, head-major LSE",
    "mixed_gqa": "mixed-policy GQA pack: 32 seqs lognormal lens (median 512) ~32k tokens, h_q=32 h_kv=8, "
                 "d=128, bf16, per-seq causal ~ Bernoulli(0.5), 0-8 pad rows, token-major LSE",
    "separate_padding": "separate Q/O vs K/V padding: 64 seqs lens U[0,4096], Q/O padded to 64, K/V 1-row gaps, "
                        "h=32, d=64, fp16, masks {none, TL, BR}, token-major LSE",
    "padded_causal": "padded THD causal: 8 seqs lens U[64,1024], 0-16 pad rows, h=16, d=128, bf16, head-major LSE",
}


def unmasked_entries(batch) -> int:
    """Visible (row, key) pairs summed over sequences and query heads."""
    lq, lk = batch.lens_q(), batch.lens_k()
    total = 0
    for b in range(batch.batch):
        mt = int(batch.mask_type[b])
        if mt == 0:
            total += int(lq[b]) * int(lk[b])
            continue
        shift = 0 if mt == 1 else (int(lk[b] - lq[b]) if batch.q_causal_offset is None
                                   else int(batch.q_causal_offset[b]))
        i = np.arange(int(lq[b]), dtype=np.int64)
        hi = np.clip(i + shift + 1, 0, int(lk[b]))
        w = -1 if batch.window_left is None else int(batch.window_left[b])
        lo = np.clip(i + shift - w, 0, int(lk[b])) if w >= 0 else 0
        total += int(np.maximum(hi - lo, 0).sum())
    return total * batch.h_q


def valid_bytes(batch) -> int:
    """Algorithmic HBM bytes: valid Q/K/V/O rows once, plus the LSE values."""
    e = batch.q.element_size()
    tq, tk = int(batch.lens_q().sum()), int(batch.lens_k().sum())
    return (2 * tq * batch.h_q * batch.d + 2 * tk * batch.h_kv * batch.d) * e + 4 * tq * batch.h_q


def recorded_traffic(workload: str):
    """DRAM bytes per attention-kernel launch from profiles/traffic.json, only while
    the kernel sources still hash to what was profiled (else None)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"fwd_tc_kernel/{workload}")
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    try:
        for rel in rec["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["sources_sha256"] else None


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed region
    runs: NVML read every 2 ms from a thread (read-only queries), else nvidia-smi
    every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None
        self.nvml = None
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self.stop_flag = threading.Event()
        self.t_begin = None

    def _nvml_open(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(dev)) != 0:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(dev, ctypes.c_int(1), ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if reasons is None:
            return None
        return lib, dev, reasons

    def _nvml_loop(self):
        import ctypes
        lib, dev, reasons = self.nvml
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            if lib.nvmlDeviceGetClockInfo(dev, ctypes.c_int(1), ctypes.byref(clk)) == 0 and \
                    reasons(dev, ctypes.byref(rs)) == 0:
                self.samples.append((time.perf_counter(), int(clk.value), int(rs.value)))
            time.sleep(0.002)

    def start(self):
        try:
            self.nvml = self._nvml_open()
        except Exception:       # no NVML here: fall back to nvidia-smi
            self.nvml = None
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def begin(self):
        """The timed region starts now: NVML samples before it are not counted."""
        self.t_begin = time.perf_counter()

    def stop(self) -> dict:
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            try:
                self.nvml[0].nvmlShutdown()
            except Exception:
                pass
            t0 = self.t_begin if self.t_begin is not None else 0.0
            kept = [(c, r) for t, c, r in self.samples if t >= t0]
            sm = [c for c, _ in kept]
            reasons = sorted({name for _, r in kept for bit, name in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(sm), "source": "nvml, 2 ms"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 100 ms"}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist, device):
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Seed of rank ``rank``'s batch: in a multi-GPU run every rank draws its own
    batch of the workload's shape (its shard of the job; the units are independent,
    so no data crosses ranks); rank 0 keeps the workload's own seed."""
    return base + 1000 * rank


def oracle_sample_time(batch, budget_s: float, max_rows: int | None = None):
    """Run the oracle on row slices of the workload until ``budget_s`` elapses.

    Returns (seconds, unmasked FLOPs computed, description)."""
    from oracle import attention_one_head, causal_shift, window_lower_shift
    q = batch.q
    scale = 1.0 / math.sqrt(batch.d) if batch.softmax_scale is None else batch.softmax_scale
    lq, lk = batch.lens_q(), batch.lens_k()
    group = batch.h_q // batch.h_kv
    rows_per_call = 64
    flops = 0
    done = []
    t0 = time.perf_counter()
    stop = False
    for b in range(batch.batch):
        if stop:
            break
        shift = causal_shift(int(batch.mask_type[b]), int(lq[b]), int(lk[b]),
                             None if batch.q_causal_offset is None else batch.q_causal_offset[b])
        lower = window_lower_shift(int(batch.mask_type[b]), shift,
                                   None if batch.window_left is None else batch.window_left[b])
        for r0 in range(0, int(lq[b]), rows_per_call):
            r1 = min(int(lq[b]), r0 + rows_per_call)
            for h in range(batch.h_q):
                g = h // group
                qb = q[batch.off_q[b]:batch.off_q[b] + lq[b], h].to(torch.float64).numpy()
                kb = batch.k[batch.off_k[b]:batch.off_k[b] + lk[b], g].to(torch.float64).numpy()
                vb = batch.v[batch.off_v[b]:batch.off_v[b] + lk[b], g].to(torch.float64).numpy()
                ts = time.perf_counter()
                attention_one_head(qb, kb, vb, scale, shift, rows=slice(r0, r1), lower=lower)
                t_step = time.perf_counter() - ts
                i = np.arange(r0, r1, dtype=np.int64)
                if shift is None:
                    n = (r1 - r0) * int(lk[b])
                else:
                    hi = np.clip(i + shift + 1, 0, int(lk[b]))
                    lo = 0 if lower is None else np.clip(i + lower, 0, int(lk[b]))
                    n = int(np.maximum(hi - lo, 0).sum())
                flops += 4 * batch.d * n
                done.append(t_step)
                if sum(done) >= budget_s or (max_rows is not None and len(done) * rows_per_call >= max_rows):
                    stop = True
                    break
            if stop:
                break
    secs = sum(done)
    desc = (f"{len(done)} (row-slice x head) oracle calls of {rows_per_call} query rows each, "
            f"starting at row 0 of sequence 0, float64 numpy; conversion of inputs excluded")
    return secs, flops, desc


def run_reference(args, batch):
    """CPU oracle timed on the host cores over a bounded sample per step (the
    forward, or with --bwd / --indexer the backward or indexer oracle)."""
    dist, rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return
    cores = os.cpu_count()
    per_step_budget = args.ref_step_seconds
    if args.indexer:
        sample = oracle_indexer_sample_time
    elif args.bwd:
        sample = oracle_bwd_sample_time
    else:
        sample = oracle_sample_time
    for _ in range(args.warmup):
        sample(batch, per_step_budget / 4)
    times, flops = [], []
    desc = ""
    for _ in range(args.steps):
        s, f, desc = sample(batch, per_step_budget)
        times.append(s)
        flops.append(f)
    total_s, total_f = sum(times), sum(flops)
    value = total_f / total_s / 1e12
    metric = IDX_METRIC if args.indexer else (BWD_METRIC if args.bwd else METRIC)
    config = ({"workload": IDX_DESC, "name": "indexer_cp", "pass": "indexer"} if args.indexer
              else {**config_block(args, batch), **({"pass": "backward"} if args.bwd else {})})
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}; budget {per_step_budget:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(args, batch):
    return {"workload": WORKLOAD_DESC.get(args.workload, args.workload), "name": args.workload,
            "batch": batch.batch, "h_q": batch.h_q, "h_kv": batch.h_kv, "d": batch.d,
            "tokens_q": int(batch.lens_q().sum()), "tokens_k": int(batch.lens_k().sum()),
            "unmasked_entries": unmasked_entries(batch),
            "window_left": None if batch.window_left is None else int(batch.window_left[0]),
            "l2": "inputs larger than L2 (K/V alone exceed 129 MB); no flush between steps"
            if valid_bytes(batch) > 129e6 else "inputs smaller than L2; L2 flushed between timed steps",
            "parallelism": (f"data-parallel x{args.gpus}, a batch per rank" if args.gpus > 1
                            else "single GPU")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="cp_chunks")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tcgen05"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kv-split", action="store_true", help="plan with THD_FLAG_NO_KV_SPLIT")
    ap.add_argument("--indexer", action="store_true",
                    help="time the indexer top-k (thd_indexer_topk) on the context-parallel indexer workload")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward pass (thd_attn_bwd) instead of the forward")
    ap.add_argument("--window-left", type=int, default=None,
                    help="left window (keys) on every causal sequence, through thd_attn_fwd_window")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from ragged_varlen_attention_gb300 import workloads as wl
    if args.indexer:
        if args.impl == "reference":
            run_reference(args, wl.indexer_cp())
        else:
            bench_indexer(args)
        return
    env_rank = int(os.environ.get("RANK", "0"))
    batch = wl.make(args.workload, seed=rank_seed(wl.WORKLOAD_SEEDS[args.workload], env_rank))
    if args.window_left is not None:
        import dataclasses
        batch = dataclasses.replace(batch, window_left=np.full(batch.batch, args.window_left, dtype=np.int32))
    if args.impl == "reference":
        run_reference(args, batch)
        return

    from ragged_varlen_attention_gb300 import binding as bd
    from ragged_varlen_attention_gb300 import build
    dist, rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(bd.library_path()):
        build.build()
    if dist is not None:
        dist.barrier()
    kernel = {"auto": bd.KERNEL_AUTO, "simt": bd.KERNEL_SIMT, "tcgen05": bd.KERNEL_TCGEN05}[args.kernel]
    if args.bwd:
        bench_backward(args, batch, bd, kernel, device, dist, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    # host (pinned) inputs and device copies
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt))
    host = {"q": batch.q.pin_memory(), "k": batch.k.pin_memory(), "v": batch.v.pin_memory(),
            "cu_q": ints(batch.cu_seqlens_q).pin_memory(), "cu_k": ints(batch.cu_seqlens_kv).pin_memory(),
            "offs": [ints(x).pin_memory() for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o,
                                                    batch.off_s)],
            "mask": ints(batch.mask_type, np.int8).pin_memory(),
            "qco": None if batch.q_causal_offset is None else ints(batch.q_causal_offset).pin_memory(),
            "win": None if batch.window_left is None else ints(batch.window_left).pin_memory()}
    dev = {k: (None if v is None else ([t.to(device) for t in v] if isinstance(v, list) else v.to(device)))
           for k, v in host.items()}
    o = torch.zeros((batch.cap_o, batch.h_q, batch.d), dtype=batch.torch_dtype, device=device)
    stats = torch.zeros((batch.stats_numel,), dtype=torch.float32, device=device)
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    stats_host = torch.empty(stats.shape, dtype=stats.dtype).pin_memory()
    plan = bd.plan_for_tensors(dev["q"], dev["k"], dev["v"], o, batch.batch, batch.cap_s,
                               batch.stats_layout, batch.softmax_scale, kernel,
                               bd.FLAG_NO_KV_SPLIT if args.no_kv_split else 0)
    ws = bd.alloc_workspace(plan, device)
    stream = torch.cuda.current_stream(device)
    small_inputs = valid_bytes(batch) <= 129e6
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device) if small_inputs else None

    def step():
        bd.thd_attn_fwd_window(plan, dev["q"], dev["k"], dev["v"], o, stats, dev["cu_q"], dev["cu_k"],
                               *dev["offs"], dev["mask"], dev["qco"], dev["win"], ws, stream)

    for _ in range(args.warmup):
        step()
    status = bd.thd_attn_read_status(plan, ws, stream)
    if status != 0:
        raise SystemExit(f"device status word {status:#x} on the benchmark workload")

    flop_per_step = 4 * batch.d * unmasked_entries(batch)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    sampler = ClockSampler(gpu_index)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bd.profile_enable(plan, args.steps)
    sampler.start()
    time.sleep(0.3)
    barrier(dist, device)
    sampler.begin()
    step_ms = []
    if flush is None:
        # one event between consecutive steps: the total and each step's duration
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        barrier(dist, device)
        total_ms = evs[0].elapsed_time(evs[-1])
        step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    else:
        # L2 flushed between steps; only the fwd calls are inside the timed events
        total_ms = 0.0
        for _ in range(args.steps):
            flush.fill_(1)
            ev0.record(stream)
            step()
            ev1.record(stream)
            ev1.synchronize()
            step_ms.append(ev0.elapsed_time(ev1))
            total_ms += step_ms[-1]
        barrier(dist, device)
    clocks = sampler.stop()
    kernel_ms, kernel_launches = bd.profile_read(plan)
    bd.profile_enable(plan, 0)
    ms_per_step = max_over_ranks(dist, total_ms / args.steps, device)
    flop_all = sum_over_ranks(dist, flop_per_step, device)      # every rank's own batch
    value = flop_all / (ms_per_step * 1e-3) / 1e12

    # the same step replayed from a CUDA graph (the call is capturable: no host
    # synchronisation, no allocation)
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            bd.thd_attn_fwd_window(plan, dev["q"], dev["k"], dev["v"], o, stats, dev["cu_q"], dev["cu_k"],
                                   *dev["offs"], dev["mask"], dev["qco"], dev["win"], ws, cap)
        cap.synchronize()
        with torch.cuda.graph(g, stream=cap):
            bd.thd_attn_fwd_window(plan, dev["q"], dev["k"], dev["v"], o, stats, dev["cu_q"], dev["cu_k"],
                                   *dev["offs"], dev["mask"], dev["qco"], dev["win"], ws, cap)
        torch.cuda.synchronize(device)
        g.replay()
        torch.cuda.synchronize(device)
        gs, ge = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if flush is None:
            gs.record(stream)
            for _ in range(args.steps):
                g.replay()
            ge.record(stream)
            ge.synchronize()
            graph_ms = gs.elapsed_time(ge) / args.steps
        else:
            # as in the timed loop: L2 flushed before each replay, outside the events
            acc = 0.0
            for _ in range(args.steps):
                flush.fill_(1)
                gs.record(stream)
                g.replay()
                ge.record(stream)
                ge.synchronize()
                acc += gs.elapsed_time(ge)
            graph_ms = acc / args.steps
    except RuntimeError as exc:          # capture unsupported here: report why, keep the line
        graph_ms = f"unavailable: {exc}".splitlines()[0][:200]

    # end-to-end through the public API: pinned host inputs -> device -> fwd -> host outputs
    h2d = sum(t.numel() * t.element_size() for t in (host["q"], host["k"], host["v"], host["cu_q"],
                                                      host["cu_k"], host["mask"], *host["offs"]))
    for name in ("qco", "win"):
        if host[name] is not None:
            h2d += host[name].numel() * host[name].element_size()
    d2h = o_host.numel() * o_host.element_size() + stats_host.numel() * 4

    # end to end, pipelined the way a serving loop runs: two sets of device inputs and
    # outputs; while step i computes, step i+1's inputs are copied in on one stream and
    # step i-1's outputs copied out on another. Every step's copies are inside the timed
    # region, which runs from before the first input copy to after the last output copy.
    sets = [dict(dev=dev, o=o, stats=stats)]
    sets.append(dict(dev={k_: (None if v_ is None else ([t.clone() for t in v_] if isinstance(v_, list) else v_.clone()))
                          for k_, v_ in dev.items()},
                     o=torch.empty_like(o), stats=torch.empty_like(stats)))
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def copy_in(b):
        d = sets[b]["dev"]
        with torch.cuda.stream(h2d_s):
            for name in ("q", "k", "v", "cu_q", "cu_k", "mask", "qco", "win"):
                if host[name] is not None:
                    d[name].copy_(host[name], non_blocking=True)
            for dt, ht in zip(d["offs"], host["offs"]):
                dt.copy_(ht, non_blocking=True)

    def compute(b):
        d, ob, sb = sets[b]["dev"], sets[b]["o"], sets[b]["stats"]
        bd.thd_attn_fwd_window(plan, d["q"], d["k"], d["v"], ob, sb, d["cu_q"], d["cu_k"], *d["offs"], d["mask"],
                               d["qco"], d["win"], ws, stream)

    def copy_out(b):
        with torch.cuda.stream(d2h_s):
            o_host.copy_(sets[b]["o"], non_blocking=True)
            stats_host.copy_(sets[b]["stats"], non_blocking=True)

    def e2e_run(n_steps):
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [], [], []
        copy_in(0)
        in_done.append(ev()); in_done[0].record(h2d_s)
        for i in range(n_steps):
            b = i % 2
            stream.wait_event(in_done[i])
            if i >= 2:
                stream.wait_event(out_done[i - 2])      # outputs of this set copied out
            compute(b)
            comp_done.append(ev()); comp_done[i].record(stream)
            if i + 1 < n_steps:
                if i >= 1:
                    h2d_s.wait_event(comp_done[i - 1])  # the other set's inputs are free
                copy_in(1 - b)
                in_done.append(ev()); in_done[i + 1].record(h2d_s)
            d2h_s.wait_event(comp_done[i])
            copy_out(b)
            out_done.append(ev()); out_done[i].record(d2h_s)
        stream.wait_event(out_done[-1])

    e2e_run(2)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    ev0.record(stream)
    h2d_s.wait_stream(stream)
    e2e_run(args.e2e_steps)
    ev1.record(stream)
    barrier(dist, device)
    e2e_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / args.e2e_steps, device)
    e2e_value = flop_all / (e2e_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    kernel_tflops = flop_per_step / (kernel_ms * 1e-3) / 1e12 if kernel_ms > 0 else None
    # below the ridge (peak FLOP/s over HBM bytes/s) a launch is bound by HBM: report GB/s
    bytes_per_step = valid_bytes(batch)
    ridge = peak * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    hbm_bound = flop_per_step / max(bytes_per_step, 1) < ridge
    src = (f"of {peak_src} MEASURED_PEAKS.json" if peak_src == "measured" else "fallback")
    if hbm_bound:
        achieved = bytes_per_step / (kernel_ms * 1e-3) / 1e9 if kernel_ms > 0 else None
        roof = {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": None if achieved is None else achieved / float(peaks["hbm_gbs"]),
                "peak_source": f"hbm_gbs {src}", "bytes_per_launch": bytes_per_step,
                "arithmetic_intensity": flop_per_step / max(bytes_per_step, 1), "ridge": ridge}
    else:
        roof = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": None if kernel_tflops is None else kernel_tflops / peak,
                "peak_source": f"bf16_tflops (burst) {src}" if peak_src == "measured" else "fallback 1.9 PFLOP/s",
                "arithmetic_intensity": flop_per_step / max(bytes_per_step, 1), "ridge": ridge}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if batch.dtype == "bf16" else batch.dtype, "data": "synthetic",
        "config": {**config_block(args, batch),
                   "kernel": "tcgen05" if plan.kernel == bd.KERNEL_TCGEN05 else "simt",
                   "kv_split_allowed": plan.kernel == bd.KERNEL_TCGEN05 and not args.no_kv_split,
                   "flop_per_step": flop_per_step},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "roofline": {**roof,
                     "kernel": "attention kernel alone (CUDA events on its stream)",
                     "kernel_ms": kernel_ms, "launches": kernel_launches,
                     "traffic": recorded_traffic(args.workload) if plan.kernel == bd.KERNEL_TCGEN05
                     and args.window_left is None else None,
                     "traffic_unit": "bytes per launch (ncu dram read+write)"},
        "step_ms_median": statistics.median(step_ms) if step_ms else None,
        "graph_replay_ms_per_step": graph_ms,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "steps": args.e2e_steps,
                "pipeline": "step i+1's inputs copied in and step i-1's outputs copied out on two "
                            "streams while step i computes (two device buffer sets)"},
        "gpu_launches": (3 if plan.kernel == bd.KERNEL_TCGEN05 and not args.no_kv_split else 2) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, flops, desc = oracle_sample_time(batch, args.cpu_baseline_seconds)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc + f"; {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


BWD_METRIC = "packed-THD attn bwd TFLOP/s (10 * d * unmasked entries: QK^T, dO V^T, P^T dO, dS^T Q, dS K)"


def oracle_bwd_sample_time(batch, budget_s: float):
    """Backward oracle on growing prefixes of sequence 0, head 0 (a crop of the
    workload: rows [0, R) with the keys they see) until ``budget_s`` elapses.
    Returns (seconds, algorithmic FLOPs, description)."""
    from oracle import attention_one_head_bwd, causal_shift, window_lower_shift
    lq, lk = batch.lens_q(), batch.lens_k()
    scale = 1.0 / math.sqrt(batch.d) if batch.softmax_scale is None else batch.softmax_scale
    shift = causal_shift(int(batch.mask_type[0]), int(lq[0]), int(lk[0]),
                         None if batch.q_causal_offset is None else batch.q_causal_offset[0])
    lower = window_lower_shift(int(batch.mask_type[0]), shift,
                               None if batch.window_left is None else batch.window_left[0])
    rng = np.random.default_rng(0)
    cap = min(int(lq[0]), 512)            # bounds the [rows, keys] float64 temporaries
    secs, flops, calls, rows = 0.0, 0, 0, min(64, cap)
    while secs < budget_s and rows > 0:
        r = rows
        kmax = int(lk[0]) if shift is None else max(0, min(int(lk[0]), r - 1 + shift + 1))
        qb = batch.q[batch.off_q[0]:batch.off_q[0] + r, 0].to(torch.float64).numpy()
        kb = batch.k[batch.off_k[0]:batch.off_k[0] + kmax, 0].to(torch.float64).numpy()
        vb = batch.v[batch.off_v[0]:batch.off_v[0] + kmax, 0].to(torch.float64).numpy()
        gb = rng.standard_normal((r, batch.d))
        t0 = time.perf_counter()
        attention_one_head_bwd(qb, kb, vb, gb, scale, shift, lower)
        secs += time.perf_counter() - t0
        i = np.arange(r, dtype=np.int64)
        if shift is None:
            n = r * kmax
        else:
            hi = np.clip(i + shift + 1, 0, kmax)
            lo = 0 if lower is None else np.clip(i + lower, 0, kmax)
            n = int(np.maximum(hi - lo, 0).sum())
        flops += 10 * batch.d * n
        calls += 1
        rows = min(2 * rows, cap)
    desc = (f"{calls} oracle backward calls on the first R rows of sequence 0, head 0 (R doubling from 64 "
            f"to {cap}, then repeated) with the keys they see, float64 numpy")
    return secs, flops, desc


def bench_backward(args, batch, bd, kernel, device, dist, rank, world):
    """Backward timing: O and Stats come from this library's forward on the same
    inputs, dO is seeded N(0, 1); each step is one thd_attn_bwd."""
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt))
    g = torch.Generator().manual_seed(1234)
    d_o_host = torch.randn((batch.cap_o, batch.h_q, batch.d), generator=g).to(batch.torch_dtype)
    host = {"q": batch.q.pin_memory(), "k": batch.k.pin_memory(), "v": batch.v.pin_memory(),
            "d_o": d_o_host.pin_memory(),
            "cu_q": ints(batch.cu_seqlens_q).pin_memory(), "cu_k": ints(batch.cu_seqlens_kv).pin_memory(),
            "offs": [ints(x).pin_memory() for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o,
                                                    batch.off_s)],
            "mask": ints(batch.mask_type, np.int8).pin_memory(),
            "qco": None if batch.q_causal_offset is None else ints(batch.q_causal_offset).pin_memory(),
            "win": None if batch.window_left is None else ints(batch.window_left).pin_memory()}
    dev = {k: (None if v is None else ([t.to(device) for t in v] if isinstance(v, list) else v.to(device)))
           for k, v in host.items()}
    o = torch.zeros((batch.cap_o, batch.h_q, batch.d), dtype=batch.torch_dtype, device=device)
    stats = torch.zeros((batch.stats_numel,), dtype=torch.float32, device=device)
    fplan = bd.plan_for_tensors(dev["q"], dev["k"], dev["v"], o, batch.batch, batch.cap_s, batch.stats_layout,
                                batch.softmax_scale, kernel, 0)
    fws = bd.alloc_workspace(fplan, device)
    stream = torch.cuda.current_stream(device)
    bd.thd_attn_fwd_window(fplan, dev["q"], dev["k"], dev["v"], o, stats, dev["cu_q"], dev["cu_k"], *dev["offs"],
                           dev["mask"], dev["qco"], dev["win"], fws, stream)
    if bd.thd_attn_read_status(fplan, fws, stream) != 0:
        raise SystemExit("device status word set by the forward on the benchmark workload")
    o_host = o.cpu().pin_memory()
    stats_host = stats.cpu().pin_memory()
    dq, dk, dv = (torch.zeros_like(dev[n]) for n in ("q", "k", "v"))
    dq_host, dk_host, dv_host = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
    plan = bd.plan_bwd_for_tensors(dev["q"], dev["k"], dev["v"], o, dev["d_o"], dq, dk, dv, batch.batch,
                                   batch.cap_s, batch.stats_layout, batch.softmax_scale, kernel, 0)
    ws = bd.alloc_workspace(plan, device)
    small_inputs = valid_bytes(batch) * 2 <= 129e6
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device) if small_inputs else None

    def step():
        bd.thd_attn_bwd(plan, dev["q"], dev["k"], dev["v"], o, dev["d_o"], stats, dq, dk, dv, dev["cu_q"],
                        dev["cu_k"], *dev["offs"], dev["mask"], dev["qco"], dev["win"], ws, stream)

    for _ in range(args.warmup):
        step()
    if bd.thd_attn_read_status(plan, ws, stream) != 0:
        raise SystemExit("device status word set by the backward on the benchmark workload")
    flop_per_step = 10 * batch.d * unmasked_entries(batch)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else 0
    sampler = ClockSampler(gpu_index)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bd.profile_enable(plan, args.steps)
    sampler.start()
    time.sleep(0.3)
    barrier(dist, device)
    sampler.begin()
    total_ms = 0.0
    if flush is None:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier(dist, device)
        total_ms = ev0.elapsed_time(ev1)
    else:
        for _ in range(args.steps):
            flush.fill_(1)
            ev0.record(stream)
            step()
            ev1.record(stream)
            ev1.synchronize()
            total_ms += ev0.elapsed_time(ev1)
        barrier(dist, device)
    clocks = sampler.stop()
    kernel_ms, kernel_launches = bd.profile_read(plan)
    bd.profile_enable(plan, 0)
    ms_per_step = max_over_ranks(dist, total_ms / args.steps, device)
    flop_all = sum_over_ranks(dist, flop_per_step, device)      # every rank's own batch
    value = flop_all / (ms_per_step * 1e-3) / 1e12

    h2d_t = [host[n] for n in ("q", "k", "v", "d_o", "cu_q", "cu_k", "mask")] + host["offs"] + [o_host, stats_host]
    h2d_t += [host[n] for n in ("qco", "win") if host[n] is not None]
    h2d = sum(t.numel() * t.element_size() for t in h2d_t)
    d2h = sum(t.numel() * t.element_size() for t in (dq_host, dk_host, dv_host))

    def e2e_step():
        for name in ("q", "k", "v", "d_o", "cu_q", "cu_k", "mask", "qco", "win"):
            if host[name] is not None:
                dev[name].copy_(host[name], non_blocking=True)
        for dt, ht in zip(dev["offs"], host["offs"]):
            dt.copy_(ht, non_blocking=True)
        o.copy_(o_host, non_blocking=True)
        stats.copy_(stats_host, non_blocking=True)
        step()
        for dt, ht in ((dq, dq_host), (dk, dk_host), (dv, dv_host)):
            ht.copy_(dt, non_blocking=True)

    e2e_step()
    barrier(dist, device)
    ev0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    ev1.record(stream)
    barrier(dist, device)
    e2e_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / args.e2e_steps, device)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    kernel_tflops = flop_per_step / (kernel_ms * 1e-3) / 1e12 if kernel_ms > 0 else None
    tc = plan.kernel == bd.KERNEL_TCGEN05
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": batch.dtype, "data": "synthetic",
        "config": {**config_block(args, batch), "pass": "backward",
                   "kernel": "tcgen05" if tc else "simt", "flop_per_step": flop_per_step,
                   "hardware_flop_per_step": (14 if tc else 10) * batch.d * unmasked_entries(batch)},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": None if kernel_tflops is None else kernel_tflops / peak,
                     "peak_source": f"bf16_tflops (burst) of {peak_src} MEASURED_PEAKS.json"
                     if peak_src == "measured" else "fallback 1.9 PFLOP/s",
                     "kernel": "dQ kernel + dK/dV kernel (CUDA events on their stream around both)",
                     "kernel_ms": kernel_ms, "launches": kernel_launches, "traffic": None},
        "e2e": {"value": flop_all / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "steps": args.e2e_steps},
        "gpu_launches": 5 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, flops, desc = oracle_bwd_sample_time(batch, args.cpu_baseline_seconds)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc + f"; {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


IDX_METRIC = "packed-THD indexer top-k TFLOP/s (2 * H * d per visible (row, key) pair)"
IDX_DESC = ("context-parallel indexer chunks: 2 docs x 65536 keys, a 4096-row query chunk per doc at "
            "q_causal_offset = k_len - q_len (bottom-right causal), H=64 indexer heads, d=128, bf16, "
            "W ~ N(0,1)/sqrt(H) float32, top-2048 per row")


def indexer_visible_pairs(b) -> int:
    lq, lk = b.lens_q(), b.lens_k()
    total = 0
    for s_ in range(b.batch):
        mt = int(b.mask_type[s_])
        if mt == 0:
            total += int(lq[s_]) * int(lk[s_])
            continue
        c = 0 if mt == 1 else (int(lk[s_] - lq[s_]) if b.q_causal_offset is None else int(b.q_causal_offset[s_]))
        i = np.arange(int(lq[s_]), dtype=np.int64)
        total += int(np.clip(i + c + 1, 0, int(lk[s_])).sum())
    return total


def oracle_indexer_sample_time(b, budget_s: float):
    """Indexer oracle on rows of document 0 (growing prefixes of the chunk, each row
    against its visible keys) until ``budget_s`` elapses."""
    from oracle import indexer_scores_one, select_topk
    q64 = b.q[:int(b.lens_q()[0])].to(torch.float64).numpy()
    k64 = b.k[:int(b.lens_k()[0])].to(torch.float64).numpy()
    w64 = b.w[:int(b.lens_q()[0])].to(torch.float64).numpy()
    c = int(b.q_causal_offset[0])
    secs, flops, rows_done, r0 = 0.0, 0, 0, 0
    while secs < budget_s and r0 < q64.shape[0]:
        r1 = min(q64.shape[0], r0 + 2)
        kmax = min(k64.shape[0], r1 - 1 + c + 1)
        t0 = time.perf_counter()
        sc = indexer_scores_one(q64[r0:r1], k64[:kmax], w64[r0:r1])
        vis = np.arange(kmax)[None, :] <= (np.arange(r0, r1)[:, None] + c)
        select_topk(sc, vis, b.topk)
        secs += time.perf_counter() - t0
        flops += 2 * b.heads * b.d * int(vis.sum())
        rows_done += r1 - r0
        r0 = r1
    return secs, flops, f"{rows_done} query rows of document 0 (2 rows per oracle call, each against its visible keys), float64 numpy"


def bench_indexer(args):
    from ragged_varlen_attention_gb300 import binding as bd
    from ragged_varlen_attention_gb300 import build
    from ragged_varlen_attention_gb300 import workloads as wl
    dist, rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or not os.path.exists(bd.library_path()):
        build.build()
    if dist is not None:
        dist.barrier()
    kernel = {"auto": bd.KERNEL_AUTO, "simt": bd.KERNEL_SIMT, "tcgen05": bd.KERNEL_TCGEN05}[args.kernel]
    b = wl.indexer_cp(seed=rank_seed(wl.INDEXER_CP_SEED, rank))
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt))
    host = {"q": b.q.pin_memory(), "k": b.k.pin_memory(), "w": b.w.pin_memory(),
            "cu_q": ints(b.cu_seqlens_q).pin_memory(), "cu_k": ints(b.cu_seqlens_kv).pin_memory(),
            "off_q": ints(b.off_q).pin_memory(), "off_k": ints(b.off_k).pin_memory(),
            "off_o": ints(b.off_out).pin_memory(), "mask": ints(b.mask_type, np.int8).pin_memory(),
            "qco": ints(b.q_causal_offset).pin_memory()}
    dev = {n: t.to(device) for n, t in host.items()}
    idx = torch.empty((b.cap_out, b.topk), dtype=torch.int32, device=device)
    sc = torch.empty((b.cap_out, b.topk), dtype=torch.float32, device=device)
    idx_host = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
    sc_host = torch.empty(sc.shape, dtype=sc.dtype).pin_memory()
    plan = bd.indexer_plan_for_tensors(dev["q"], dev["k"], dev["w"], idx, b.batch, b.topk,
                                       int(b.lens_k().max()), kernel)
    ws = bd.alloc_workspace(plan, device)
    stream = torch.cuda.current_stream(device)

    def step():
        bd.thd_indexer_topk(plan, dev["q"], dev["k"], dev["w"], idx, sc, dev["cu_q"], dev["cu_k"], dev["off_q"],
                            dev["off_k"], dev["off_o"], dev["mask"], dev["qco"], ws, stream)

    for _ in range(args.warmup):
        step()
    if bd.thd_attn_read_status(plan, ws, stream) != 0:
        raise SystemExit("device status word set on the indexer workload")
    pairs = indexer_visible_pairs(b)
    flop_per_step = 2 * b.heads * b.d * pairs
    sampler = ClockSampler(0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bd.profile_enable(plan, args.steps)
    sampler.start()
    time.sleep(0.3)
    barrier(dist, device)
    sampler.begin()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier(dist, device)
    total_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop()
    kernel_ms, launches = bd.profile_read(plan)
    bd.profile_enable(plan, 0)
    ms_per_step = max_over_ranks(dist, total_ms / args.steps, device)
    flop_all = sum_over_ranks(dist, flop_per_step, device)      # every rank's own batch
    value = flop_all / (ms_per_step * 1e-3) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = idx_host.numel() * 4 + sc_host.numel() * 4

    def e2e_step():
        for n in host:
            dev[n].copy_(host[n], non_blocking=True)
        step()
        idx_host.copy_(idx, non_blocking=True)
        sc_host.copy_(sc, non_blocking=True)

    e2e_step()
    barrier(dist, device)
    ev0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    ev1.record(stream)
    barrier(dist, device)
    e2e_ms = max_over_ranks(dist, ev0.elapsed_time(ev1) / args.e2e_steps, device)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    kt = flop_per_step / (kernel_ms * 1e-3) / 1e12 if kernel_ms > 0 else None
    tc = plan.kernel == bd.KERNEL_TCGEN05
    line = {
        "metric": IDX_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": b.dtype, "data": "synthetic",
        "config": {"workload": IDX_DESC, "name": "indexer_cp", "heads": b.heads, "d": b.d, "topk": b.topk,
                   "visible_pairs": pairs, "flop_per_step": flop_per_step, "pass": "indexer",
                   "kernel": "tcgen05" if tc else "simt",
                   "l2": "inputs smaller than L2 but the float32 score scratch (2 GB) is not; no flush",
                   "parallelism": (f"data-parallel x{args.gpus}, a batch per rank" if args.gpus > 1
                                   else "single GPU")},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": kt, "peak": peak, "unit": "TFLOP/s",
                     "frac": None if kt is None else kt / peak,
                     "peak_source": f"bf16_tflops (burst) of {peak_src} MEASURED_PEAKS.json"
                     if peak_src == "measured" else "fallback 1.9 PFLOP/s",
                     "kernel": "indexer score kernel (CUDA events on its stream)",
                     "kernel_ms": kernel_ms, "launches": launches, "traffic": None},
        "e2e": {"value": flop_all / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "steps": args.e2e_steps},
        "gpu_launches": (4 if tc else 3) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, flops, desc = oracle_indexer_sample_time(b, args.cpu_baseline_seconds)
        line["cpu_baseline"] = {"value": flops / secs / 1e12, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc + f"; {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
