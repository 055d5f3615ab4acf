"""Timeline of the forward tensor-core kernel's hand-offs on cuda:0.

``python -m ragged_varlen_attention_gb300.profiling.fwd_timeline [workload]`` builds a copy of
the library with the kernel's clock64() stamps compiled in (-DTHD_FWD_TRACE, under
_build/trace), runs the workload's forward pass (default cp_chunks) and prints, as
medians over CTAs and KV tiles 4..59 of each CTA's first unit, how long the softmax
warps and the MMA-issuing thread spend in each phase of a tile, in SM clock cycles.
With ``--units`` it prints instead where the launch's time goes unit by unit
(%globaltimer, ns): CTA start and end against the earliest start, and per unit the
wait from claim to first MMA, the tile loop, and the epilogue.
The library itself is built without the stamps.
"""
from __future__ import annotations

import ctypes
import glob
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
CTAS, ROLES, TILES, EVENTS = 160, 3, 64, 8
UNITS, UEVENTS = 16, 8


def build_traced() -> str:
    sys.path.insert(0, ROOT)
    from ragged_varlen_attention_gb300 import build as b
    out_dir = os.path.join(ROOT, "_build", "trace")
    os.makedirs(out_dir, exist_ok=True)
    objs, procs = [], []
    for src in sorted(glob.glob(os.path.join(b.CSRC, "*.cu"))):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        procs.append(subprocess.Popen([b.nvcc(), *b.ARCH, *b.NVCC_FLAGS, "-DTHD_FWD_TRACE", "-c", src, "-o", obj]))
        objs.append(obj)
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("nvcc failed")
    lib = os.path.join(out_dir, "libthd_attn_trace.so")
    subprocess.check_call([b.nvcc(), *b.ARCH, "-shared", "-cudart", "static", "-o", lib, *objs])
    return lib


def main() -> int:
    import torch
    args = [a for a in sys.argv[1:] if not a.startswith("--")]
    units_mode = "--units" in sys.argv[1:]
    name = args[0] if args else "cp_chunks"
    lib_path = build_traced()
    from ragged_varlen_attention_gb300 import binding as bd
    from ragged_varlen_attention_gb300 import workloads as wl
    bd.library_path = lambda: lib_path
    lib = bd.load_library()
    lib.thd_fwd_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    batch = wl.make(name)
    dev = torch.device("cuda", 0)
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)
    q, k, v = batch.q.to(dev), batch.k.to(dev), batch.v.to(dev)
    o, st = batch.o_init().to(dev), batch.stats_init().to(dev)
    meta = [ints(x) for x in (batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.off_q, batch.off_k, batch.off_v,
                              batch.off_o, batch.off_s)]
    mask = ints(batch.mask_type, np.int8)
    qco = None if batch.q_causal_offset is None else ints(batch.q_causal_offset)
    plan = bd.plan_for_tensors(q, k, v, o, batch.batch, batch.cap_s, batch.stats_layout)
    ws = bd.alloc_workspace(plan, dev)
    for _ in range(4):
        if lib.thd_fwd_trace_clear() != 0:
            raise RuntimeError("trace clear failed")
        bd.thd_attn_fwd(plan, q, k, v, o, st, *meta, mask, qco, ws)
    status = bd.thd_attn_read_status(plan, ws)
    torch.cuda.synchronize()
    if units_mode:
        return report_units(lib, name, status, int(os.environ.get("THD_TRACE_SMS", "0")) or
                            torch.cuda.get_device_properties(0).multi_processor_count)
    buf = np.zeros(CTAS * ROLES * TILES * EVENTS, dtype=np.uint64)
    if lib.thd_fwd_trace_read(buf.ctypes.data, buf.nbytes) != 0:
        raise RuntimeError("trace read failed")
    tr = buf.reshape(CTAS, ROLES, TILES, EVENTS).astype(np.float64)
    tr[tr == 0] = np.nan
    span = slice(4, 60)

    def med(x):
        x = x[np.isfinite(x)]
        return float(np.median(x)) if x.size else float("nan")

    print(f"workload {name}, status {status}; cycles per KV tile (medians over CTAs, tiles 4..59)")
    for t in (0, 1):
        s = tr[:, t]
        print(f"softmax {t}: wait for S {med(s[:, span, 1] - s[:, span, 0]):7.0f}  load S {med(s[:, span, 2] - s[:, span, 1]):5.0f}  "
              f"compute P {med(s[:, span, 3] - s[:, span, 2]):5.0f}  store P {med(s[:, span, 4] - s[:, span, 3]):5.0f}  "
              f"arrive {med(s[:, span, 5] - s[:, span, 4]):5.0f}  period {med(s[:, 5:61, 1] - s[:, 4:60, 1]):6.0f}")
    i = tr[:, 2]
    print(f"issuer: V/K waits {med(i[:, span, 1] - i[:, span, 0]):5.0f}  P0 wait {med(i[:, span, 2] - i[:, span, 1]):5.0f}  "
          f"batch 0 {med(i[:, span, 3] - i[:, span, 2]):5.0f}  P1 wait {med(i[:, span, 4] - i[:, span, 3]):5.0f}  "
          f"batch 1 {med(i[:, span, 5] - i[:, span, 4]):5.0f}  releases {med(i[:, span, 6] - i[:, span, 5]):5.0f}  "
          f"period {med(i[:, 5:61, 0] - i[:, 4:60, 0]):6.0f}")
    s0, s1 = tr[:, 0], tr[:, 1]
    print(f"P0 stored -> issuer past its wait {med(i[:, span, 2] - s0[:, span, 5]):6.0f}; "
          f"P1 {med(i[:, span, 4] - s1[:, span, 5]):6.0f}; batch 0 issued -> S0(j+1) seen "
          f"{med(s0[:, 5:61, 1] - i[:, 4:60, 3]):5.0f}; batch 1 -> S1(j+1) {med(s1[:, 5:61, 1] - i[:, 4:60, 5]):5.0f}")
    return 0


def report_units(lib, name: str, status: int, n_sms: int) -> int:
    lib.thd_fwd_trace_units_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    buf = np.zeros(CTAS * UNITS * UEVENTS + CTAS * 2, dtype=np.uint64)
    if lib.thd_fwd_trace_units_read(buf.ctypes.data, buf.nbytes) != 0:
        raise RuntimeError("trace read failed")
    u = buf[:CTAS * UNITS * UEVENTS].reshape(CTAS, UNITS, UEVENTS)
    cta = buf[CTAS * UNITS * UEVENTS:].reshape(CTAS, 2)[:n_sms].astype(np.int64)
    n_sms = int((cta[:, 0] > 0).sum())           # CTAs of the launch (grid <= SMs)
    cta = cta[:n_sms]
    t0 = int(cta[:, 0].min())
    rel = lambda x: (x.astype(np.int64) - t0) / 1000.0    # microseconds after the earliest CTA start
    start, end = rel(cta[:, 0]), rel(cta[:, 1])
    print(f"workload {name}, status {status}; times in us after the earliest CTA start")
    print(f"CTA start: min {start.min():.2f} median {np.median(start):.2f} max {start.max():.2f}; "
          f"CTA end: min {end.min():.2f} median {np.median(end):.2f} max {end.max():.2f}")
    rows = []
    for c in range(n_sms):
        for k in range(UNITS):
            ev = u[c, k]
            if ev[2] == 0 or ev[3] == 0:      # not reached, or a unit without KV tiles
                continue
            tiles = int(ev[7] & 0xffffffff)
            epi = max(int(ev[5]), int(ev[6]))
            rows.append((c, k, tiles, rel(ev[0]), rel(ev[2]), rel(ev[3]), rel(ev[4]), rel(np.uint64(epi)) if epi else np.nan))
    a = np.array([r[2:] for r in rows], dtype=np.float64)
    n_units = np.bincount([r[0] for r in rows], minlength=n_sms)
    print(f"units per CTA: min {n_units.min()} median {np.median(n_units):.0f} max {n_units.max()}")
    tiles, claim, got, first, last, epi = a.T
    print(f"per unit (medians): claim -> first QK committed {np.median(first - claim):.2f}; "
          f"first QK -> last MMA committed {np.median(last - first):.2f} for {np.median(tiles):.0f} tiles; "
          f"last MMA -> epilogue stored {np.nanmedian(epi - last):.2f}")
    for n in sorted(set(tiles.astype(int))):
        m = tiles == n
        print(f"  {n:3d} tiles: {int(m.sum()):4d} units, loop {np.median(last[m] - first[m]):6.2f} us "
              f"({np.median(last[m] - first[m]) / max(n, 1):.2f} per tile), claim -> first QK "
              f"{np.median(first[m] - claim[m]):5.2f}, epilogue {np.nanmedian(epi[m] - last[m]):5.2f}")
    worst = int(np.argmax(end))
    print(f"last CTA to finish ({worst}, end {end[worst]:.2f}):")
    for r in rows:
        if r[0] == worst:
            print(f"  unit {r[1]}: {r[2]} tiles, claimed {r[3]:.2f}, first QK {r[5]:.2f}, last MMA {r[6]:.2f}, "
                  f"stored {r[7]:.2f}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
