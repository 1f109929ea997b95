"""Pipeline trace of the tensor-core passes: where block 0 of each pass spends
its cycles, from the clock64 stamps that a trace build records.

    FLAREPP_TRACE=1 python -m rank_latent_routing_gb300.micro.trace [--workload pde2d]

Builds the library with FLAREPP_TRACE, runs a few forward calls of the
workload, then one traced call per pass (synthesis, encode, decode), and
prints for each pass: the pipeline fill (kernel start to the first scores),
the median softmax step and the wait for the next scores of the same stream,
the issuing threads' median time to issue the products and the next
scores, and the drain and epilogue after the last step.
"""
from __future__ import annotations

import argparse
import ctypes
import os

import numpy as np

ROLES, LEN = 16, 4096
START, LOAD, NORM, ISSUE, SOFTMAX, EPI = 0, 1, 2, 6, 10, 12


def _med(x):
    x = [v for v in x if v is not None and v >= 0]
    return float(np.median(x)) if x else float("nan")


def report(name, st, mhz):
    t0, t1 = int(st[START, 0]), int(st[START, 1])
    if not t0:
        print(f"== {name}: no stamps")
        return
    print(f"== {name}: block 0, {t1 - t0} cycles ({(t1 - t0) / mhz:.2f} us at {mhz:.0f} MHz)")
    loads = st[LOAD][st[LOAD] > 0] - t0
    if len(loads):
        print(f"  tiles loaded: {len(loads)}, first issued +{loads.min()}, last +{loads.max()}")
    for p in range(4):
        nz = np.sort(st[NORM + p][st[NORM + p] > 0])
        if len(nz) > 1:
            print(f"  N0 rows {32 * p}-{32 * p + 31}: {len(nz)} tiles, first +{nz[0] - t0}, "
                  f"median gap {np.median(np.diff(nz)):.0f}")
    last = 0
    for g in range(2):
        row = st[SOFTMAX + g]
        steps, waits, first = [], [], None
        j = 0
        while 2 * j + 1 < LEN and row[2 * j]:
            s, f = int(row[2 * j]), int(row[2 * j + 1])
            first = s if first is None else min(first, s)
            if f:
                steps.append(f - s)
                last = max(last, f)
            if f and 2 * (j + 1) < LEN and row[2 * (j + 1)]:
                waits.append(int(row[2 * (j + 1)]) - f)
            j += 1
        if first is not None:
            print(f"  softmax stream {g}: {len(steps)} steps, first scores +{first - t0}, median step "
                  f"{_med(steps):.0f}, median wait for the next scores {_med(waits):.0f}")
    for q in range(2):
        row = st[ISSUE + q]
        pv, sc, wp = [], [], []
        j = 0
        while 3 * j + 2 < LEN and row[3 * j]:
            a, b, c = int(row[3 * j]), int(row[3 * j + 1]), int(row[3 * j + 2])
            if b:
                pv.append(b - a)
            if b and c:
                sc.append(c - b)
            if c and 3 * (j + 1) < LEN and row[3 * (j + 1)]:
                wp.append(int(row[3 * (j + 1)]) - c)
            j += 1
        if j:
            print(f"  issuer of stream {q}: {j} steps, median cycles: products {_med(pv):.0f}, "
                  f"next scores {_med(sc):.0f}, wait for P {_med(wp):.0f}")
    epi = [int(v) - t0 if v else None for v in st[EPI, :3]]
    print(f"  last softmax step done +{last - t0 if last else -1}; epilogue (drain, partials written, "
          f"arrived) {epi}; end +{t1 - t0}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="pde2d")
    ap.add_argument("--mhz", type=float, default=2070.0, help="SM clock for the microsecond column")
    ap.add_argument("--save", default=None, help="write the raw stamps of each pass to <save>_<pass>.npy")
    args = ap.parse_args()
    if os.environ.get("FLAREPP_TRACE") != "1":
        raise SystemExit("set FLAREPP_TRACE=1: the trace needs a trace build of the library")
    from rank_latent_routing_gb300 import build
    build.build(force=True)
    import torch
    from rank_latent_routing_gb300 import flarepp, workloads

    wl = workloads.config(args.workload)
    dev = {}
    for k in ("K", "V", "Ks_raw", "Qseed", "Qf"):
        a = wl.bits[k] if wl.dtype == "bf16" else getattr(wl, k)
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if wl.dtype == "bf16" else np.float32))
        dev[k] = t.cuda().view(torch.bfloat16) if wl.dtype == "bf16" else t.cuda()
    dev["gate"] = torch.from_numpy(wl.gate).cuda()
    call = lambda: flarepp.forward(dev["K"], dev["V"], dev["Ks_raw"], dev["Qseed"], dev["Qf"], dev["gate"])
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    lib = flarepp._lib
    lib.flarepp_debug_trace.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
    lib.flarepp_debug_trace.restype = ctypes.c_int
    print(f"workload {args.workload}: {wl.shape}, {wl.dtype}")
    for pass_id, name in ((1, "synthesis"), (2, "encode"), (3, "decode")):
        if lib.flarepp_debug_trace(pass_id, None, 0) != 0:
            raise SystemExit("flarepp_debug_trace failed (not a trace build?)")
        call()
        torch.cuda.synchronize()
        buf = (ctypes.c_ulonglong * (ROLES * LEN))()
        if lib.flarepp_debug_trace(0, buf, ROLES * LEN) != 0:
            raise SystemExit("reading the trace failed")
        st = np.frombuffer(buf, dtype=np.uint64).astype(np.int64).reshape(ROLES, LEN)
        if args.save:
            np.save(f"{args.save}_{name}.npy", st)
        report(name, st, args.mhz)
    if flarepp.sync_status() != 0:
        raise SystemExit("device error during the traced calls")


if __name__ == "__main__":
    main()
