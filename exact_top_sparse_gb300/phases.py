"""Per-phase time split of the persistent selector kernel (a diagnostic).

Builds a second copy of the library with -DTOPK_PHASE_TIMING (the kernel
then adds thread 0's clock64 deltas between its phase marks into a device
array) into lib/libtopk_phases.so, runs the selector on synthetic causal
indexer-like rows and prints, per workload, the call's time and the
microseconds one CTA spends per row in each phase:

  claim        taking the row from the queue
  first_load   the first ring copies, the sample loads and their range
  sample_rank  the two sample ranks that give tau0 and tau1 (with a sampler
               warp, which took them during the previous row's pass: the
               first ring copies only)
  scan         the certify + collect pass over the whole row
  tally        C(tau0) and the seeded histogram from the candidates
  next         without a sampler warp: claiming the next row and warming L2
               with its sample points
  select       refinement (and, on rare rows, recovery or a re-read)
  finish       closing the row (padding, flags, diagnostics)
  unsampled    rows served without sampling (sentinel or exact path)

and the refinement rounds per row.  With --timeline it also records, for
one more call, every CTA's global-timer stamps (start, exit, and for each of
its first four rows the claim, the start and end of the full-row pass and
the close) and prints their spread over the CTAs in microseconds from the
first CTA's start: where a call of few rows per CTA spends its time.  The
library used by everything else is not touched.  Needs a GPU.

    python -m exact_top_sparse_gb300.phases [--dtype f32|bf16|e4m3] [--timeline] NxM ...
"""
import argparse
import ctypes
import json
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

from . import build as B

PHASE_LIB = os.path.join(B.LIBDIR, "libtopk_phases.so")
NAMES = {0: "claim", 8: "first_load", 1: "sample_rank", 2: "scan", 3: "tally", 4: "next",
         5: "select", 6: "finish", 7: "unsampled"}
ROUNDS_SLOT = 9
SLOTS = 12
SM_MHZ = 2070.0  # clock the cycle counts are converted with (GB300 maximum SM clock)


def build_phase_library() -> str:
    """Compile every translation unit with -DTOPK_PHASE_TIMING and link them
    (skipped while the library is newer than every source)."""
    if os.path.exists(PHASE_LIB) and all(os.path.getmtime(p) <= os.path.getmtime(PHASE_LIB)
                                         for p in B._inputs()):
        return PHASE_LIB
    objdir = os.path.join(B.HERE, "_build_phases")
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(B.LIBDIR, exist_ok=True)
    incs = ["-I", os.path.join(B.ROOT, "include"), "-I", B.CSRC]

    def one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [B._nvcc()] + B.ARCH + B.FLAGS + ["-DTOPK_PHASE_TIMING"] + incs + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s" % (src, r.stderr))
        return obj

    with ThreadPoolExecutor(max_workers=max(1, len(B.sources()))) as ex:
        objs = list(ex.map(one, B.sources()))
    cmd = [B._nvcc()] + B.ARCH + ["-shared", "-cudart", "shared", "-o", PHASE_LIB] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s" % r.stderr)
    return PHASE_LIB


def _spread(v):
    """min / median / 90th percentile / max of v, rounded to 0.1."""
    v = sorted(v)
    if not v:
        return []
    return [round(v[min(len(v) - 1, int(q * (len(v) - 1) + 0.5))], 1) for q in (0, 0.5, 0.9, 1)]


def timeline_summary(shape, tl, grid, slots):
    """Spread over the CTAs of one launch's timeline stamps (microseconds from
    the first CTA's start)."""
    recs = [tl[i * slots:(i + 1) * slots] for i in range(grid)]
    recs = [r for r in recs if r[0] > 0]
    if not recs:  # the call ran no persistent launch (direct or KV-split plan)
        return {"shape": shape, "timeline_ctas": 0}
    t0 = min(r[0] for r in recs)
    us = lambda t: (t - t0) / 1000.0  # noqa: E731
    nrows = [sum(1 for j in range((slots - 2) // 5) if r[2 + 5 * j] > 0) for r in recs]
    out = {"shape": shape, "timeline_ctas": len(recs),
           "ctas_by_rows": {str(n): nrows.count(n) for n in sorted(set(nrows))},
           "start_us": _spread([us(r[0]) for r in recs]),
           "exit_us": _spread([us(r[1]) for r in recs])}
    for j in range((slots - 2) // 5):
        rows = [r[2 + 5 * j:7 + 5 * j] for r in recs if r[2 + 5 * j] > 0]
        sampled = [f for f in rows if f[2] > 0 and f[3] > 0]
        if not rows:
            break
        out["row%d" % j] = {
            "ctas": len(rows),
            "claim_us": _spread([us(f[1]) for f in rows]),
            "close_us": _spread([us(f[4]) for f in rows]),
            "before_pass_us": _spread([(f[2] - f[1]) / 1000.0 for f in sampled]),
            "pass_us": _spread([(f[3] - f[2]) / 1000.0 for f in sampled]),
            "after_pass_us": _spread([(f[4] - f[3]) / 1000.0 for f in sampled]),
        }
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("shapes", nargs="*", default=["131072x8192", "262144x8192", "524288x8192",
                                                  "1048576x8192"])
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16", "e4m3"])
    ap.add_argument("--K", type=int, default=2048)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--timeline", action="store_true")
    args = ap.parse_args()

    import torch

    import exact_top_sparse_gb300 as ets
    from exact_top_sparse_gb300 import synth

    path = build_phase_library()
    ets._lib = None
    lib = ets.load_library(path)
    lib.topk_debug_phase_cycles.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
    lib.topk_debug_phase_cycles.restype = ctypes.c_int
    lib.topk_debug_timeline.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int,
                                        ctypes.c_int]
    lib.topk_debug_timeline.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    K = args.K
    for shape in args.shapes:
        N, M = (int(v) for v in shape.split("x"))
        lens = synth.causal_lens(N, M, 0, window=max(M, 8192))
        x = synth.indexer_rows(lens, N, seed=7, device=dev)
        if args.dtype == "bf16":
            x = x.to(torch.bfloat16)
        elif args.dtype == "e4m3":
            x = (x * 4.0).clamp(max=448.0).to(torch.float8_e4m3fn)
        d = lens.to(dev)
        out = torch.empty((M, K), dtype=torch.int32, device=dev)
        for _ in range(2):
            ets.topk_ragged(x, d, K, out=out)
        torch.cuda.synchronize()
        buf = (ctypes.c_ulonglong * SLOTS)()
        lib.topk_debug_phase_cycles(buf, 1)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.reps)]
        for a, b in evs:
            a.record()
            ets.topk_ragged(x, d, K, out=out)
            b.record()
        torch.cuda.synchronize()
        ms = sorted(a.elapsed_time(b) for a, b in evs)[args.reps // 2]
        lib.topk_debug_phase_cycles(buf, 1)
        per_row = {NAMES[i]: round(buf[i] / args.reps / M / SM_MHZ, 2) for i in NAMES}
        vb = float(x.element_size()) * float(lens.to("cpu").to(torch.int64).sum())
        print(json.dumps({"shape": shape, "dtype": args.dtype, "plan": ets.plan(M, N, K)["kind"],
                          "ms_per_call": round(ms, 4), "gbps_valid": round(vb / ms / 1e6, 1),
                          "us_per_row_per_cta": per_row,
                          "refine_rounds_per_row": round(buf[ROUNDS_SLOT] / args.reps / M, 2)}),
              flush=True)
        if args.timeline:
            grid = int(ets.plan(M, N, K)["grid"])
            if lib.topk_debug_timeline(None, 0, 1) < 0:
                raise RuntimeError("timeline reset failed")
            ets.topk_ragged(x, d, K, out=out)
            slots = lib.topk_debug_timeline(None, 0, 0)
            tl = (ctypes.c_ulonglong * (grid * slots))()
            if lib.topk_debug_timeline(tl, grid, 0) < 0:
                raise RuntimeError("timeline read failed")
            print(json.dumps(timeline_summary(shape, list(tl), grid, slots)), flush=True)
        del x, out
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
