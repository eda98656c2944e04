"""Benchmark: exact Top-K (K = 2048) over causal ragged FP32 score rows.

One step = one topk_ragged call over one batch of M rows of N_alloc columns
(the whole hot path: sampling, certify+collect, refinement, recovery), with
the inputs already resident in HBM.  Default workload: N_alloc = 1,048,576,
M = 8192 causal rows (row j has length N_alloc - 8192 + j + 1), K = 2048; the
inputs (34.2 GB of valid scores) exceed L2, so no flush is needed between
steps.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank selects its own batch (weak scaling, no data-path
collective); the timed region is bracketed by a barrier and a device
synchronisation, and the slowest rank's time is reported.

--impl reference times the CPU oracle (the plain std::nth_element
definition) on the host cores, on a bounded sample of the same rows.
"""
import argparse
import json
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
import torch  # noqa: E402

METRIC = ("exact Top-K(K=2048) rows/s and achieved HBM GB/s (% of peak) at 128K–1M cols")
UNIT = "rows/s"
K_DEFAULT = 2048


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--N", type=int, default=1048576)
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--K", type=int, default=K_DEFAULT)
    ap.add_argument("--no-matrix", action="store_true", help="skip the 20-shape operator matrix")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the sampled-vs-exact proposal ablation and the rho / stride sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16", "e4m3"],
                    help="score type of the timed rows (the headline is f32)")
    ap.add_argument("--no-narrow", action="store_true",
                    help="skip the bfloat16 / FP8 E4M3 rows of the headline workload")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the indexer-score + Top-K chain (tensor-core) line")
    ap.add_argument("--chain-T", type=int, default=2048, help="queries of the chain line")
    ap.add_argument("--no-trace", action="store_true",
                    help="skip the replays of 245K- and 430K-token prefills (26 and 71 Top-K calls)")
    ap.add_argument("--chain-S", type=int, default=262144, help="keys of the chain line")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--force-kind", default="auto",
                    choices=["auto", "direct", "persistent", "kvsplit"])
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch from an ncu capture of this kernel")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time); a
    no-op for one rank."""
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if ws > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def copy_only_step(h, K, chunk_bytes=1 << 30):
    """One step of the copies the host-buffer call makes, without selection:
    the pinned host rows h [M, N] go to the device in chunks of about 1 GiB,
    alternating between two streams as topk_ragged_host does, and K indices
    per row come back.  Returns (step, release): step() runs and waits for
    one step; release() frees its buffers."""
    M, N = h.shape
    rows = max(1, min(M, chunk_bytes // max(1, N * 4)))
    dev = torch.device("cuda", torch.cuda.current_device())
    bufs = [torch.empty((rows, N), dtype=torch.float32, device=dev) for _ in range(2)]
    outs = [torch.zeros((rows, K), dtype=torch.int32, device=dev) for _ in range(2)]
    ho = torch.empty((M, K), dtype=torch.int32, pin_memory=True)
    sts = [torch.cuda.Stream(device=dev) for _ in range(2)]

    def step():
        for c, r0 in enumerate(range(0, M, rows)):
            n = min(rows, M - r0)
            with torch.cuda.stream(sts[c & 1]):
                bufs[c & 1][:n].copy_(h[r0:r0 + n], non_blocking=True)
                ho[r0:r0 + n].copy_(outs[c & 1][:n], non_blocking=True)
        for st in sts:
            st.synchronize()

    def release():
        bufs.clear()
        outs.clear()
        torch.cuda.empty_cache()

    return step, release


def step_gbs(nbytes: float, seconds) -> list:
    """GB/s of each timed step that moved nbytes (one figure per step)."""
    return [round(nbytes / t / 1e9, 1) for t in seconds]


def job_rows_per_s(ws: int, M: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank selects its own M-row batch per step
    (weak scaling, no data-path collective), timed by the slowest rank."""
    return ws * M * steps / (total_ms / 1000.0)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 peak for a kernel timed alone (the burst figure)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# The pages' timing protocol (codexqa.cn, section "什么叫精确，时间怎么量"):
# CUDA-graph replays, timed per call with CUDA events on the stream, median
# per call after warm-up and conditioning replays; mechanism runs take 10
# warm-up replays, 2 blocks of 50 conditioning replays and 7 rounds of 100
# timed replays rotated over the shape's groups.
PROTOCOL = {"warmup": 10, "condition": (2, 50), "rounds": 7, "per_round": 100}


def capture_graphs(stream, calls):
    """One CUDA graph per zero-argument call (each enqueues its launches on
    the current stream), captured on `stream` after one eager run of every
    call (which creates the library's workspace before any capture)."""
    with torch.cuda.stream(stream):
        for fn in calls:
            fn()
    stream.synchronize()
    graphs = []
    for fn in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs.append(g)
    stream.synchronize()
    return graphs


def replay_median(stream, graphs, warmup, condition, rounds, per_round):
    """Median device time (ms) of one replay: `warmup` replays, then
    condition[0] blocks of condition[1] replays, then `rounds` rounds of
    `per_round` timed replays; every replay takes the next graph in turn."""
    n = len(graphs)
    k = 0
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graphs[k % n].replay()
            k += 1
        for _ in range(condition[0]):
            for _ in range(condition[1]):
                graphs[k % n].replay()
                k += 1
            stream.synchronize()
    times = []
    for _ in range(rounds):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(per_round)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                graphs[k % n].replay()
                b.record(stream)
                k += 1
        stream.synchronize()
        times += [a.elapsed_time(b) for a, b in evs]
    return statistics.median(times), len(times)


def operator_matrix_leg(ets, dev, stream, peak, K, inputs_1m=None):
    """The pages' operator matrix (codexqa.cn, section "20 个形状都最快"):
    widths 128K-1M x M in {512 .. 8192}; each width's last 8192 causal rows
    are cut into non-overlapping groups of M rows, every group is captured as
    one graph, and the shape's latency is the median per call over the
    protocol's replays rotated across the groups."""
    mat = {}
    for w in (131072, 262144, 524288, 1048576):
        if w == 1048576 and inputs_1m is not None:
            xw, lw = inputs_1m
        else:
            xw, lw = make_inputs(w, 8192, 0, seed=11, device=dev)
        dlw = lw.to(dev)
        outw = torch.empty((8192, K), dtype=torch.int32, device=dev)
        for m in (512, 1024, 2048, 4096, 8192):
            ng = 8192 // m
            calls = [(lambda g0=g0: ets.topk_ragged(xw[g0:g0 + m], dlw[g0:g0 + m], K,
                                                    out=outw[g0:g0 + m]))
                     for g0 in range(0, 8192, m)]
            graphs = capture_graphs(stream, calls)
            ms, n = replay_median(stream, graphs, **PROTOCOL)
            del graphs
            vb = 4.0 * float(lw.to(torch.int64).sum()) / ng  # mean valid bytes of a group
            gbps = vb / (ms / 1000.0) / 1e9
            mat["%dx%d" % (w, m)] = {"ms": ms, "rows_per_s": m / (ms / 1000.0), "gbps": gbps,
                                     "frac": gbps / peak, "path": ets.plan(m, w, K)["kind"],
                                     "groups": ng, "replays_timed": n,
                                     "protocol": "graph-replay median"}
        del xw, lw, dlw, outw
        ets.release_workspaces()
        torch.cuda.empty_cache()
    return mat


def proposal_ablation_leg(ets, dev, stream, peak, K):
    """Sampled proposal against the exact one, the selector otherwise
    unchanged (codexqa.cn, section "采样不是处处都该开"): the exact form
    serves every row on the library's exact path (a histogram pass over the
    whole row, then refinement passes), which is what a selector without a
    sampled proposal has to do to find its boundary.  Graph replays, median
    per call (3 warm-up, 2 x 20 conditioning, 3 x 40 timed)."""
    from exact_top_sparse_gb300 import synth
    res = {}
    for w, m, gi in ((131072, 2048, 1), (1048576, 1024, 3)):
        lens = synth.causal_lens(w, m, gi)
        x = synth.indexer_rows(lens, w, seed=23, device=dev)
        dl = lens.to(dev)
        o = torch.empty((m, K), dtype=torch.int32, device=dev)
        vb = 4.0 * float(lens.to(torch.int64).sum())
        cell = {}
        old = ets.get_params()
        try:
            for name, kw in (("sampled", {}), ("exact", {"sample_min_len": w + 1})):
                ets.set_params(**kw)
                graphs = capture_graphs(stream, [lambda: ets.topk_ragged(x, dl, K, out=o)])
                ms, _ = replay_median(stream, graphs, 3, (2, 20), 3, 40)
                del graphs
                with torch.cuda.stream(stream):
                    _, dg = ets.topk_ragged_diag(x, dl, K, stream=stream)
                cell[name] = {"ms": ms, "gbps": vb / (ms / 1000.0) / 1e9,
                              "frac": vb / (ms / 1000.0) / 1e9 / peak,
                              "row_paths": path_counts(ets, dg)}
                ets.set_params(**old)
        finally:
            ets.set_params(**old)
        cell["exact_over_sampled"] = cell["exact"]["ms"] / cell["sampled"]["ms"]
        res["%dx%d" % (w, m)] = cell
        del x, o
        ets.release_workspaces()
        torch.cuda.empty_cache()
    return res


def sampling_sweep_leg(ets, dev, stream, K):
    """Primary targets rho0 and strides s swept with the selector unchanged
    (codexqa.cn, section "采样不是处处都该开": rho = 1 leaves about a third of
    the rows to recovery, 1.25K 5.7-7.8 %, 1.5K under 1 %; at 1.5K, s = 16
    recovers almost nothing, s = 64 under 0.01 %, s = 128 under 0.9 %,
    s = 256 2.48-3.26 %; H20, captured Hy4-Preview rows).  Every row uses
    the swept values (no long tier); rho1 = rho0 + 0.25.  Per cell: the
    primary miss rate (rows with C(tau0) < K: served by tau1 or recovery),
    the exact-recovery rate (C(tau1) < K) and the median of 5 calls."""
    from exact_top_sparse_gb300 import synth
    res = {"pages_context": {"rho_1.0": "~1/3", "rho_1.25": "5.7-7.8 %", "rho_1.5": "< 1 %",
                             "s_16": "~0", "s_64": "< 0.01 %", "s_128": "< 0.9 %",
                             "s_256": "2.48-3.26 %"}}
    cells = [(128, r_) for r_ in (1.0, 1.25, 1.5, 1.75, 2.0)] + \
            [(s_, 1.5) for s_ in (16, 64, 256, 512)]
    for w, m in ((131072, 2048), (1048576, 1024)):
        lens = synth.causal_lens(w, m, 0)
        x = synth.indexer_rows(lens, w, seed=29, device=dev)
        dl = lens.to(dev)
        o = torch.empty((m, K), dtype=torch.int32, device=dev)
        old = ets.get_params()
        out = {}
        try:
            for s_, r_ in cells:
                ets.set_params(stride=s_, rho0=r_, rho1=r_ + 0.25, long_len=0)
                with torch.cuda.stream(stream):
                    _, dg = ets.topk_ragged_diag(x, dl, K, stream=stream)
                    ts = []
                    for _ in range(6):
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        ets.topk_ragged(x, dl, K, out=o, stream=stream)
                        b.record(stream)
                        ts.append((a, b))
                stream.synchronize()
                ms = statistics.median([a.elapsed_time(b) for a, b in ts[1:]])
                pc = path_counts(ets, dg)
                sampled = pc["tau0"] + pc["tau1"] + pc["recovery"]
                out["s%d_rho%.2f" % (s_, r_)] = {
                    "stride": s_, "rho0": r_, "rho1": r_ + 0.25, "ms": ms,
                    "primary_miss_rate": (pc["tau1"] + pc["recovery"]) / max(1, sampled),
                    "exact_recovery_rate": pc["recovery"] / max(1, sampled),
                    "overflow_rows": pc["overflow"], "sampled_rows": sampled}
        finally:
            ets.set_params(**old)
        res["%dx%d" % (w, m)] = out
        del x, o
        torch.cuda.empty_cache()
    return res


def path_counts(ets, dg):
    """Rows per path (and rows that overflowed) of one call's diagnostics."""
    paths = {name: int((dg["path"] == code).sum()) for name, code in
             (("sentinel", 0), ("direct", 1), ("tau0", 2), ("tau1", 3), ("recovery", 4))}
    paths["overflow"] = int(((dg["flags"] & ets.FLAG_OVERFLOW) != 0).sum())
    return paths


def trace_leg(ets, dev, stream, tokens=430 * 1024, K=2048):
    """Replay the Top-K calls of one synthetic prefill (exact_top_sparse_gb300.trace):
    first the selector alone over indexer-like score rows of each call's shape,
    then the whole score -> select chain.  As the pages report a trace (codexqa.cn,
    section "什么叫精确，时间怎么量": trace latency is the sum of per-call medians),
    every call is captured as a CUDA graph and timed by replays (selector: 3
    warm-up, 20 timed; chain: 2 warm-up, 5 timed), and the totals are the sums
    of the per-call medians.  The whole sequence of eager calls is also timed
    once (`*_sequence_ms`)."""
    from exact_top_sparse_gb300 import synth, trace
    calls = trace.calls(tokens)
    W = trace.WORKSPACE_FLOATS
    buf = synth.trace_scores(W, seed=17, device=dev)
    lens_all = torch.arange(1, tokens + 1, dtype=torch.int32, device=dev)
    outs = torch.empty((max(c.rows for c in calls), K), dtype=torch.int32, device=dev)
    valid = sum(4.0 * (c.row0 * c.rows + c.rows * (c.rows + 1) / 2.0) for c in calls)

    def run_topk():
        for c in calls:
            x = buf[:c.rows * c.width].view(c.rows, c.width)
            ets.topk_ragged(x, lens_all[c.row0:c.row0 + c.rows], K, out=outs[:c.rows],
                            stream=stream)

    # every call's width is a multiple of 128 and its rows a multiple of 4
    assert all(c.width % 128 == 0 and c.rows % 4 == 0 for c in calls)
    q, k, w, _ = synth.index_inputs(tokens + (-tokens) % 4, tokens + (-tokens) % 128, seed=19,
                                    device=dev)
    flops = sum(2.0 * c.rows * c.width * 64 * 128 for c in calls)

    def run_chain():
        for c in calls:
            ets.topk_index_topk(q[c.row0:c.row0 + c.rows], k[:c.width],
                                w[c.row0:c.row0 + c.rows], lens_all[c.row0:c.row0 + c.rows], K,
                                scores=buf[:c.rows * c.width].view(c.rows, c.width),
                                out=outs[:c.rows], stream=stream)

    res = {"tokens": tokens, "calls": len(calls), "steps": len({c.step for c in calls}),
           "workspace_floats": W, "valid_score_bytes": valid,
           "protocol": "sum of per-call graph-replay medians"}
    for name, fn in (("topk", run_topk), ("chain", run_chain)):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            fn()
            b.record(stream)
        stream.synchronize()
        res[name + "_sequence_ms"] = a.elapsed_time(b)

    def one_topk(c):
        return lambda: ets.topk_ragged(buf[:c.rows * c.width].view(c.rows, c.width),
                                       lens_all[c.row0:c.row0 + c.rows], K, out=outs[:c.rows])

    def one_chain(c):
        return lambda: ets.topk_index_topk(
            q[c.row0:c.row0 + c.rows], k[:c.width], w[c.row0:c.row0 + c.rows],
            lens_all[c.row0:c.row0 + c.rows], K,
            scores=buf[:c.rows * c.width].view(c.rows, c.width), out=outs[:c.rows])

    def one_fused(c):
        return lambda: ets.topk_index_topk_fused(
            q[c.row0:c.row0 + c.rows], k[:c.width], w[c.row0:c.row0 + c.rows],
            lens_all[c.row0:c.row0 + c.rows], K,
            scores=buf[:c.rows * c.width].view(c.rows, c.width), out=outs[:c.rows])

    for name, make, reps in (("topk", one_topk, (3, 20)), ("chain", one_chain, (2, 5)),
                             ("chain_fused", one_fused, (2, 5))):
        medians = []
        for c in calls:
            g = capture_graphs(stream, [make(c)])
            ms, _ = replay_median(stream, g, reps[0], (0, 0), 1, reps[1])
            medians.append(ms)
            del g
        res[name + "_total_ms"] = sum(medians)
        res[name + "_call_medians_ms"] = [round(v, 4) for v in medians]
    res["topk_gbps"] = valid / (res["topk_total_ms"] / 1000.0) / 1e9
    res["score_flops_dense"] = flops
    res["chain_score_share_ms"] = res["chain_total_ms"] - res["topk_total_ms"]
    res["status_flags"] = ets.read_status(dev, stream) | ets.index_read_status(dev, stream)
    del buf, q, k, w
    torch.cuda.empty_cache()
    return res


def chain_leg(ets, dev, stream, reps, T=2048, S=262144, K=2048):
    """Indexer scores (tcgen05) followed by the exact Top-K, timed with CUDA
    events on the launching stream; the score kernel's roofline is tensor."""
    from exact_top_sparse_gb300 import synth
    q, k, w, lens = synth.index_inputs(T, S, seed=13, device=dev)
    dl = lens.to(dev)
    scores = torch.empty((T, S), dtype=torch.float32, device=dev)
    out = torch.empty((T, K), dtype=torch.int32, device=dev)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        ts = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                fn()
                b.record(stream)
            stream.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    score_ms = timed(lambda: ets.topk_index_scores(q, k, w, row_lens=dl, scores=scores,
                                                   stream=stream))
    chain_ms = timed(lambda: ets.topk_index_topk(q, k, w, dl, K, scores=scores, out=out,
                                                 stream=stream))
    out_f = torch.empty((T, K), dtype=torch.int32, device=dev)
    fused_ms = timed(lambda: ets.topk_index_topk_fused(q, k, w, dl, K, scores=scores, out=out_f,
                                                       stream=stream))
    status = ets.index_read_status(dev, stream)
    flops = 2.0 * T * S * 64 * 128
    peak, kind = measured_bf16_tflops()
    tflops = flops / (score_ms / 1000.0) / 1e12
    import oracle
    rows = np.array([0, T // 3, T - 1])
    xr = scores[torch.as_tensor(rows, device=dev)].cpu().numpy()
    v = oracle.compare(xr, lens.numpy()[rows], K, out[torch.as_tensor(rows, device=dev)].cpu().numpy())
    vf = oracle.compare(xr, lens.numpy()[rows], K,
                        out_f[torch.as_tensor(rows, device=dev)].cpu().numpy())
    del scores, q, k
    torch.cuda.empty_cache()
    return {
        "workload": "indexer scores I[t,s] = sum_j w[t,j]*ReLU(q[t,j].k[s]) then exact Top-%d; "
                    "T=%d queries, S=%d keys, H=64, D=128, bf16 q/k, f32 w and scores, causal "
                    "lengths S-T+t+1" % (K, T, S),
        "ms_per_call": chain_ms, "score_ms": score_ms, "topk_ms": chain_ms - score_ms,
        "rows_per_s": T / (chain_ms / 1000.0), "reps": reps, "gpu_launches_per_call": 2,
        "status_flags": status,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "peak_kind": kind + " (bf16 dense, burst)",
                     "flops_per_launch": flops, "kernel": "k_index_scores"},
        "spot_check": {"rows": int(rows.size), "contract_failures": int((v["check"] != 0).sum()),
                       "set_mismatches": int(v["set_mismatch"].sum())},
        "fused": {"api": "topk_index_topk_fused (sample-key score pass, gated score pass, "
                         "selection from the candidates)",
                  "ms_per_call": fused_ms, "rows_per_s": T / (fused_ms / 1000.0),
                  "selection_ms_beyond_scores": fused_ms - score_ms, "gpu_launches_per_call": 5,
                  "spot_check": {"rows": int(rows.size),
                                 "contract_failures": int((vf["check"] != 0).sum()),
                                 "set_mismatches": int(vf["set_mismatch"].sum())}},
    }


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# Sources whose text decides a selector launch's DRAM traffic (the kernels and
# the host defaults that reach them, such as the L2 prefetch distance).
FINGERPRINT_SOURCES = ("score_elem.cuh", "topk_device.cuh", "topk_kernels.cu", "topk_launch.h",
                       "topk_api.cu")

SAMPLING_KNOBS = ("stride", "rho0", "rho1", "sample_min_len", "long_len", "long_stride",
                  "long_rho0", "long_rho1")


def kernel_fingerprint(params, kind, grid, elem_bytes=4):
    """Hash of what decides a selector launch's DRAM traffic: the kernel
    sources, the sampling parameters in effect, the launch shape and the
    score element size."""
    import hashlib
    h = hashlib.sha256()
    for name in FINGERPRINT_SOURCES:
        with open(os.path.join(ROOT, "exact_top_sparse_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    launch = {"sampling": {k: params[k] for k in SAMPLING_KNOBS}, "kind": kind, "grid": grid,
              "elem_bytes": elem_bytes}
    h.update(json.dumps(launch, sort_keys=True).encode())
    return h.hexdigest()[:16]


def profiled_traffic(params, plan, valid_bytes, elem_bytes=4):
    """DRAM bytes per launch from the committed ncu capture of this kernel.

    profiles/k_persistent_traffic.json holds the DRAM-bytes-per-valid-byte
    ratio of one capture and the kernel fingerprint (sources, sampling
    parameters, launch shape) it was taken with; the figure is reported only
    while the fingerprint still matches (else None).
    """
    p = os.path.join(ROOT, "profiles", "k_persistent_traffic.json")
    if plan["kind"] != "persistent" or not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if (kernel_fingerprint(params, plan["kind"], plan["grid"], elem_bytes)
            != d.get("kernel_fingerprint")):
        return None
    return float(d["dram_bytes_per_valid_byte"]) * valid_bytes


def narrow_leg(ets, dev, stream, N, M, K, peak, reps=5):
    """The headline workload with its scores rounded to bfloat16 and to FP8
    E4M3 (scaled by 4 and held below 448 first), selected exactly as their
    widened values; device time of `reps` consecutive calls after two
    untimed ones, and 4 rows spot-checked against the oracle."""
    import oracle
    res = {}
    for name in ("bf16", "e4m3"):
        x32, lens = make_inputs(N, M, 0, seed=7, device=dev)
        if name == "bf16":
            x = x32.to(torch.bfloat16)
        else:
            x = (x32 * 4.0).clamp(max=448.0).to(torch.float8_e4m3fn)
        del x32
        d_lens = lens.to(dev)
        out = torch.empty((M, K), dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(2):
                ets.topk_ragged(x, d_lens, K, out=out, stream=stream)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                ets.topk_ragged(x, d_lens, K, out=out, stream=stream)
            b.record(stream)
        stream.synchronize()
        ms = a.elapsed_time(b) / reps
        nbytes = float(lens.to(torch.int64).sum()) * x.element_size()
        rows = torch.linspace(0, M - 1, 4).round().long()
        xr = x[rows.to(dev)].float().cpu().numpy()
        v = oracle.compare(xr, lens[rows].numpy(), K, out[rows.to(dev)].cpu().numpy())
        res[name] = {"ms_per_call": ms, "rows_per_s": M / (ms / 1000.0),
                     "gbps_valid_scores": nbytes / (ms / 1000.0) / 1e9,
                     "frac": nbytes / (ms / 1000.0) / 1e9 / peak, "reps": reps,
                     "spot_check": {"rows": 4, "contract_failures": int((v["check"] != 0).sum()),
                                    "set_mismatches": int(v["set_mismatch"].sum())}}
        del x, out
        torch.cuda.empty_cache()
    return res


def make_inputs(N, M, group, seed, device):
    from exact_top_sparse_gb300 import synth
    lens = synth.causal_lens(N, M, group)
    x = synth.indexer_rows(lens, N, seed=seed, device=device)
    return x, lens


def time_steps(ets, x, d_lens, K, steps, warmup, ws, stream):
    """Device time of `steps` consecutive calls (events on the launching stream)."""
    out = torch.empty((x.shape[0], K), dtype=torch.int32, device=x.device)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            ets.topk_ragged(x, d_lens, K, out=out)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        t0 = time.perf_counter()
        for a, b in evs:
            a.record(stream)
            ets.topk_ragged(x, d_lens, K, out=out)
            b.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - t0
    per = [a.elapsed_time(b) for a, b in evs]  # ms
    total_ms = evs[0][0].elapsed_time(evs[-1][1])
    return total_ms, per, wall, out


def cpu_oracle_rate(x_rows_host, lens_host, K, budget_s=12.0):
    """Rows/s of the CPU oracle, repeating a host sample until ~budget_s of work."""
    import oracle
    threads = oracle.default_threads()
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.topk(x_rows_host, lens_host, K, threads=threads)
        n += x_rows_host.shape[0]
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return n / el, threads, el


def host_sample(N, M, K, rows=64, seed=7):
    """A bounded host copy of the workload: `rows` evenly spaced rows of the batch."""
    from exact_top_sparse_gb300 import synth
    lens_all = synth.causal_lens(N, M, 0)
    pick = torch.linspace(0, M - 1, rows).round().long()
    lens = lens_all[pick]
    x = synth.indexer_rows(lens, N, seed=seed, device="cpu")
    return x.numpy(), lens.numpy()


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    N, M, K = args.N, args.M, args.K
    xs, ls = host_sample(N, M, K, rows=32)
    threads = oracle.default_threads()
    for _ in range(max(args.warmup, 0)):
        oracle.topk(xs[:4], ls[:4], K, threads=threads)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.topk(xs, ls, K, threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > 150:
            break
    steps = len(times)
    rate = xs.shape[0] * steps / sum(times)
    ms = 1000.0 * M / rate
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "causal ragged FP32 score rows N_alloc=%d M=%d K=%d" % (N, M, K),
                   "N_alloc": N, "M": M, "K": K},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "each step: the CPU oracle (std::nth_element per row) on 32 "
                                   "evenly spaced rows of the %d-row batch; rows/s scaled to "
                                   "the full batch" % M},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args):
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import __graft_entry__ as g
    g.build()
    import exact_top_sparse_gb300 as ets

    N, M, K = args.N, args.M, args.K
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    if args.force_kind != "auto":
        ets.set_params(force_kind={"direct": ets.KIND_DIRECT, "persistent": ets.KIND_PERSISTENT,
                                   "kvsplit": ets.KIND_KVSPLIT}[args.force_kind])

    x, lens = make_inputs(N, M, 0, seed=7 + rank, device=dev)
    if args.dtype == "bf16":
        x = x.to(torch.bfloat16)
    elif args.dtype == "e4m3":
        # scaled by 4 and held below the largest E4M3 value before rounding
        x = (x * 4.0).clamp(max=448.0).to(torch.float8_e4m3fn)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    d_lens = lens.to(dev)
    elem_bytes = x.element_size()
    valid_bytes = float(elem_bytes) * float(lens.to(torch.int64).sum())
    type_name = {"f32": "FP32", "bf16": "bfloat16", "e4m3": "FP8 E4M3"}[args.dtype]
    plan = ets.plan(M, N, K)
    launches_per_step = 2 if plan["kind"] == "kvsplit" else 1

    clocks = ClockSampler(local)
    clocks.start()
    total_ms, per, wall, out = time_steps(ets, x, d_lens, K, args.steps, args.warmup, ws, stream)
    clk = clocks.stop()

    total_ms = max_over_ranks(total_ms, ws, dev)
    ms_per_step = total_ms / args.steps
    rows_per_s = job_rows_per_s(ws, M, args.steps, total_ms)
    kern_ms = statistics.mean(per)
    achieved = valid_bytes / (kern_ms / 1000.0) / 1e9
    status = ets.read_status(dev, stream)
    # per-row paths of one (untimed) call with diagnostics
    with torch.cuda.stream(stream):
        _, dg = ets.topk_ragged_diag(x, d_lens, K)
    paths = path_counts(ets, dg)

    result = {
        "metric": METRIC, "value": rows_per_s, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded indexer-like rows: Normal(30+N(0,1), 2.5) body, 0.2% "
                "Exponential(mean 6) upper tail, -inf causal suffix)",
        "config": {"workload": "causal ragged %s score rows N_alloc=%d M=%d K=%d"
                               % (type_name, N, M, K),
                   "N_alloc": N, "M": M, "K": K, "path": plan["kind"],
                   "grid": plan["grid"], "segments": plan["segments"],
                   "l2": "inputs (%.1f GB of valid scores) exceed the 129 MB L2; no flush"
                         % (valid_bytes / 1e9),
                   "gbps_valid_scores": achieved},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": (args.traffic if args.traffic is not None
                                 else profiled_traffic(ets.get_params(), plan, valid_bytes,
                                                       elem_bytes)),
                     "bytes_per_launch": valid_bytes,
                     "kernel": "k_kv_segment" if plan["kind"] == "kvsplit" else
                               ("k_direct" if plan["kind"] == "direct" else "k_persistent")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "status_flags": status,
        "row_paths": paths,
    }
    # a short exactness spot check of the timed output (8 rows, oracle)
    if rank == 0:
        import oracle
        rows = torch.linspace(0, M - 1, 8).round().long()
        xr = x[rows.to(dev)].float().cpu().numpy()
        v = oracle.compare(xr, lens[rows].numpy(), K, out[rows.to(dev)].cpu().numpy())
        result["spot_check"] = {"rows": 8, "contract_failures": int((v["check"] != 0).sum()),
                                "set_mismatches": int(v["set_mismatch"].sum())}

    # the operator matrix (informational) with the pages' timing protocol,
    # then the proposal ablation and the sampling sweep
    full_f32 = args.dtype == "f32" and N == 1048576 and M == 8192
    if not args.no_matrix and rank == 0 and full_f32:
        del out
        torch.cuda.empty_cache()
        result["operator_matrix"] = operator_matrix_leg(ets, dev, stream, peak, K,
                                                        inputs_1m=(x, lens))
        del x
        x = None
        torch.cuda.empty_cache()
    if not args.no_ablation and rank == 0 and full_f32:
        if x is not None:
            del x
            x = None
            torch.cuda.empty_cache()
        result["proposal_ablation"] = proposal_ablation_leg(ets, dev, stream, peak, K)
        result["sampling_sweep"] = sampling_sweep_leg(ets, dev, stream, K)

    if not args.no_narrow and rank == 0 and full_f32:
        if x is not None:
            del x
            x = None
            torch.cuda.empty_cache()
        try:
            result["narrow_rows"] = narrow_leg(ets, dev, stream, N, M, K, peak)
        except RuntimeError as e:
            result["narrow_rows"] = {"error": str(e)[:200]}

    if not args.no_chain and rank == 0:
        if x is not None:
            del x
            x = None
            torch.cuda.empty_cache()
        try:
            result["chain"] = chain_leg(ets, dev, stream, max(5, args.steps // 2),
                                        T=args.chain_T, S=args.chain_S)
        except RuntimeError as e:
            result["chain"] = {"error": str(e)[:200]}
    if not args.no_trace and rank == 0:
        for name, tokens in (("trace_245k", 245 * 1024), ("trace_430k", 430 * 1024)):
            try:
                result[name] = trace_leg(ets, dev, stream, tokens=tokens)
            except RuntimeError as e:
                result[name] = {"error": str(e)[:200]}

    # end to end through the host-buffer C ABI: pinned host rows in, indices out
    if not args.no_e2e and rank == 0 and args.dtype == "f32":
        if x is None:
            x, _ = make_inputs(N, M, 0, seed=7, device=dev)
        try:
            h = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
            h.copy_(x)
            del x
            torch.cuda.empty_cache()
            hl = lens.numpy().copy()
            ho = np.empty((M, K), dtype=np.int32)
            hn = h.numpy()
            copy_step, copy_release = copy_only_step(h, K)
            ets.topk_ragged_host(hn, hl, K, out=ho)
            copy_step()
            # The call's steps run back to back, then the copy-only steps: on
            # these hosts the page-locked link can switch speed from one step
            # to the next, and in two runs strictly alternating the two legs
            # gave every fast step to the call.
            ts, tc = [], []
            for _ in range(args.e2e_steps):
                t0 = time.perf_counter()
                ets.topk_ragged_host(hn, hl, K, out=ho)
                ts.append(time.perf_counter() - t0)
            for _ in range(args.e2e_steps):
                t0 = time.perf_counter()
                copy_step()
                tc.append(time.perf_counter() - t0)
            copy_release()
            e2e_rate = M * len(ts) / sum(ts)
            copy_rate = M * len(tc) / sum(tc)
            h2d_gbs = M * N * 4 * len(tc) / sum(tc) / 1e9
            result["e2e"] = {"value": e2e_rate, "unit": UNIT,
                             "h2d_bytes_per_step": M * N * 4 + M * 4,
                             "d2h_bytes_per_step": M * K * 4,
                             "steps": len(ts), "api": "topk_ragged_host (pinned host buffers)",
                             "h2d_gbs_per_step": step_gbs(M * N * 4, ts),
                             "copy_only": {"value": copy_rate, "unit": UNIT, "h2d_gbs": h2d_gbs,
                                           "h2d_gbs_per_step": step_gbs(M * N * 4, tc),
                                           "what": "the same host->device and device->host "
                                                   "bytes in the same 1 GiB chunks on two "
                                                   "streams, no selection, timed in as many "
                                                   "steps right after the call's"}}
            del h
        except RuntimeError as e:
            result["e2e"] = {"value": None, "unit": UNIT, "error": str(e)[:200]}
    if not args.no_cpu and rank == 0 and args.dtype == "f32":
        xs, ls = host_sample(N, M, K, rows=32)
        rate, threads, el = cpu_oracle_rate(xs, ls, K)
        result["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads,
                                  "kind": "oracle",
                                  "sample": "the CPU oracle (std::nth_element per row) on 32 "
                                            "evenly spaced rows of the batch, repeated for "
                                            "%.1f s on %d threads" % (el, threads)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
