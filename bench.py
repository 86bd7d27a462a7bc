"""Benchmark of the fused reduce + residual add + RMSNorm step on GB300.

One step = one launch of the fused kernel over one batch of the headline
workload (N=8 dense row-parallel bf16 partials, T=1024 tokens, H=8192), with
inputs already resident in HBM.  Prints ONE JSON line (rank 0):

  value     tokens/s over all ranks (device time, CUDA events, max over ranks)
  roofline  achieved algorithmic GB/s of the kernel vs the measured HBM copy
            peak; algorithmic bytes per token = (N + 1 + n_out + 1) * H * 2
  e2e       the same metric through the C ABI with pinned HOST buffers: every
            step copies its inputs host->device, runs the kernel and copies the
            outputs back, all inside the timed region
  cpu_baseline  the fp64 oracle timed on this host's cores on a bounded sample
  sm_budget the same kernel held to 8 SMs

L2 (129 MB) is defeated by rotating through several buffer sets whose total
is above 3x the L2 size, so every step streams from HBM.

--impl reference times the oracle (the only reference this path has) on the
host cores instead.  --sweep adds the SM-budget sweep, the decode sweep, the
two-stream split and the fp32 column-split workload as extra fields.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused reduce+add+RMSNorm tokens/s and HBM GB/s (% of roofline) on 1 GB300"
HEADLINE = "tp8_t1024_h8192_bf16"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["tw", "reference"], default="tw")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (e.g. decode sizes)")
    ap.add_argument("--path", default="auto", choices=["auto", "rows", "warp", "cluster"],
                    help="kernel of the timed leg")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="add the GEMM / fused-kernel overlap measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# The sources that define the timed rows-kernel launch: the kernel with its
# launch plan (stage sizes, ring depth, producers), its device helpers and
# its parameters.
ROWS_KERNEL_SOURCES = ("tw_device.cuh", "tw_internal.h", "tw_rows.cu")


def code_only(text):
    """C/C++ source without comments and whitespace (string and character
    literals kept), so that edits to comments leave the hash unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            i = text.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash():
    """Hash of the rows kernel's code (comments and whitespace left out): a
    stored ncu traffic figure is only reported while it still describes the
    kernel being timed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "reduce_residual_rmsnorm_tw_gb300", "csrc")
    for name in ROWS_KERNEL_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + b"\0" + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(workload):
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][1]),
                "samples": len(rows), "power_w_max": max(float(r[2]) for r in rows
                                                         if r[2].strip() not in ("", "[N/A]")),
                "reasons": reasons}


# ------------------------------------------------------------ workloads ---
class Resident:
    """n_sets batches of a workload resident in HBM as ONE [n_sets * T, H]
    allocation per tensor; batch i is token range [i*T, (i+1)*T).  Rotating
    through the batches keeps every step streaming from HBM: the sets total
    more than 3x the L2 size."""

    def __init__(self, wl, min_sets=2):
        import torch
        from reduce_residual_rmsnorm_tw_gb300 import inputs
        l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or (132 << 20)
        per_set = wl.bytes_per_token() * wl.T
        self.n_sets = max(min_sets, -(-3 * l2 // per_set))
        self.l2_bytes = l2
        self.wl = wl
        self.big = wl.with_tokens(wl.T * self.n_sets)
        d = inputs.make_inputs(self.big, device="cuda")
        self.partials, self.residual, self.weight = d["partials"], d["residual"], d["weight"]
        self.out = [torch.empty_like(self.residual) for _ in range(wl.n_out)]
        self.residual_out = torch.empty_like(self.residual)

    def ranges(self):
        T = self.wl.T
        return [(i * T, (i + 1) * T) for i in range(self.n_sets)]

    def launchers(self, max_sms=None, path="auto"):
        from reduce_residual_rmsnorm_tw_gb300 import tw
        return [tw.prepare(self.partials, self.residual, self.weight, self.out,
                           self.residual_out, self.wl.eps, t0, t1, max_sms=max_sms, path=path)
                for t0, t1 in self.ranges()]

    def l2_note(self):
        total = self.wl.bytes_per_token() * self.big.T
        return (f"inputs larger than L2: {self.n_sets} rotating batches, "
                f"{total / 1e6:.0f} MB total vs {self.l2_bytes / 1e6:.0f} MB L2")


def time_launches(launchers, steps, warmup, stream, sync_ranks=None, per_launch=False):
    """Launch launchers[i % n] for warmup + steps steps on `stream` and time
    the steps with CUDA events around the region; the average launch is the
    region divided by the steps (the launches run back to back, each may
    overlap its start with the previous one's drain).  With per_launch=True
    every launch is also bracketed by its own events (a diagnostic: events
    between kernels add the launch gap to every step).
    Returns (region_ms, per_launch_ms list or None)."""
    import torch
    n = len(launchers)
    h = stream.cuda_stream
    torch.cuda.synchronize()  # inputs were drawn on the default stream
    with torch.cuda.stream(stream):
        for i in range(warmup):
            launchers[i % n](h)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if per_launch else None
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if per_launch else None
    begin = torch.cuda.Event(enable_timing=True)
    finish = torch.cuda.Event(enable_timing=True)
    if sync_ranks:
        sync_ranks()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("tw_timed")  # lets ncu --nvtx-include select this region
    with torch.cuda.stream(stream):
        begin.record(stream)
        if per_launch:
            for i in range(steps):
                starts[i].record(stream)
                launchers[(warmup + i) % n](h)
                ends[i].record(stream)
        else:
            for i in range(steps):
                launchers[(warmup + i) % n](h)
        finish.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if sync_ranks:
        sync_ranks()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)] if per_launch else None
    return begin.elapsed_time(finish), per


def graph_latency(launchers, reps=200):
    """Per-launch time of `reps` back-to-back launches replayed from one CUDA
    graph (no host launch overhead in the timed region)."""
    import torch
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(3):  # warm: per-device library state is set up outside capture
            launchers[i % len(launchers)](s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(reps):
            launchers[i % len(launchers)](h)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def summarize(per):
    ps = sorted(per)
    return {"mean_launch_ms": sum(ps) / len(ps), "median_launch_ms": ps[len(ps) // 2],
            "min_launch_ms": ps[0]}


def check_status():
    from reduce_residual_rmsnorm_tw_gb300 import tw
    status = tw.tw_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: a kernel gave up on a bounded wait")


def device_leg(res, steps, warmup, max_sms=None, path="auto", sync_ranks=None,
               per_launch=False):
    """Time the fused kernel on the resident batches of `res`: mean_launch_ms
    is the region over the steps; with per_launch, the per-launch event
    statistics are added under "events"."""
    import torch
    stream = torch.cuda.Stream()
    region_ms, per = time_launches(res.launchers(max_sms, path), steps, warmup, stream,
                                   sync_ranks, per_launch)
    check_status()
    out = {"region_ms": region_ms, "mean_launch_ms": region_ms / steps}
    if per is not None:
        out["events"] = summarize(per)
    return out


# ------------------------------------------------------------------ e2e ---
def e2e_leg(wl, steps, warmup, chunks=(64, 128, 256, 512), sync_ranks=None):
    """The same step from pinned HOST buffers through the C ABI's host entry
    point (tw_fused_reduce_add_rmsnorm_host): every step moves that step's
    inputs host->device, runs the kernel and moves the outputs back, with the
    copies of one token chunk overlapping the kernel on the previous chunk.
    Returns the best chunk's (ms per step, chunk) and all chunks' ms."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
    d = inputs.make_inputs(wl, device="cuda")
    h_parts = [p.cpu().pin_memory() for p in d["partials"]]
    h_res, h_w = d["residual"].cpu().pin_memory(), d["weight"].cpu().pin_memory()
    del d
    h_out = [torch.empty(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory() for _ in range(wl.n_out)]
    h_res_out = torch.empty(wl.T, wl.H, dtype=wl.torch_dtype).pin_memory()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    per_chunk = {}
    for chunk in chunks:
        ws = torch.empty(tw.tw_host_workspace_bytes(wl.n_parts, wl.n_out, wl.H, chunk,
                                                    wl.torch_dtype),
                         dtype=torch.uint8, device="cuda")

        def step():
            tw.tw_fused_reduce_add_rmsnorm_host(h_parts, h_res, h_w, h_out, h_res_out, wl.eps,
                                                ws, chunk, stream=stream)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        begin, finish = (torch.cuda.Event(enable_timing=True),
                         torch.cuda.Event(enable_timing=True))
        if sync_ranks:
            sync_ranks()
        begin.record(stream)
        for _ in range(steps):
            step()
        finish.record(stream)
        torch.cuda.synchronize()
        if sync_ranks:
            sync_ranks()
        per_chunk[chunk] = begin.elapsed_time(finish) / steps
        del ws
    check_status()
    best = min(per_chunk, key=per_chunk.get)
    es = wl.elem_bytes
    h2d = (wl.n_parts + 1) * wl.T * wl.H * es + wl.H * es
    d2h = (wl.n_out + 1) * wl.T * wl.H * es
    return per_chunk[best], best, per_chunk, h2d, d2h


# ---------------------------------------------------------- CPU oracle ---
def oracle_sample(wl, n_tokens):
    """fp64 inputs of the first n_tokens tokens of the workload (CPU draw)."""
    from reduce_residual_rmsnorm_tw_gb300 import inputs
    d = inputs.make_inputs(wl.with_tokens(n_tokens), device="cpu")
    return ([inputs.to_f64(p) for p in d["partials"]], inputs.to_f64(d["residual"]),
            inputs.to_f64(d["weight"]))


def host_cores():
    """Cores this process may run on (torchrun's OMP_NUM_THREADS=1 aside)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, seconds, threads=None):
    """The oracle (reordered order, fp64, as it stands) on this host's cores
    (or `threads` of them), repeated on a bounded sample of the workload for
    about `seconds`."""
    import oracle
    oracle.set_threads(threads or host_cores())
    n_tok = min(wl.T, 64)
    parts, res, w = oracle_sample(wl, n_tok)
    oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)  # build + warm
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)
        runs += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= seconds:
            break
    return {"value": runs * n_tok / elapsed, "unit": "tokens/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"first {n_tok} tokens of {wl.name}, fp64 reordered order, "
                      f"{runs} runs in {elapsed:.1f} s"}


def reference_main(args):
    """--impl reference: the oracle timed on the host cores, one bounded
    sample of the workload per step, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import oracle
    from reduce_residual_rmsnorm_tw_gb300.inputs import WORKLOADS
    oracle.set_threads(host_cores())
    wl = WORKLOADS[args.workload]
    if args.tokens is not None:
        wl = wl.with_tokens(args.tokens)
    calib_tok = min(wl.T, 16)
    parts, res, w = oracle_sample(wl, calib_tok)
    oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)
    t0 = time.perf_counter()
    oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)
    per_tok = (time.perf_counter() - t0) / calib_tok
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_tok = int(max(1, min(wl.T, budget / max(per_tok, 1e-9))))
    parts, res, w = oracle_sample(wl, n_tok)
    for _ in range(args.warmup):
        oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.reordered(parts, res, w, wl.eps, n_out=wl.n_out)
    elapsed = time.perf_counter() - t0
    value = args.steps * n_tok / elapsed
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "n_parts": wl.n_parts, "T": wl.T, "H": wl.H,
                       "n_out": wl.n_out, "eps": wl.eps,
                       "step": f"{n_tok} tokens of the batch per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle",
                             "cores": oracle.threads(),
                             "sample": f"{n_tok} of {wl.T} tokens per step, fp64 "
                                       "reordered order"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- sweep ---
def sweep(args, sync_ranks):
    """SM-budget sweep, decode sweep, fp32 column split, the two-stream split
    and the same tokens as one launch, the unfused torch chain, and the oracle
    on one host thread and on all cores."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
    W = inputs.WORKLOADS
    peak, _ = measured_peaks()
    out = {}

    def entry(wl, ms):
        gbs = wl.bytes_per_token() * wl.T / (ms * 1e-3) / 1e9
        return {"launch_us": round(ms * 1e3, 2), "tokens_per_s": wl.T / (ms * 1e-3),
                "gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4)}

    steps = max(50, min(args.steps, 2000))
    for name in (HEADLINE, "tp2_t2048_h4096_bf16"):
        res = Resident(W[name])
        out[f"sm_budget:{name}"] = {
            str(b): entry(res.wl, device_leg(res, steps, 20, max_sms=b)["mean_launch_ms"])
            for b in (2, 4, 8, 16, 148, 10 ** 6)}
        del res
    dec = {}
    for T in sorted(set(inputs.DECODE_TOKENS) | {12, 16, 24, 32, 48, 96, 128}):
        res = Resident(W["decode_tp8_h8192_bf16"].with_tokens(T))
        dec[str(T)] = {path: entry(res.wl, graph_latency(res.launchers(path=path)))
                       for path in ("warp", "cluster", "rows", "auto")}
        del res
    out["decode_tp8_h8192_bf16"] = dec
    out["decode_note"] = ("per-launch time of 200 back-to-back launches replayed from one "
                          "CUDA graph, rotating resident batches")
    # fp32 column split, four destinations: the dense read of all N zero-padded
    # partials, and the column-split mode that reads each rank's slice only
    # (GB/s counted against the dense algorithmic bytes; the column-split
    # algorithmic bytes per token are (1 + 1 + n_out + 1) * H * 4).
    res = Resident(W["colsplit_tp4_t8192_h5120_f32_out4"])
    cs = {}
    for mode in ("auto", "colsplit"):
        ms = device_leg(res, max(20, steps // 20), 5, path=mode)["mean_launch_ms"]
        cs["dense" if mode == "auto" else "colsplit"] = entry(res.wl, ms)
    wl = res.wl
    cs_bytes = (1 + 1 + wl.n_out + 1) * wl.H * wl.elem_bytes * wl.T
    cs["colsplit"]["colsplit_gbs"] = round(cs_bytes / (cs["colsplit"]["launch_us"] * 1e-6) / 1e9, 1)
    cs["colsplit"]["colsplit_frac_of_measured_hbm"] = round(cs["colsplit"]["colsplit_gbs"] / peak, 4)
    out["colsplit_tp4_t8192_h5120_f32_out4"] = cs
    del res
    # Two-chunk split on two streams (fork/join inside the library).
    wl = W["split_tp8_t16384_h8192_bf16"]
    res = Resident(wl)
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    split = {}
    for b in (2, 4, 8, 16, 148):
        n_rep = 3 if b <= 4 else 20
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for rep in range(n_rep + 1):
            if rep == 1:
                evs[0].record(s0)
            t0, t1 = res.ranges()[rep % res.n_sets]
            parts = [p[t0:t1] for p in res.partials]
            tw.tw_split_launch(parts, res.residual[t0:t1], res.weight,
                               [o[t0:t1] for o in res.out], res.residual_out[t0:t1],
                               wl.eps, t_split=-1, max_sms=b, s0=s0, s1=s1)
        evs[1].record(s0)
        torch.cuda.synchronize()
        split[str(b)] = entry(wl, evs[0].elapsed_time(evs[1]) / n_rep)
    check_status()
    out["split_tp8_t16384_h8192_bf16"] = split
    # The same 16 384 tokens as one launch at the same budgets.
    out["single_launch:split_tp8_t16384_h8192_bf16"] = {
        str(b): entry(wl, device_leg(res, 3 if b <= 4 else 20, 2, max_sms=b)["mean_launch_ms"])
        for b in (2, 4, 8, 16, 148)}
    del res
    out["flags_raised:" + HEADLINE] = flags_leg(W[HEADLINE], steps)
    out["unfused_torch_chain"] = unfused_leg(W[HEADLINE], steps)
    out["oracle_threads"] = {str(n): cpu_baseline(W[HEADLINE], 5.0, threads=n)
                             for n in (1, host_cores())}
    return out


def flags_leg(wl, steps):
    """The readiness-flag entry point with every flag already raised (one
    flag per token, and one per 64 tokens) against the plain launch: the cost
    of checking the flags, and of giving up the L2 warming that flag launches
    do not do (their rows may not exist before the flag)."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import tw
    res = Resident(wl)
    peak, _ = measured_peaks()
    stream = torch.cuda.Stream()
    out = {}

    def entry(ms):
        gbs = wl.bytes_per_token() * wl.T / (ms * 1e-3) / 1e9
        return {"launch_us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                "frac_of_measured_hbm": round(gbs / peak, 4)}

    region, _ = time_launches(res.launchers(), steps, 20, stream)
    out["plain"] = entry(region / steps)
    for bt in (1, 64):
        ready = torch.ones(-(-res.big.T // bt), dtype=torch.int32, device="cuda")
        launchers = [tw.prepare(res.partials, res.residual, res.weight, res.out,
                                res.residual_out, wl.eps, t0, t1, ready=ready,
                                block_tokens=bt, epoch=1) for t0, t1 in res.ranges()]
        region, _ = time_launches(launchers, steps, 20, stream)
        out[f"flags_block_{bt}"] = entry(region / steps)
    check_status()
    del res
    torch.cuda.empty_cache()
    return out


def unfused_leg(wl, steps):
    """Context comparator: the unfused chain the fused step replaces, in
    plain torch ops (a stacked sum of the partials, the residual add, then
    torch's RMSNorm), on the same rotating resident batches.  GB/s is counted
    with the fused step's algorithmic bytes, so it compares times."""
    import torch
    import torch.nn.functional as F
    res = Resident(wl)
    peak, _ = measured_peaks()
    stream = torch.cuda.Stream()

    def step(i):
        t0, t1 = res.ranges()[i % res.n_sets]
        x = torch.stack([p[t0:t1] for p in res.partials]).sum(0) + res.residual[t0:t1]
        res.residual_out[t0:t1] = x
        res.out[0][t0:t1] = F.rms_norm(x, (wl.H,), res.weight, wl.eps)

    n = max(20, steps // 10)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    gbs = wl.bytes_per_token() * wl.T / (ms * 1e-3) / 1e9
    del res
    torch.cuda.empty_cache()
    return {"workload": wl.name, "step_us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4),
            "chain": "torch.stack(partials).sum(0) + residual; rms_norm(x, weight, eps); "
                     "copies into residual_out and out"}


# --------------------------------------------------------------- overlap ---
def overlap_leg(budgets=(2, 4, 8, 16, 32), gemm_reps=20):
    """The pages' overlap claim on one GPU ("Der intelligente Split", "Der
    Fused Kernel"): a compute-bound bf16 GEMM (torch.matmul, cuBLAS) on one
    stream while the fused kernel, held to a few SMs, runs on a second,
    higher-priority stream.  Reports the GEMM's slowdown and the fused
    kernel's throughput alone and under overlap, and a two-chunk layer step
    (GEMM(A); GEMM(B) beside fused(A); fused(B)) against the sequential order
    (GEMM(A+B); fused(A+B)), the GEMM writing partial 0 of each chunk."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
    W = inputs.WORKLOADS
    peak, _ = measured_peaks()
    res = Resident(W[HEADLINE])
    wl = res.wl
    M = N_ = K = 8192
    a = torch.randn(M, K, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(K, N_, device="cuda", dtype=torch.bfloat16)
    c = torch.empty(M, N_, device="cuda", dtype=torch.bfloat16)
    g = torch.cuda.Stream()
    f = torch.cuda.Stream(priority=-1)
    torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def gemms(n):
        with torch.cuda.stream(g):
            for _ in range(n):
                torch.matmul(a, b, out=c)

    gemms(3)
    e0, e1 = ev(), ev()
    e0.record(g)
    gemms(gemm_reps)
    e1.record(g)
    torch.cuda.synchronize()
    gemm_ms = e0.elapsed_time(e1) / gemm_reps
    out = {"gemm": {"shape": [M, N_, K], "ms": round(gemm_ms, 4),
                    "tflops": round(2 * M * N_ * K / (gemm_ms * 1e-3) / 1e12, 1)}}
    bytes_launch = wl.bytes_per_token() * wl.T
    for bud in budgets:
        launchers = res.launchers(max_sms=bud)
        alone = device_leg(res, 10, 3, max_sms=bud)["mean_launch_ms"]
        n_fused = max(2, int(gemm_reps * gemm_ms / alone))
        gemms(2)
        g0, g1, f0, f1 = ev(), ev(), ev(), ev()
        g0.record(g)
        gemms(gemm_reps)
        g1.record(g)
        f0.record(f)
        for i in range(n_fused):
            launchers[i % len(launchers)](f.cuda_stream)
        f1.record(f)
        torch.cuda.synchronize()
        gemm_ov = g0.elapsed_time(g1) / gemm_reps
        fused_ov = f0.elapsed_time(f1) / n_fused
        out[str(bud)] = {
            "fused_alone_us": round(alone * 1e3, 1), "fused_overlap_us": round(fused_ov * 1e3, 1),
            "fused_overlap_gbs": round(bytes_launch / (fused_ov * 1e-3) / 1e9, 1),
            "gemm_overlap_ms": round(gemm_ov, 4), "gemm_slowdown": round(gemm_ov / gemm_ms, 4)}
    check_status()
    del res, a, b, c
    torch.cuda.empty_cache()

    # Two-chunk layer step on the 16384-token batch: the GEMM of each chunk
    # writes that chunk's rows of partial 0, the fused step reads them.
    wl = W["split_tp8_t16384_h8192_bf16"]
    d = inputs.make_inputs(wl, device="cuda")
    o = [torch.empty_like(d["residual"])]
    ro = torch.empty_like(d["residual"])
    x = torch.randn(wl.T, 8192, device="cuda", dtype=torch.bfloat16)
    wmat = torch.randn(8192, wl.H, device="cuda", dtype=torch.bfloat16) * 0.01
    half = wl.T // 2
    torch.cuda.synchronize()

    def fused(t0, t1, budget, stream):
        tw.tw_fused_reduce_add_rmsnorm(d["partials"], d["residual"], d["weight"], o, ro,
                                       wl.eps, t0, t1, max_sms=budget, stream=stream)

    def sequential():
        with torch.cuda.stream(g):
            torch.matmul(x, wmat, out=d["partials"][0])
            fused(0, wl.T, None, g)

    def two_chunk(budget):
        done_a, done_b = torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(g):
            torch.matmul(x[:half], wmat, out=d["partials"][0][:half])
            done_a.record(g)
            torch.matmul(x[half:], wmat, out=d["partials"][0][half:])
            done_b.record(g)
        f.wait_event(done_a)
        fused(0, half, budget, f)
        f.wait_event(done_b)
        fused(half, wl.T, None, f)
        g.wait_stream(f)

    def timed(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        s0, s1 = ev(), ev()
        s0.record(g)
        for _ in range(reps):
            fn()
        s1.record(g)
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / reps

    layer = {"sequential_ms": round(timed(sequential), 4)}
    for bud in (8, 16, 32, 48, 64):
        layer[f"two_chunk_budget_{bud}_ms"] = round(timed(lambda: two_chunk(bud)), 4)
    check_status()
    out["layer_step_t16384"] = layer
    return out


# ------------------------------------------------------------------ main ---
def max_over_ranks(values, world):
    """Element-wise max of a list of floats over all ranks (host-side gloo
    all-reduce; the data path itself has no collective)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tokens_per_s(world, tokens_per_step, steps, max_region_ms):
    """Replicas: every rank processes its own batch each step (weak scaling)."""
    return world * tokens_per_step * steps / (max_region_ms * 1e-3)


def tw_main(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    # One GPU per rank; with fewer GPUs than ranks, replicas share them.
    device = local_rank % max(1, torch.cuda.device_count())
    torch.cuda.set_device(device)
    sync_ranks = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # host-side barrier and timing reduce only
        sync_ranks = dist.barrier
    if rank == 0:
        from reduce_residual_rmsnorm_tw_gb300 import build as twbuild
        twbuild.build()
    if sync_ranks:
        sync_ranks()
    from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
    tw.load()
    wl = inputs.WORKLOADS[args.workload]
    if args.tokens is not None:
        wl = wl.with_tokens(args.tokens)
    res = Resident(wl)
    l2_note = res.l2_note()

    sampler = ClockSampler(device) if rank == 0 else None
    dev = device_leg(res, args.steps, args.warmup, path=args.path, sync_ranks=sync_ranks)
    clocks = sampler.stop() if sampler else None

    region_ms, launch_ms = max_over_ranks([dev["region_ms"], dev["mean_launch_ms"]], world)
    value = whole_job_tokens_per_s(world, wl.T, args.steps, region_ms)
    peak, peak_kind = measured_peaks()
    algo_bytes = wl.bytes_per_token() * wl.T
    achieved = algo_bytes / (launch_ms * 1e-3) / 1e9

    diag = device_leg(res, min(args.steps, 2000), 20, path=args.path, per_launch=True)["events"]
    sm8 = device_leg(res, max(50, min(args.steps, 2000)), 20, max_sms=8, path=args.path)
    sm8_gbs = algo_bytes / (sm8["mean_launch_ms"] * 1e-3) / 1e9
    del res
    torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(10, min(100, args.steps // 200))
        step_ms, chunk, per_chunk, h2d, d2h = e2e_leg(wl, e2e_steps, 3, sync_ranks=sync_ranks)
        (step_ms,) = max_over_ranks([step_ms], world)
        e2e = {"value": whole_job_tokens_per_s(world, wl.T, 1, step_ms),
               "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "ms_per_step": round(step_ms, 4),
               "link_gbs": round((h2d + d2h) / (step_ms * 1e-3) / 1e9, 1),
               "chunk_tokens": chunk,
               "ms_per_step_by_chunk": {str(k): round(v, 4) for k, v in per_chunk.items()},
               "path": "tw_fused_reduce_add_rmsnorm_host: pinned host buffers, "
                       "chunked host->device copies overlapping the kernel on the previous "
                       "chunk, which stores its results straight into the mapped host "
                       "outputs (device->host copies where they are not mapped)"}
    extra = sweep(args, None) if args.sweep and rank == 0 else None
    overlap = overlap_leg() if args.overlap and rank == 0 else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "n_parts": wl.n_parts, "T": wl.T, "H": wl.H,
                   "n_out": wl.n_out, "eps": wl.eps, "l2": l2_note, "path": args.path,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "sm_count": torch.cuda.get_device_properties(device).multi_processor_count},
        "hbm_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": stored_traffic(wl.name), "peak_kind": peak_kind,
                     "frac_of_8tbs": round(achieved / 8000.0, 4),
                     "algorithmic_bytes_per_launch": algo_bytes,
                     "mean_launch_us": round(launch_ms * 1e3, 2),
                     "launch_timing": "timed-region events over back-to-back launches "
                                      "divided by the steps",
                     "events_per_launch_us": {
                         "mean": round(diag["mean_launch_ms"] * 1e3, 2),
                         "median": round(diag["median_launch_ms"] * 1e3, 2),
                         "min": round(diag["min_launch_ms"] * 1e3, 2),
                         "note": "diagnostic pass with an event pair around every launch "
                                 "(adds the launch gap, disables launch overlap)"}},
        "sm_budget_8": {"tokens_per_s": wl.T / (sm8["mean_launch_ms"] * 1e-3),
                        "gbs": round(sm8_gbs, 1), "frac": round(sm8_gbs / peak, 4)},
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps, "clocks": clocks,
    }
    if extra is not None:
        line["sweep"] = extra
    if overlap is not None:
        line["overlap"] = overlap
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return reference_main(args)
    return tw_main(args)


if __name__ == "__main__":
    sys.exit(main())
