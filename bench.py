"""Benchmark of the fused reduce + residual add + RMSNorm step on GB300.

One step = one launch of the fused kernel over one batch of the headline
workload (N=8 dense row-parallel bf16 partials, T=1024 tokens, H=8192), with
inputs already resident in HBM.  Prints ONE JSON line (rank 0):

  value     tokens/s over all ranks (device time, CUDA events, max over ranks)
  roofline  achieved algorithmic GB/s of the kernel vs the measured HBM copy
            peak; algorithmic bytes per token = (N + 1 + n_out + 1) * H * 2;
            also the launch right after a different kernel (no launch of the
            fused kernel before it to overlap with)
  e2e       the same metric through the C ABI with pinned HOST buffers: every
            step copies its inputs host->device, runs the kernel and copies the
            outputs back, all inside the timed region
  cpu_baseline  the fp64 oracle timed on this host's cores on a bounded sample
  configs   every benchmark workload: the SM-budget sweep (2/4/8/16/148 and
            the whole GPU) of the headline and of the 16384-token two-stream
            split, the N=2 workload, the decode sizes on every kernel, the fp32
            column split (dense read and column-split mode), the split
            workload as one launch, the unfused torch chain
  overlap   the fused kernel on a few SMs beside a bf16 GEMM, and the
            two-chunk layer step
  flags     readiness flags raised before the launch, and a live producer
  clocks    nvidia-smi samples across every GPU leg of the run

L2 (129 MB) is defeated by rotating through several buffer sets whose total
is above 3x the L2 size, so every step streams from HBM.

--impl reference times the oracle (the only reference this path has) on the
host cores instead.  --sweep adds the oracle on one thread and on all cores;
--overlap the full GEMM-overlap sweep; --no-extra keeps only the headline,
e2e and CPU legs.
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
    ap.add_argument("--max-sms", type=int, default=None,
                    help="SM budget of the timed leg (default: the whole GPU)")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="add the GEMM / fused-kernel overlap measurement")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload, overlap and flag legs")
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
                 "--format=csv,noheader,nounits", "-lms", "50"],
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
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        power = [num(r[2]) for r in rows if num(r[2]) is not None]
        if not sm:
            return None
        # Samples under load: power at least 1.5x the lowest sample (idle
        # moments between legs are left out of the median).
        loaded = [num(r[0]) for r in rows if num(r[0]) is not None and num(r[2]) is not None
                  and power and num(r[2]) >= 1.5 * min(power)]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(loaded or sm), "sm_mhz_all_samples":
                statistics.median(sm), "sm_max_mhz": num(rows[0][1]), "samples": len(rows),
                "samples_under_load": len(loaded), "power_w_max": max(power) if power else None,
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
    the steps with CUDA events around the region (a spin kernel queued just
    before the start event covers the host's enqueue time); the average
    launch is the region divided by the steps (the launches run back to back,
    each may overlap its start with the previous one's drain).  With
    per_launch=True every launch is also bracketed by its own events (a
    diagnostic: events between kernels add the launch gap to every step).
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
        # A ~50 us spin ahead of the start event keeps the stream busy while
        # the host enqueues the event and the first launches, so the region
        # holds device time only (not the host's time to issue the first
        # launch).  The first timed launch still follows a foreign kernel.
        torch.cuda._sleep(100_000)
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
def e2e_leg(wl, steps, warmup, chunks=(0, 128, 256, 512), sync_ranks=None):
    """The same step from pinned HOST buffers through the C ABI's host entry
    point (tw_fused_reduce_add_rmsnorm_host): every step moves that step's
    inputs host->device, runs the kernel and moves the outputs back.  Chunk 0:
    one kernel reads the host tensors in place over the host link and stores
    straight into the host outputs; chunks >= 1: host->device copies of one
    token chunk overlap the kernel on the previous chunk.  Returns the best
    chunk's (ms per step, chunk) and all chunks' ms."""
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
        ws = None if chunk == 0 else torch.empty(
            tw.tw_host_workspace_bytes(wl.n_parts, wl.n_out, wl.H, chunk, wl.torch_dtype),
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


# -------------------------------------------------------- workload legs ---
def rate(wl, ms, peak, tokens=None, bytes_per_token=None):
    """Time per launch, tokens/s and algorithmic GB/s (fraction of `peak`)."""
    tokens = wl.T if tokens is None else tokens
    bpt = wl.bytes_per_token() if bytes_per_token is None else bytes_per_token
    gbs = bpt * tokens / (ms * 1e-3) / 1e9
    return {"launch_us": round(ms * 1e3, 2), "tokens_per_s": round(tokens / (ms * 1e-3)),
            "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}


def budget_steps(max_sms):
    """Launches per budget point: about 20 ms of work at the small budgets."""
    if max_sms is None or max_sms >= 16:
        return 200
    return 20


def budget_sweep(res, peak, budgets):
    """The same launches held to each SM budget (None: the whole GPU, whose
    launches may overlap the previous one's drain)."""
    out = {}
    for b in budgets:
        ms = device_leg(res, budget_steps(b), 3, max_sms=b)["mean_launch_ms"]
        out["all" if b is None else str(b)] = rate(res.wl, ms, peak)
    return out


def after_foreign_leg(res, peak, steps=200, spin_cycles=40000, gemm_k=8192):
    """The headline launch right after a DIFFERENT kernel, so that it cannot
    overlap the drain of a previous launch of itself: the region of `steps`
    pairs [foreign kernel, fused launch] minus the region of the foreign
    kernels alone, per step.  Two foreign kernels: a one-thread spin that
    touches no memory (the fused launch starts on an idle memory system),
    and a bf16 GEMM that writes partial 0 of the batch the fused launch then
    reads (the row-parallel linear layer before it).  Each region is timed
    twice, alternating, and the smaller is kept."""
    import torch
    stream = torch.cuda.Stream()
    launchers = res.launchers()
    n = len(launchers)
    h = stream.cuda_stream
    wl = res.wl
    x = torch.randn(wl.T, gemm_k, device="cuda", dtype=torch.bfloat16)
    wmat = torch.randn(gemm_k, wl.H, device="cuda", dtype=torch.bfloat16) * (1.0 / gemm_k) ** 0.5
    ranges = res.ranges()

    def spin(i):
        torch.cuda._sleep(spin_cycles)

    def gemm(i):
        t0, t1 = ranges[i % n]
        torch.matmul(x, wmat, out=res.partials[0][t0:t1])

    def region(foreign, with_fused):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(5):
                foreign(i)
                if with_fused:
                    launchers[i % n](h)
            e0.record(stream)
            for i in range(steps):
                foreign(i)
                if with_fused:
                    launchers[i % n](h)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    out = {}
    for name, foreign in (("spin", spin), ("gemm", gemm)):
        both = min(region(foreign, True), region(foreign, True))
        alone = min(region(foreign, False), region(foreign, False))
        e = rate(wl, both - alone, peak)
        e["foreign_us"] = round(alone * 1e3, 2)
        out[name] = e
    check_status()
    del x, wmat
    return out


def decode_leg(W, peak, tokens=(1, 8, 12, 16, 24, 32, 48, 64, 96, 128, 256)):
    """Decode-size ranges on every kernel: per-launch time of 200 launches
    replayed from one CUDA graph."""
    dec = {}
    for T in tokens:
        res = Resident(W["decode_tp8_h8192_bf16"].with_tokens(T))
        dec[str(T)] = {path: round(graph_latency(res.launchers(path=path)) * 1e3, 2)
                       for path in ("auto", "warp", "cluster", "rows")}
        del res
    return {"latency_us": dec,
            "note": "per-launch time of 200 back-to-back launches replayed from one CUDA "
                    "graph, rotating resident batches; auto is the library's choice"}


def split_leg(wl, peak, budgets):
    """tw_split_launch (the two-chunk split on two streams, default split
    point) at each budget per chunk, and the same tokens as one launch."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import tw
    res = Resident(wl)
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    split = {}
    for b in budgets:
        n_rep = 3 if b is not None and b <= 4 else 10
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for rep in range(n_rep + 1):
            if rep == 1:
                evs[0].record(s0)
            t0, t1 = res.ranges()[rep % res.n_sets]
            tw.tw_split_launch([p[t0:t1] for p in res.partials], res.residual[t0:t1],
                               res.weight, [o[t0:t1] for o in res.out], res.residual_out[t0:t1],
                               wl.eps, t_split=-1, max_sms=b, s0=s0, s1=s1)
        evs[1].record(s0)
        torch.cuda.synchronize()
        split["all" if b is None else str(b)] = rate(wl, evs[0].elapsed_time(evs[1]) / n_rep, peak)
    check_status()
    single = {}
    for b in budgets:
        steps = 3 if b is not None and b <= 4 else 10
        ms = device_leg(res, steps, 2, max_sms=b)["mean_launch_ms"]
        single["all" if b is None else str(b)] = rate(wl, ms, peak)
    del res
    return {"tw_split_launch": split, "one_launch": single,
            "note": "budget per chunk for tw_split_launch (both chunks run at once: up to "
                    "twice the budget while both run); budget per launch for one_launch"}


def colsplit_leg(wl, peak):
    """fp32 zero-padded column split, four destinations: the dense read of
    all N partials, and the column-split mode that reads each rank's slice
    only (its own algorithmic bytes per token: (1 + 1 + n_out + 1) * H * 4)."""
    res = Resident(wl)
    out = {}
    for mode in ("auto", "colsplit"):
        ms = device_leg(res, 20, 3, path=mode)["mean_launch_ms"]
        out["dense" if mode == "auto" else "colsplit"] = rate(wl, ms, peak)
    own = (1 + 1 + wl.n_out + 1) * wl.H * wl.elem_bytes
    c = out["colsplit"]
    c["own_bytes_per_token"] = own
    c["own_gbs"] = round(own * wl.T / (c["launch_us"] * 1e-6) / 1e9, 1)
    c["own_frac"] = round(c["own_gbs"] / peak, 4)
    del res
    return out


def configs_leg(peak):
    """Every benchmark workload: budgets, decode sizes, split, column split."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs
    W = inputs.WORKLOADS
    budgets = list(inputs.SM_BUDGETS) + [None]
    out = {}
    for name in (HEADLINE, "tp2_t2048_h4096_bf16"):
        res = Resident(W[name])
        out[name] = {"sm_budget": budget_sweep(res, peak, budgets)}
        del res
        torch.cuda.empty_cache()
    out["decode_tp8_h8192_bf16"] = decode_leg(W, peak)
    out["split_tp8_t16384_h8192_bf16"] = split_leg(W["split_tp8_t16384_h8192_bf16"], peak, budgets)
    torch.cuda.empty_cache()
    out["colsplit_tp4_t8192_h5120_f32_out4"] = colsplit_leg(W["colsplit_tp4_t8192_h5120_f32_out4"],
                                                            peak)
    torch.cuda.empty_cache()
    out["unfused_torch_chain"] = unfused_leg(W[HEADLINE], 200)
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
    region, _ = time_launches(res.launchers(), steps, 20, stream)
    out["plain"] = rate(wl, region / steps, peak)
    for bt in (1, 64):
        ready = torch.ones(-(-res.big.T // bt), dtype=torch.int32, device="cuda")
        launchers = [tw.prepare(res.partials, res.residual, res.weight, res.out,
                                res.residual_out, wl.eps, t0, t1, ready=ready,
                                block_tokens=bt, epoch=1) for t0, t1 in res.ranges()]
        region, _ = time_launches(launchers, steps, 20, stream)
        out[f"raised_block_{bt}"] = rate(wl, region / steps, peak)
    check_status()
    del res
    torch.cuda.empty_cache()
    out["live_producer"] = flags_live_leg(wl)
    return out


def flags_live_leg(wl, block_tokens=64, budgets=(8, 32), gap_cycles=20000):
    """A live producer: a second stream copies one block of 64 tokens' partial
    and residual rows at a time into the buffers the consumer reads, raises
    the block's flag with tw_set_ready and pauses (a spin of `gap_cycles`);
    the consumer (tw_fused_reduce_add_rmsnorm_flags) was launched first, on a
    budget that leaves SMs free for the producer.  Reports the producer's
    span from its first copy to its last flag, the consumer's span from launch
    to end, and how long the consumer ran after the last flag rose.  A
    consumer wait that ran out (status word nonzero) is reported, and the
    word cleared, rather than raised."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs, tw
    src = inputs.make_inputs(wl, device="cuda")
    src_t = src["partials"] + [src["residual"]]
    dst = [torch.empty_like(t) for t in src_t]
    out_t = [torch.empty_like(src["residual"]) for _ in range(wl.n_out)]
    res_out = torch.empty_like(src["residual"])
    n_blocks = -(-wl.T // block_tokens)
    ready = torch.zeros(n_blocks, dtype=torch.int32, device="cuda")
    consumer, producer = torch.cuda.Stream(), torch.cuda.Stream()
    # The producer's kernels run once before any consumer waits (a kernel's
    # first launch may load it, and a load can wait for running kernels).
    with torch.cuda.stream(producer):
        torch.cuda._sleep(10)
        dst[0][:1].copy_(src_t[0][:1])
        tw.tw_set_ready(ready, 0, first_block=0, n_blocks=1, stream=producer)
    torch.cuda.synchronize()
    result = {}
    epoch = 0
    for b_sms in budgets:
        spans = []
        for rep in range(3):
            epoch += 1
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[0].record(consumer)
            tw.tw_fused_reduce_add_rmsnorm_flags(dst[:-1], dst[-1], src["weight"], out_t, res_out,
                                                 wl.eps, ready, block_tokens, epoch,
                                                 max_sms=b_sms, stream=consumer)
            ev[1].record(consumer)
            with torch.cuda.stream(producer):
                torch.cuda._sleep(100000)
                ev[2].record(producer)
                for b in range(n_blocks):
                    rows = slice(b * block_tokens, min((b + 1) * block_tokens, wl.T))
                    for d_t, s_t in zip(dst, src_t):
                        d_t[rows].copy_(s_t[rows])
                    tw.tw_set_ready(ready, epoch, first_block=b, n_blocks=1, stream=producer)
                    if b + 1 < n_blocks:
                        torch.cuda._sleep(gap_cycles)
                ev[3].record(producer)
            torch.cuda.synchronize()
            spans.append((ev[2].elapsed_time(ev[3]), ev[0].elapsed_time(ev[1]),
                          ev[3].elapsed_time(ev[1])))
        status = tw.tw_device_status(clear=True)
        prod, cons, tail = min(spans, key=lambda x: x[1])
        result[str(b_sms)] = {
            "producer_ms": round(prod, 4), "consumer_ms": round(cons, 4),
            "consumer_after_last_flag_us": round(tail * 1e3, 1), "device_status": status}
    result["note"] = (f"{n_blocks} blocks of {block_tokens} tokens; budget per consumer "
                      f"launch; producer pauses {gap_cycles} cycles between blocks")
    del src, dst, out_t, res_out
    torch.cuda.empty_cache()
    return result


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
    del res
    torch.cuda.empty_cache()
    e = rate(wl, ms, peak)
    e["chain"] = ("torch.stack(partials).sum(0) + residual; rms_norm(x, weight, eps); "
                  "copies into residual_out and out")
    return e


# --------------------------------------------------------------- overlap ---
def overlap_leg(budgets=(8,), layer_budgets=(16, 48), gemm_reps=20):
    """The pages' overlap claim on one GPU ("Der intelligente Split", "Der
    Fused Kernel"): a compute-bound bf16 GEMM (torch.matmul, cuBLAS) on one
    stream while the fused kernel, held to a few SMs, runs on a second,
    higher-priority stream.  Reports the GEMM's slowdown and the fused
    kernel's throughput alone and under overlap, and the two-chunk layer
    step (layer_step.two_chunk_layer_step) against the sequential order."""
    import torch
    from reduce_residual_rmsnorm_tw_gb300 import inputs, layer_step
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
        out[f"fused_{bud}_sms_beside_gemm"] = {
            "fused_alone": rate(wl, alone, peak), "fused_beside_gemm": rate(wl, fused_ov, peak),
            "gemm_beside_fused_ms": round(gemm_ov, 4), "gemm_slowdown": round(gemm_ov / gemm_ms, 4)}
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
    torch.cuda.synchronize()
    args = (x, wmat, d["partials"], d["residual"], d["weight"], o, ro, wl.eps)

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

    layer = {"sequential_ms": round(timed(lambda: layer_step.sequential_layer_step(*args, g)), 4)}
    for bud in layer_budgets:
        layer[f"two_chunk_budget_{bud}_ms"] = round(
            timed(lambda: layer_step.two_chunk_layer_step(*args, bud, g, f)), 4)
    check_status()
    out["layer_step_t16384"] = layer
    del d, o, ro, x, wmat
    torch.cuda.empty_cache()
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
    # Clocks are sampled from before the first launch to after the last GPU
    # leg, so that even a short timed region is covered.
    sampler = ClockSampler(device) if rank == 0 else None
    res = Resident(wl)
    l2_note = res.l2_note()
    peak, peak_kind = measured_peaks()

    dev = device_leg(res, args.steps, args.warmup, max_sms=args.max_sms, path=args.path,
                     sync_ranks=sync_ranks)
    region_ms, launch_ms = max_over_ranks([dev["region_ms"], dev["mean_launch_ms"]], world)
    value = whole_job_tokens_per_s(world, wl.T, args.steps, region_ms)
    algo_bytes = wl.bytes_per_token() * wl.T
    achieved = algo_bytes / (launch_ms * 1e-3) / 1e9

    extra = not args.no_extra and rank == 0
    diag = device_leg(res, max(20, min(args.steps, 2000)), 20, path=args.path,
                      per_launch=True)["events"]
    sm8 = device_leg(res, max(50, min(args.steps, 200)), 20, max_sms=8, path=args.path)
    sm8_gbs = algo_bytes / (sm8["mean_launch_ms"] * 1e-3) / 1e9
    foreign = after_foreign_leg(res, peak) if extra else None
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
               "path": "tw_fused_reduce_add_rmsnorm_host on pinned host buffers: chunk 0 = "
                       "one kernel reading the host tensors in place over the host link and "
                       "storing into the host outputs; chunks >= 1 = host->device copies of "
                       "one chunk overlapping the kernel on the previous chunk"}
    configs = configs_leg(peak) if extra else None
    overlap = overlap_leg() if extra else None
    if args.overlap and rank == 0:
        overlap = overlap_leg(budgets=(2, 4, 8, 16, 32), layer_budgets=(8, 16, 32, 48, 64))
    flags = flags_leg(inputs.WORKLOADS[HEADLINE], 200) if extra else None
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if clocks:
        clocks["note"] = "nvidia-smi every 50 ms from before the first launch to after the last GPU leg"
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)
    threads = None
    if args.sweep and rank == 0:
        threads = {str(n): cpu_baseline(inputs.WORKLOADS[HEADLINE], 5.0, threads=n)
                   for n in (1, host_cores())}
    if rank != 0:
        return 0
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
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
                            "(adds the launch gap, disables launch overlap)"}}
    if foreign:
        # Strict case: after a kernel that shares nothing with it.  After the
        # GEMM a layer runs before this step the figure is a marginal time
        # (part of the launch overlaps the GEMM's end and the GEMM's output,
        # partial 0, is partly read from L2), not a bandwidth.
        roofline["frac_after_foreign_kernel"] = foreign["spin"]["frac"]
        roofline["frac_after_gemm_marginal"] = foreign["gemm"]["frac"]
        roofline["after_foreign_kernel"] = foreign
        roofline["after_foreign_kernel_note"] = (
            "fused launch right after a different kernel: [foreign, fused] pairs minus the "
            "foreign kernels alone; spin = a one-thread spin touching no memory "
            "(frac_after_foreign_kernel), gemm = a bf16 GEMM writing partial 0 of the batch "
            "the fused launch reads (frac_after_gemm_marginal: the launch's marginal cost in "
            "the pair, partly hidden behind the GEMM's end)")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "n_parts": wl.n_parts, "T": wl.T, "H": wl.H,
                   "n_out": wl.n_out, "eps": wl.eps, "l2": l2_note, "path": args.path,
                   "max_sms": args.max_sms or "all",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "sm_count": torch.cuda.get_device_properties(device).multi_processor_count},
        "hbm_gbs": round(achieved, 1),
        "roofline": roofline,
        "sm_budget_8": {"tokens_per_s": wl.T / (sm8["mean_launch_ms"] * 1e-3),
                        "gbs": round(sm8_gbs, 1), "frac": round(sm8_gbs / peak, 4)},
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps, "clocks": clocks,
    }
    if configs is not None:
        line["configs"] = configs
    if overlap is not None:
        line["overlap"] = overlap
    if flags is not None:
        line["flags"] = flags
    if threads is not None:
        line["oracle_threads"] = threads
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return reference_main(args)
    return tw_main(args)


if __name__ == "__main__":
    sys.exit(main())
