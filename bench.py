"""MoE block-verify benchmark on GB300: per-layer us and achieved HBM GB/s vs the
block size k, and the verify/decode latency ratio.

Workload (one "step"): a block of k=16 positions verified through 40 MoE layers
of the Qwen3-A3B-like shape (d=2048, 128 experts, top-8, d_ff=768, bf16, SwiGLU,
independent seeded weights per layer, 48 GB in HBM), each layer called through
the C ABI (router + top-8 + woken union + grouped expert FFN + combine).  The
40 distinct weight sets are far larger than L2, so no step reads weights from
L2.  `value` = algorithmic HBM bytes (woken experts x expert bytes + router
bytes, summed over the layers) / device time, in GB/s.

Also reported: the k=1 decode pass (verify/decode ratio against the woken-byte
ratio), a k=1..16 sweep for repeated-token and independent blocks, the 40-layer
pre-norm residual stack with greedy acceptance on logits[17, 151936], per-kernel
roofline of the dominant kernel, an end-to-end number through the host-buffer
entry point, and the CPU oracle on a bounded sample.

python bench.py [--gpus N --steps K --warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE block-verify layer µs and HBM GB/s (% of roofline) vs k; verify/decode ratio"
N_LAYERS = 40   # layers per step (--layers overrides, for profiling runs only)
KBLOCK = 16
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}

# DRAM bytes (read + write) per launch from one ncu capture of each single-launch
# kernel at k=16 (the capture and its command are summarised under profiles/),
# keyed by a hash of the kernel's sources: a kernel edited since the capture
# reports traffic null.
KERNEL_SOURCES = {
    "moe_fused_kernel": ["layer_fused.cu", "fused_common.cuh", "dfv_internal.cuh"],
    "moe_fused_kernel_shared": ["layer_fused.cu", "fused_common.cuh", "dfv_internal.cuh"],
    "moe_fused_bs_kernel_mxfp4": ["layer_fused_bs.cu", "fused_common.cuh", "mxfp4_common.cuh", "dfv_internal.cuh"],
    "moe_fused_bs_kernel_q8": ["layer_fused_bs.cu", "fused_common.cuh", "mxfp4_common.cuh", "dfv_internal.cuh"],
    "tc_group_kernel_gateup": ["batch.cu", "tc05.cuh", "dfv_internal.cuh"],
}
# kernel -> (source hash, dram read+write bytes of one captured launch, algorithmic bytes of that launch);
# the captures and their commands are summarised under profiles/ (one file per kernel and workload)
NCU_TRAFFIC = {
    "moe_fused_kernel": ("8cafc0fbfcdc4fea", 727380480 + 4437504, 77 * 9437184 + 524288),
    "moe_fused_kernel_shared": ("8cafc0fbfcdc4fea", 647156736 + 5038336, 102 * 6291456 + 1048576),
    "moe_fused_bs_kernel_mxfp4": ("934bcf6738e1707c", 171702016 + 4564224, 102 * 1671168 + 1048576),
    "moe_fused_bs_kernel_q8": ("934bcf6738e1707c", 342161920 + 4358144, 102 * 3342336 + 1048576),
    "tc_group_kernel_gateup": ("39054c6688135d8c", 822216960 + 3193088, 128 * 6291456),
}


def kernel_hash(name: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, "speculative_decoding_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(name: str, algorithmic_bytes: float):
    """Traffic of the captured launch scaled to a launch of `algorithmic_bytes`
    (by the woken experts processed), or None when the kernel changed since."""
    t = NCU_TRAFFIC.get(name)
    if t is None or t[0] != kernel_hash(name):
        return None
    return t[1] * algorithmic_bytes / t[2]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return PEAKS_FALLBACK, "fallback"


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over the ranks of the default process group (the
    slowest replica's time), or `value` itself for a single process.  `device`
    is where the collective's tensor lives: a CUDA device under NCCL, the CPU
    under gloo."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.05)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- reference arm (CPU oracle)


class OracleSample:
    """The CPU oracle on Qwen3-A3B-like layers: `n_layers` layers drawn once, then
    timed calls with fresh hidden rows, alternating layers."""

    def __init__(self, n_layers: int = 2):
        import oracle
        from speculative_decoding_moe_gb300 import inputs
        from tests._util import np_of, oracle_layer
        oracle.build()
        self.oracle, self.inputs, self.np_of = oracle, inputs, np_of
        self.lws = [inputs.make_layer(inputs.A3B, seed=9000 + i) for i in range(n_layers)]
        self.ols = [oracle_layer(lw) for lw in self.lws]
        self.seed = 9100

    def run(self, n_threads: int, budget_s: float, k: int = KBLOCK, max_calls: int = 2000):
        """Calls at block k on `n_threads` threads until `budget_s` seconds of timed
        oracle work; returns (GB/s of woken-expert + router bytes, calls, seconds)."""
        o, A3B = self.oracle, self.inputs.A3B
        total_bytes, total_s, calls = 0.0, 0.0, 0
        while calls < max_calls and (calls == 0 or total_s < budget_s):
            lw, ol = self.lws[calls % len(self.lws)], self.ols[calls % len(self.ols)]
            x = self.np_of(self.inputs.make_hidden(k, A3B.d, "bf16", seed=self.seed))
            self.seed += 1
            _, idx, _ = o.route(ol, x)
            W = len(o.woken(idx, A3B.n_experts)[0])
            t0 = time.perf_counter()
            o.moe_forward(ol, x, nthreads=n_threads)
            total_s += time.perf_counter() - t0
            total_bytes += W * lw.expert_bytes() + lw.router_bytes()
            calls += 1
        return total_bytes / total_s / 1e9, calls, total_s


def oracle_stack_sample(ols, d: int, n_threads: int, n_total: int = 40, V: int = 151936):
    """The oracle's pre-norm stack over the given layers at k=16 plus greedy
    acceptance on [k+1, V] logits, timed once; the stack time is scaled to
    `n_total` layers (every layer costs the same work at a fixed woken count)."""
    import oracle
    from speculative_decoding_moe_gb300 import inputs
    from tests._util import np_of
    x = np_of(inputs.make_hidden(KBLOCK, d, "bf16", seed=9400))
    t0 = time.perf_counter()
    oracle.stack_forward(ols, x, nthreads=n_threads)
    t_stack = time.perf_counter() - t0
    lg, toks = inputs.spiked_logits(KBLOCK + 1, V, "bf16", 2.0, seed=9401)
    draft = toks[:KBLOCK].contiguous().numpy()
    t0 = time.perf_counter()
    tau, _ = oracle.accept_greedy(np_of(lg), draft)
    t_acc = time.perf_counter() - t0
    return {"layers_timed": len(ols), "stack_ms": t_stack * 1e3, "accept_ms": t_acc * 1e3, "tau": tau,
            "threads": n_threads, "stack%d_accept_ms_extrapolated" % n_total:
                t_stack * 1e3 * n_total / len(ols) + t_acc * 1e3}


def cpu_baseline_line(budget_s: float):
    """`cpu_baseline`: the oracle at k=16 on every host thread (the headline, about
    `budget_s` seconds), plus shorter samples single-threaded and at k=1, and the
    40-layer stack + acceptance of the bf16 and mxfp4 layers, timed on two
    layers and scaled."""
    nthr = host_threads()
    smp = OracleSample()
    gbs, calls, secs = smp.run(nthr, budget_s)
    side = {}
    for name, nt, k in (("k16_1thread", 1, KBLOCK), ("k1_all_threads", nthr, 1), ("k1_1thread", 1, 1)):
        g, c, t = smp.run(nt, budget_s / 4, k=k)
        side[name] = {"value": g, "unit": "GB/s", "threads": nt, "k": k, "calls": c,
                      "us_per_layer": t / c * 1e6}
    from speculative_decoding_moe_gb300 import inputs
    from tests._util import oracle_layer
    side["stack_bf16"] = oracle_stack_sample(smp.ols, inputs.A3B.d, nthr)
    mx = [oracle_layer(inputs.make_layer(inputs.MXFP4, seed=9500 + i)) for i in range(2)]
    side["stack_mxfp4"] = oracle_stack_sample(mx, inputs.MXFP4.d, nthr)
    return {"value": gbs, "unit": "GB/s", "cores": nthr, "kind": "oracle",
            "us_per_layer": secs / calls * 1e6,
            "sample": "%d Qwen3-A3B-like layer call(s) at k=16 over 2 layers (oracle moe_forward, fp64, "
                      "%d threads, %.1f s timed)" % (calls, nthr, secs),
            "also": side}


def achieved_gbs(nbytes: float, ms: float) -> float:
    """Bytes moved over a time in ms, as GB/s (1e9 bytes per second)."""
    return nbytes / (ms * 1e-3) / 1e9


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from speculative_decoding_moe_gb300 import inputs
    from tests._util import np_of, oracle_layer
    oracle.build()
    nthr = host_threads()
    lw = inputs.make_layer(inputs.A3B, seed=9000)
    ol = oracle_layer(lw)
    x = np_of(inputs.make_hidden(KBLOCK, inputs.A3B.d, "bf16", seed=9100))
    _, idx, _ = oracle.route(ol, x)
    W = len(oracle.woken(idx, inputs.A3B.n_experts)[0])
    step_bytes = W * lw.expert_bytes() + lw.router_bytes()
    for _ in range(args.warmup):
        oracle.moe_forward(ol, x, nthreads=nthr)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.moe_forward(ol, x, nthreads=nthr)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = step_bytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": nthr, "kind": "oracle",
                         "sample": "a bounded sample of the 40-layer workload: each step is one of its Qwen3-A3B-like "
                                   "layers (d=2048, E=128, top-8, d_ff=768, bf16 weights) at k=16, W=%d woken experts, "
                                   "oracle moe_forward on %d host threads; GB/s counts that layer's woken-expert and "
                                   "router bytes, as the GPU arm counts each of its 40" % (W, nthr)},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config():
    return {"workload": "qwen3-a3b-like MoE layer x %d (d=2048, E=128, top-8, d_ff=768, bf16, SwiGLU), "
                        "k=16 verify block" % N_LAYERS,
            "d": 2048, "n_experts": 128, "top_k": 8, "d_ff": 768, "k": KBLOCK, "layers_per_step": N_LAYERS,
            # 40 layers x (128 experts x 3 x 768 x 2048 bf16 + the 128 x 2048 bf16 router)
            "weights_gb": round(N_LAYERS * (128 * 3 * 768 * 2048 * 2 + 128 * 2048 * 2) / 1e9, 2),
            "l2": "inputs larger than L2: 40 distinct layer weight sets (48 GB), each step streams every woken "
                  "expert from HBM"}


# ---------------------------------------------------------------------------- GPU arm


def progress(msg: str):
    """One line on stderr per bench section (stdout carries only the JSON line)."""
    print("[bench] %s" % msg, file=sys.stderr, flush=True)


def graph_time(fn, warmup: int, steps: int, barrier=None, sampler=None, per_step=None):
    """Capture one step into a CUDA graph, replay `warmup` untimed then `steps`
    timed replays bracketed by CUDA events; returns ms per step.  With a list
    `per_step`, an event between consecutive replays also gives each step's
    own time (appended to the list, in ms)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps - 1)] if per_step is not None else []
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        a.record()
        for i in range(steps):
            g.replay()
            if mids and i < steps - 1:
                mids[i].record()
        b.record()
        b.synchronize()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    if per_step is not None:
        marks = [a] + mids + [b]
        per_step.extend(marks[i].elapsed_time(marks[i + 1]) for i in range(steps))
    return a.elapsed_time(b) / steps


def spread_us(per_step_ms, per: int):
    """Median, p10 and p90 of per-step times, in µs per `per` (e.g. per layer)."""
    v = sorted(x * 1e3 / per for x in per_step_ms)
    q = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]
    return {"median": statistics.median(v), "p10": q(0.1), "p90": q(0.9), "steps": len(v)}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def stream_time(fn, warmup: int, steps: int):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / steps


def run_gpu(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

        def barrier():
            dist.barrier()
    else:
        barrier = None

    from speculative_decoding_moe_gb300 import build as bld
    bld.build()
    from speculative_decoding_moe_gb300 import dfv, inputs

    peaks, peak_kind = load_peaks()
    shape = inputs.A3B
    t_gen = time.time()
    layers = [inputs.make_layer(shape, seed=1000 * rank + l, device=dev) for l in range(N_LAYERS)]
    torch.cuda.synchronize()
    t_gen = time.time() - t_gen
    Ls = [dfv.Layer(w) for w in layers]
    exp_bytes = layers[0].expert_bytes()
    router_bytes = layers[0].router_bytes()
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], KBLOCK), device=dev)

    def make_pass(k, mode="independent", seed=5, pert_std=0.3):
        x = inputs.make_hidden(k, shape.d, "bf16", seed=seed + 100 * rank, mode=mode, device=dev,
                               pert_std=pert_std)
        out = torch.empty_like(x)
        nws = torch.zeros(N_LAYERS, dtype=torch.int32, device=dev)

        def fn():
            for l in range(N_LAYERS):
                dfv.moe_block_forward(Ls[l], x, ws, out=out, n_woken=nws[l:l + 1])
        return fn, nws

    def pass_bytes(nws):
        W = nws.to(torch.int64).cpu()
        return float(W.sum().item() * exp_bytes + N_LAYERS * router_bytes), W

    # ---- headline: k=16 verify pass over 40 layers (CUDA graph replay)
    progress("headline k=16")
    torch.cuda.nvtx.range_push("headline")
    fn16, nw16 = make_pass(KBLOCK)
    sampler = ClockSampler(local)
    steps16 = []
    ms16 = graph_time(fn16, args.warmup, args.steps, barrier, sampler, per_step=steps16)
    clocks = sampler.summary()
    bytes16, W16 = pass_bytes(nw16)
    ms_max = max_over_ranks(ms16, dev)
    value = achieved_gbs(world * bytes16, ms_max)

    torch.cuda.nvtx.range_pop()

    # ---- decode: k=1 pass, same layers
    progress("decode k=1")
    fn1, nw1 = make_pass(1, seed=6)
    ms1 = graph_time(fn1, args.warmup, args.steps, barrier)
    bytes1, W1 = pass_bytes(nw1)

    # ---- stream-launch numbers (no graph) for context
    progress("stream launches")
    ms16_stream = stream_time(fn16, 2, max(3, args.steps // 4))
    ms1_stream = stream_time(fn1, 2, max(3, args.steps // 4))

    # ---- per-launch timing with CUDA events.  The fused path runs one kernel per
    # layer (the dominant and only kernel); the multi-kernel path is timed too.
    x16 = inputs.make_hidden(KBLOCK, shape.d, "bf16", seed=5 + 100 * rank, device=dev)
    out16 = torch.empty_like(x16)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(N_LAYERS)]

    def per_phase(reps=3):
        tot = [0.0, 0.0, 0.0]
        for r in range(reps + 1):
            for l in range(N_LAYERS):
                dfv.profile_set_events(evs[l])
                dfv.moe_block_forward(Ls[l], x16, ws, out=out16)
            dfv.profile_set_events(None)
            torch.cuda.synchronize()
            if r == 0:
                continue
            for l in range(N_LAYERS):
                e = evs[l]
                tot[0] += e[0].elapsed_time(e[1])
                tot[1] += e[1].elapsed_time(e[2])
                tot[2] += e[2].elapsed_time(e[3])
        n = reps * N_LAYERS
        return [t / n for t in tot]

    layer_bytes = float(W16.sum().item()) * exp_bytes / N_LAYERS + router_bytes  # per launch
    ph = per_phase()
    fused_used = dfv.last_layer_path() == 1
    fused_ms = ph[0] + ph[1] + ph[2]
    fused_gbs = layer_bytes / (fused_ms * 1e-3) / 1e9
    dfv.set_path(False)
    torch.cuda.nvtx.range_push("multi_kernel")
    phm = per_phase()
    ms16_multi = graph_time(fn16, 2, max(3, args.steps // 4))
    torch.cuda.nvtx.range_pop()
    dfv.set_path(True)
    gate_bytes = float(W16.sum().item()) * (2 * shape.d_ff * shape.d * 2) / N_LAYERS
    down_bytes = float(W16.sum().item()) * (shape.d * shape.d_ff * 2) / N_LAYERS
    peak_bw = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    # The timed region runs this kernel alone, one launch per layer (the ncu
    # launch list of the same command shows no other kernel there), so its
    # average launch duration is the region's device time over its launches.
    # Events around each launch (stream launches) are reported too: they
    # break the programmatic chaining of consecutive layers and add their own
    # gap, so they give the launch in isolation.
    per_launch_ms = ms_max / N_LAYERS
    launch_gbs = layer_bytes / (per_launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "moe_fused_kernel<2> (one launch per layer, k=16)", "achieved": launch_gbs,
                "peak": peak_bw, "unit": "GB/s", "frac": launch_gbs / peak_bw,
                "traffic": ncu_traffic("moe_fused_kernel", layer_bytes),
                "traffic_note": "ncu dram read+write of one k=16 launch, scaled to this average launch by woken experts",
                "peak_kind": peak_kind + " (STREAM-style copy, burst)",
                "per_launch_us": per_launch_ms * 1e3,
                "per_launch_note": "timed region (CUDA-graph replay, events at its ends) / its 40 launches",
                "isolated_launch_us": fused_ms * 1e3, "isolated_launch_frac": fused_gbs / peak_bw,
                "algorithmic_bytes_per_launch": layer_bytes,
                "multi_kernel_per_launch_us": {"router": phm[0] * 1e3, "gate_up": phm[1] * 1e3,
                                               "down_combine": phm[2] * 1e3},
                "multi_kernel_gate_up_gbs": gate_bytes / (phm[1] * 1e-3) / 1e9,
                "multi_kernel_down_gbs": down_bytes / (phm[2] * 1e-3) / 1e9}

    # ---- k sweep (repeated-token vs independent blocks).  "repeated" is the
    # stated recipe (base + N(0, 0.3^2) per position, ~19 woken at k=16);
    # "repeated_w30" widens the perturbation to N(0, 0.55^2), which lands at the
    # ~30 woken experts part 2 reports for its repeated-token block.
    sweep = {}
    if not args.no_sweep:
        for name, mode, pstd in (("repeated", "repeated", 0.3), ("repeated_w30", "repeated", 0.55),
                                 ("independent", "independent", 0.3)):
            rows = []
            for k in range(1, 17):
                progress("sweep %s k=%d" % (name, k))
                fnk, nwk = make_pass(k, mode=mode, seed=50 + k, pert_std=pstd)
                msk = graph_time(fnk, 2, max(3, args.steps // 4))
                bk, Wk = pass_bytes(nwk)
                rows.append({"k": k, "woken_mean": float(Wk.double().mean().item()),
                             "layer_us": msk * 1e3 / N_LAYERS, "gbs": bk / (msk * 1e-3) / 1e9})
            sweep[name] = rows

    # ---- 40-layer pre-norm residual stack + greedy acceptance (one verify cycle)
    progress("stack")
    stack = None
    if not args.no_stack:
        V = 151936
        xs0 = inputs.make_hidden(KBLOCK, shape.d, "bf16", seed=7 + 100 * rank, device=dev)
        xs = xs0.clone()
        logits, toks = inputs.spiked_logits(KBLOCK + 1, V, "bf16", 2.0, seed=8, device=dev)
        nacc = 5
        draft = toks[:KBLOCK].clone()
        draft[nacc] = (draft[nacc] + 1) % V
        aws = dfv.alloc_workspace(dfv.accept_workspace_size(KBLOCK, V), device=dev)
        tau = torch.zeros(1, dtype=torch.int32, device=dev)
        com = torch.zeros(KBLOCK + 1, dtype=torch.int32, device=dev)

        def fn_stack():
            xs.copy_(xs0)
            dfv.moe_stack_forward(Ls, xs, ws)
            dfv.accept_greedy(logits, draft, aws, tau=tau, committed=com)

        ms_stack = graph_time(fn_stack, 2, max(3, args.steps // 4))
        stack = {"ms": ms_stack, "layer_us": ms_stack * 1e3 / N_LAYERS, "tau": int(tau.item()),
                 "tau_expected": nacc + 1, "finite": bool(torch.isfinite(xs.float()).all().item())}

    # ---- end to end through the host-buffer entry point (plain stream launches)
    progress("end to end")
    hx = x16.cpu().pin_memory()
    ho = torch.empty_like(hx).pin_memory()

    def fn_e2e():
        for l in range(N_LAYERS):
            dfv.moe_block_forward_host(Ls[l], hx, ho, ws)
        _ = None

    e2e_ms = stream_time(fn_e2e, 2, max(3, args.steps // 2))
    e2e = {"value": world * bytes16 / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": N_LAYERS * hx.numel() * hx.element_size(),
           "d2h_bytes_per_step": N_LAYERS * ho.numel() * ho.element_size(), "ms_per_step": e2e_ms,
           "api": "dfv_moe_block_forward_host per layer, pinned host buffers"}

    # each section in its own NVTX range, so a profiler can select one (ncu --nvtx --nvtx-include "q8/")
    def section(name, skip, fn, *a, **kw):
        if skip:
            return None
        torch.cuda.nvtx.range_push(name)
        try:
            return fn(*a, **kw)
        finally:
            torch.cuda.nvtx.range_pop()

    stk = section("stack40", args.no_stack, stack_section, args, dev, rank, barrier, dfv, inputs, peak_bw, Ls,
                  exp_bytes, router_bytes, ws, shape)
    bt = section("batch", args.no_batch, batch_section, args, dev, rank, barrier, dfv, inputs, peaks, peak_bw, Ls,
                 exp_bytes, router_bytes)
    mx = section("mxfp4", args.no_mxfp4, mxfp4_section, args, dev, rank, barrier, dfv, inputs, peak_bw)
    q8 = section("q8", args.no_q8, mxfp4_section, args, dev, rank, barrier, dfv, inputs, peak_bw, fmt="q8")
    sh = section("shared_expert", args.no_shared, shared_section, args, dev, rank, barrier, dfv, inputs, peak_bw)
    wd = section("wide", args.no_wide, wide_section, args, dev, rank, barrier, dfv, inputs, peak_bw)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        progress("cpu oracle sample")
        cpu = cpu_baseline_line(args.cpu_budget)

    ratio = ms16 / ms1
    byte_ratio = bytes16 / bytes1
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random-init weights and hidden rows)",
        "config": workload_config(),
        "layer_us_spread_k16": spread_us(steps16, N_LAYERS),
        "layer_us": {"k16": ms16 * 1e3 / N_LAYERS, "k1": ms1 * 1e3 / N_LAYERS,
                     "k16_multi_kernel": ms16_multi * 1e3 / N_LAYERS,
                     "k16_stream": ms16_stream * 1e3 / N_LAYERS, "k1_stream": ms1_stream * 1e3 / N_LAYERS},
        "frac_of_hbm_peak": {"measured": value / world / peak_bw, "nominal_8tbs": value / world / 8000.0},
        "woken_mean": {"k16": float(W16.double().mean().item()), "k1": float(W1.double().mean().item())},
        "verify_decode": {"latency_ratio": ratio, "woken_byte_ratio": byte_ratio,
                          "quotient": byte_ratio / ratio},
        "kernel_path": {"fused": fused_used, "why_not": dfv.fused_unavailable_reason()},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": N_LAYERS * args.steps, "clocks": clocks,
        "sweep": sweep, "stack40": stk, "stack40_accept": stack, "weight_gen_s": t_gen, "batch": bt, "mxfp4": mx, "q8": q8, "shared_expert": sh, "wide_layers": wd,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def stack_section(args, dev, rank, barrier, dfv, inputs, peak_bw, Ls, exp_bytes, router_bytes, ws, shape):
    """The 40-layer pre-norm residual stack through dfv_moe_stack_forward at k = 16
    (verify) and k = 1 (decode): one persistent launch for all layers against
    one launch per layer.  Bytes are each layer's woken experts (reported by the
    call) plus its router."""
    res = {"config": "Qwen3-A3B-like layer x %d (d=2048, E=128, top-8, d_ff=768, bf16), pre-norm residual stack"
                     % N_LAYERS}
    outs = {}
    for k in (KBLOCK, 1):
        x0 = inputs.make_hidden(k, shape.d, "bf16", seed=9 + 100 * rank + k, device=dev)
        xs = x0.clone()
        nw = torch.zeros(N_LAYERS, dtype=torch.int32, device=dev)

        def fn():
            xs.copy_(x0)
            dfv.moe_stack_forward(Ls, xs, ws, n_woken=nw)

        row = {}
        for name, mode in (("persistent", 2), ("per_layer", 0)):
            progress("stack k=%d %s" % (k, name))
            dfv.set_stack_launch(mode)
            try:
                ms = graph_time(fn, max(3, args.warmup), max(5, args.steps // 2), barrier)
                fn()
                torch.cuda.synchronize()
                path = dfv.last_layer_path()
            finally:
                dfv.set_stack_launch(1)
            outs[(k, name)] = xs.clone()
            W = nw.to(torch.int64).cpu()
            nbytes = float(W.sum().item() * exp_bytes + N_LAYERS * router_bytes)
            row[name] = {"ms": ms, "layer_us": ms * 1e3 / N_LAYERS, "gbs": achieved_gbs(nbytes, ms),
                         "frac_of_measured_hbm": achieved_gbs(nbytes, ms) / peak_bw, "path": path,
                         "woken_mean": float(W.double().mean().item()), "bytes": nbytes}
        row["identical"] = bool(torch.equal(outs[(k, "persistent")], outs[(k, "per_layer")]))
        # eager calls (no graph): each launch pays the host's launch cost, which
        # is what the default mode's choice of the persistent kernel at k <= 8 saves
        eager = {}
        for name, mode in (("persistent", 2), ("per_layer", 0), ("default", 1)):
            progress("stack k=%d eager %s" % (k, name))
            dfv.set_stack_launch(mode)
            try:
                if barrier:
                    barrier()
                ms_e = max_over_ranks(stream_time(fn, max(3, args.warmup), max(5, args.steps // 2)), dev)
                path = dfv.last_layer_path()
            finally:
                dfv.set_stack_launch(1)
            eager[name] = {"ms": ms_e, "layer_us": ms_e * 1e3 / N_LAYERS, "path": path,
                           "gbs": achieved_gbs(row["per_layer"]["bytes"], ms_e)}
        row["eager"] = eager
        res["k%d" % k] = row
    for name in ("persistent", "per_layer"):
        a, b = res["k%d" % KBLOCK][name], res["k1"][name]
        res["verify_decode_" + name] = {"latency_ratio": a["ms"] / b["ms"], "woken_byte_ratio": a["bytes"] / b["bytes"],
                                        "quotient": (a["bytes"] / b["bytes"]) / (a["ms"] / b["ms"])}
    # the default launch mode on eager calls: one launch per layer at k = 16,
    # persistent at k = 1 (inside a graph it launches per layer at every k)
    a, b = res["k%d" % KBLOCK]["eager"]["default"], res["k1"]["eager"]["default"]
    wb = res["k%d" % KBLOCK]["per_layer"]["bytes"] / res["k1"]["per_layer"]["bytes"]
    res["verify_decode_default_mode_eager"] = {"latency_ratio": a["ms"] / b["ms"], "woken_byte_ratio": wb,
                                               "quotient": wb / (a["ms"] / b["ms"])}
    res["device_error"] = dfv.read_device_error(ws)
    return res


def batch_section(args, dev, rank, barrier, dfv, inputs, peaks, peak_bw, Ls, exp_bytes, router_bytes):
    """Batched verify: 32 blocks of k=16 (512 rows) through the same 40
    Qwen3-A3B-like layers, expert contractions on tcgen05.  Bytes count each
    woken expert once per layer (the batch shares the weights) plus the
    router; FLOPs count 2 * rows * K * 3 * d * d_ff per layer.  Also timed:
    the same rows as 32 single-block calls per layer (legacy mma.sync path,
    weights streamed once per block)."""
    progress("batched verify")
    shape = inputs.A3B
    n_blocks, k = 32, KBLOCK
    T = n_blocks * k
    x = inputs.make_hidden(T, shape.d, "bf16", seed=61 + 100 * rank, device=dev)
    out = torch.empty_like(x)
    bws = dfv.alloc_workspace(dfv.batch_workspace_size(Ls[0], T), device=dev)
    nws = torch.zeros(N_LAYERS, dtype=torch.int32, device=dev)

    def fn():
        for l in range(N_LAYERS):
            dfv.moe_batch_forward(Ls[l], x, n_blocks, bws, out=out, n_woken=nws[l:l + 1])

    ms = graph_time(fn, args.warmup, args.steps, barrier)
    W = nws.to(torch.int64).cpu()
    nbytes = float(W.sum().item() * exp_bytes + N_LAYERS * router_bytes)
    flops = 2.0 * T * shape.top_k * 3 * shape.d * shape.d_ff * N_LAYERS
    # per-phase events over the 40 layers (stream launches)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(N_LAYERS)]
    tot = [0.0, 0.0, 0.0]
    reps = 3
    for r in range(reps + 1):
        for l in range(N_LAYERS):
            dfv.profile_set_events(evs[l])
            dfv.moe_batch_forward(Ls[l], x, n_blocks, bws, out=out)
        dfv.profile_set_events(None)
        torch.cuda.synchronize()
        if r:
            for l in range(N_LAYERS):
                for i in range(3):
                    tot[i] += evs[l][i].elapsed_time(evs[l][i + 1])
    ph = [t / (reps * N_LAYERS) for t in tot]
    Wm = float(W.double().mean().item())
    gate_bytes = Wm * 2 * shape.d_ff * shape.d * 2
    down_bytes = Wm * shape.d * shape.d_ff * 2
    gate_flops = 2.0 * T * shape.top_k * 2 * shape.d * shape.d_ff
    # the same rows as single-block calls (mma.sync path), 40 layers
    ws1 = dfv.alloc_workspace(dfv.workspace_size(Ls[0], k), device=dev)
    o1 = torch.empty(k, shape.d, dtype=torch.bfloat16, device=dev)
    xb = [x[b * k:(b + 1) * k].contiguous() for b in range(n_blocks)]

    def fn_single():
        for l in range(N_LAYERS):
            for b in range(n_blocks):
                dfv.moe_block_forward(Ls[l], xb[b], ws1, out=o1)

    ms_single = graph_time(fn_single, 2, max(3, args.steps // 5))

    # the small-M contraction choice: one block of 16 rows through the tcgen05
    # path (M = 128 weight rows per tile, N = the expert's rows) against the
    # single-launch kernel's mma.sync (M = 16, N = 8 tokens per tile)
    def fn_one_tc():
        for l in range(N_LAYERS):
            dfv.moe_batch_forward(Ls[l], xb[0], 1, bws, out=o1)

    def fn_one_mma():
        for l in range(N_LAYERS):
            dfv.moe_block_forward(Ls[l], xb[0], ws1, out=o1)

    ms_one_tc = graph_time(fn_one_tc, 2, max(3, args.steps // 5))
    ms_one_mma = graph_time(fn_one_mma, 2, max(3, args.steps // 5))
    tot1 = [0.0, 0.0, 0.0]
    for r in range(reps + 1):
        for l in range(N_LAYERS):
            dfv.profile_set_events(evs[l])
            dfv.moe_batch_forward(Ls[l], xb[0], 1, bws, out=o1)
        dfv.profile_set_events(None)
        torch.cuda.synchronize()
        if r:
            for l in range(N_LAYERS):
                for i in range(3):
                    tot1[i] += evs[l][i].elapsed_time(evs[l][i + 1])
    ph1 = [t / (reps * N_LAYERS) for t in tot1]
    tf_sus = peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops")
    return {
        "config": "32 blocks x k=16 (512 rows), Qwen3-A3B-like layer x 40 (d=2048, E=128, top-8, d_ff=768, bf16)",
        "ms_per_pass": ms, "layer_us": ms * 1e3 / N_LAYERS, "woken_mean": Wm,
        "value_gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_measured_hbm": nbytes / (ms * 1e-3) / 1e9 / peak_bw,
        "tflops": flops / (ms * 1e-3) / 1e12,
        "rows_per_s": T * 1.0 / (ms * 1e-3) * N_LAYERS / N_LAYERS,
        "phase_us": {"routing_gather": ph[0] * 1e3, "gate_up": ph[1] * 1e3, "down_combine": ph[2] * 1e3},
        "roofline": {"bound": "hbm", "kernel": "tc_group_kernel<gate/up> (tcgen05, one launch per layer)",
                     "achieved": gate_bytes / (ph[1] * 1e-3) / 1e9, "peak": peak_bw, "unit": "GB/s",
                     "frac": gate_bytes / (ph[1] * 1e-3) / 1e9 / peak_bw,
                     "traffic": ncu_traffic("tc_group_kernel_gateup", gate_bytes),
                     "per_launch_us": ph[1] * 1e3, "algorithmic_bytes_per_launch": gate_bytes,
                     "tensor_tflops": gate_flops / (ph[1] * 1e-3) / 1e12,
                     "tensor_frac_of_sustained": gate_flops / (ph[1] * 1e-3) / 1e12 / tf_sus if tf_sus else None},
        "down_gbs": down_bytes / (ph[2] * 1e-3) / 1e9,
        "single_block_calls": {"ms_per_pass": ms_single, "layer_us": ms_single * 1e3 / N_LAYERS,
                               "speedup_of_batched": ms_single / ms},
        "one_block_16_rows": {"tcgen05_path_layer_us": ms_one_tc * 1e3 / N_LAYERS,
                              "mma_sync_single_launch_layer_us": ms_one_mma * 1e3 / N_LAYERS,
                              "tcgen05_phase_us": {"routing_gather": ph1[0] * 1e3, "gate_up": ph1[1] * 1e3,
                                                   "down_combine": ph1[2] * 1e3}},
        "device_error": dfv.read_device_error(bws),
    }


def mxfp4_section(args, dev, rank, barrier, dfv, inputs, peak_bw, fmt="mxfp4"):
    """Block-scaled experts, E=256, top-8, d=2048, d_ff=512, 40 layers, bf16
    activations: mxfp4 (e2m1 codes + e8m0 per 32) or, with fmt="q8", 8-bit
    codes + a binary16 scale per 32 (the pages' "Q8" target).  Bytes per woken
    expert count the codes and the scale bytes."""
    progress("%s section" % fmt)
    shape = inputs.MXFP4 if fmt == "mxfp4" else inputs.Q8
    layers = [inputs.make_layer(shape, seed=5000 + 1000 * rank + l, device=dev) for l in range(N_LAYERS)]
    Ls = [dfv.Layer(w) for w in layers]
    exp_bytes = layers[0].expert_bytes()
    router_bytes = layers[0].router_bytes()
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], KBLOCK), device=dev)

    def make_pass(k, mode="independent", seed=5):
        x = inputs.make_hidden(k, shape.d, "bf16", seed=seed + 100 * rank, mode=mode, device=dev)
        out = torch.empty_like(x)
        nws = torch.zeros(N_LAYERS, dtype=torch.int32, device=dev)

        def fn():
            for l in range(N_LAYERS):
                dfv.moe_block_forward(Ls[l], x, ws, out=out, n_woken=nws[l:l + 1])
        return fn, nws, x

    def pass_bytes(nws):
        W = nws.to(torch.int64).cpu()
        return float(W.sum().item() * exp_bytes + N_LAYERS * router_bytes), W

    fn16, nw16, x16 = make_pass(KBLOCK, seed=15)
    ms16 = graph_time(fn16, args.warmup, args.steps, barrier)
    b16, W16 = pass_bytes(nw16)
    fn1, nw1, _ = make_pass(1, seed=16)
    ms1 = graph_time(fn1, args.warmup, args.steps, barrier)
    b1, W1 = pass_bytes(nw1)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(N_LAYERS)]
    out16 = torch.empty_like(x16)
    tot = [0.0, 0.0, 0.0]
    reps = 3
    for r in range(reps + 1):
        for l in range(N_LAYERS):
            dfv.profile_set_events(evs[l])
            dfv.moe_block_forward(Ls[l], x16, ws, out=out16)
        dfv.profile_set_events(None)
        torch.cuda.synchronize()
        if r:
            for l in range(N_LAYERS):
                e = evs[l]
                for i in range(3):
                    tot[i] += e[i].elapsed_time(e[i + 1])
    ph = [t / (reps * N_LAYERS) for t in tot]
    fused = dfv.last_layer_path() == 1
    Wm = float(W16.double().mean().item())
    gate_bytes = Wm * 2 * (shape.d_ff * shape.d // 2 + shape.d_ff * shape.d // 32)
    down_bytes = Wm * (shape.d * shape.d_ff // 2 + shape.d * shape.d_ff // 32)
    layer_bytes = Wm * exp_bytes + router_bytes
    desc = "mxfp4 experts (e2m1 + e8m0/32)" if fmt == "mxfp4" else "8-bit experts (int8 + binary16/32)"
    res = {
        "config": "E=256 top-8 d=2048 d_ff=512 %s, bf16 router and activations, "
                  "40 layers, k=16; inputs > L2 (%.1f GB of weights)" % (desc, N_LAYERS * (exp_bytes * 256 + router_bytes) / 1e9),
        "value_gbs": b16 / (ms16 * 1e-3) / 1e9, "frac_of_measured_hbm": b16 / (ms16 * 1e-3) / 1e9 / peak_bw,
        "ms_per_pass": {"k16": ms16, "k1": ms1},
        "layer_us": {"k16": ms16 * 1e3 / N_LAYERS, "k1": ms1 * 1e3 / N_LAYERS},
        "woken_mean": {"k16": Wm, "k1": float(W1.double().mean().item())},
        "verify_decode": {"latency_ratio": ms16 / ms1, "woken_byte_ratio": b16 / b1, "quotient": (b16 / b1) / (ms16 / ms1)},
        "kernel_path": "moe_fused_bs_kernel<%s> (one launch per layer)" % fmt if fused else "router + gate/up + down launches",
        "layer_gbs_events": layer_bytes / (sum(ph) * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "moe_fused_bs_kernel<%s, 2> (k=16)" % fmt if fused else "multi-launch",
                     "achieved": layer_bytes / (ms16 / N_LAYERS * 1e-3) / 1e9, "peak": peak_bw, "unit": "GB/s",
                     "frac": layer_bytes / (ms16 / N_LAYERS * 1e-3) / 1e9 / peak_bw,
                     "traffic": ncu_traffic("moe_fused_bs_kernel_" + fmt, layer_bytes) if fused else None,
                     "per_launch_us": ms16 / N_LAYERS * 1e3,
                     "per_launch_note": "timed k=16 pass (CUDA-graph replay) / its 40 launches",
                     "isolated_launch_us": sum(ph) * 1e3,
                     "algorithmic_bytes_per_launch": layer_bytes},
        "device_error": dfv.read_device_error(ws),
    }
    if not fused:
        res["per_launch_us"] = {"router": ph[0] * 1e3, "gate_up": ph[1] * 1e3, "down_combine": ph[2] * 1e3}
        res["gate_up_gbs"] = gate_bytes / (ph[1] * 1e-3) / 1e9
        res["down_combine_gbs"] = down_bytes / (ph[2] * 1e-3) / 1e9
    if not args.no_stack:
        V = 151936
        xs0 = inputs.make_hidden(KBLOCK, shape.d, "bf16", seed=17 + 100 * rank, device=dev)
        xs = xs0.clone()
        logits, toks = inputs.spiked_logits(KBLOCK + 1, V, "bf16", 2.0, seed=18, device=dev)
        nacc = 5
        draft = toks[:KBLOCK].clone()
        draft[nacc] = (draft[nacc] + 1) % V
        aws = dfv.alloc_workspace(dfv.accept_workspace_size(KBLOCK, V), device=dev)
        tau = torch.zeros(1, dtype=torch.int32, device=dev)
        com = torch.zeros(KBLOCK + 1, dtype=torch.int32, device=dev)

        def fn_stack():
            xs.copy_(xs0)
            dfv.moe_stack_forward(Ls, xs, ws)
            dfv.accept_greedy(logits, draft, aws, tau=tau, committed=com)

        ms_stack = graph_time(fn_stack, 2, max(3, args.steps // 4))
        res["stack40_accept"] = {"ms": ms_stack, "layer_us": ms_stack * 1e3 / N_LAYERS, "tau": int(tau.item()),
                                 "tau_expected": nacc + 1, "finite": bool(torch.isfinite(xs.float()).all().item())}
    del layers, Ls
    return res


def shared_section(args, dev, rank, barrier, dfv, inputs, peak_bw):
    """256 routed experts (top-8) plus one always-on shared expert of the same
    size, d=2048, d_ff=512, bf16, 40 layers.  The shared expert is read once
    per block whatever k is, so a block's bytes are (W + 1) experts + router."""
    progress("shared-expert section")
    shape = inputs.E256_SHARED
    layers = [inputs.make_layer(shape, seed=7000 + 1000 * rank + l, device=dev) for l in range(N_LAYERS)]
    Ls = [dfv.Layer(w) for w in layers]
    exp_bytes = layers[0].expert_bytes()
    router_bytes = layers[0].router_bytes()
    ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], KBLOCK), device=dev)

    def make_pass(k, seed):
        x = inputs.make_hidden(k, shape.d, "bf16", seed=seed + 100 * rank, device=dev)
        out = torch.empty_like(x)
        nws = torch.zeros(N_LAYERS, dtype=torch.int32, device=dev)  # routed experts woken per layer

        def fn():
            for l in range(N_LAYERS):
                dfv.moe_block_forward(Ls[l], x, ws, out=out, n_woken=nws[l:l + 1])
        return fn, nws, x

    def pass_bytes(nws):
        W = nws.to(torch.int64).cpu()
        return float((W.sum().item() + N_LAYERS) * exp_bytes + N_LAYERS * router_bytes), W

    fn16, nw16, x16 = make_pass(KBLOCK, seed=25)
    ms16 = graph_time(fn16, args.warmup, args.steps, barrier)
    b16, W16 = pass_bytes(nw16)
    fn1, nw1, _ = make_pass(1, seed=26)
    ms1 = graph_time(fn1, args.warmup, args.steps, barrier)
    b1, W1 = pass_bytes(nw1)

    # per-launch event timing of the single-launch kernel at k=16
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(N_LAYERS)]
    out16 = torch.empty_like(x16)
    tot = 0.0
    reps = 3
    for r in range(reps + 1):
        for l in range(N_LAYERS):
            dfv.profile_set_events(evs[l])
            dfv.moe_block_forward(Ls[l], x16, ws, out=out16)
        dfv.profile_set_events(None)
        torch.cuda.synchronize()
        if r:
            tot += sum(evs[l][0].elapsed_time(evs[l][3]) for l in range(N_LAYERS))
    per_launch_ms = tot / (reps * N_LAYERS)
    fused = dfv.last_layer_path() == 1
    Wm, Wm1 = float(W16.double().mean().item()), float(W1.double().mean().item())
    layer_bytes = (Wm + 1) * exp_bytes + router_bytes
    res = {
        "config": "E=256 top-8 + 1 shared expert, d=2048, d_ff=512, bf16, 40 layers, k=16; inputs > L2 "
                  "(%.1f GB of weights)" % (N_LAYERS * (exp_bytes * 257 + router_bytes) / 1e9),
        "value_gbs": b16 / (ms16 * 1e-3) / 1e9, "frac_of_measured_hbm": b16 / (ms16 * 1e-3) / 1e9 / peak_bw,
        "ms_per_pass": {"k16": ms16, "k1": ms1},
        "layer_us": {"k16": ms16 * 1e3 / N_LAYERS, "k1": ms1 * 1e3 / N_LAYERS},
        "routed_woken_mean": {"k16": Wm, "k1": Wm1},
        "verify_decode": {"latency_ratio": ms16 / ms1, "woken_byte_ratio": b16 / b1,
                          "quotient": (b16 / b1) / (ms16 / ms1),
                          "routed_only_byte_ratio": Wm / Wm1},
        "kernel_path": "moe_fused_kernel (one launch per layer)" if fused else "router + gate/up + down launches",
        "roofline": {"bound": "hbm", "kernel": "moe_fused_kernel<2> (k=16)" if fused else "multi-launch",
                     "achieved": layer_bytes / (ms16 / N_LAYERS * 1e-3) / 1e9, "peak": peak_bw, "unit": "GB/s",
                     "frac": layer_bytes / (ms16 / N_LAYERS * 1e-3) / 1e9 / peak_bw,
                     "traffic": ncu_traffic("moe_fused_kernel_shared", layer_bytes) if fused else None,
                     "per_launch_us": ms16 / N_LAYERS * 1e3,
                     "per_launch_note": "timed k=16 pass (CUDA-graph replay) / its 40 launches",
                     "isolated_launch_us": per_launch_ms * 1e3,
                     "algorithmic_bytes_per_launch": layer_bytes},
        "device_error": dfv.read_device_error(ws),
    }
    del layers, Ls
    return res


def wide_section(args, dev, rank, barrier, dfv, inputs, peak_bw):
    """Layers wider than the single-launch bf16 kernel takes (d_ff > 768), on
    the general router + gate/up + down + combine path: 8 distinct layers per
    shape (more than L2 holds), k = 16 and k = 1, graph replay.  Bytes are
    each layer's woken experts plus its router."""
    shapes = [("OLMoE-like: d=2048, E=64, top-8, d_ff=1024", inputs.LayerShape(d=2048, n_experts=64, top_k=8, d_ff=1024)),
              ("Qwen1.5-MoE-like: d=2048, E=60, top-4, d_ff=1408",
               inputs.LayerShape(d=2048, n_experts=60, top_k=4, d_ff=1408)),
              ("Qwen3-235B-like: d=4096, E=128, top-8, d_ff=1536",
               inputs.LayerShape(d=4096, n_experts=128, top_k=8, d_ff=1536))]
    nl = 8
    res = []
    for name, shape in shapes:
        progress("wide layers: " + name)
        layers = [inputs.make_layer(shape, seed=2000 + 10 * rank + l, device=dev) for l in range(nl)]
        Ls = [dfv.Layer(w) for w in layers]
        ws = dfv.alloc_workspace(dfv.workspace_size(Ls[0], KBLOCK), device=dev)
        eb, rb = layers[0].expert_bytes(), layers[0].router_bytes()
        row = {"shape": name, "layers": nl}
        for k in (KBLOCK, 1):
            x = inputs.make_hidden(k, shape.d, "bf16", seed=2100 + k, device=dev)
            out = torch.empty_like(x)
            nws = torch.zeros(nl, dtype=torch.int32, device=dev)

            def fn():
                for l in range(nl):
                    dfv.moe_block_forward(Ls[l], x, ws, out=out, n_woken=nws[l:l + 1])

            ms = graph_time(fn, max(3, args.warmup), max(5, args.steps // 2), barrier)
            W = nws.to(torch.int64).cpu()
            nbytes = float(W.sum().item() * eb + nl * rb)
            row["k%d" % k] = {"layer_us": ms * 1e3 / nl, "gbs": achieved_gbs(nbytes, ms),
                              "frac_of_measured_hbm": achieved_gbs(nbytes, ms) / peak_bw,
                              "woken_mean": float(W.double().mean().item()), "path": dfv.last_layer_path()}
        row["device_error"] = dfv.read_device_error(ws)
        res.append(row)
        del layers, Ls, ws
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dfv", choices=["dfv", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-mxfp4", action="store_true", help="skip the mxfp4-expert section")
    ap.add_argument("--no-shared", action="store_true", help="skip the shared-expert section")
    ap.add_argument("--no-wide", action="store_true", help="skip the section of layers wider than the fused kernel takes")
    ap.add_argument("--no-q8", action="store_true", help="skip the 8-bit-expert section")
    ap.add_argument("--no-batch", action="store_true", help="skip the batched-verify section")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=40, help="layers per step (profiling runs only)")
    args = ap.parse_args()
    global N_LAYERS
    N_LAYERS = args.layers
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
