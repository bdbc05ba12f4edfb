"""Device-timed benchmark of paged-KV decode attention on GB300.

One step = one pass of the whole hot path over one batch: the scheduling
metadata kernel, the split-KV kernel and the LSE combine kernel. Inputs are
seeded synthetic tensors resident in HBM before timing starts. Workloads whose
KV is smaller than twice the L2 (129 MB) rotate through enough copies of the
inputs that every step reads its KV from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the workload (the path shards by request / KV head
with no exchange); value = all ranks' calls / max-over-ranks time.
"""
import argparse
import ctypes
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

L2_BYTES = 129 * 1024 * 1024
# the largest single-GPU workload (2.15 GB of e4m3 KV per call); the others via --workload
DEFAULT_WORKLOAD = "fp8_gqa"
METRIC = "decode attn us/call (KV-read HBM GB/s, % of GB300 peak), device-timed"
# the pages' own figure for this exact workload (MetaX C500, 25% compute slice, graph mode, batch 8)
PAGE_NUMBERS_US = {"gqa_bf16_b8": 248.43}
# the pages' timing protocol (MetaX PR page, note above its performance table):
# 10 groups of 100 calls, median of the group means
PROTOCOL_GROUPS, PROTOCOL_CALLS = 10, 100
MAIN_KERNEL_SOURCES = {
    "gqa": "paged_kv_cache_60_gb300/csrc/decode_gqa.cu",
    "mla": "paged_kv_cache_60_gb300/csrc/decode_mla.cu",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--eager", action="store_true", help="launch every step from the host (no CUDA graph)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed
def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if n > 0 and torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML every ~2 ms."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, bus_id):
        self.samples, self.reasons, self.max_mhz, self.ok = [], 0, None, False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            assert self.nvml.nvmlInit_v2() == 0
            self.dev = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.dev)) != 0:
                assert self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev)) == 0
            m = ctypes.c_uint(0)
            self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(m))
            self.max_mhz = m.value
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        mhz, r = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        get_r = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if get_r(self.dev, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(v for k, v in self.REASONS.items() if self.reasons & k),
                "samples": len(self.samples)}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source): the measured copy bandwidth
    and cuBLAS bf16 GEMM rate of this machine, else one earlier GB300 measurement."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def profile_traffic(kernel_key, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (sha recorded in the summary)."""
    src = os.path.join(ROOT, MAIN_KERNEL_SOURCES[kernel_key])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", f"{kernel_key}_decode_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for ln in open(path):
        if ":" in ln and ln.startswith("- "):
            k, v = ln[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def make_desc(da, w):
    s = w.spec
    return da.Desc.make(B=s.B, H_kv=s.H_kv, G=s.G, D_qk=s.D_qk, D_v=s.D_v, page_size=s.page_size,
                        max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages, kv_dtype=s.kv_dtype,
                        splits=s.splits, softmax_scale=s.softmax_scale, s_q=s.s_q, window=s.window,
                        topk=s.topk)


class DevCopy:
    def __init__(self, torch, w, desc, da):
        dev = "cuda"
        self.q = w.q.to(dev)
        self.k_pool = w.k_pool.to(dev)
        self.v_pool = w.v_pool.to(dev) if w.v_pool is not None else None
        self.k_scale = w.k_scale.to(dev) if w.k_scale is not None else None
        self.v_scale = w.v_scale.to(dev) if w.v_scale is not None else None
        self.block_table = w.block_table.to(dev)
        self.cache_seqlens = w.cache_seqlens.to(dev)
        self.sinks = w.sinks.to(dev) if w.sinks is not None else None
        self.indices = w.indices.to(dev) if w.indices is not None else None
        s = w.spec
        self.meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device=dev)
        self.out = torch.empty(s.B, s.s_q * s.H_q, s.D_v, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(s.B, s.s_q * s.H_q, dtype=torch.float32, device=dev)
        # one new token per request, written at its last position (decode_attn_append_kv)
        from workloads import make_append_batch
        k_new, v_new, pos = make_append_batch(w, seed=s.seed + 1)
        self.k_new = k_new.to(dev)
        self.v_new = v_new.to(dev) if v_new is not None else None
        self.positions = pos.to(dev)

    def append(self, da, desc, stream):
        da.append_kv(desc, self.k_new, self.v_new, self.positions, self.block_table, self.k_pool, self.v_pool,
                     self.k_scale, self.v_scale, stream=stream)

    def sched(self, da, desc, stream):
        da.sched_meta(desc, self.cache_seqlens, self.meta, stream=stream)

    def fwd(self, da, desc, stream, **kw):
        da.fwd(desc, self.q, self.k_pool, self.v_pool, self.k_scale, self.v_scale, self.block_table,
               self.cache_seqlens, self.meta, self.out, self.lse, stream=stream, sinks=self.sinks,
               indices=self.indices, **kw)

    def step(self, da, desc, stream, **kw):
        self.sched(da, desc, stream)
        self.fwd(da, desc, stream, **kw)


def append_at_scale(torch, da, spec, stream, hbm_peak, reps=50):
    """decode_attn_append_kv on a large batch of the workload's KV format
    (65536 requests, or 262144 latent tokens: 0.2-0.5 GB moved per call, so
    that launch and tail costs are a small share), one page of 16 slots per
    request, new rows rotating over enough copies to exceed 2x L2: the append
    kernel's HBM roofline, which decode batch sizes are too small to show."""
    P = 16
    mla = spec.kv_dtype == da.KV_MLA656
    B = 262144 if mla else 65536
    H, D = (1, 576) if mla else (spec.H_kv, spec.D_qk)
    g = torch.Generator(device="cuda").manual_seed(spec.seed + 3)
    desc = da.Desc.make(B=B, H_kv=H, G=spec.G, D_qk=D, D_v=spec.D_v, page_size=P, max_pages_per_seq=1,
                        num_pages=B, kv_dtype=spec.kv_dtype)
    if mla:
        k_pool, v_pool = torch.zeros(B, P, 1, 656, dtype=torch.uint8, device="cuda"), None
        row_bytes = 2 * 576 + 656
    else:
        dt = torch.uint8 if spec.kv_dtype == da.KV_FP8 else torch.bfloat16
        k_pool = torch.zeros(B, P, H, D, dtype=dt, device="cuda")
        v_pool = torch.zeros_like(k_pool)
        es = 1 if spec.kv_dtype == da.KV_FP8 else 2
        row_bytes = 2 * H * D * (2 + es)
    scales = torch.rand(H, generator=g, device="cuda") * 0.05 + 0.01
    bt = torch.randperm(B, generator=g, device="cuda").to(torch.int32).view(B, 1)
    pos = torch.randint(0, P, (B,), generator=g, device="cuda", dtype=torch.int32)
    in_bytes = B * H * D * 2 * (1 if mla else 2)
    ncopy = max(1, -(-2 * L2_BYTES // in_bytes))
    rows = [(torch.randn(B, H, D, generator=g, device="cuda").to(torch.bfloat16),
             None if mla else torch.randn(B, H, D, generator=g, device="cuda").to(torch.bfloat16))
            for _ in range(ncopy)]

    def call(k):
        kn, vn = rows[k % ncopy]
        da.append_kv(desc, kn, vn, pos, bt, k_pool, v_pool, None if mla else scales, None if mla else scales,
                     stream=stream)
    with torch.cuda.stream(stream):
        for k in range(5):
            call(k)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(reps):
            call(k)
        b.record(stream)
        torch.cuda.synchronize()
    us = a.elapsed_time(b) / reps * 1000.0
    nbytes = B * row_bytes + 8 * B
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"requests": B, "us_per_call": round(us, 3), "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
            "frac": round(gbs / hbm_peak, 4), "bound": "hbm",
            "note": "one page of 16 slots per request, random pages and slots, eager launches, "
                    "new rows rotating over %d copies" % ncopy}


def oracle_time_per_call(w, budget_s):
    """Oracle (float64, host cores) on a bounded sample of (request, KV head)
    units, scaled to one whole call. Returns (us_per_call, cores, sample text)."""
    import oracle
    s = w.spec
    if s.topk > 0:
        attend = oracle.attend_sparse
    elif s.s_q > 1 or s.window > 0 or s.sinks:
        attend = oracle.attend_multi
    else:
        attend = oracle.attend
    units_all = [(b, h) for b in range(s.B) for h in range(s.H_kv)]
    def unit_cost(L):   # tokens one (request, KV head) unit reads
        if s.topk > 0:
            return min(L, s.topk)
        if s.window > 0:
            return min(L, s.window + s.s_q - 1)
        return L
    cost = {u: unit_cost(w.lengths[u[0]]) for u in units_all}
    total_cost = sum(cost.values())
    # cheap probe on the shortest unit to size the sample
    probe = min(units_all, key=lambda u: cost[u])
    t0 = time.perf_counter()
    attend(w, heads=[probe])
    t_probe = max(time.perf_counter() - t0, 1e-6)
    per_token = t_probe / max(1, cost[probe])
    cores = oracle.num_threads()
    # spread units in a fixed order, take a prefix until the budget is used
    order = sorted(units_all, key=lambda u: (u[0] * 7919 + u[1] * 104729) % len(units_all))
    sample, est = [], 0.0
    for u in order:
        sample.append(u)
        est += per_token * cost[u] / max(1, min(cores, len(sample)))
        if est >= budget_s:
            break
    reps = 1
    t0 = time.perf_counter()
    attend(w, heads=sample)
    el = time.perf_counter() - t0
    while el * (reps + 1) / reps < budget_s and reps < 1000:
        attend(w, heads=sample)
        reps += 1
        el = time.perf_counter() - t0
    sample_cost = sum(cost[u] for u in sample)
    us = el / reps * (total_cost / sample_cost) * 1e6
    text = (f"{len(sample)} of {len(units_all)} (request, KV head) units, {sample_cost} of {total_cost} "
            f"tokens x heads, {reps} repetition(s), scaled to one whole call")
    return us, cores, text


# ----------------------------------------------------------------------------- arms
def workload_config(name, w):
    """The workload's shape, as both arms report it."""
    spec = w.spec
    return {"workload": name, "desc": spec.description, "B": spec.B, "s_q": spec.s_q, "window": spec.window,
            "sinks": spec.sinks, "topk": spec.topk, "H_q": spec.H_q, "H_kv": spec.H_kv, "D_qk": spec.D_qk,
            "D_v": spec.D_v, "page_size": spec.page_size, "splits": spec.splits, "kv_bytes_per_call": w.kv_bytes()}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from workloads import make_workload, spec_by_name
    w = make_workload(spec_by_name(args.workload))
    # each step times the oracle on a bounded sample; the whole run stays within a few minutes
    budget = max(0.05, min(4.0, 150.0 / (args.steps + args.warmup + 1)))
    oracle_time_per_call(w, budget)
    times = []
    cores, text = 0, ""
    for _ in range(args.steps):
        us, cores, text = oracle_time_per_call(w, budget)
        times.append(us)
    v = statistics.median(times)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "us/call", "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": round(v / 1000.0, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args.workload, w),
            "cpu_baseline": {"value": round(v, 3), "unit": "us/call", "cores": cores, "kind": "oracle",
                             "sample": text},
            "e2e": {"value": round(v, 3), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_60_gb300 as da
    from paged_kv_cache_60_gb300 import build as dabuild
    from workloads import make_workload, spec_by_name

    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        dabuild.build()
    dist_barrier(world)
    da.load_library()
    spec = spec_by_name(args.workload)
    w = make_workload(spec)
    desc = make_desc(da, w)
    kv_bytes = w.kv_bytes()
    copies = 1 if kv_bytes >= 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / kv_bytes))
    devs = [DevCopy(torch, w, desc, da) for _ in range(copies)]
    stream = torch.cuda.Stream()
    steps, warm = args.steps, max(3, args.warmup)
    # A call is decode_attn_fwd (split-KV kernel + combine) on scheduling
    # metadata built once beforehand and reused, as every layer of a decode
    # step reuses it; decode_attn_sched_meta is timed on its own and together
    # with the call (sched_meta_us, with_sched_meta_us).
    # split-KV kernel + combine; a fixed split count of 2..8 merges inside the split-KV kernel
    launches_per_step = 1 if (spec.kv_dtype != da.KV_MLA656 and 2 <= spec.splits <= 8) else 2

    # ---- CUDA graphs of several calls each (calls rotate over the input
    # copies, so consecutive calls read different memory), or eager launches.
    # A graph holds cpg calls; n calls replay it n // cpg times plus a graph of
    # the remaining n % cpg calls, so exactly n calls run.
    cpg = copies * max(1, -(-8 // copies))
    fns = {"fwd": lambda d: d.fwd(da, desc, stream), "both": lambda d: d.step(da, desc, stream),
           "sched": lambda d: d.sched(da, desc, stream), "append": lambda d: d.append(da, desc, stream),
           "append_fwd": lambda d: (d.append(da, desc, stream), d.fwd(da, desc, stream))}
    graph_cache = {}
    with torch.cuda.stream(stream):
        for d in devs:
            d.step(da, desc, stream)
        torch.cuda.synchronize()

    def graph_of(which, ncalls):
        key = (which, ncalls)
        if key not in graph_cache:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    for j in range(ncalls):
                        fns[which](devs[j % copies])
            torch.cuda.synchronize()
            graph_cache[key] = g
        return graph_cache[key]

    def run_calls(n, which="fwd"):
        if args.eager:
            for k in range(n):
                fns[which](devs[k % copies])
            return
        for _ in range(n // cpg):
            graph_of(which, cpg).replay()
        if n % cpg:
            graph_of(which, n % cpg).replay()

    def timed(which, n):
        if not args.eager:  # capture before timing
            graph_of(which, cpg)
            if n % cpg:
                graph_of(which, n % cpg)
        with torch.cuda.stream(stream):
            run_calls(min(n, 3 * cpg), which)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run_calls(n, which)
            b.record(stream)
            torch.cuda.synchronize()
        return a.elapsed_time(b) / n * 1000.0

    bus = torch.cuda.get_device_properties(local)
    bus_id = getattr(bus, "pci_bus_id", None)
    bus_str = f"{getattr(bus, 'pci_domain_id', 0):08x}:{bus_id:02x}:{getattr(bus, 'pci_device_id', 0):02x}.0" \
        if isinstance(bus_id, int) else ""

    if not args.eager:
        graph_of("fwd", cpg)
        if steps % cpg:
            graph_of("fwd", steps % cpg)
        if warm % cpg:
            graph_of("fwd", warm % cpg)
    with torch.cuda.stream(stream):
        run_calls(warm)
        torch.cuda.synchronize()
        dist_barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk = ClockSampler(bus_str)
        clk.__enter__()
        e0.record(stream)
        run_calls(steps)
        e1.record(stream)
        torch.cuda.synchronize()
        clk_region_samples = len(clk.samples)
        dist_barrier(world)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ms = dist_max(ms, world)
    value_us = ms * 1000.0 / world     # whole-job: world replicas per step time
    # the pages' protocol (10 groups of 100 calls, median of the group means),
    # whatever --steps is; the clock sampler keeps running through it
    if not args.eager:
        graph_of("fwd", cpg)
        if PROTOCOL_CALLS % cpg:
            graph_of("fwd", PROTOCOL_CALLS % cpg)
    group_us = [timed("fwd", PROTOCOL_CALLS) for _ in range(PROTOCOL_GROUPS)]
    clk.__exit__(None, None, None)
    median_group_us = statistics.median(group_us)
    err = da.get_error(devs[0].meta, stream=stream)

    # ---- dominant kernel: events around the split-KV kernel, every step (eager)
    n_main = min(steps, 400)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_main)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize()
        for k, (a, b) in enumerate(evs):
            devs[k % copies].fwd(da, desc, stream, main_begin=a, main_end=b)
        torch.cuda.synchronize()
    event_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    n_side = max(3, min(steps, 200))
    # the same calls launched eagerly; and, for workloads that fit in L2, one input copy (L2-hot)
    saved_eager = args.eager
    args.eager = True
    eager_us = timed("fwd", n_side)
    args.eager = saved_eager
    hot_us = None
    if copies > 1:
        fns["hot"] = lambda d: devs[0].fwd(da, desc, stream)
        hot_us = timed("hot", n_side)
    sched_us = timed("sched", n_side)
    both_us = timed("both", n_side)
    append_us = timed("append", n_side)
    append_fwd_us = timed("append_fwd", n_side)
    n_app = sum(1 for L in w.lengths if L > 0)
    if spec.kv_dtype == da.KV_MLA656:
        app_bytes = n_app * (2 * (spec.D_qk) + 656) + 8 * spec.B
    else:
        es = 1 if spec.kv_dtype == da.KV_FP8 else 2
        app_bytes = n_app * 2 * spec.H_kv * spec.D_qk * (2 + es) + 8 * spec.B
    hbm_peak0, _, _ = load_peaks()
    app_scale = append_at_scale(torch, da, spec, stream, hbm_peak0)
    append = {"us_per_call": round(append_us, 3), "algorithmic_bytes": app_bytes, "at_scale": app_scale,
              "gbs": round(app_bytes / (append_us * 1e-6) / 1e9, 1), "with_fwd_us": round(append_fwd_us, 3),
              "call": "decode_attn_append_kv: one new token per request into its page slot "
                      "(bf16 rows in, pool format out), then optionally decode_attn_fwd"}
    hbm_peak, tc_peak, peak_kind = load_peaks()
    key = "mla" if spec.kv_dtype == da.KV_MLA656 else "gqa"
    traffic = profile_traffic(key, args.workload)
    # The split-KV kernel's time per launch: the per-call time of the timed
    # region (one split-KV launch per call, plus the PDL-chained combine where
    # one runs), so it can never exceed `value` and reads as a lower bound on
    # the kernel's own rate. Events around single eager launches break the
    # dependent-launch chain and add their own overhead; they are reported
    # beside it only as a cross-check.
    main_ms = value_us * 1e-3
    hbm_achieved = kv_bytes / (main_ms * 1e-3) / 1e9
    if key == "mla":
        # tensor-bound: 2 (D_qk + D_v) flops per (token, query head, query token); 424 flop per KV byte
        ntok = sum(min(L, spec.topk) for L in w.lengths) if spec.topk > 0 else sum(w.lengths)
        flops = 2.0 * (spec.D_qk + spec.D_v) * spec.H_q * spec.s_q * ntok
        achieved = flops / (main_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": round(achieved / tc_peak, 4), "traffic": traffic,
                    "peak_kind": peak_kind + " (cuBLAS bf16 burst)", "flops_per_launch": flops,
                    "hbm_achieved_gbs": round(hbm_achieved, 1), "hbm_frac": round(hbm_achieved / hbm_peak, 4)}
    else:
        roofline = {"bound": "hbm", "achieved": round(hbm_achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(hbm_achieved / hbm_peak, 4), "traffic": traffic, "peak_kind": peak_kind}
    roofline.update({"kernel": f"{key}_decode_kernel", "main_kernel_us": round(main_ms * 1000.0, 3),
                     "algorithmic_bytes_per_launch": kv_bytes,
                     "kernel_time_source": "per-call time of the timed region (CUDA events on the launch "
                                           "stream around all K calls): split-KV kernel%s per call"
                                           % ("" if launches_per_step == 1 else " + PDL-chained combine"),
                     "eager_event_split_kv_us": round(event_ms * 1000.0, 3)})
    assert roofline["main_kernel_us"] <= round(value_us, 4) + 1e-3

    # ---- end to end: host buffers in, host results out, every step. Two device
    # input sets: step k + 1's inputs cross the host link on a copy stream while
    # step k computes (the link, ~210 GB/s here, bounds the large workloads);
    # every step still copies all of its inputs in and reads its results back.
    e2e = None
    with torch.cuda.stream(stream):
        host = {k: getattr(devs[0], k).cpu().pin_memory() for k in
                ("q", "k_pool", "v_pool", "k_scale", "v_scale", "block_table", "cache_seqlens", "sinks",
                 "indices")
                if getattr(devs[0], k) is not None}
        h_out = torch.empty_like(devs[0].out, device="cpu").pin_memory()
        h_lse = torch.empty_like(devs[0].lse, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        n_e2e = max(3, min(steps, 50))
        sets = devs[:2] if copies >= 2 else [devs[0], DevCopy(torch, w, desc, da)]
        cstream = torch.cuda.Stream()
        ready = [torch.cuda.Event() for _ in sets]  # inputs of set i copied in
        done = [torch.cuda.Event() for _ in sets]   # the step that last used set i has finished

        def copy_in(k):
            d = sets[k % 2]
            cstream.wait_event(done[k % 2])
            with torch.cuda.stream(cstream):
                for name, t in host.items():
                    getattr(d, name).copy_(t, non_blocking=True)
                ready[k % 2].record(cstream)

        def compute(k):
            d = sets[k % 2]
            stream.wait_event(ready[k % 2])
            d.step(da, desc, stream)
            h_out.copy_(d.out, non_blocking=True)
            h_lse.copy_(d.lse, non_blocking=True)
            done[k % 2].record(stream)

        def run_e2e(n, start=None):
            if start is not None:
                cstream.wait_event(start)
            copy_in(0)
            for k in range(n):
                if k + 1 < n:
                    copy_in(k + 1)
                compute(k)
        run_e2e(3)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_e2e(n_e2e, start=a)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_us = a.elapsed_time(b) / n_e2e * 1000.0
        e2e_us = dist_max(e2e_us, world) / world
        e2e = {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
               "includes": "pinned host inputs to device (next step's copy overlapping this step's compute), "
                           "decode_attn_sched_meta, decode_attn_fwd, out and lse to host",
               "d2h_bytes_per_step": d2h, "steps": n_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, cores, text = oracle_time_per_call(w, 12.0)
        cpu = {"value": round(us, 1), "unit": "us/call", "cores": cores, "kind": "oracle", "sample": text}

    if rank == 0:
        page = PAGE_NUMBERS_US.get(args.workload)
        line = {
            "metric": METRIC, "value": round(value_us, 4), "unit": "us/call", "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": round(ms, 6), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": round(value_us / page, 5) if page else None,
            "dtype": {da.KV_BF16: "bf16", da.KV_FP8: "fp8-e4m3 kv / bf16 q,out"}.get(
                spec.kv_dtype, "fp8-e4m3 656-byte kv dequantised to bf16 / bf16 q,out"),
            "data": "synthetic",
            "config": {**workload_config(args.workload, w),
                       "l2": ("inputs rotate over %d copies (%.0f MB > 2x L2)" % (copies, copies * kv_bytes / 1e6))
                       if copies > 1 else "inputs larger than 2x L2",
                       "launch": "eager" if args.eager else f"cuda graphs of {cpg} calls",
                       "call": "decode_attn_fwd (split-KV kernel + PDL-chained combine) on scheduling "
                               "metadata built once and reused; decode_attn_sched_meta timed separately",
                       "parallelism": f"replicas x{world}"},
            "kv_read_gbs": round(kv_bytes / (ms * 1e-3) / 1e9 * world, 1),
            "median_of_10_groups_us": round(median_group_us, 3),
            "protocol": "%d groups of %d calls, CUDA events per group, median of the group means"
                        % (PROTOCOL_GROUPS, PROTOCOL_CALLS),
            "eager_us": round(eager_us, 3),
            "l2_hot_us": None if hot_us is None else round(hot_us, 3),
            "sched_meta_us": round(sched_us, 3),
            "with_sched_meta_us": round(both_us, 3),
            "append": append,
            "roofline": roofline,
            "clocks": dict(clk.summary() or {}, window="timed region (%d samples) and the 10 x 100-call protocol "
                           "that follows it" % clk_region_samples) if clk.summary() else None,
            "gpu_launches": launches_per_step * steps,
            "device_error": err,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
