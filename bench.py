"""Benchmark: one sharded MLA decode step (all shards' partial attention, then
the LSE combine) on the bimodal agentic batch, on N GPUs of one node.

Workload (seeded, synthetic; stands in for the agentic long-context trace of
"Decode Context Parallelism", section 2.1): 32 requests, 64 query heads,
q_len 1, bf16 paged latent cache (576 = 512 c_kv + 64 k_rope, page size 64,
pages scattered by a random block table), context lengths from a stratified
log-uniform mix (~47% below 64k, ~18% below 8k, median ~67k, tail to ~1M,
total <= 4M tokens), 4 logical shards interleaved, merged by LSE combine.

metric: KV HBM GB/s = algorithmic KV bytes (every token < L_b once, 1152 B)
        / device time of one whole step.  Inputs (3.4 GB) exceed L2.
Also printed: decode steps/s per layer, the partial kernel's roofline
fraction against the measured copy bandwidth, the oracle timed on host
cores (cpu_baseline), and the same metric end to end through host buffers
(e2e: pinned host -> device copies of the step's inputs and device -> host
read of its outputs inside the timed region).

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload.

With --gpus N > 1 (one process per GPU under torchrun) the step is the
multi-GPU DCP step over one global batch ("Decode Context Parallelism",
section 4.1): rank r holds shard r of every request's cache and query heads
[r H/N, (r + 1) H/N); query all-gather, partial, head-sliced all-to-all of
the partials, combine (strong scaling).  --independent runs N independent
batches instead.
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

METRIC = "MLA sharded decode: KV HBM GB/s (% of ~8 TB/s peak), decode steps/s per layer"
DEFAULT_CONFIG = 2     # the bimodal agentic batch the metric is quoted on
GQA_CONFIG = 6         # the grouped-query backend on the same length mix


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s: the sustained measurement (the
    partial kernel runs inside a long loop of steps), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured bf16_tflops_sustained"
    except Exception:
        return 1700.0, "fallback"


def kernel_sha(kernel_src):
    return hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]


def traffic_for(kernel_src, workload):
    """ncu DRAM bytes (read + write) per launch of the partial kernel on this
    workload, as recorded in profiles/traffic.json for this exact kernel
    source; None when no record matches (the kernel changed since)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        ent = rec[kernel_sha(kernel_src)][workload]
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            res = parse_clock_samples(f)
        os.unlink(self.path)
        return res


def parse_clock_samples(lines):
    """Summarise nvidia-smi rows of ClockSampler.FIELDS (csv, no header, no
    units): median SM clock, max SM clock, and every throttle reason seen
    active in any sample."""
    sms, maxes, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sms.append(float(parts[1]))
            maxes.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sms) if sms else None,
            "sm_max_mhz": max(maxes) if maxes else None,
            "reasons": sorted(reasons), "samples": len(sms)}


def dist_setup(args, backend="nccl"):
    """World, rank and local rank from the launcher's environment; joins the
    process group when there is more than one rank.  The reference arm runs
    on rank 0 alone and joins nothing."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def rank_workload_params(config, rank, requests=0, wuv=False):
    """Arguments of the batch rank ``rank`` decodes: rank 0 the configuration
    itself, every other rank an independently seeded batch of the same shape
    (weak scaling: ranks share nothing on the data path).  ``requests`` > 0
    keeps the first K requests (profiling runs only)."""
    import mla_inputs as mi
    p = mi.config_params(config)
    if rank > 0:
        p["seed"] += 1000 * rank
        if config == 2:
            p["seq_lens"] = mi.agentic_lengths(p["seed"], p["batch"])
    if requests:
        p["name"] += f"-first{requests}"
        p["batch"] = requests
        p["seq_lens"] = list(p["seq_lens"])[:requests]
    if wuv and not p.get("with_w_uv"):
        p["name"] += "+wuv"
        p["with_w_uv"] = True
    return p


_WORKLOADS = {}


def rank_workload(config, rank, requests=0, pinned=True, wuv=False):
    """The rank's workload, generated once per process (the shard-count sweep
    runs one cache at several shard counts and layouts)."""
    import mla_inputs as mi
    key = (config, rank, requests, pinned, wuv)
    if key not in _WORKLOADS:
        _WORKLOADS[key] = mi.build_workload(pinned=pinned,
                                            **rank_workload_params(config, rank, requests, wuv))
    return _WORKLOADS[key]


def reduce_over_ranks(dist, times, kv_bytes, device):
    """Max of the per-rank times (the slowest rank ends the job) and sum of
    the per-rank KV bytes (the whole job's work)."""
    import torch
    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    b = torch.tensor([float(kv_bytes)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return t.tolist(), b.item()


def cpu_sample(w, budget_s, oracle, threads=0):
    """Oracle on whole requests (all heads, unsharded, W_UV if present) until
    about ``budget_s`` of CPU time; returns (KV bytes covered, seconds, desc).
    ``threads`` > 0 runs the oracle on that many host threads."""
    import numpy as np
    oracle.set_threads(threads)
    order = np.argsort(w.seq_lens)            # short to long, one of each band first
    picked, t_used, kv_bytes = [], 0.0, 0
    per = 1152 if w.kv_dtype == "bf16" else 580
    H, q_len = w.num_heads, w.q_len
    for b in order[::max(1, len(order) // 8)]:
        rows = np.arange(b * q_len * H, (b + 1) * q_len * H, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.reference_step(w, rows=rows)
        dt = time.perf_counter() - t0
        picked.append(int(b))
        t_used += dt
        kv_bytes += int(w.seq_lens[b]) * per
        if t_used >= budget_s:
            break
    desc = (f"requests {picked} of the workload (all {H} heads each, unsharded "
            f"attention{', W_UV' if w.w_uv is not None else ''}), "
            f"{int(sum(int(w.seq_lens[b]) for b in picked))} tokens")
    return kv_bytes, t_used, desc


def gqa_cpu_sample(w, budget_s, oracle, threads=0):
    """The GQA oracle on whole requests (all heads, unsharded) until about
    ``budget_s`` of CPU time; returns (K/V bytes covered, seconds, desc)."""
    import numpy as np
    oracle.set_threads(threads)
    order = np.argsort(w.seq_lens)
    picked, t_used, kv_bytes = [], 0.0, 0
    per = 2 * w.num_kv_heads * w.head_dim * 2
    H, q_len = w.num_heads, w.q_len
    for b in order[::max(1, len(order) // 8)]:
        rows = np.arange(b * q_len * H, (b + 1) * q_len * H, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.gqa_attend(w, shard=-1, rows=rows)
        t_used += time.perf_counter() - t0
        picked.append(int(b))
        kv_bytes += int(w.seq_lens[b]) * per
        if t_used >= budget_s:
            break
    desc = (f"requests {picked} of the workload (all {H} heads each, unsharded attention), "
            f"{int(sum(int(w.seq_lens[b]) for b in picked))} tokens")
    return kv_bytes, t_used, desc


def run_reference(args, world, rank):
    if rank != 0:
        return
    import mla_inputs as mi
    import oracle
    if args.config == GQA_CONFIG:
        w = mi.config_gqa_workload()
        sample, name = gqa_cpu_sample, mi.GQA_CONFIG_NAME
        kv_dtype = "bf16"
    else:
        w = mi.config_workload(args.config)
        sample, name = cpu_sample, mi.CONFIG_NAMES[args.config]
        kv_dtype = w.kv_dtype
    threads = oracle.num_threads()
    # one step = the oracle over a bounded sample of the workload
    budget = args.ref_step_seconds
    results = []
    for step in range(args.warmup + args.steps):
        kv_bytes, dt, desc = sample(w, budget, oracle)
        if step >= args.warmup:
            results.append((kv_bytes, dt))
    tot_b = sum(r[0] for r in results)
    tot_t = sum(r[1] for r in results)
    value = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / len(results) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "batch": w.batch,
                       "heads": w.num_heads, "q_len": w.q_len, "num_shards": w.num_shards,
                       "layout": w.layout, "kv_dtype": kv_dtype,
                       "total_tokens": w.total_tokens},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class Case:
    """One benchmark workload on the device: pinned host inputs and their
    device copies, output buffers, and the step (the library calls)."""

    def __init__(self, name, kv_bytes, config, pairs, outputs, workspace, step, dtype, kernel,
                 kernel_src, cpu, flops=0.0, combine_bytes=0.0, tensor_bound=False,
                 tensor_fp8=False, launches_per_step=4, fused_step=False):
        self.name, self.kv_bytes, self.config = name, kv_bytes, config
        self.pairs = pairs            # [(pinned host tensor, device tensor)] copied per e2e step
        self.outputs = outputs        # [(device tensor, pinned host tensor)] read per e2e step
        self.workspace, self.step, self.dtype, self.kernel = workspace, step, dtype, kernel
        self.kernel_src = kernel_src  # source file of the timed kernel (traffic record key)
        self.cpu = cpu                # cpu(budget_s, oracle) -> (KV bytes, seconds, sample)
        self.flops = flops            # useful MMA flops of the partial kernel per step
        self.combine_bytes = combine_bytes   # bytes the combine kernel reads and writes
        self.tensor_bound = tensor_bound     # the dense contractions bound the partial kernel
        self.tensor_fp8 = tensor_fp8         # the contractions run on e4m3 operands
        self.launches_per_step = launches_per_step
        # fused_step: the step is one mla_decode_step call (plan, partial,
        # combine); the combine is timed from the end of the partial kernel
        self.fused_step = fused_step


def visible_pairs(seq_lens, q_len, causal):
    """Sum over requests and query positions of the tokens each query sees."""
    tot = 0
    for L in seq_lens:
        L = int(L)
        tot += sum(max(0, L - q_len + i + 1) for i in range(q_len)) if causal else L * q_len
    return tot


def _pinned_pair(h, dev):
    h = h.pin_memory() if not h.is_pinned() else h
    return h, h.to(dev)


def mla_case(args, rank, dev, stream, ev_p, ev_k, ev_c):
    import numpy as np
    import torch

    import mla_inputs as mi
    import sequence_sharded_mla_gb300 as mla
    w = rank_workload(args.config, rank, args.requests, wuv=getattr(args, "wuv", False))
    B, H, q_len = w.batch, w.num_heads, w.q_len
    N = args.num_shards or w.num_shards
    layout = args.layout or w.layout
    key = ("device", args.config, rank, args.requests, getattr(args, "wuv", False))
    if key not in _WORKLOADS:
        q = _pinned_pair(torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16), dev)
        if w.kv_dtype == "bf16":
            kv = _pinned_pair(torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16), dev)
            sc = None
        else:
            kv = _pinned_pair(torch.from_numpy(w.kv), dev)
            sc = _pinned_pair(torch.from_numpy(w.kv_scale), dev)
        bt = _pinned_pair(torch.from_numpy(w.block_table), dev)
        sl = _pinned_pair(torch.from_numpy(w.seq_lens), dev)
        _WORKLOADS[key] = (q, kv, sc, bt, sl)
    q, kv, sc, bt, sl = _WORKLOADS[key]
    d_wuv = None
    if w.w_uv is not None:
        d_wuv = torch.from_numpy(w.w_uv.view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((B, q_len, H, 512 if d_wuv is None else 128), dtype=torch.bfloat16,
                      device=dev)
    lse = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    ws = torch.empty((mla.mla_decode_step_workspace_size(B, q_len, H, N),), dtype=torch.uint8,
                     device=dev)

    def step(i=None):
        # one call: plan, partial kernel (events around it recorded by the
        # library), then the combine that also merges split pieces
        if i is not None:
            ev_p[2 * i].record(stream)
            mla.mla_set_profile_events(ev_k[2 * i], ev_k[2 * i + 1])
        mla.mla_decode_step(q[1], kv[1], bt[1], sl[1], N, layout,
                            kv_scale=None if sc is None else sc[1], causal=w.causal,
                            w_uv=d_wuv, out=out, lse_out=lse, workspace=ws, stream=stream)
        if i is not None:
            mla.mla_set_profile_events(None, None)
            ev_c[i].record(stream)

    pairs = [q, kv, bt, sl] + ([sc] if sc is not None else [])
    outputs = [(out, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)),
               (lse, torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True))]
    name = w.name + (f"-n{N}-{layout}" if args.config == 3 else "")
    config = {"workload": name, "batch": B, "heads": H, "q_len": q_len,
              "num_shards": N, "layout": layout, "kv_dtype": w.kv_dtype,
              "causal": bool(w.causal), "fused_w_uv": d_wuv is not None,
              "total_tokens_per_gpu": w.total_tokens}
    fp8 = w.kv_dtype == "fp8"
    # the template instance the library launches: cache kind (0 whole
    # requests, 2 interleaved shards that do not divide the page), and for
    # bf16 whether the producer waits once for chunk groups 1 and 2 (four or
    # more boxes per chunk group)
    pad = layout == "interleaved" and 64 % N != 0
    kind = 2 if pad else 0
    boxes = 8 if pad else (N if layout == "interleaved" else 1)
    kernel = (f"mla_partial_fp8_kernel<{kind}, false>" if fp8 else
              f"mla_partial_kernel<{kind}, false, {'true' if boxes >= 4 else 'false'}>")
    rows = B * q_len * H
    flops = 2.0 * H * (576 + 512) * visible_pairs(w.seq_lens, q_len, w.causal)
    comb = N * rows * (512 * 4 + 4) + rows * ((128 if d_wuv is not None else 512) * 2 + 4)
    if d_wuv is not None:
        comb += d_wuv.numel() * 2
    return Case(config["workload"], w.kv_bytes(), config, pairs, outputs, ws, step,
                "e4m3" if fp8 else "bf16", kernel, "partial_fp8.cu" if fp8 else "partial.cu",
                lambda budget, orc, threads=0: cpu_sample(w, budget, orc, threads), flops=flops,
                combine_bytes=comb, tensor_bound=q_len * H > 64, tensor_fp8=fp8,
                launches_per_step=3, fused_step=True)


def gqa_case(args, rank, dev, stream, ev_p, ev_k, ev_c):
    import numpy as np
    import torch

    import mla_inputs as mi
    import sequence_sharded_mla_gb300 as mla
    lens = mi.agentic_lengths(6 + 1000 * rank, 32)
    name = mi.GQA_CONFIG_NAME
    if args.requests:   # a reduced copy (first K requests) for profiling runs
        lens, name = lens[:args.requests], name + f"-first{args.requests}"
    w = mi.build_gqa_workload(name, len(lens), 1, 64, 4, 128, lens, 2, "interleaved", False,
                              seed=6 + 1000 * rank, pinned=True)
    B, H, q_len, N, D = w.batch, w.num_heads, w.q_len, w.num_shards, w.head_dim
    f = lambda a: _pinned_pair(torch.from_numpy(a.view(np.int16)).view(torch.bfloat16), dev)
    q, k, v = f(w.q), f(w.k_cache), f(w.v_cache)
    bt = _pinned_pair(torch.from_numpy(w.block_table), dev)
    sl = _pinned_pair(torch.from_numpy(w.seq_lens), dev)
    part = torch.empty((N, B, q_len, H, D), dtype=torch.float32, device=dev)
    lsep = torch.empty((N, B, q_len, H), dtype=torch.float32, device=dev)
    out = torch.empty((B, q_len, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    ws = torch.empty((mla.gqa_workspace_size(B, q_len, H, w.num_kv_heads, N),), dtype=torch.uint8,
                     device=dev)

    def step(i=None):
        if i is not None:
            ev_p[2 * i].record(stream)
            mla.mla_set_profile_events(ev_k[2 * i], ev_k[2 * i + 1])
        mla.gqa_decode_partial(q[1], k[1], v[1], bt[1], sl[1], N, w.layout, causal=w.causal,
                               out_partial=part, lse_partial=lsep, workspace=ws, stream=stream)
        if i is not None:
            mla.mla_set_profile_events(None, None)
            ev_p[2 * i + 1].record(stream)
        mla.gqa_shard_combine(part, lsep, out=out, lse_out=lse, stream=stream)
        if i is not None:
            ev_c[i].record(stream)

    outputs = [(out, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)),
               (lse, torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True))]
    config = {"workload": name, "batch": B, "heads": H,
              "kv_heads": w.num_kv_heads, "head_dim": D, "q_len": q_len, "num_shards": N,
              "layout": w.layout, "kv_dtype": "bf16", "causal": bool(w.causal),
              "total_tokens_per_gpu": w.total_tokens}
    rows = B * q_len * H
    return Case(mi.GQA_CONFIG_NAME, w.kv_bytes(), config, [q, k, v, bt, sl], outputs, ws, step,
                "bf16", "gqa_partial_kernel", "gqa.cu",
                lambda budget, orc, threads=0: gqa_cpu_sample(w, budget, orc, threads),
                flops=2.0 * H * (D + D) * visible_pairs(w.seq_lens, q_len, w.causal),
                combine_bytes=N * rows * (D * 4 + 4) + rows * (D * 2 + 4))


L2_BYTES = 129 * 1024 * 1024


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(case, args):
    """The oracle as it stands on a bounded sample of the workload: all host
    cores, then one core (a smaller sample)."""
    import oracle
    kvb, dt, desc = case.cpu(args.cpu_seconds, oracle)
    cores = oracle.num_threads()
    kvb1, dt1, desc1 = case.cpu(args.cpu_seconds / 3.0, oracle, 1)
    oracle.set_threads(0)
    return {"value": kvb / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": desc, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "one_core": {"value": kvb1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                         "sample": desc1}}


def time_case(case, args, dev, stream, ev_p, ev_k, ev_c, barrier, flush):
    """Warm-up, then args.steps timed steps.  Returns per-step times (ms) of
    the whole step, the partial kernel alone, the calls before it and the
    combine, and the clock record.

    Inputs larger than L2 (flush is None): the timed steps run back to back
    with one event before and one after them, nothing in between (an event
    between two kernels keeps the second from launching early), and a second,
    untimed pass of as many steps records the events inside every step for
    the per-kernel breakdown.  Otherwise each step is timed between its own
    events, with L2 flushed before it."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    for _ in range(args.warmup):
        case.step()
    assert mla.mla_get_device_error(case.workspace, stream) == 0
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    if flush is None:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            case.step()
        t1.record(stream)
        barrier()
        total_ms = t0.elapsed_time(t1)
        for i in range(args.steps):
            case.step(i)
    else:
        for i in range(args.steps):
            flush.zero_()          # evict the previous step's data from L2 (not timed)
            case.step(i)
    barrier()
    clk = clocks.stop()
    status = mla.mla_get_device_error(case.workspace, stream)
    if status != 0:
        raise RuntimeError(f"device error status {status}")
    if flush is None:
        step_ms = [total_ms / args.steps] * args.steps
    else:
        step_ms = [ev_p[2 * i].elapsed_time(ev_c[i]) for i in range(args.steps)]
    kernel_ms = [ev_k[2 * i].elapsed_time(ev_k[2 * i + 1]) for i in range(args.steps)]
    if case.fused_step:
        before_ms = [ev_p[2 * i].elapsed_time(ev_k[2 * i + 1]) for i in range(args.steps)]
        combine_ms = [ev_k[2 * i + 1].elapsed_time(ev_c[i]) for i in range(args.steps)]
    else:
        before_ms = [ev_p[2 * i].elapsed_time(ev_p[2 * i + 1]) for i in range(args.steps)]
        combine_ms = [ev_p[2 * i + 1].elapsed_time(ev_c[i]) for i in range(args.steps)]
    case.profiled_step_ms = statistics.mean(
        ev_p[2 * i].elapsed_time(ev_c[i]) for i in range(args.steps))
    return step_ms, kernel_ms, before_ms, combine_ms, clk


def make_events(n):
    import torch
    return ([torch.cuda.Event(enable_timing=True) for _ in range(2 * n)],
            [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)],
            [torch.cuda.Event(enable_timing=True) for _ in range(n)])


def run_sweep(args, dev, stream, barrier):
    """Config 3's shard-count sweep: one seeded cache at N = 1, 2, 4, 8 in
    both layouts; the partial kernel's and the combine's bandwidth per run."""
    import torch
    peak, peak_kind = load_peaks()
    rows = []
    for layout in ("interleaved", "contiguous"):
        for N in (1, 2, 4, 8):
            args.num_shards, args.layout = N, layout
            ev_p, ev_k, ev_c = make_events(args.steps)
            for ev in ev_p + ev_k + ev_c:
                ev.record(stream)
            case = mla_case(args, 0, dev, stream, ev_p, ev_k, ev_c)
            step_ms, kernel_ms, _, combine_ms, clk = time_case(case, args, dev, stream, ev_p,
                                                               ev_k, ev_c, barrier, None)
            km, cm, sm = (statistics.mean(kernel_ms), statistics.mean(combine_ms),
                          statistics.mean(step_ms))
            rows.append({"num_shards": N, "layout": layout,
                         "partial_kernel_ms": km,
                         "partial_kernel_gbps": case.kv_bytes / km / 1e6,
                         "partial_frac_of_peak": case.kv_bytes / km / 1e6 / peak,
                         "combine_ms": cm,
                         "combine_gbps": case.combine_bytes / cm / 1e6,
                         "combine_bytes": case.combine_bytes,
                         "step_ms": sm, "step_gbps": case.kv_bytes / sm / 1e6,
                         "sm_mhz": clk["sm_mhz"], "reasons": clk["reasons"]})
            del case
            torch.cuda.empty_cache()
    print(json.dumps({"sweep": "shard-count-sweep", "peak_gbs": peak,
                      "peak_source": f"{peak_kind} hbm_gbs", "steps": args.steps,
                      "warmup": args.warmup, "runs": rows}), flush=True)


def dcp_rank_inputs(w, world, rank, device):
    """Rank ``rank``'s inputs of a multi-GPU DCP step over the global workload
    ``w``: its query heads [B, q_len, H/N, 576], the cache slice holding only
    its shard's positions (the *_LOCAL layout), that slice's block table,
    the global lengths and its heads' W_UV."""
    import numpy as np
    import torch
    import mla_inputs as mi
    H = w.num_heads
    if H % world != 0:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    Hl = H // world
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16)
    d = mi.local_shard_cache(w, world, rank, w.layout, seed=rank)
    if w.kv_dtype == "bf16":
        kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16)
        sc = None
    else:
        kv = torch.from_numpy(d["kv"])
        sc = torch.from_numpy(d["kv_scale"]).to(device)
    w_uv = None
    if w.w_uv is not None:
        w_uv = torch.from_numpy(w.w_uv.view(np.int16)).view(torch.bfloat16)[
            rank * Hl:(rank + 1) * Hl].contiguous().to(device)
    return dict(q_local=q[:, :, rank * Hl:(rank + 1) * Hl].contiguous().to(device),
                kv=kv.to(device), kv_scale=sc,
                block_table=torch.from_numpy(d["block_table"]).to(device),
                seq_lens=torch.from_numpy(w.seq_lens).to(device), w_uv_local=w_uv,
                local_tokens=int(d["local_lens"].sum()))


def dcp_exchange_bytes(w, world):
    """Bytes one rank sends per DCP step: its query heads to every peer (the
    all-gather) and, to every peer, that peer's head slice of its shard
    partial (the all-to-all: 512 fp32 values and one LSE per row)."""
    rows_l = w.batch * w.q_len * (w.num_heads // world)
    return {"q_allgather_bytes_per_rank": (world - 1) * rows_l * 576 * 2,
            "partial_alltoall_bytes_per_rank": (world - 1) * rows_l * (512 + 1) * 4}


def run_dcp(args, world, rank, dist, device, workload=None, partial_fn=None, combine_fn=None):
    """The multi-GPU DCP step ("Decode Context Parallelism", section 4.1) on
    ``world`` ranks, one per GPU: rank r holds query heads
    [r H/N, (r + 1) H/N) and shard r of every request's cache; a step is the
    query all-gather, the rank's partial over its shard, the head-sliced
    all-to-all of the partials and the combine of its heads.  The total work
    is one global batch (strong scaling): value = the batch's KV bytes / the
    step time (max over ranks).  Returns the JSON line on rank 0 (None
    elsewhere).  ``workload``, ``partial_fn``, ``combine_fn`` and a CPU
    ``device`` are for tests of this host logic on gloo ranks."""
    import torch
    from sequence_sharded_mla_gb300 import dcp
    import mla_inputs as mi
    w = workload if workload is not None else rank_workload(args.config, 0, args.requests)
    w.layout = args.layout or w.layout
    inp = dcp_rank_inputs(w, world, rank, device)
    cuda = device.type == "cuda"

    def step():
        return dcp.dcp_decode_step(inp["q_local"], inp["kv"], inp["block_table"],
                                   inp["seq_lens"], layout=w.layout, kv_scale=inp["kv_scale"],
                                   causal=w.causal, softmax_scale=w.softmax_scale,
                                   w_uv_local=inp["w_uv_local"], partial_fn=partial_fn,
                                   combine_fn=combine_fn, chunks=args.dcp_chunks)

    def barrier():
        if dist is not None:
            dist.barrier()
        if cuda:
            torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        result = step()
    clk = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
    clocks = ClockSampler(device.index) if cuda else None
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    barrier()
    if cuda:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            result = step()
        t1.record()
        barrier()
        elapsed = t0.elapsed_time(t1) / 1e3
    else:
        c0 = time.perf_counter()
        for _ in range(args.steps):
            result = step()
        barrier()
        elapsed = time.perf_counter() - c0
    if clocks is not None:
        clk = clocks.stop()
    # the rank's partial kernels alone, from an untimed profiled step: one
    # event pair around each request group's launch, summed
    kernel_ms = None
    if cuda and partial_fn is None:
        import sequence_sharded_mla_gb300 as mla
        pairs = []

        def timed_partial(*a, **k):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            mla.mla_set_profile_events(e0, e1)
            try:
                return dcp._cuda_partial(*a, **k)
            finally:
                mla.mla_set_profile_events(None, None)
                pairs.append((e0, e1))

        dcp.dcp_decode_step(inp["q_local"], inp["kv"], inp["block_table"], inp["seq_lens"],
                            layout=w.layout, kv_scale=inp["kv_scale"], causal=w.causal,
                            softmax_scale=w.softmax_scale, w_uv_local=inp["w_uv_local"],
                            partial_fn=timed_partial, chunks=args.dcp_chunks)
        barrier()
        kernel_ms = sum(e0.elapsed_time(e1) for e0, e1 in pairs)
    local_kv = inp["local_tokens"] * (1152 if w.kv_dtype == "bf16" else 580)
    (elapsed, kms), _ = reduce_over_ranks(dist, [elapsed, kernel_ms or 0.0], 0,
                                          device if cuda else torch.device("cpu"))
    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    ms = elapsed / args.steps * 1e3
    name = f"{w.name}-dcp{world}-{w.layout}"
    line = {
        "metric": METRIC, "value": w.kv_bytes() * args.steps / elapsed / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3", "data": "synthetic",
        "config": {"workload": name, "batch": w.batch, "heads": w.num_heads, "q_len": w.q_len,
                   "num_shards": world, "layout": w.layout, "kv_dtype": w.kv_dtype,
                   "total_kv_bytes": w.kv_bytes(), "kv_bytes_rank0": local_kv,
                   "l2": "inputs larger than L2" if w.kv_bytes() > 4 * L2_BYTES else
                         "inputs not flushed from L2",
                   "parallelism": f"dcp{world}: one sequence shard per GPU, query all-gather, "
                                  "head-sliced all-to-all of the partials, combine per head "
                                  f"slice; {args.dcp_chunks} request group(s)"
                                  + (", each group's exchange overlapping the next group's "
                                     "partial" if args.dcp_chunks > 1 else "")},
        "exchange": dict(dcp_exchange_bytes(w, world), chunks=args.dcp_chunks,
                         step_ms=ms, partial_kernel_ms_max=kms if kernel_ms is not None else None,
                         outside_partial_kernel_ms=(ms - kms) if kernel_ms is not None else None),
        "clocks": clk,
    }
    if kernel_ms is not None:
        achieved = local_kv / (kms / 1e3) / 1e9
        line["roofline"] = {"kernel": "mla_partial_kernel<1, true, false> (local cache, DCP I/O)"
                            if w.kv_dtype == "bf16" else
                            "mla_partial_fp8_kernel<1, true> (local cache, DCP I/O)",
                            "launches": args.dcp_chunks, "bound": "hbm",
                            "achieved": achieved, "peak": peak, "unit": "GB/s",
                            "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                            "traffic": None}
    line["gpu_launches"] = 4 * args.dcp_chunks * args.steps   # plan, partial, merge, combine
    return line


def run_gpu(args, world, rank, local, dist):
    import torch

    import sequence_sharded_mla_gb300 as mla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.lib()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    if args.sweep:
        if args.config != 3 or world != 1:
            raise SystemExit("--sweep is the shard-count sweep of --config 3 on one GPU")
        run_sweep(args, dev, stream, barrier)
        return
    if (world > 1 and not args.independent) or args.dcp:
        if args.config == GQA_CONFIG:
            raise SystemExit("the DCP step runs the MLA configurations")
        line = run_dcp(args, world, rank, dist, dev)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    # per timed step: events at its start, around the partial kernel
    # (recorded by the library itself) and at its end
    ev_p, ev_k, ev_c = make_events(args.steps)
    for ev in ev_p + ev_k + ev_c:
        ev.record(stream)
    # each rank decodes its own batch of the same shape (independent requests)
    make = gqa_case if args.config == GQA_CONFIG else mla_case
    case = make(args, rank, dev, stream, ev_p, ev_k, ev_c)
    kv_bytes = case.kv_bytes
    step = case.step
    # inputs not well above L2 (the tiny batch, the q_len-9 batch's 148 MB)
    # are evicted by writing a buffer twice L2's size before every timed step
    flush = None
    if kv_bytes < 4 * L2_BYTES:
        flush = torch.empty((2 * L2_BYTES // 4,), dtype=torch.float32, device=dev)
    step_ms, kernel_ms, before_ms, combine_ms, clk = time_case(case, args, dev, stream, ev_p,
                                                               ev_k, ev_c, barrier, flush)
    elapsed = sum(step_ms) / 1e3

    # end to end through host buffers: copy the step's inputs in, read results out
    h2d = sum(h.numel() * h.element_size() for h, _ in case.pairs)
    d2h = sum(d.numel() * d.element_size() for d, _ in case.outputs)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        for h, d in case.pairs:
            d.copy_(h, non_blocking=True)
        step()
        for d, h in case.outputs:
            h.copy_(d, non_blocking=True)

    e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_elapsed = e0.elapsed_time(e1) / 1e3

    (elapsed, e2e_per_step, before_avg_ms, kernel_avg_ms, combine_avg_ms), total_kv = \
        reduce_over_ranks(dist, [elapsed, e2e_elapsed / e2e_steps, statistics.mean(before_ms),
                                 statistics.mean(kernel_ms), statistics.mean(combine_ms)],
                          kv_bytes, dev)
    if rank != 0:
        return
    peak, peak_kind = load_peaks()
    tpeak, tpeak_kind = load_tensor_peak()
    value = total_kv * args.steps / elapsed / 1e9
    ms_per_step = elapsed / args.steps * 1e3
    achieved = kv_bytes / (kernel_avg_ms / 1e3) / 1e9
    traffic = traffic_for(os.path.join(ROOT, "sequence_sharded_mla_gb300", "csrc",
                                       case.kernel_src), case.name)
    hbm_roof = {"kernel": case.kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": traffic}
    tflops = case.flops / (kernel_avg_ms / 1e3) / 1e12
    if case.tensor_fp8:
        # e4m3 contractions: the measured bf16 rate x the nominal fp8 / bf16
        # ratio (4.5 / 2.25); the kernel executes twice the useful flops
        # (two-term query and probabilities)
        tpeak = tpeak * 2.0
        tsrc = (f"{tpeak_kind} x 2 (nominal e4m3 / bf16 dense ratio); useful MMA flops "
                "2*H*(Dk+Dv) per visible token and query, executed twice (two-term q and P)")
    else:
        tsrc = (f"{tpeak_kind} (dense fp16/bf16 rate; useful MMA flops "
                "2*H*(Dk+Dv) per visible token and query)")
    tensor_roof = {"kernel": case.kernel, "bound": "tensor", "achieved": tflops, "peak": tpeak,
                   "unit": "TFLOP/s", "frac": tflops / tpeak, "peak_source": tsrc,
                   "traffic": traffic}
    if flush is not None:
        l2 = (f"L2 flushed before every timed step (a {2 * L2_BYTES >> 20} MiB buffer written, "
              f"outside the timed interval); {kv_bytes / 1e6:.1f} MB of KV per GPU")
    else:
        l2 = f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB of KV per GPU vs 129 MB)"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.dtype, "data": "synthetic",
        "config": dict(case.config, kv_bytes_per_gpu=kv_bytes, l2=l2,
                       parallelism=f"{world} GPU(s), independent batches; "
                                   f"{case.config['num_shards']} logical shards each"),
        "steps_per_s": args.steps / elapsed,
        "pct_of_peak_hbm": value / world / peak,
        "roofline": hbm_roof if not case.tensor_bound else tensor_roof,
        "roofline_other": tensor_roof if not case.tensor_bound else hbm_roof,
        "combine": {"kernel_ms": combine_avg_ms,
                    "gbps": case.combine_bytes / (combine_avg_ms / 1e3) / 1e9,
                    "bytes_per_step": case.combine_bytes},
        "partial_kernel_ms": kernel_avg_ms,
        "partial_call_ms": before_avg_ms,
        "profiled_step_ms": case.profiled_step_ms,   # a step with events between its kernels
        "e2e": {"value": total_kv / e2e_per_step / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": case.launches_per_step * args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5, 6],
                    help="workload: one of the five benchmark configurations (default 2), "
                         "or 6: the grouped-query batch")
    ap.add_argument("--requests", type=int, default=0,
                    help="profiling only: keep the first K requests of the workload")
    ap.add_argument("--wuv", action="store_true",
                    help="attach a W_UV projection to the configuration (fused into the step)")
    ap.add_argument("--num-shards", type=int, default=0,
                    help="override the configuration's logical shard count (1..8)")
    ap.add_argument("--layout", default="", choices=["", "interleaved", "contiguous"],
                    help="override the configuration's shard layout")
    ap.add_argument("--independent", action="store_true",
                    help="with --gpus N > 1: N independent batches (no exchange) instead of "
                         "the DCP step over one global batch")
    ap.add_argument("--dcp", action="store_true",
                    help="run the DCP step also at --gpus 1 (an exchange-free check of its path)")
    ap.add_argument("--dcp-chunks", type=int, default=1,
                    help="DCP step: request groups whose exchange overlaps the next group's "
                         "partial attention (each group is a launch of its own, with its own "
                         "start and tail: more than one pays only when the exchange is long)")
    ap.add_argument("--sweep", action="store_true",
                    help="with --config 3: the shard-count sweep, N = 1, 2, 4, 8 in both "
                         "layouts over one seeded cache (one JSON line with a table)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local, dist = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
