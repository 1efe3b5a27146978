"""Throughput of the routed-MoE layer on GB300 (one JSON line on stdout).

Headline workload: the GLM-5.2-shaped MoE layer at decode batch 1 (hidden
6144, 256 routed experts in 8 groups, topk_group 4, top-8, moe_inter 2048,
one shared expert, packed int4 per-row-scaled weights, all experts resident
in HBM); one step = 1000 independent seeded positions, one coli_moe_layer
call each (router and expert layer in one fused launch, through the C ABI),
back to back.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

* value: tokens/s with inputs resident in HBM, timed with CUDA events around
  K steps replayed from a CUDA graph; L2 is defeated by rotating 8 identical
  copies of the layer's weights (≈39 GB), so consecutive calls never find a
  weight byte in L2.
* roofline: the layer kernel's algorithmic bytes per launch (9 expert
  records: 8 routed + the shared one, plus the fp32 router weights and bias)
  over its average launch duration, measured with CUDA events on its stream,
  against the measured HBM copy bandwidth.
* e2e: the same tokens/s through the public API called per position from
  Python with host buffers: pinned x copied in, y copied out, inside the timed
  region.
* cpu_baseline / --impl reference: the CPU oracle (numpy, one thread) timed on
  a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own 1000 positions on its own copy
of the layer (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")  # the CPU oracle runs on one thread
os.environ.setdefault("OMP_NUM_THREADS", "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "routed-MoE layer tokens/s + achieved HBM GB/s (decode) / int8 TOPS (prefill)"
UNIT = "tokens/s"
EXPERT_BYTES = synth.GLM.record_bytes() + 4 * synth.GLM.scale_count()   # 18,915,328
ROUTER_BYTES = 4 * synth.GLM.n_experts * synth.GLM.hidden + 4 * synth.GLM.n_experts
DECODE_TOKENS = 1000
REPLICAS = 8
# DRAM bytes (read + write) of one layer-kernel launch on this workload, from
# an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one position,
# cold L2); reported only while the kernel's sources hash to the value the
# capture was taken on, null otherwise.
LAYER_KERNEL_SOURCES = ("quantized_expert_ffn_sigmoid_gb300/csrc/decode.cu",
                        "quantized_expert_ffn_sigmoid_gb300/csrc/select_cta.cuh",
                        "quantized_expert_ffn_sigmoid_gb300/csrc/gemv_common.cuh",
                        "quantized_expert_ffn_sigmoid_gb300/csrc/colimoe_internal.cuh")
LAYER_KERNEL_TRAFFIC = {"bytes": 178367744, "sources_sha256": "31eefbaf7cb71ffae1c8110737a05d84d735aa3cdd5db4105cf5ceb3d781dcf3"}
WORKLOAD = ("glm_decode_b1: GLM-5.2-shaped MoE layer (H 6144, E 256 in 8 groups, topk_group 4, top-8, "
            "moe_inter 2048, 1 shared expert, int4 per-row scales, rsf 2.5), decode batch 1, "
            "1000 independent seeded positions per step, one layer call each")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def layer_kernel_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in LAYER_KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    ok = LAYER_KERNEL_TRAFFIC["sources_sha256"] == h.hexdigest()
    return LAYER_KERNEL_TRAFFIC["bytes"] if ok else None


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1937.1)), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons; only samples taken
    between mark_start() and mark_end() are summarised."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.out, _ = self.proc.communicate()

    def summary(self):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or 1e18)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({n for r in use for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_window": bool(inside)}


# ----------------------------------------------------------------- GPU arm
class DecodeBench:
    def __init__(self, device, rank, replicas=REPLICAS, tokens=DECODE_TOKENS):
        import torch
        import synth.gpu as sg
        import quantized_expert_ffn_sigmoid_gb300 as cm
        self.torch, self.cm = torch, cm
        self.dev = device
        self.shape = synth.GLM
        self.seed = synth.WORKLOADS["glm_decode_b1"][1]
        self.n = tokens
        self.R = replicas
        self.cfg = cm.Cfg.of(self.shape)
        t0 = time.time()
        recs, scs = sg.expert_records(self.shape, self.seed, 0, "routed", self.shape.n_experts, device)
        srec, ssc = sg.expert_records(self.shape, self.seed, 0, "shared", 1, device)
        wr = torch.from_numpy(synth.router_weight(self.shape, self.seed)).to(device)
        bias = torch.from_numpy(synth.router_bias(self.shape, self.seed)).to(device)
        self.rep = []
        for r in range(self.R):
            if r == 0:
                t = (recs, scs, srec, ssc, wr, bias)
            else:
                t = tuple(a.clone() for a in (recs, scs, srec, ssc, wr, bias))
            self.rep.append(t)
        self.W = [cm.make_weights(t[0], t[1], t[2], t[3]) for t in self.rep]
        torch.cuda.synchronize()
        log(f"[bench] weights: {self.R} x {(recs.numel() + srec.numel()) / 1e9:.2f} GB in {time.time() - t0:.1f}s")
        self.x = sg.token_batch(self.shape, self.seed, ("bench", rank), range(self.n), device)
        k = self.shape.top_k
        self.idx = torch.empty((self.n, k), dtype=torch.int32, device=device)
        self.w = torch.empty((self.n, k), dtype=torch.float32, device=device)
        self.y = torch.empty((self.n, self.shape.hidden), dtype=torch.float32, device=device)
        self.ws = cm.new_workspace(self.cfg, 1)
        self.launches_per_token = 1   # one fused layer kernel (router + experts)

    def step(self):
        cm = self.cm
        for i in range(self.n):
            r = i % self.R
            rec = self.rep[r]
            cm.coli_moe_layer(self.cfg, self.W[r], self.x[i:i + 1], rec[4], rec[5], self.idx[i:i + 1],
                              self.w[i:i + 1], self.y[i:i + 1], self.ws)

    def capture(self):
        torch = self.torch
        self.step()  # warm the attribute calls outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.step()
        torch.cuda.synchronize()
        self.graph = g

    def expert_kernel_ms(self, n=None):
        """Average duration of the layer kernel (the one launch of
        coli_moe_layer per position), from CUDA events on its stream; the host
        enqueues everything behind a sleep so that launches run back to back."""
        torch, cm = self.torch, self.cm
        n = n or self.n
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        torch.cuda.synchronize()
        torch.cuda._sleep(int(6e8))   # keeps the GPU busy while the host enqueues
        for i in range(n):
            r = i % self.R
            rec = self.rep[r]
            starts[i].record()
            cm.coli_moe_layer(self.cfg, self.W[r], self.x[i:i + 1], rec[4], rec[5], self.idx[i:i + 1],
                              self.w[i:i + 1], self.y[i:i + 1], self.ws)
            ends[i].record()
        torch.cuda.synchronize()
        d = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return statistics.mean(d), statistics.median(d)

    def e2e_step(self, x_host, y_host):
        """Public API per position with host buffers: each position's x is
        copied in from pinned host memory before its own layer call and its y
        copied out after it (a decode caller's per-token pattern)."""
        cm = self.cm
        for i in range(self.n):
            r = i % self.R
            rec = self.rep[r]
            self.x[i:i + 1].copy_(x_host[i:i + 1], non_blocking=True)
            cm.coli_moe_layer(self.cfg, self.W[r], self.x[i:i + 1], rec[4], rec[5], self.idx[i:i + 1],
                              self.w[i:i + 1], self.y[i:i + 1], self.ws)
            y_host[i:i + 1].copy_(self.y[i:i + 1], non_blocking=True)
        self.torch.cuda.synchronize()


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    b = DecodeBench(device, rank, replicas=args.replicas, tokens=args.tokens)
    b.capture()
    for _ in range(args.warmup):
        b.graph.replay()
    torch.cuda.synchronize()
    st = cm_status(b)
    if st:
        raise RuntimeError(f"device status {st} after warm-up")

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        clk.mark_start()
        e0.record()
        for _ in range(args.steps):
            b.graph.replay()
        e1.record()
        barrier()
        clk.mark_end()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world, device)
    tokens = sum_over_ranks(float(args.steps * b.n), world, device)
    value = tokens / (ms_max / 1e3)

    # roofline of the dominant kernel: the timed region runs that kernel alone,
    # one launch per position, so its average launch duration is the timed
    # region over the launches; an isolated launch (events around each one,
    # no overlap with its neighbours) is reported beside it
    k_mean, k_med = b.expert_kernel_ms()
    hbm, _, peak_kind = read_peaks()
    kbytes = 9 * EXPERT_BYTES + ROUTER_BYTES
    launch_ms = ms_max / (args.steps * b.n * b.launches_per_token)
    achieved = kbytes / (launch_ms / 1e3) / 1e9

    # end to end through the public API with host buffers
    x_host = b.x.cpu().pin_memory()
    y_host = torch.empty(b.y.shape, dtype=torch.float32).pin_memory()
    b.e2e_step(x_host, y_host)
    barrier()
    t0 = time.perf_counter()
    e2e_steps = max(1, min(args.steps, 5))
    for _ in range(e2e_steps):
        b.e2e_step(x_host, y_host)
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
    e2e_val = sum_over_ranks(float(e2e_steps * b.n), world, device) / e2e_s
    st = cm_status(b)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "positions_per_call": 1, "positions_per_step": b.n,
                   "l2": f"inputs larger than L2: {b.R} identical weight copies rotated per call "
                         f"({b.R * (256 + 1) * EXPERT_BYTES / 1e9:.1f} GB)",
                   "launch": "CUDA graph of the per-position coli_moe_layer calls",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "layer_bytes_per_token": 9 * EXPERT_BYTES + ROUTER_BYTES,
                   "layer_gbs": round(value / world * (9 * EXPERT_BYTES + ROUTER_BYTES) / 1e9, 1)},
        "roofline": {"bound": "hbm", "kernel": "decode_layer_kernel", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "peak_source": f"{peak_kind} (HBM copy)", "traffic": args.traffic if args.traffic is not None else layer_kernel_traffic(),
                     "bytes_per_launch": kbytes, "launch_ms_mean": round(launch_ms, 5),
                     "isolated_launch_ms_mean": round(k_mean, 5), "isolated_launch_ms_median": round(k_med, 5),
                     "achieved_isolated": round(kbytes / (k_mean / 1e3) / 1e9, 1)},
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": int(b.x.numel() * 4),
                "d2h_bytes_per_step": int(b.y.numel() * 4)},
        "gpu_launches": int(args.steps * b.n * b.launches_per_token),
        "clocks": clk.summary(),
        "status": st,
    }
    if rank == 0 and args.secondary:
        out["secondary"] = secondary(device, b)
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(b, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cm_status(b):
    return b.cm.coli_moe_status(b.ws)


def secondary(device, b):
    """Other workloads: MTP verify (4 positions/call) and prefill (2048
    positions/call) on the decode layer's resident experts, and the 25-layer
    stack at batch 32 on its own resident layers."""
    import torch
    cm = b.cm
    res = {}
    shape = b.shape
    # MTP verify: 4 correlated positions per call
    seed = synth.WORKLOADS["glm_mtp_verify_t4"][1]
    calls = synth.WORKLOADS["glm_mtp_verify_t4"][3]   # 500 calls of 4 positions
    xs = np.stack([synth.mtp_chain(shape, seed, c) for c in range(calls)])
    x = torch.from_numpy(xs).to(device)
    wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    bias = torch.from_numpy(synth.router_bias(shape, seed)).to(device)
    ws = cm.new_workspace(b.cfg, 4)
    idx = torch.empty((calls, 4, 8), dtype=torch.int32, device=device)
    w = torch.empty((calls, 4, 8), dtype=torch.float32, device=device)
    y = torch.empty((calls, 4, shape.hidden), dtype=torch.float32, device=device)
    L = cm.coli_moe_workspace_layout(b.cfg, 4)
    uniq = 0
    for c in range(calls):
        cm.coli_moe_route(b.cfg, x[c], wr, bias, idx[c], w[c], ws)
        cm.coli_moe_dispatch(b.cfg, x[c], idx[c], ws)
        uniq += int(ws[L.n_entries:L.n_entries + 4].view(torch.int32).item()) - 1

    wrs = [wr] + [wr.clone() for _ in range(b.R - 1)]

    def mtp():
        for c in range(calls):
            r = c % b.R
            cm.coli_moe_layer(b.cfg, b.W[r], x[c], wrs[r], bias, idx[c], w[c], y[c], ws)
    ms = time_graph(mtp, 3)
    byt = (uniq + calls) * EXPERT_BYTES + calls * ROUTER_BYTES
    res["glm_mtp_verify_t4"] = {"tokens_per_s": round(4 * calls / (ms / 1e3), 1),
                                "unique_experts_per_call": round(uniq / calls, 2),
                                "gbs": round(byt / (ms / 1e3) / 1e9, 1), "ms_per_call": round(ms / calls, 4),
                                "note": "router of the MTP workload, routed experts of the decode workload"}
    # prefill: 2048 positions, uniform routing
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    import synth.gpu as sg
    T = 2048
    xp = sg.token_batch(shape, seed, 0, range(T), device)
    wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    bias = torch.from_numpy(synth.zero_router_bias(shape)).to(device)
    ws = cm.new_workspace(b.cfg, T)
    idx = torch.empty((T, 8), dtype=torch.int32, device=device)
    w = torch.empty((T, 8), dtype=torch.float32, device=device)
    y = torch.empty((T, shape.hidden), dtype=torch.float32, device=device)

    def pre():
        cm.coli_moe_layer(b.cfg, b.W[0], xp, wr, bias, idx, w, y, ws)
    ms = time_graph(pre, 2)
    ops = 2.0 * (T * 8 + T) * 3 * shape.inter * shape.hidden
    byt = (256 + 1) * EXPERT_BYTES + ROUTER_BYTES
    tops = ops / (ms / 1e3) / 1e12
    i8 = int8_gemm_tops(device)
    _, bf16, kind = read_peaks()
    res["glm_prefill_s2048"] = {"tokens_per_s": round(T / (ms / 1e3), 1), "ms_per_call": round(ms, 3),
                                "int8_tops": round(tops, 2),
                                "gbs_min_bytes": round(byt / (ms / 1e3) / 1e9, 1),
                                "int8_gemm_tops_measured": round(i8, 1),
                                "frac_of_int8_gemm": round(tops / i8, 3) if i8 else None,
                                "frac_of_bf16_peak": round(tops / bf16, 4),
                                "peak_note": "int8: the library int8 GEMM (cuBLASLt through torch._int_mm, 8192^3) "
                                             "on this GPU, which has no tcgen05 int8 MMA; bf16: " + kind +
                                             " dense bf16, the rate of the kind::f16 MMA the kernel uses"}
    del xp, ws, idx, w, y
    res["glm_gs64_decode_b1"] = weight_format_bench(device, b)
    res["glm_gs64_mtp_verify_t4"] = weight_format_bench(device, b, calls=100, T=4)
    res["glm_int2_decode_b1"] = weight_format_bench(device, b, shape=synth.GLM_INT2)
    res["glm_int2_mtp_verify_t4"] = weight_format_bench(device, b, calls=100, T=4, shape=synth.GLM_INT2)
    res["glm_int2_b32"] = weight_format_bench(device, b, calls=20, T=32, shape=synth.GLM_INT2)
    res["glm_gs64_b32"] = weight_format_bench(device, b, calls=20, T=32)
    res["glm_prefill_sweep"] = prefill_sweep(device, b)
    res["glm_stack24_mtp1_b32"] = stack_bench(device, b)
    return res


def int8_gemm_tops(device, n=8192, reps=3):
    """Measured int8 tensor throughput of the library GEMM (int8 x int8 -> int32,
    n^3), the reference point for the prefill's int8-equivalent rate."""
    import torch
    try:
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device)
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=device)
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        del a, b
        return 2.0 * n ** 3 / (ms / 1e3) / 1e12
    except (RuntimeError, AttributeError):
        return 0.0


def prefill_only(args):
    """--only prefill: the prefill workload alone (no decode replicas), for
    profiling; --prefill-experts / --prefill-t shrink it to a small case with
    the same kernels.  Prints one JSON line with the call time."""
    import dataclasses
    import torch
    import synth.gpu as sg
    import quantized_expert_ffn_sigmoid_gb300 as cm
    device = torch.device("cuda", 0)
    shape = dataclasses.replace(synth.GLM, n_experts=args.prefill_experts)
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    T = args.prefill_t
    recs, scs = sg.expert_records(shape, seed, 0, "routed", shape.n_experts, device)
    srec, ssc = sg.expert_records(shape, seed, 0, "shared", 1, device)
    W = cm.make_weights(recs, scs, srec, ssc)
    cfg = cm.Cfg.of(shape)
    xp = sg.token_batch(shape, seed, 0, range(T), device)
    wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    bias = torch.from_numpy(synth.zero_router_bias(shape)).to(device)
    ws = cm.new_workspace(cfg, T)
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device=device)
    w = torch.empty((T, shape.top_k), dtype=torch.float32, device=device)
    y = torch.empty((T, shape.hidden), dtype=torch.float32, device=device)
    for _ in range(args.warmup):
        cm.coli_moe_layer(cfg, W, xp, wr, bias, idx, w, y, ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        cm.coli_moe_layer(cfg, W, xp, wr, bias, idx, w, y, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"workload": f"prefill: GLM-5.2-shaped layer with {shape.n_experts} routed experts, T={T}",
                      "ms_per_call": round(ms, 3), "tokens_per_s": round(T / (ms / 1e3), 1),
                      "status": cm.coli_moe_status(ws)}), flush=True)


def sweep_only(args):
    """--only sweep: the GLM-5.2-shaped layer at 64 .. 2048 positions per call
    on one resident copy (the bench's prefill sweep alone)."""
    import torch
    import synth.gpu as sg
    import quantized_expert_ffn_sigmoid_gb300 as cm
    device = torch.device("cuda", 0)

    class _B:  # the attributes prefill_sweep reads
        pass
    b = _B()
    b.cm, b.shape, b.cfg = cm, synth.GLM, cm.Cfg.of(synth.GLM)
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    recs, scs = sg.expert_records(synth.GLM, seed, 0, "routed", synth.GLM.n_experts, device)
    srec, ssc = sg.expert_records(synth.GLM, seed, 0, "shared", 1, device)
    b.W = [cm.make_weights(recs, scs, srec, ssc)]
    print(json.dumps({"workload": "GLM-5.2-shaped layer, uniform routing, positions per call sweep",
                      **prefill_sweep(device, b)}), flush=True)


def few_only(args):
    """--only mtp / --only b32: one workload with a few positions per call, on
    one resident copy of a GLM-5.2-shaped layer, for profiling.  mtp: the MTP
    verify chain (4 positions per call); b32: batch 32 with the Zipf-skewed
    correction bias of the stack's first layer.  Prints one JSON line."""
    import torch
    import synth.gpu as sg
    import quantized_expert_ffn_sigmoid_gb300 as cm
    device = torch.device("cuda", 0)
    shape = synth.GLM
    if args.only == "mtp":
        seed, T = synth.WORKLOADS["glm_mtp_verify_t4"][1], 4
        xs = torch.from_numpy(np.stack([synth.mtp_chain(shape, seed, c) for c in range(args.calls)])).to(device)
        bias = torch.from_numpy(synth.router_bias(shape, seed)).to(device)
        wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    else:
        seed, T = synth.WORKLOADS["glm_stack24_mtp1_b32"][1], 32
        xs = torch.stack([sg.token_batch(shape, seed, ("b32", c), range(T), device) for c in range(args.calls)])
        bias = torch.from_numpy(synth.zipf_router_bias(shape, seed, 0)).to(device)
        wr = torch.from_numpy(synth.router_weight(shape, seed, 0)).to(device)
    recs, scs = sg.expert_records(shape, seed, 0, "routed", shape.n_experts, device)
    srec, ssc = sg.expert_records(shape, seed, 0, "shared", 1, device)
    W = cm.make_weights(recs, scs, srec, ssc)
    cfg = cm.Cfg.of(shape)
    ws = cm.new_workspace(cfg, T)
    idx = torch.empty((args.calls, T, shape.top_k), dtype=torch.int32, device=device)
    w = torch.empty((args.calls, T, shape.top_k), dtype=torch.float32, device=device)
    y = torch.empty((args.calls, T, shape.hidden), dtype=torch.float32, device=device)

    def calls():
        for c in range(args.calls):
            cm.coli_moe_layer(cfg, W, xs[c], wr, bias, idx[c], w[c], y[c], ws)
    for _ in range(args.warmup):
        calls()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        calls()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (args.steps * args.calls)
    print(json.dumps({"workload": f"{args.only}: GLM-5.2-shaped layer, {T} positions per call, {args.calls} calls",
                      "ms_per_call": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1),
                      "status": cm.coli_moe_status(ws)}), flush=True)


def weight_format_bench(device, b, calls=300, T=1, shape=synth.GLM_GS64):
    """The decode workload on another weight format of the same layer --
    group-scaled int4 (one fp32 scale per 64 weights of a row, the default) or
    packed int2 with per-row scales: 8 rotated copies of the layer, one
    coli_moe_layer call per call of T positions."""
    import torch
    import synth.gpu as sg
    cm = b.cm
    seed = synth.WORKLOADS["glm_decode_b1"][1]
    cfg = cm.Cfg.of(shape)
    recs, scs = sg.expert_records(shape, seed, 0, "routed", shape.n_experts, device)
    srec, ssc = sg.expert_records(shape, seed, 0, "shared", 1, device)
    wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    bias = torch.from_numpy(synth.router_bias(shape, seed)).to(device)
    reps = [(recs, scs, srec, ssc, wr, bias)] + [
        tuple(a.clone() for a in (recs, scs, srec, ssc, wr, bias)) for _ in range(b.R - 1)]
    Ws = [cm.make_weights(r[0], r[1], r[2], r[3]) for r in reps]
    if T == 1:
        x = sg.token_batch(shape, seed, ("gs64", 0), range(calls), device).view(calls, 1, -1)
    elif T > 4:  # a decode batch: T independent positions per call
        x = sg.token_batch(shape, seed, ("batch", T), range(calls * T), device).view(calls, T, -1)
    else:  # the MTP-verify chain: T correlated positions per call
        mseed = synth.WORKLOADS["glm_mtp_verify_t4"][1]
        x = torch.from_numpy(np.stack([synth.mtp_chain(shape, mseed, c, n_pos=T) for c in range(calls)])).to(device)
    ws = cm.new_workspace(cfg, T)
    idx = torch.empty((calls, T, shape.top_k), dtype=torch.int32, device=device)
    w = torch.empty((calls, T, shape.top_k), dtype=torch.float32, device=device)
    y = torch.empty((calls, T, shape.hidden), dtype=torch.float32, device=device)
    L = cm.coli_moe_workspace_layout(cfg, T)
    uniq = 0
    for i in range(calls):
        r = reps[i % b.R]
        cm.coli_moe_layer(cfg, Ws[i % b.R], x[i], r[4], r[5], idx[i], w[i], y[i], ws)
        uniq += int(ws[L.n_entries:L.n_entries + 4].view(torch.int32).item())  # routed + shared

    def run():
        for i in range(calls):
            r = reps[i % b.R]
            cm.coli_moe_layer(cfg, Ws[i % b.R], x[i], r[4], r[5], idx[i], w[i], y[i], ws)
    ms = time_graph(run, 3)
    rec_bytes = shape.record_bytes() + 4 * shape.scale_count()
    byt = uniq * rec_bytes + calls * ROUTER_BYTES
    out = {"tokens_per_s": round(T * calls / (ms / 1e3), 1), "us_per_call": round(1e3 * ms / calls, 2),
           "gbs": round(byt / (ms / 1e3) / 1e9, 1), "experts_per_call": round(uniq / calls, 2),
           "status": cm.coli_moe_status(ws),
           "note": (("packed int2, per-row scales" if shape.weight_bits == 2 else "group-scaled int4 (gs64)") +
                    (", the fused single-position kernel" if T == 1 else
                     ", the few-position kernels" if shape.weight_bits == 2 and T <= 4 else
                     ", the small-batch kernels") +
                    f", {T} position(s) per call; 8 rotated copies")}
    del reps, Ws, recs, scs, srec, ssc
    torch.cuda.empty_cache()
    return out


def weight_format_only(args, shape=synth.GLM_GS64, name="gs64", fmt="group-scaled int4"):
    """--only gs64 / int2: one weight format's decode and MTP-verify
    measurements alone (for profiling)."""
    import torch

    class _B:  # the two attributes weight_format_bench reads
        import quantized_expert_ffn_sigmoid_gb300 as cm
        R = REPLICAS
    for T in (1, 4, 32):
        print(json.dumps({"workload": f"{name}: GLM-5.2-shaped layer, {fmt}, {T} position(s) per call",
                          **weight_format_bench(torch.device("cuda", 0), _B,
                                                calls=300 if T == 1 else 100 if T == 4 else 20, T=T, shape=shape)}),
              flush=True)


def stack_bench(device, b, steps=None):
    """24 int4 GLM layers + 1 int8 layer resident, decode batch 32, Zipf-skewed
    correction bias per layer.  A step is one coli_moe_stack_forward call: the
    25 layers chained on the device (x_{l+1} = x_l + delta_l, the seeded
    residual of every (step, layer), independent of y_l), replayed from one
    CUDA graph whose input buffers are refilled from that step's seeded inputs
    (the device-to-device refill is inside the timed region)."""
    import torch
    import synth.gpu as sg
    cm = b.cm
    seed = synth.WORKLOADS["glm_stack24_mtp1_b32"][1]
    steps = steps or synth.WORKLOADS["glm_stack24_mtp1_b32"][3]
    T, n_layers, H = 32, 25, synth.GLM.hidden
    t0 = time.time()
    layers = []
    for l in range(n_layers):
        shape = synth.GLM_INT8 if l == 24 else synth.GLM
        recs, scs = sg.expert_records(shape, seed, l, "routed", shape.n_experts, device)
        srec, ssc = sg.expert_records(shape, seed, l, "shared", 1, device)
        wr = torch.from_numpy(synth.router_weight(shape, seed, l)).to(device)
        bias = torch.from_numpy(synth.zipf_router_bias(shape, seed, l)).to(device)
        layers.append((shape, cm.Cfg.of(shape), (recs, scs, srec, ssc), cm.make_weights(recs, scs, srec, ssc),
                       wr, bias))
    resident = sum(sum(a.numel() * a.element_size() for a in L[2]) for L in layers)
    # every step's inputs: x_0 ~ N(0,1) per sequence and the seeded residual of every layer
    x0_all = torch.empty((steps, T, H), device=device)
    res_all = torch.empty((steps, n_layers, T, H), device=device)
    for st in range(steps):
        x0_all[st] = sg.token_batch(synth.GLM, seed, ("stack", st), range(T), device)
        for l in range(n_layers):
            d = sg.normal_f32(synth.make_key(seed, "residual", st, l), 32 * H, 0.1, device)
            res_all[st, l] = d[:T * H].view(T, H)
    arr = cm.stack_layers([(L[1], L[3], L[4], L[5]) for L in layers])
    xs = torch.empty((n_layers + 1, T, H), device=device)
    res = torch.empty((n_layers, T, H), device=device)
    idx = torch.empty((n_layers, T, 8), dtype=torch.int32, device=device)
    w = torch.empty((n_layers, T, 8), device=device)
    y = torch.empty((n_layers, T, H), device=device)
    ws = cm.new_workspace(max((L[1] for L in layers), key=lambda c: cm.coli_moe_workspace_size(c, T)), T)
    torch.cuda.synchronize()
    log(f"[bench] stack: {resident / 1e9:.1f} GB resident, {steps} steps of inputs in {time.time() - t0:.1f}s")
    # unique experts per layer (for the bytes moved), from step 0
    xs[0].copy_(x0_all[0])
    res.copy_(res_all[0])
    g = cm.capture_stack_step(arr, xs, res, idx, w, y, ws)
    uniq = [int(torch.unique(idx[l]).numel()) for l in range(n_layers)]

    def ebytes(sh):
        return sh.record_bytes() + 4 * sh.scale_count()
    byt = sum((u + 1) * ebytes(synth.GLM_INT8 if l == 24 else synth.GLM) for l, u in enumerate(uniq)) \
        + n_layers * ROUTER_BYTES

    def one(st):
        xs[0].copy_(x0_all[st])
        res.copy_(res_all[st])
        g.replay()
    for st in range(min(3, steps)):
        one(st)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for st in range(steps):
        one(st)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    st_code = cm.coli_moe_status(ws)
    del layers, x0_all, res_all, ws
    torch.cuda.empty_cache()
    return {"tokens_per_s": round(T / (ms / 1e3), 1), "ms_per_step": round(ms, 3),
            "unique_experts_per_layer": round(sum(uniq) / n_layers, 1),
            "gbs": round(byt / (ms / 1e3) / 1e9, 1), "resident_gb": round(resident / 1e9, 1),
            "steps": steps, "status": st_code,
            "note": "coli_moe_stack_forward (24 int4 + 1 int8 layers chained on the device) per step of 32 "
                    "positions, one CUDA graph; input refill inside the timed region; bytes from step 0's "
                    "unique experts"}


def prefill_sweep(device, b, Ts=(64, 128, 256, 512, 1024, 2048)):
    """The GLM-5.2-shaped layer on the tensor-core path at several call sizes
    (uniform routing, every position's own experts): time per call, positions
    per second, bytes of the distinct experts per second and int8-equivalent
    operations per second."""
    import torch
    import synth.gpu as sg
    cm = b.cm
    shape = b.shape
    seed = synth.WORKLOADS["glm_prefill_s2048"][1]
    wr = torch.from_numpy(synth.router_weight(shape, seed)).to(device)
    bias = torch.from_numpy(synth.zero_router_bias(shape)).to(device)
    xall = sg.token_batch(shape, seed, 0, range(max(Ts)), device)
    out = {}
    for T in Ts:
        x = xall[:T]
        ws = cm.new_workspace(b.cfg, T)
        idx = torch.empty((T, 8), dtype=torch.int32, device=device)
        w = torch.empty((T, 8), dtype=torch.float32, device=device)
        y = torch.empty((T, shape.hidden), dtype=torch.float32, device=device)
        ms = time_graph(lambda: cm.coli_moe_layer(b.cfg, b.W[0], x, wr, bias, idx, w, y, ws), 3)
        uniq = int(torch.unique(idx).numel())
        byt = (uniq + 1) * EXPERT_BYTES + ROUTER_BYTES
        ops = 2.0 * (T * 8 + T) * 3 * shape.inter * shape.hidden
        out[str(T)] = {"ms_per_call": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1),
                       "unique_experts": uniq, "gbs_min_bytes": round(byt / (ms / 1e3) / 1e9, 1),
                       "int8_equiv_tops": round(ops / (ms / 1e3) / 1e12, 2), "status": cm.coli_moe_status(ws)}
        del ws, idx, w, y
    return out


def time_graph(fn, reps):
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# ----------------------------------------------------------------- CPU oracle
def oracle_tokens_per_s(get_record, router_w, bias, xs, budget_s):
    """The oracle as it stands, one position per call, until ``budget_s``."""
    import oracle
    shape = synth.GLM
    n = 0
    t0 = time.perf_counter()
    while n < len(xs):
        oracle.moe_layer(shape, get_record, xs[n:n + 1], router_w, bias)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return n, time.perf_counter() - t0


def host_records(recs, scs, srec, ssc):
    """Host copies of a layer's records (generator output), made before any timing."""
    R, S, SR, SS = recs.cpu().numpy(), scs.cpu().numpy(), srec.cpu().numpy(), ssc.cpu().numpy()
    return lambda kind, e: (R[e], S[e]) if kind == "routed" else (SR[e], SS[e])


def oracle_parallel_tokens_per_s(get_record, router_w, bias, xs, budget_s, threads):
    """The oracle as it stands on ``threads`` host threads: independent
    positions, one oracle layer call each, dealt to the threads in waves until
    ``budget_s`` (numpy releases the GIL in its array work; BLAS itself runs
    single-threaded)."""
    import concurrent.futures as cf
    import oracle
    shape = synth.GLM
    n = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        while n < len(xs) and time.perf_counter() - t0 < budget_s:
            wave = range(n, min(n + threads, len(xs)))
            list(ex.map(lambda i: oracle.moe_layer(shape, get_record, xs[i:i + 1], router_w, bias), wave))
            n += len(wave)
    return n, time.perf_counter() - t0


def cpu_baseline(b, budget_s):
    """The oracle on the host cores: one thread (serial) and every core."""
    cores = os.cpu_count() or 1
    xs = b.x[:max(16, 4 * cores)].cpu().numpy()
    rep = b.rep[0]
    get_record = host_records(rep[0], rep[1], rep[2], rep[3])
    wr = rep[4].cpu().numpy()
    bias = rep[5].cpu().numpy()
    n1, s1 = oracle_tokens_per_s(get_record, wr, bias, xs, budget_s / 2)
    nc, sc = oracle_parallel_tokens_per_s(get_record, wr, bias, xs, budget_s / 2, cores)
    return {"value": round(nc / sc, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "serial_value": round(n1 / s1, 4), "serial_cores": 1,
            "sample": f"{nc} positions of the decode workload on {cores} threads and {n1} on one thread, "
                      f"one oracle layer call each (numpy)"}


def run_reference(args):
    """The oracle as the reference arm: same workload, metric and unit."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle  # noqa: F401
    shape = synth.GLM
    seed = synth.WORKLOADS["glm_decode_b1"][1]
    wr = synth.router_weight(shape, seed)
    bias = synth.router_bias(shape, seed)
    cores = os.cpu_count() or 1
    per_step = cores          # one position per host thread and step
    xs = synth.token_batch(shape, seed, ("bench", 0), range((args.warmup + args.steps) * per_step))
    # the layer's records, made by the generator before any timing (on the
    # device twin when a GPU is present: 4.9 GB in seconds instead of minutes)
    try:
        import torch
        import synth.gpu as sg
        if not torch.cuda.is_available():
            raise RuntimeError
        recs, scs = sg.expert_records(shape, seed, 0, "routed", shape.n_experts, "cuda")
        srec, ssc = sg.expert_records(shape, seed, 0, "shared", 1, "cuda")
        get_record = host_records(recs, scs, srec, ssc)
        del recs, scs, srec, ssc
    except (ImportError, RuntimeError, OSError):
        import oracle as _o
        need = set()
        idx, _ = _o.route(_o.router_logits(xs, wr), bias, shape)
        need.update(int(e) for e in idx.ravel())
        cache = {("routed", e): synth.expert_record(shape, seed, 0, "routed", e) for e in sorted(need)}
        cache[("shared", 0)] = synth.expert_record(shape, seed, 0, "shared", 0)
        get_record = lambda kind, e: cache[(kind, e)]
    def step(i):
        oracle_parallel_tokens_per_s(get_record, wr, bias, xs[i * per_step:(i + 1) * per_step], 1e9, cores)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    s = time.perf_counter() - t0
    value = args.steps * per_step / s
    out = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(1e3 * s / args.steps, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic", "impl": "reference",
           "config": {"workload": WORKLOAD, "positions_per_step": per_step},
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": f"{per_step} positions per step of the decode workload, one per host "
                                      f"thread ({cores} threads, numpy)"},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--replicas", type=int, default=REPLICAS)
    ap.add_argument("--tokens", type=int, default=DECODE_TOKENS)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--only", choices=["prefill", "mtp", "b32", "gs64", "int2", "sweep"], default=None,
                    help="time one secondary workload alone (profiling)")
    ap.add_argument("--calls", type=int, default=20, help="calls per step of --only mtp / b32")
    ap.add_argument("--prefill-experts", type=int, default=256)
    ap.add_argument("--prefill-t", type=int, default=2048)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per expert-kernel launch, if measured for this build")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300" and args.steps > 2:
        log("[bench] warm-up raised to 3")
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only == "prefill":
        prefill_only(args)
    elif args.only in ("mtp", "b32"):
        few_only(args)
    elif args.only == "gs64":
        weight_format_only(args)
    elif args.only == "int2":
        weight_format_only(args, shape=synth.GLM_INT2, name="int2", fmt="packed int2 with per-row scales")
    elif args.only == "sweep":
        sweep_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
