"""Benchmark of the routed-MoE layer decode step on GB300.

Default workload: the GLM-scale layer (hidden 6144, expert intermediate 2048,
256 routed experts, top-8, one shared expert, affine group-64 4-bit experts,
fp32 router, bf16 activations). One step = 1000 seeded tokens decoded one
after another, each a separate moe_decode call. Weights are synthetic
(seeded), inputs are seeded N(0,1) rounded to bf16.

L2 is defeated by rotating 4 device replicas of the layer (token t uses
replica t mod 4): between two uses of the same bytes ~600 MB of other weights
stream through the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. Under torchrun with N > 1 every rank runs its own
replica of the workload on its own GPU (the decode path has no exchange
step); rank 0 prints tokens/s summed over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# the CPU baseline is the oracle on one core: keep BLAS single-threaded
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s vs 8 TB/s roofline"
UNIT = "tokens/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def algorithmic_bytes(spec: si.LayerSpec):
    """Bytes one decode token must read: router + (top_k + n_shared) experts (canonical format)."""
    router = spec.n_experts * spec.hidden * 4 if spec.router_fmt == "f32" else \
        spec.n_experts * spec.hidden + spec.n_experts * spec.hidden // 64 * 4
    ns = spec.top_k + spec.n_shared
    b = spec.expert_bits
    gu = ns * 2 * spec.inter * (spec.hidden * b // 8 + spec.hidden // 16)
    down = ns * spec.hidden * (spec.inter * b // 8 + spec.inter // 16)
    return router + gu + down, gu, down, router


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the first sample takes a moment: wait for it (bounded) so that a
            # short timed region still falls inside the sampled span
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


KERNEL_SOURCES = {"gateup_decode": ("decode.cu", "common.cuh"),
                  "prefill_gemm_gateup": ("prefill.cu", "sm100.cuh", "common.cuh")}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the sources that define `kernel`: a stored ncu traffic figure is
    only used while it matches."""
    import hashlib
    d = os.path.join(ROOT, "quantized_routed_expert_moe_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def max_over_ranks(vals, device):
    """Elementwise maximum of `vals` over every rank of the default process
    group (the values themselves when there is one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def oracle_sample(layer, X, n_tokens):
    """Time the fp64 oracle on n_tokens tokens; returns tokens/s."""
    import oracle
    Wr = oracle.router_weights_f64(layer.router)
    t0 = time.perf_counter()
    for t in range(n_tokens):
        oracle.moe_token(layer, X[t], Wr=Wr)
    return n_tokens / (time.perf_counter() - t0)


def run_reference(args, spec, workload):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    layer = si.gen_layer(0, 0, spec)
    X = si.gen_tokens(0, 0, 4, spec)
    per_step = 2
    for _ in range(args.warmup):
        oracle_sample(layer, X, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(layer, X, per_step)
    dt = time.perf_counter() - t0
    v = args.steps * per_step / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "tokens_per_step": per_step},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{per_step} tokens per step of the same layer, fp64 numpy, 1 BLAS thread"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PREFILL_DESC = {
    "glm_verify": "GLM-scale verify batches: H6144 I2048 E256 top-8 + 1 shared, T tokens per batch through the "
                  "batch-union path (each distinct expert read once per batch), router bias from Zipf(1.1)",
    "glm_prefill": "GLM-scale prefill chunk: H6144 I2048 E256 top-8 + 1 shared, 128 tokens, "
                   "router bias from Zipf(1.1) expert popularity (uneven expert loads)",
    "glm_prefill_dense": "GLM-scale prefill chunk, all 128 tokens on the same 8 experts "
                         "(router bias +30 on experts 0..7, -30 elsewhere): 9 full 128-token groups",
}


def prefill_layer(workload, seed=0, experts=None):
    import dataclasses
    spec = si.CONFIGS["glm_prefill"]
    if experts:
        spec = dataclasses.replace(spec, n_experts=experts)
    layer = si.gen_layer(seed, 0, spec)
    if workload == "glm_prefill_dense":
        bias = np.full(layer.spec.n_experts, -30.0, np.float32)
        bias[:8] = 30.0
        layer = dataclasses.replace(layer, router_bias=bias)
    return layer


def run_prefill(args, emit=True):
    """One step = one 128-token chunk through each of R rotating layer replicas."""
    ws, rank, local = dist_info()
    T = args.chunk or (4 if args.workload == "glm_verify" else 128)
    layer = prefill_layer(args.workload, experts=args.experts)
    spec = layer.spec
    workload = PREFILL_DESC[args.workload]
    if args.workload == "glm_verify":
        workload = workload.replace("T tokens", f"{T} tokens")
    if args.experts:
        workload = workload.replace("E256", f"E{args.experts}")
    X = si.gen_tokens(1000 * rank, 0, T, spec)
    flops_gu = 2.0 * T * (spec.top_k + spec.n_shared) * 2 * spec.inter * spec.hidden
    flops_down = 2.0 * T * (spec.top_k + spec.n_shared) * spec.hidden * spec.inter
    flops_router = 2.0 * T * spec.n_experts * spec.hidden
    if args.impl == "reference":
        if rank != 0:
            return
        n = 1
        for _ in range(args.warmup):
            oracle_sample(layer, X, n)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_sample(layer, X, n)
        dt = time.perf_counter() - t0
        v = args.steps * n / dt
        print(json.dumps({"impl": "reference", "metric": "MoE-layer prefill tokens/s", "value": v, "unit": UNIT,
                          "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": {"workload": workload, "tokens_per_step": n},
                          "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": f"{n} token of the chunk per step, fp64 numpy, 1 BLAS thread"},
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return

    import torch
    import torch.distributed as dist

    import quantized_routed_expert_moe_gb300 as moe
    from quantized_routed_expert_moe_gb300 import build as _b
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        _b.build()
    if ws > 1:
        dist.barrier()
    R = args.replicas or 4
    reps = [moe.MoELayer(layer, device=local, max_tokens=T) for _ in range(R)]
    x_host = torch.from_numpy(np.ascontiguousarray(X.view(np.int16))).view(torch.bfloat16).pin_memory()
    x_dev = x_host.to("cuda")
    y_dev = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device="cuda")
    y_host = torch.empty((T, spec.hidden), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream()

    def step():
        for r in reps:
            r.prefill_chunk(x_dev, T, y_dev, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    for r in reps:
        st, bits = r.check()
        if st:
            raise RuntimeError(f"prefill reported device error bits {bits:#x}")

    for r in reps:
        moe.moe_profile_start(r.handle, 16 * args.steps)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = {}
    for r in reps:
        for name, (n, t) in moe.moe_profile_stop(r.handle).items():
            a, b = prof.get(name, (0, 0.0))
            prof[name] = (a + n, b + t)

    # end to end: pinned host chunk -> device, prefill, device -> pinned host output
    for _ in range(args.warmup):
        x_dev.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(y_dev, non_blocking=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(y_dev, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0

    # the chunk's expert groups (outside the timed region): the gate/up GEMM
    # streams each group's gate/up block once
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    reps[0].route(x_dev, T, ids, wts)
    torch.cuda.synchronize()
    n_groups = len(np.unique(ids.cpu().numpy())) + spec.n_shared
    rows = T * (spec.top_k + spec.n_shared)
    gu_bytes = (n_groups * 2 * spec.inter * (spec.hidden // 2 + spec.hidden // 16)
                + rows * spec.hidden * 2 + rows * spec.inter * 2)

    ms, e2e_s = max_over_ranks([ms, e2e_s], "cuda")
    total_tokens = T * R * args.steps * ws
    value = total_tokens / (ms / 1e3)
    hbm, tflops, peak_kind = peaks()
    kernels = {k: {"launches": n, "avg_us": t / max(n, 1) * 1e3} for k, (n, t) in prof.items()}
    n_gu, t_gu = prof.get("prefill_gemm_gateup", (0, 0.0))
    gu_avg_s = t_gu / max(n_gu, 1) / 1e3
    achieved = flops_gu / gu_avg_s / 1e12 if n_gu else None
    gbs = gu_bytes / gu_avg_s / 1e9 if n_gu else None
    tensor_roof = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                   "frac": achieved / tflops if achieved else None,
                   "peak_source": f"{peak_kind} bf16_tflops (cuBLAS), burst; fp16 and bf16 share the dense rate",
                   "algorithmic_flops_per_launch": flops_gu}
    hbm_roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                "frac": gbs / hbm if gbs else None, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": gu_bytes,
                "bytes_note": f"{n_groups} expert groups x gate/up block (codes + fp16 scale/bias) "
                              "+ gathered fp16 activations in + fp16 h out"}
    # the binding roof is the one the kernel is closer to; the other rides along
    main, other = (hbm_roof, tensor_roof) if (hbm_roof["frac"] or 0) > (tensor_roof["frac"] or 0) \
        else (tensor_roof, hbm_roof)
    # DRAM traffic per launch from a stored ncu capture of the same sources
    # (a smaller layer of the same shape), scaled to this launch by the
    # algorithmic bytes (the expert groups streamed)
    traffic = None
    tf = os.path.join(ROOT, "profiles", f"prefill_gemm_gateup_{args.workload}_traffic.json")
    if os.path.exists(tf):
        tj = json.load(open(tf))
        if tj.get("kernel_source_sha") == kernel_source_sha("prefill_gemm_gateup"):
            traffic = tj["bytes_per_launch"] * gu_bytes / tj["algorithmic_bytes_per_launch"]
    chunk_flops = flops_gu + flops_down + flops_router
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": f"MoE-layer prefill tokens/s ({T}-token chunks)", "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": workload, "tokens_per_step": T * R, "layer_replicas": R,
                   "l2": f"inputs larger than L2: {R} rotating layer replicas",
                   "parallelism": f"replicas x{ws}"},
        "chunk_tflops": chunk_flops * R * args.steps * ws / (ms / 1e3) / 1e12,
        "roofline": dict(main, traffic=traffic, kernel="prefill_gemm_gateup", avg_launch_us=gu_avg_s * 1e6,
                         other_roof=other, expert_groups=n_groups),
        "kernels": kernels,
        "e2e": {"value": total_tokens / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size()},
        "gpu_launches": sum(n for n, _ in prof.values()),
        "clocks": clk,
        "cpu_baseline": None,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_chunk_sample(layer, X, 8)
    if emit:
        print(json.dumps(line), flush=True)
    return line


def cpu_chunk_sample(layer, X, n):
    """The fp64 oracle on the first n tokens of a chunk (each distinct expert
    dequantised once for the rows that selected it): tokens/s on one core."""
    import oracle
    t0 = time.perf_counter()
    oracle.moe_tokens(layer, X[:n])
    v = n / (time.perf_counter() - t0)
    return {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"the first {n} tokens of the chunk through the fp64 numpy oracle (chunk evaluation), "
                      "1 BLAS thread"}


def run_streamed(args, emit=True):
    """Streamed decode through a stack of GLM-scale layers, each with a 16-slot
    LFU device cache filled from pinned host records. One step = one token
    through every layer; between layers the activation is renormalised
    (x <- bf16(y / rms(y)), a weightless stand-in for the rest of the model) so
    that each layer's routing depends on the previous layer's output.

    Routed expert records come from an alias pool of `pool` distinct records in
    pinned host memory (layer l's expert e uses pool record (l * E + e) * 2654435761
    mod pool): the full stack (75 x 256 records, 407 GB) does not fit in host
    memory; the host-to-device traffic per miss is the same."""
    ws, rank, local = dist_info()
    spec = si.CONFIGS["glm_prefill"]   # GLM shape with Zipf(1.1) router bias
    E, Lc, P = spec.n_experts, args.layers, args.pool
    workload = (f"streamed GLM-scale decode: {Lc} layers of H6144 I2048 E256 top-8 + 1 shared, 16-slot LFU cache "
                f"per layer, Zipf(1.1) routing bias per layer, {P}-record alias pool in pinned host memory; "
                f"chain: {args.chain}; router lookahead: {'on' if args.lookahead else 'off'}; "
                f"cache managed on the {'device' if args.device_cache else 'host'}; "
                f"pinned hottest per layer: {args.pin}" + (f" (usage learned over {args.learn} tokens)" if args.pin else ""))
    if args.impl == "reference":
        if rank != 0:
            return
        layer = si.gen_layer(0, 0, spec)
        X = si.gen_tokens(0, 0, 2, spec)
        for _ in range(args.warmup):
            oracle_sample(layer, X, 1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_sample(layer, X, 1)
        dt = time.perf_counter() - t0
        v = args.steps / dt / Lc   # one token through every layer
        print(json.dumps({"impl": "reference", "metric": "streamed MoE decode tokens/s", "value": v, "unit": UNIT,
                          "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": dt / args.steps * 1e3 * Lc, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": {"workload": workload, "tokens_per_step": 1},
                          "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": "one layer-token per step, scaled to the layer count"},
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return

    import torch
    import torch.distributed as dist

    import quantized_routed_expert_moe_gb300 as moe
    from quantized_routed_expert_moe_gb300 import build as _b
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        _b.build()
    if ws > 1:
        dist.barrier()
    desc = moe.desc_from_spec(spec, cache_slots=16)
    rb = moe.moe_expert_record_bytes(desc)
    pool = torch.empty((P, rb), dtype=torch.uint8).pin_memory()
    pool_np = pool.numpy()
    for p in range(P):
        moe.moe_pack_expert_record(desc, si.gen_expert(0, 1000, p, spec), pool_np[p])
    stack = []
    for l in range(Lc):
        recs = [pool[((l * E + e) * 2654435761) % P] for e in range(E)]
        lay = si.Layer(spec, si.gen_router(0, l, spec), [], si.gen_expert(0, l, E, spec),
                       si.gen_router_bias(0, l, spec), 0, l)
        stack.append(moe.MoELayer(lay, device=local, cache_slots=16, records=recs))
    for li in range(Lc):   # each layer warms the next one's router into L2
        stack[li].set_next(stack[(li + 1) % Lc])
        if args.device_cache:   # LFU step and fills on the device, no host round trip per layer
            stack[li].set_option(moe.MOE_OPT_CACHE_DEVICE, 1)
    X0 = si.gen_tokens(1000 * rank, 0, args.warmup + args.steps, spec)
    x_host = torch.from_numpy(np.ascontiguousarray(X0.view(np.int16))).view(torch.bfloat16).pin_memory()
    x = torch.empty(spec.hidden, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(spec.hidden, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    H = spec.hidden
    rms_norm = torch.nn.functional.rms_norm

    def chain(y):
        if args.chain == "norm":   # the layer output, renormalised
            return rms_norm(y, (H,), eps=1e-12)
        # a residual-stream stand-in: the layer adds its output at a quarter of
        # the stream's RMS, and the sum is renormalised
        return rms_norm(torch.add(x.float(), rms_norm(y, (H,), eps=1e-12), alpha=0.25), (H,), eps=1e-12)

    def token(i, src=None):
        x.copy_((x_host if src is None else src)[i], non_blocking=True)
        for li, ml in enumerate(stack):
            if args.lookahead and li + 1 < Lc:
                # the next layer's router on this layer's input: stage its predicted experts now
                stack[li + 1].cache_prefetch(x, stream=stream)
            ml.decode(x, None, y, stream=stream)
            x.copy_(chain(y))   # bf16 rounding in the copy

    if args.pin:
        # the learning cache: record which experts a run of tokens (a seeded
        # stream of their own) routes to, then pin each layer's hottest
        XL = si.gen_tokens(1000 * rank + 500, 0, args.learn, spec)
        xl_host = torch.from_numpy(np.ascontiguousarray(XL.view(np.int16))).view(torch.bfloat16).pin_memory()
        for i in range(args.learn):
            token(i, xl_host)
        torch.cuda.synchronize()
        for ml in stack:
            ml.pin_hottest(args.pin)
    # warm-up tokens, recording every layer's selection: the oracle's LFU run
    # over the same id stream must give the same hits and misses
    rec_ids = torch.empty((args.warmup, Lc, spec.top_k), dtype=torch.int32, device="cuda")
    rec_w = torch.empty((args.warmup, Lc, spec.top_k), dtype=torch.float32, device="cuda")
    pre = [ml.cache_stats() for ml in stack]

    def token_rec(i):
        x.copy_(x_host[i], non_blocking=True)
        for li, ml in enumerate(stack):
            ml.decode(x, None, y, stream=stream)
            ml.selection(1, rec_ids[i, li], rec_w[i, li], stream=stream)
            x.copy_(chain(y))

    for i in range(args.warmup):
        if args.lookahead:
            token(i)
        else:
            token_rec(i)
    torch.cuda.synchronize()
    s0 = [ml.cache_stats() for ml in stack]
    lfu_check = None
    if not args.lookahead and not args.pin:
        import oracle
        ids_np = rec_ids.cpu().numpy()
        o_hits = o_miss = 0
        for li in range(Lc):
            c = oracle.LFUCache(16)
            for i in range(args.warmup):
                h, f = c.access(ids_np[i, li])
                o_hits += len(h)
                o_miss += len(f)
        m_hits = sum(b["hits"] - a["hits"] for a, b in zip(pre, s0))
        m_miss = sum(b["misses"] - a["misses"] for a, b in zip(pre, s0))
        lfu_check = {"tokens": args.warmup, "layers": Lc, "hits": m_hits, "misses": m_miss,
                     "oracle_hits": o_hits, "oracle_misses": o_miss,
                     "hit_rate": m_hits / max(m_hits + m_miss, 1),
                     "oracle_hit_rate": o_hits / max(o_hits + o_miss, 1),
                     "note": "the warm-up tokens (from an empty cache), every layer's selection recorded and run "
                             "through the oracle's LFU simulation"}
    p0 = [ml.prefetch_stats() for ml in stack]
    clocks = ClockSampler(local)
    clocks.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.steps):
        token(args.warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    s1 = [ml.cache_stats() for ml in stack]
    pf = [{key: b[key] - a[key] for key in b} for a, b in zip(p0, [ml.prefetch_stats() for ml in stack])]
    hits = sum(b["hits"] - a["hits"] for a, b in zip(s0, s1))
    misses = sum(b["misses"] - a["misses"] for a, b in zip(s0, s1))
    # fills for misses and fills for predictions
    h2d = sum(b["bytes_h2d"] - a["bytes_h2d"] for a, b in zip(s0, s1)) + sum(p["bytes_h2d"] for p in pf)
    graph = None
    if args.device_cache:
        # the same steps with each token's pass through the stack captured once
        # as a CUDA graph (no host work per layer at all), replayed per token
        try:
            x_in = torch.empty_like(x)
            gs = torch.cuda.Stream()
            gs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()

            def token_g():
                x.copy_(x_in)
                for ml in stack:
                    ml.decode(x, None, y, stream=gs)
                    x.copy_(chain(y))
            with torch.cuda.stream(gs):
                x_in.copy_(x_host[0], non_blocking=True)
                token_g()
                gs.synchronize()
                with torch.cuda.graph(g, stream=gs):
                    token_g()
            stream.wait_stream(gs)
            for i in range(args.warmup):
                x_in.copy_(x_host[i], non_blocking=True)
                g.replay()
            torch.cuda.synchronize()
            gev0, gev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            gev0.record(stream)
            for i in range(args.steps):
                x_in.copy_(x_host[args.warmup + i], non_blocking=True)
                g.replay()
            gev1.record(stream)
            torch.cuda.synchronize()
            gms = gev0.elapsed_time(gev1)
            graph = {"value": args.steps / (gms / 1e3), "unit": UNIT, "ms_per_step": gms / args.steps,
                     "note": "each token through the stack captured once as a CUDA graph, replayed per token "
                             "(the same tokens as the timed steps)"}
            del g
        except Exception as exc:   # reported, not fatal
            graph = {"error": str(exc).splitlines()[0][:200]}
            torch.cuda.synchronize()
    # pinned host -> device copy peak on this machine, for the fraction
    big = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dst.copy_(big, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(4):
        dst.copy_(big, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_peak = 4 * (1 << 30) / (e0.elapsed_time(e1) / 1e3) / 1e9
    ms, wall = max_over_ranks([ms, wall], "cuda")
    value = args.steps * ws / (ms / 1e3)
    for ml in stack:
        ml.close()
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    h2d_gbs = h2d / (ms / 1e3) / 1e9
    line = {
        "metric": "streamed MoE decode tokens/s (every layer of the stack per token)", "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "tokens_per_step": 1, "layers": Lc, "pool_records": P,
                   "record_bytes": rb, "parallelism": f"replicas x{ws}"},
        "hit_rate": hits / max(hits + misses, 1),
        "h2d_gbs": h2d_gbs,
        "graph": graph,
        "lookahead": {"calls": sum(p["calls"] for p in pf), "predicted_resident": sum(p["resident"] for p in pf),
                      "fills": sum(p["fills"] for p in pf), "bytes_h2d": sum(p["bytes_h2d"] for p in pf)},
        "roofline": {"bound": "h2d", "achieved": h2d_gbs, "peak": h2d_peak, "unit": "GB/s",
                     "frac": h2d_gbs / h2d_peak, "traffic": None, "kernel": "cache fills (cudaMemcpyAsync)",
                     "peak_source": "measured here: pinned 1 GiB host-to-device copy"},
        "e2e": {"value": args.steps * ws / wall, "unit": UNIT, "h2d_bytes_per_step": spec.hidden * 2 + h2d / args.steps,
                "d2h_bytes_per_step": 0},
        "lfu_check": lfu_check,
        "gpu_launches": None,
        "clocks": clk,
        "cpu_baseline": None,
    }
    if ws == 1 and not args.no_cpu_baseline:
        layer0 = si.Layer(spec, si.gen_router(0, 0, spec), LazyExperts(0, 1000, spec, P, 0),
                          si.gen_expert(0, 0, E, spec), si.gen_router_bias(0, 0, spec), 0, 0)
        n = 2
        t0 = time.perf_counter()
        for i in range(n):
            import oracle
            oracle.moe_token(layer0, X0[i])
        dt = (time.perf_counter() - t0) / n
        line["cpu_baseline"] = {"value": 1.0 / (dt * Lc), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{n} layer-tokens of the first layer through the fp64 oracle, scaled to "
                                          f"{Lc} layers per token, 1 BLAS thread"}
    if emit:
        print(json.dumps(line), flush=True)
    return line


class LazyExperts:
    """The routed experts of one layer of the streamed stack, generated on
    first use (layer l's expert e is alias-pool record (l * E + e) * 2654435761
    mod P, itself seeded expert p of layer `pool_layer`)."""

    def __init__(self, seed, pool_layer, spec, P, layer):
        self.seed, self.pool_layer, self.spec, self.P, self.layer = seed, pool_layer, spec, P, layer
        self.cache = {}

    def __len__(self):
        return self.spec.n_experts

    def __getitem__(self, e):
        p = ((self.layer * self.spec.n_experts + int(e)) * 2654435761) % self.P
        if p not in self.cache:
            self.cache[p] = si.gen_expert(self.seed, self.pool_layer, p, self.spec)
        return self.cache[p]


def h2d_peak_gbs(stream):
    """Pinned host -> device copy bandwidth of this machine (1 GiB copies)."""
    import torch
    big = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dst.copy_(big, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(4):
        dst.copy_(big, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    del big, dst
    return 4 * (1 << 30) / (e0.elapsed_time(e1) / 1e3) / 1e9


def run_streamed_prefill(args):
    """Prefill chunks on one streamed GLM-scale layer: the chunk's distinct
    experts pass through the 16-slot cache in waves (batch union), routed
    records from a pinned alias pool. One step = one distinct 128-token chunk."""
    ws, rank, local = dist_info()
    spec = si.CONFIGS["glm_prefill"]
    E, P = spec.n_experts, args.pool
    T = args.chunk or 128
    workload = (f"streamed GLM-scale prefill: H6144 I2048 E256 top-8 + 1 shared, {T}-token chunks, 16-slot cache, "
                f"Zipf(1.1) routing bias, {P}-record alias pool in pinned host memory")
    if args.impl == "reference":
        if rank != 0:
            return
        layer = si.gen_layer(0, 0, spec)
        X = si.gen_tokens(0, 0, 2, spec)
        for _ in range(args.warmup):
            oracle_sample(layer, X, 1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_sample(layer, X, 1)
        v = args.steps / (time.perf_counter() - t0)
        print(json.dumps({"impl": "reference", "metric": f"streamed MoE-layer prefill tokens/s ({T}-token chunks)",
                          "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 / v, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic", "config": {"workload": workload, "tokens_per_step": 1},
                          "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": "one token per step through the fp64 oracle"},
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import torch
    import quantized_routed_expert_moe_gb300 as moe
    from quantized_routed_expert_moe_gb300 import build as _b
    torch.cuda.set_device(local)
    if rank == 0:
        _b.build()
    desc = moe.desc_from_spec(spec, cache_slots=16, max_tokens=T)
    rb = moe.moe_expert_record_bytes(desc)
    pool = torch.empty((P, rb), dtype=torch.uint8).pin_memory()
    pool_np = pool.numpy()
    for p in range(P):
        moe.moe_pack_expert_record(desc, si.gen_expert(0, 1000, p, spec), pool_np[p])
    recs = [pool[(e * 2654435761) % P] for e in range(E)]
    lay = si.Layer(spec, si.gen_router(0, 0, spec), [], si.gen_expert(0, 0, E, spec), si.gen_router_bias(0, 0, spec))
    ml = moe.MoELayer(lay, device=local, max_tokens=T, cache_slots=16, records=recs)
    n_chunks = args.warmup + args.steps
    X = si.gen_tokens(1000 * rank, 0, T * n_chunks, spec).reshape(n_chunks, T, spec.hidden)
    x_host = torch.from_numpy(np.ascontiguousarray(X.view(np.int16))).view(torch.bfloat16).pin_memory()
    x_dev = x_host.to("cuda")
    y = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        ml.prefill_chunk(x_dev[i], T, y, stream=stream)
    torch.cuda.synchronize()
    s0 = ml.cache_stats()
    clocks = ClockSampler(local)
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.steps):
        ml.prefill_chunk(x_dev[args.warmup + i], T, y, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    s1 = ml.cache_stats()
    st, bits = ml.check()
    if st:
        raise RuntimeError(f"streamed prefill reported device error bits {bits:#x}")
    ml.close()
    hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
    h2d = s1["bytes_h2d"] - s0["bytes_h2d"]
    waves = s1["tokens"] - s0["tokens"]
    peak = h2d_peak_gbs(stream)
    h2d_gbs = h2d / (ms / 1e3) / 1e9
    value = T * args.steps / (ms / 1e3)
    if rank != 0:
        return
    line = {
        "metric": f"streamed MoE-layer prefill tokens/s ({T}-token chunks)", "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": workload, "tokens_per_step": T, "pool_records": P, "record_bytes": rb,
                   "parallelism": f"replicas x{ws}"},
        "waves_per_chunk": waves / args.steps,
        "hit_rate": hits / max(hits + misses, 1),
        "h2d_gbs": h2d_gbs,
        "roofline": {"bound": "h2d", "achieved": h2d_gbs, "peak": peak, "unit": "GB/s", "frac": h2d_gbs / peak,
                     "traffic": None, "kernel": "cache fills (cudaMemcpyAsync) between the waves' GEMMs",
                     "peak_source": "measured here: pinned 1 GiB host-to-device copy"},
        "e2e": {"value": T * args.steps / wall, "unit": UNIT,
                "h2d_bytes_per_step": T * spec.hidden * 2 + h2d / args.steps, "d2h_bytes_per_step": 0},
        "gpu_launches": None,
        "clocks": clk,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


DECODE_DESC = {"glm_decode": "GLM-scale decode: H6144 I2048 E256 top-8 + 1 shared, q4g64 experts, fp32 router",
               "glm_decode_q2": "GLM-scale decode: H6144 I2048 E256 top-8 + 1 shared, q2g64 experts, fp32 router",
               "gemma_decode": "Gemma-style decode: H2816 I704 E128 top-8 + 1 shared, q4g64 experts, q8g64 router",
               "tiny": "tiny layer: H512 I256 E32 top-8 + 1 shared, fp32 I/O"}
DECODE_REPLICAS = {"glm_decode": 4, "glm_decode_q2": 4, "gemma_decode": 16, "tiny": 64}
DECODE_CPU_TOKENS = {"glm_decode": 6, "glm_decode_q2": 6, "gemma_decode": 60, "tiny": 400}
DTYPE = "int8 x int4 dp4a on 16-bit fixed-point activations per run of 32, fp32 accumulate and SwiGLU"


def decode_bench(args, name, spec, workload):
    """T seeded tokens decoded one after another per step, token t on replica t
    mod R; returns the JSON line (dict)."""
    import torch
    import torch.distributed as dist

    import quantized_routed_expert_moe_gb300 as moe

    ws, rank, local = dist_info()
    R = args.replicas or DECODE_REPLICAS[name]
    layer = si.gen_layer(0, 0, spec)
    reps = [moe.MoELayer(layer, device=local) for _ in range(R)]
    T = args.tokens
    X = si.gen_tokens(1000 * rank, 0, T, spec)   # distinct tokens per rank
    xdt = torch.bfloat16 if spec.act == "bf16" else torch.float32
    x_np_view = X.view(np.int16) if spec.act == "bf16" else X
    x_host = torch.from_numpy(np.ascontiguousarray(x_np_view)).view(xdt).pin_memory()
    x_dev = x_host.to("cuda", non_blocking=False)
    y_dev = torch.empty((T, spec.hidden), dtype=xdt, device="cuda")
    y_host = torch.empty((T, spec.hidden), dtype=xdt).pin_memory()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    handles = [r.handle for r in reps]
    dec = moe.lib().moe_decode
    row = spec.hidden * x_dev.element_size()
    xb, yb = x_dev.data_ptr(), y_dev.data_ptr()

    def step():
        for t in range(T):
            st = dec(handles[t % R], xb + t * row, yb + t * row, None, sp)
            if st:
                raise moe.MoEError(st, "moe_decode", moe.moe_last_error())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # timed region: K steps, CUDA events on the launching stream, clocks sampled alongside
    clocks = ClockSampler(local)
    clocks.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    for r in reps:
        st, bits = r.check()
        if st:
            raise RuntimeError(f"decode reported device error bits {bits:#x}")

    # the same K steps again with a CUDA event pair around every kernel the
    # library launches (recorded by the library on the launch stream)
    for h in handles:
        moe.moe_profile_start(h, (3 * T // R + 16) * args.steps)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = {}
    for h in handles:
        for kname, (n, t) in moe.moe_profile_stop(h).items():
            a, b = prof.get(kname, (0, 0.0))
            prof[kname] = (a + n, b + t)

    # phase trace (--trace): tokens decoded with MOE_OPT_TRACE on; per kernel,
    # the per-CTA global-timer stamps (start, dependency met, main work done,
    # end) relative to the router's first CTA, median and last CTA
    phases = None
    if getattr(args, "trace", False):
        phases = []
        n_tr = min(T, 8 * R)
        for rep_i in range(3):
            for h in handles:
                moe.moe_layer_set_option(h, 3, 1)
            for t in range(n_tr):
                st = dec(handles[t % R], xb + t * row, yb + t * row, None, sp)
                if st:
                    raise moe.MoEError(st, "moe_decode", moe.moe_last_error())
            torch.cuda.synchronize()
            tr = moe.moe_trace_read_split(handles[(n_tr - 1) % R])
            for h in handles:
                moe.moe_layer_set_option(h, 3, 0)
            base = min(c[0] for c in tr[0] if c[0])
            ph = {}
            for kk, kn in enumerate(("router", "gateup", "down")):
                cs = np.array([c for c in tr[kk] if c[0]], dtype=np.float64)
                if len(cs) == 0:
                    continue
                cs = (cs - base) / 1e3
                ph[kn] = {"ctas": int(len(cs)),
                          **{f"{p}_{w}": round(float(f(cs[:, i])), 2)
                             for i, p in enumerate(moe.SPLIT_TRACE_POINTS) for w, f in (("med", np.median), ("max", np.max))}}
            phases.append(ph)

    # per-token intervals: one step again with an event after every token. The
    # events sit between consecutive tokens' kernels (they block the overlap of
    # the next token's router prologue with this token's tail), so these are an
    # upper bound on the per-token time of the timed region.
    tev = [torch.cuda.Event(enable_timing=True) for _ in range(T + 1)]
    torch.cuda.synchronize()
    tev[0].record(stream)
    for t in range(T):
        st = dec(handles[t % R], xb + t * row, yb + t * row, None, sp)
        if st:
            raise moe.MoEError(st, "moe_decode", moe.moe_last_error())
        tev[t + 1].record(stream)
    torch.cuda.synchronize()
    lat = np.array([tev[t].elapsed_time(tev[t + 1]) * 1e3 for t in range(T)])
    latency = {"p50": float(np.percentile(lat, 50)), "p95": float(np.percentile(lat, 95)),
               "p99": float(np.percentile(lat, 99)), "max": float(lat.max()), "unit": "us",
               "note": "interval between events recorded after consecutive tokens of one step"}

    # the same step captured once into a CUDA graph and replayed K times
    graph = None
    try:
        gstream = torch.cuda.Stream()
        gstream.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gstream):
            gsp = gstream.cuda_stream
            step_g = lambda: [dec(handles[t % R], xb + t * row, yb + t * row, None, gsp) for t in range(T)]
            step_g()   # untimed warm-up on the capture stream
            gstream.synchronize()
            with torch.cuda.graph(g, stream=gstream):
                codes = step_g()
        if any(codes):
            raise RuntimeError(f"moe_decode returned {max(codes)} during capture")
        stream.wait_stream(gstream)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        gev0, gev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gev0.record(torch.cuda.current_stream())
        for _ in range(args.steps):
            g.replay()
        gev1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        gms = gev0.elapsed_time(gev1)
        graph = {"value": T * args.steps / (gms / 1e3), "unit": UNIT, "ms_per_step": gms / args.steps,
                 "note": "one step (T decodes, rotating replicas) captured once, replayed K times"}
        del g
    except Exception as exc:   # reported, not fatal: the plain timed region above is the headline
        graph = {"error": str(exc).splitlines()[0][:200]}
        torch.cuda.synchronize()

    # end to end with HOST buffers: every step copies its T input tokens from
    # pinned host memory to the device, decodes them through moe_decode on the
    # same R rotating replicas as the timed region, copies the T outputs back
    # to pinned host memory and synchronises
    def step_e2e():
        x_dev.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(y_dev, non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step_e2e()
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step_e2e()
    e2e_s = time.perf_counter() - t0

    ms, e2e_s = max_over_ranks([ms, e2e_s], "cuda")
    total_tokens = T * args.steps * ws
    value = total_tokens / (ms / 1e3)
    e2e = total_tokens / e2e_s

    hbm, _, peak_kind = peaks()
    tot_b, gu_b, down_b, router_b = algorithmic_bytes(spec)
    dom, dom_bytes = "gateup_decode", gu_b
    n_dom, t_dom = prof.get(dom, (0, 0.0))
    dom_avg_ms = t_dom / max(n_dom, 1)
    dom_gbs = dom_bytes / (dom_avg_ms / 1e3) / 1e9 if n_dom else None
    launches = sum(n for n, _ in prof.values())
    kernels = {k: {"launches": n, "avg_us": t / max(n, 1) * 1e3, "share": t / max(sum(v[1] for v in prof.values()), 1e-9)}
               for k, (n, t) in prof.items()}
    for r in reps:
        r.close()

    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        n_cpu = DECODE_CPU_TOKENS[name]
        v = oracle_sample(layer, X, n_cpu)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n_cpu} tokens of the same layer through the fp64 numpy oracle, 1 BLAS thread"}
        if name == "glm_decode":
            cpu["all_cores"] = oracle_all_cores(name, X, 2 * (os.cpu_count() or 1))

    traffic = None
    tf = os.path.join(ROOT, "profiles", f"{dom}_{name}_traffic.json")
    if os.path.exists(tf):
        tj = json.load(open(tf))
        if tj.get("kernel_source_sha") == kernel_source_sha(dom):
            traffic = tj.get("bytes_per_launch")

    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": workload, "tokens_per_step": T, "layer_replicas": R,
                   "l2": f"inputs larger than L2: {R} rotating layer replicas "
                         f"({R * (len(layer.experts) + 1) * spec.expert_bytes() / 1e9:.1f} GB of weights)",
                   "weights": f"affine group-64 {spec.expert_bits}-bit experts, dequantised on the fly",
                   "parallelism": f"replicas x{ws}"},
        "effective_hbm_gbs": tot_b * value / ws / 1e9,
        "hbm_roofline_frac_nominal_8tbs": tot_b * value / ws / 8e12,
        "hbm_roofline_frac_measured": tot_b * value / ws / 1e9 / hbm,
        "roofline": {"bound": "hbm", "achieved": dom_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": (dom_gbs / hbm) if dom_gbs else None, "traffic": traffic,
                     "kernel": dom, "peak_source": f"{peak_kind} hbm_gbs (copy), burst",
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "avg_launch_us": dom_avg_ms * 1e3},
        "kernels": kernels,
        **({"phase_trace_us": phases} if phases is not None else {}),
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size(),
                "path": "pinned host -> device copy of the step's tokens, moe_decode per token over the same "
                        "rotating replicas as the timed region, device -> pinned host copy, synchronize"},
        "gpu_launches": launches,
        "per_token_latency": latency,
        "graph": graph,
        "clocks": clk,
        "cpu_baseline": cpu,
    }


def _oracle_worker(job):
    """One token of the oracle (a spawned process): the layer's router, the
    shared expert and the 8 selected experts are generated here."""
    import oracle
    name, x, seed = job
    spec = si.CONFIGS[name]

    class Lazy:
        def __init__(self):
            self.c = {}

        def __len__(self):
            return spec.n_experts

        def __getitem__(self, e):
            e = int(e)
            if e not in self.c:
                self.c[e] = si.gen_expert(seed, 0, e, spec)
            return self.c[e]

    layer = si.Layer(spec, si.gen_router(seed, 0, spec), Lazy(),
                     si.gen_expert(seed, 0, spec.n_experts, spec) if spec.n_shared else None,
                     si.gen_router_bias(seed, 0, spec), seed, 0)
    t0 = time.perf_counter()
    oracle.moe_token(layer, x)
    return time.perf_counter() - t0


def oracle_all_cores(name, X, n):
    """The oracle on every host core at once: n tokens over a pool of
    os.cpu_count() spawned processes (one BLAS thread each); tokens/s of the
    whole pool, counting only the oracle's time per token in each worker."""
    import concurrent.futures as cf
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    jobs = [(name, X[i % len(X)], 0) for i in range(n)]
    t0 = time.perf_counter()
    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        per = list(ex.map(_oracle_worker, jobs))
    wall = time.perf_counter() - t0
    busy = sum(per)
    return {"value": n / (busy / cores) if busy else None, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} tokens over {cores} spawned worker processes (each generates the layer's router "
                      "and the experts a token needs, then times the fp64 oracle on it); value = tokens / "
                      "(summed oracle seconds / cores)",
            "wall_s_including_generation": wall}


def sub_args(args, **kw):
    import copy
    a = copy.copy(args)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="glm_decode",
                    choices=["glm_decode", "glm_decode_q2", "gemma_decode", "tiny", "glm_prefill", "glm_prefill_dense",
                             "glm_verify", "glm_streamed", "glm_streamed_prefill"])
    ap.add_argument("--layers", type=int, default=75, help="glm_streamed: layers in the stack")
    ap.add_argument("--pool", type=int, default=256,
                    help="glm_streamed: distinct expert records in pinned host memory (alias pool)")
    ap.add_argument("--tokens", type=int, default=1000)
    ap.add_argument("--chain", default="norm", choices=["norm", "residual"],
                    help="glm_streamed: how one layer's output becomes the next layer's input")
    ap.add_argument("--lookahead", action="store_true",
                    help="glm_streamed: stage each next layer's predicted experts (moe_cache_prefetch)")
    ap.add_argument("--pin", type=int, default=0,
                    help="glm_streamed: pin each layer's N most used experts after --learn tokens (learning cache)")
    ap.add_argument("--learn", type=int, default=32, help="glm_streamed: tokens whose routing --pin learns from")
    ap.add_argument("--device-cache", action="store_true",
                    help="glm_streamed: device-managed caches (MOE_OPT_CACHE_DEVICE); also times the token as a CUDA graph")
    ap.add_argument("--chunk", type=int, default=None,
                    help="tokens per prefill chunk / verify batch (default 128; glm_verify: 4)")
    ap.add_argument("--replicas", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="default workload: print the GLM-scale decode line without the other configurations")
    ap.add_argument("--trace", action="store_true",
                    help="decode workloads: add the kernels' per-CTA phase stamps of a few tokens to the line")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the routed-expert count (a smaller layer of the same shape, for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.workload.startswith("glm_prefill") or args.workload == "glm_verify":
        run_prefill(args)
        return
    if args.workload == "glm_streamed" and args.device_cache and args.lookahead:
        ap.error("--lookahead stages on the host; it does not combine with --device-cache")
    if args.workload == "glm_streamed":
        run_streamed(args)
        return
    if args.workload == "glm_streamed_prefill":
        run_streamed_prefill(args)
        return
    spec = si.CONFIGS[args.workload]
    if args.experts:
        import dataclasses
        spec = dataclasses.replace(spec, n_experts=args.experts)
    desc = DECODE_DESC[args.workload]
    if args.experts:
        desc = desc.replace(f"E{si.CONFIGS[args.workload].n_experts}", f"E{args.experts}")
    workload = f"{desc}; {args.tokens} sequential single-token decodes per step"
    if args.impl == "reference":
        run_reference(args, spec, workload)
        return

    import torch
    import torch.distributed as dist

    from quantized_routed_expert_moe_gb300 import build as _b

    ws, rank, local = dist_info()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        _b.build()
    if ws > 1:
        dist.barrier()

    line = decode_bench(args, args.workload, spec, workload)
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    if args.workload == "glm_decode" and ws == 1 and not args.headline_only and not args.experts:
        # the other configurations of the same path, each with its own
        # roofline, oracle baseline and clock record
        subs = {
            "gemma_decode": lambda: decode_bench(
                sub_args(args, replicas=None), "gemma_decode", si.CONFIGS["gemma_decode"],
                DECODE_DESC["gemma_decode"] + f"; {args.tokens} sequential single-token decodes per step"),
            "glm_prefill_dense": lambda: run_prefill(sub_args(args, workload="glm_prefill_dense", replicas=None,
                                                              chunk=None), emit=False),
            "glm_prefill": lambda: run_prefill(sub_args(args, workload="glm_prefill", replicas=None, chunk=None),
                                               emit=False),
            "glm_streamed": lambda: run_streamed(sub_args(args, workload="glm_streamed", layers=75, pool=256,
                                                          steps=20, warmup=16, device_cache=True, lookahead=False,
                                                          pin=0, chain="norm"), emit=False),
        }
        line["configs"] = {}
        for name, fn in subs.items():
            try:
                line["configs"][name] = fn()
            except Exception as exc:   # reported in the line, the headline stands
                line["configs"][name] = {"error": f"{type(exc).__name__}: {str(exc).splitlines()[0][:300]}"}
            torch.cuda.empty_cache()
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
