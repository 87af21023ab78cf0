"""Benchmark: NVFP4 linear-layer step (Fprop + Dgrad + Wgrad) on GB300.

Workload: the MLP up-projection layer, M=8192 tokens, K=5120, N=20480, BF16
inputs drawn by nvfp4_bit_numerics_gb300.workloads (X ~ N(0,1) with 8 outlier
channels x30, W ~ N(0, 0.014), dY ~ N(0, 1e-4)).  One step = every part of
the path: amax (plain and Hadamard-transformed), X -> rowwise + transposed
Hadamard quantization, W -> 2D 16x16 quantization (W and W^T), dY ->
rowwise + transposed Hadamard quantization with stochastic rounding, and
the three block-scaled FP4 GEMMs.  Throughput = 6*M*K*N flops per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  Under torchrun every rank runs its own layer step on
its own token shard (weak scaling; data-parallel ranks need no exchange on
this path); rank 0 prints.  --impl reference times the CPU oracle on a
64-token slice of the same layer step.
"""

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, K, N = 8192, 5120, 20480
FLOPS_PER_STEP = 6 * M * K * N          # three GEMMs of 2*M*N*K
FLOPS_PER_GEMM = 2 * M * K * N
WORKLOAD = "nvfp4_linear_fwd_bwd_mlp_up_8192x5120x20480"
SEED = 2
ORACLE_TOKENS = 64
FP4_OVER_BF16 = 13.5 / 2.25             # nominal dense FP4 : BF16 tensor-core ratio
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_over_ranks(x, world, device=None):
    """Max of a per-rank scalar over all ranks (the slowest rank sets the step
    time); a no-op on one rank."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(ms_per_step, world):
    """Weak scaling: every rank runs one full layer step per step."""
    return FLOPS_PER_STEP * world / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", HBM_FALLBACK_GBS), d.get("bf16_tflops", BF16_FALLBACK_TFLOPS), "measured"
    return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gemm_code_hash():
    """sha256 of gemm_kernel.cu with its comments and blank lines removed:
    the code the counters were taken on (comment edits keep it)."""
    import re

    src = os.path.join(ROOT, "nvfp4_bit_numerics_gb300", "csrc", "gemm_kernel.cu")
    with open(src) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()


def traffic_record():
    """DRAM bytes per GEMM launch from the committed ncu summary, valid only
    while the GEMM code is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("gemm_kernel_code_sha256") != gemm_code_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def time_ms(fn, stream, reps=10, warm=2):
    """Mean device time of fn() on `stream` (CUDA events)."""
    import torch

    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def library_gemms(pairs, stream):
    """For context only (never the product path): the same GEMMs through
    cuBLAS BF16 (torch.matmul) and cuBLASLt's NVFP4 GEMM (torch._scaled_mm on
    this library's own quantized operands, whose scale layout it accepts).
    pairs: {name: (a_bf16, b_bf16, out_bf16, a_q, b_q)} with out = a @ b^T."""
    import torch

    res = {"cublas_bf16_ms": {}, "cublaslt_nvfp4_ms": {}}
    for name, (a, b, out, qa, qb) in pairs.items():
        res["cublas_bf16_ms"][name] = time_ms(lambda: torch.matmul(a, b.t(), out=out), stream)
        try:
            fa, fb = qa.codes.view(torch.float4_e2m1fn_x2), qb.codes.view(torch.float4_e2m1fn_x2)
            sa, sb = qa.scales.view(torch.float8_e4m3fn), qb.scales.view(torch.float8_e4m3fn)
            res["cublaslt_nvfp4_ms"][name] = time_ms(
                lambda: torch._scaled_mm(fa, fb.t(), sa, sb, out_dtype=torch.bfloat16), stream)
        except Exception as e:  # an older torch without FP4 types
            res["cublaslt_nvfp4_ms"][name] = None
            res["cublaslt_nvfp4_error"] = type(e).__name__
    return res


def cpu_oracle_step(x_f, w_f, dy_f, threads=0):
    """One bounded oracle sample: the whole layer step for a 64-token slice of
    X and dY (all of W), through the plain C++ oracle on the host's cores.
    Returns (seconds, flops)."""
    from oracle import cxx

    xs, dys = x_f[:ORACLE_TOKENS], dy_f[:ORACLE_TOKENS]
    t0 = time.perf_counter()
    f = cxx.linear_fwd(xs, w_f, SEED, threads=threads)
    cxx.linear_bwd(dys, f, SEED, threads=threads)
    return time.perf_counter() - t0, 6 * ORACLE_TOKENS * K * N


def cpu_quantize_full(x_f, w_f, dy_f, threads=0, tensors=("x", "w", "dy")):
    """The layer step's three quantize passes in full through the plain C++
    oracle: X [8192, 5120] (amax, amax of the transform along tokens, rowwise
    RNE, transposed Hadamard RNE), W [20480, 5120] (amax, 16x16 blocks, W and
    W^T), dY [8192, 20480] (amax, amax of the transform, rowwise SR, transposed
    Hadamard SR).  Returns {tensor: seconds} for the tensors named."""
    from oracle import cxx

    out = {}
    if "x" in tensors:
        t0 = time.perf_counter()
        cxx.quantize_1d(x_f, "rne", amax=cxx.tensor_amax(x_f, threads), threads=threads)
        cxx.quantize_transpose(x_f, "rne", rht_seed=SEED, amax=cxx.amax_rht(x_f, SEED, 0, threads),
                               threads=threads)
        out["x"] = time.perf_counter() - t0
    if "w" in tensors:
        t0 = time.perf_counter()
        cxx.quantize_2d(w_f, threads=threads)
        out["w"] = time.perf_counter() - t0
    if "dy" in tensors:
        t0 = time.perf_counter()
        cxx.quantize_1d(dy_f, "sr", seed=SEED, stream_id=0, amax=cxx.tensor_amax(dy_f, threads), threads=threads)
        cxx.quantize_transpose(dy_f, "sr", seed=SEED, stream_id=1, rht_seed=SEED,
                               amax=cxx.amax_rht(dy_f, SEED, 0, threads), threads=threads)
        out["dy"] = time.perf_counter() - t0
    return out


def cpu_baseline_record(x_f, w_f, dy_f):
    """The bench line's cpu_baseline: the C++ oracle with one std::thread per
    host core, timed on the layer step's quantize passes in full and on a
    64-token slice of the whole layer step (the GEMMs, float64 on the
    dequantized operands, are the bulk of the oracle's work)."""
    cores = os.cpu_count()
    s, flops = cpu_oracle_step(x_f, w_f, dy_f, threads=cores)
    q = cpu_quantize_full(x_f, w_f, dy_f, threads=cores)
    # one thread, on X (the 8192x5120 tensor size of the quantize sweep) only,
    # to keep the run short
    q1 = cpu_quantize_full(x_f, w_f, dy_f, threads=1, tensors=("x",))
    elems = {"x": M * K, "w": N * K, "dy": M * N}
    # algorithmic bytes: BF16 read once per amax pass and once per quantize
    # pass, 0.5625 B per element per NVFP4 output
    qbytes = {"x": elems["x"] * (2 * 2 + 2 * 0.5625), "w": elems["w"] * (2 * 2 + 2 * 0.5625),
              "dy": elems["dy"] * (2 * 2 + 2 * 0.5625)}
    return {
        "value": flops / s / 1e12, "unit": "TFLOP/s", "cores": cores, "threads": cores, "kind": "oracle",
        "sample": "plain C++ oracle (oracle/cxx), one std::thread per core: the layer step on a %d-token "
                  "slice of X and dY with all of W (%.1f GFLOP, float64 GEMMs), %.2f s" % (ORACLE_TOKENS,
                                                                                         flops / 1e9, s),
        "quantize_full": {k: {"s": v, "gbs": qbytes[k] / v / 1e9} for k, v in q.items()},
        "quantize_full_note": "each tensor's amax and quantize passes of the layer step in full "
                              "(X 8192x5120, W 20480x5120, dY 8192x20480)",
        "quantize_full_1thread": {k: {"s": v, "gbs": qbytes[k] / v / 1e9, "threads": 1} for k, v in q1.items()},
    }


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    from nvfp4_bit_numerics_gb300 import workloads

    x, w, dy = workloads.mlp_up()
    x_f, w_f, dy_f = (workloads.bf16_to_f32_numpy(t) for t in (x, w, dy))
    cores = os.cpu_count()
    for _ in range(args.warmup):
        cpu_oracle_step(x_f, w_f, dy_f, threads=cores)
    times = []
    flops = 0
    for _ in range(args.steps):
        dt, fl = cpu_oracle_step(x_f, w_f, dy_f, threads=cores)
        times.append(dt)
        flops = fl
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    sample = ("plain C++ oracle, one std::thread per core: the layer step on a %d-token slice of X and dY "
              "with all of W, %.1f GFLOP per step" % (ORACLE_TOKENS, flops / 1e9))
    line = {
        "impl": "reference", "metric": "NVFP4 linear fwd+bwd TFLOPS", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "sample_tokens": ORACLE_TOKENS},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "threads": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, rank, world, local):
    import numpy as np
    import torch

    from nvfp4_bit_numerics_gb300 import binding as B
    from nvfp4_bit_numerics_gb300 import build as nbuild
    from nvfp4_bit_numerics_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    nbuild.build()
    B.load_library()

    # each rank draws its own token shard (weak scaling)
    x_h, w_h, dy_h = workloads.mlp_up(seed=SEED + 1000 * rank)
    x, w, dy = x_h.to(dev), w_h.to(dev), dy_h.to(dev)
    ws = B.linear_workspace(M, K, N, device=dev)
    v = B.nvfp4_linear_get_views(ws, M, K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(marks=None):
        # the launches of nvfp4_linear_fwd / nvfp4_linear_bwd, issued through
        # the public primitives so that events can bracket each part
        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        mark(0)
        B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_ROUND_RNE, rht=True, seed=SEED,
                         out=v["xq"], out_t=v["xtq"])
        mark(1)
        B.nvfp4_quantize(w, B.NVFP4_Q_2D, out=v["wq"], out_t=v["wtq"])
        mark(2)
        B.nvfp4_gemm(v["xq"], v["wq"], out=y)
        mark(3)
        B.nvfp4_quantize(dy, B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_ROUND_SR, rht=True, seed=SEED, sr_stream=0,
                         sr_stream_t=1, out=v["dyq"], out_t=v["dytq"])
        mark(4)
        B.nvfp4_gemm2(v["dyq"], v["wtq"], v["dytq"], v["xtq"], out0=dx, out1=dw)  # Dgrad + Wgrad, one launch
        mark(5)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    def api_step():
        # the layer step as a user runs it: nvfp4_linear_fwd (which quantizes W
        # on the library's side stream while X is quantized) + nvfp4_linear_bwd
        B.nvfp4_linear_fwd(x, w, SEED, ws, y=y, stream=stream)
        B.nvfp4_linear_bwd(dy, K, SEED, ws, dx=dx, dw=dw, stream=stream)

    for _ in range(args.warmup):
        api_step()
        step()
    if B.nvfp4_get_status() != B.NVFP4_OK:
        raise RuntimeError("device status after warm-up")

    marks = [[ev() for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.3)
    launches0 = B.nvfp4_kernel_launch_count()
    t_start, t_end = ev(), ev()
    barrier()
    t_start.record(stream)
    for i in range(args.steps):
        api_step()
    t_end.record(stream)
    barrier()
    launches = B.nvfp4_kernel_launch_count() - launches0
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    st = B.nvfp4_get_status()
    if st != B.NVFP4_OK:
        raise RuntimeError("device status %d in the timed region" % st)

    # per-part times: a separate pass of the same launches issued one after
    # another through the primitives, with events between the parts
    barrier()
    for i in range(args.steps):
        step(marks[i])
    barrier()
    part = np.array([[marks[i][j].elapsed_time(marks[i][j + 1]) for j in range(5)] for i in range(args.steps)])
    # the step's two GEMM launches: Fprop, and Dgrad + Wgrad in one launch
    gemm_ms = float(np.mean(part[:, 2] + part[:, 4]))
    ms_per_step = reduce_max_over_ranks(total_ms / args.steps, world, dev)

    # e2e: the public layer API on pinned host buffers.  Every step uploads
    # its X, W, dY from pinned host memory and downloads Y, dX, dW, all inside
    # the timed region; the copies of neighbouring steps run on their own
    # streams, overlapping the current step's kernels (double-buffered device
    # inputs and outputs, one workspace on the compute stream).
    xp, wp, dyp = (t.pin_memory() for t in (x_h, w_h, dy_h))
    outs_h = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory(),
              torch.empty((M, K), dtype=torch.bfloat16).pin_memory(),
              torch.empty((N, K), dtype=torch.bfloat16).pin_memory()]
    ins_d = [[x, w, dy], [torch.empty_like(x), torch.empty_like(w), torch.empty_like(dy)]]
    outs_d = [[y, dx, dw], [torch.empty_like(y), torch.empty_like(dx), torch.empty_like(dw)]]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])  # step i-2 finished reading these inputs
            for d, h in zip(ins_d[b], (xp, wp, dyp)):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])  # step i-2's outputs have left the device
        xb, wb, dyb = ins_d[b]
        yb, dxb, dwb = outs_d[b]
        B.nvfp4_linear_fwd(xb, wb, SEED, ws, y=yb, stream=stream)
        B.nvfp4_linear_bwd(dyb, K, SEED, ws, dx=dxb, dw=dwb, stream=stream)
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            for h, d in zip(outs_h, outs_d[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    barrier()
    e0, e1 = ev(), ev()
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)
    barrier()
    e2e_ms = reduce_max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    if B.nvfp4_get_status() != B.NVFP4_OK:
        raise RuntimeError("device status in the e2e region")
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    h2d = sum(t.numel() * t.element_size() for t in (x_h, w_h, dy_h))

    # library GEMMs of the same three shapes, for context (after the timed
    # regions; the quantized operands are the last step's workspace)
    dyt, xt = dy.t().contiguous(), x.t().contiguous()
    context = library_gemms({
        "fprop": (x, w, y, v["xq"], v["wq"]),
        "dgrad": (dy, w.t().contiguous(), dx, v["dyq"], v["wtq"]),
        "wgrad": (dyt, xt, dw, v["dytq"], v["xtq"]),
    }, stream)
    del dyt, xt

    if rank != 0:
        return 0
    hbm, bf16, src = measured_peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    achieved = 3 * FLOPS_PER_GEMM / (gemm_ms * 1e-3) / 1e12  # the three GEMMs' flops over their two launches
    # quantize GB/s of the dY pass (algorithmic: two reads of dY for amax and
    # quantize, two NVFP4 outputs of 0.5625 B per element each)
    dy_elems = M * N
    q_bytes = dy_elems * (2 + 2 + 2 * 0.5625)
    q_ms = float(np.mean(part[:, 3]))
    cpu = cpu_baseline_record(*(workloads.bf16_to_f32_numpy(t) for t in (x_h, w_h, dy_h)))
    value = whole_job_tflops(ms_per_step, world)
    line = {
        "metric": "NVFP4 linear fwd+bwd TFLOPS", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "parallelism": "dp%d" % world,
                   "l2": "inputs larger than L2 (X+W+dY = 629 MB read per step)",
                   "pct_fp4_peak": 100.0 * value / world / fp4_peak},
        "parts_ms": {"quant_x": float(np.mean(part[:, 0])), "quant_w2d": float(np.mean(part[:, 1])),
                     "gemm_fprop": float(np.mean(part[:, 2])), "quant_dy": q_ms,
                     "gemm_dgrad_wgrad": float(np.mean(part[:, 4])),
                     "note": "a separate pass issuing the step's launches one after another through the "
                             "primitives (Dgrad and Wgrad in one nvfp4_gemm2 launch, as nvfp4_linear_bwd runs "
                             "them); the timed step (nvfp4_linear_fwd + nvfp4_linear_bwd) overlaps quant_x with "
                             "quant_w2d"},
        "quantize_gbs": {"dy_fused_sr_rht": q_bytes / (q_ms * 1e-3) / 1e9, "unit": "GB/s",
                         "bytes": "2 reads of BF16 dY (amax, quantize) + 2 x 0.5625 B/elem written"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp4_peak, "traffic": traffic_record(),
                     "kernel": "nvfp4_gemm_pair_kernel, the step's two launches (Fprop; Dgrad + Wgrad): "
                               "3 x 2MNK flops over their summed time, DRAM traffic averaged per launch",
                     "peak_source": "%s bf16 burst %.1f TFLOP/s x %.0f (nominal FP4:BF16)" % (src, bf16,
                                                                                         FP4_OVER_BF16)},
        "e2e": {"value": whole_job_tflops(e2e_ms, world), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "api": "nvfp4_linear_fwd + nvfp4_linear_bwd",
                "overlap": "uploads of step i+1 and downloads of step i-1 overlap step i's kernels"},
        "gpu_launches": int(launches),
        "context": dict(context, note="library GEMMs of the same shapes for comparison; not this "
                                      "library's path (out = A B^T: Fprop X W^T, Dgrad dY W, Wgrad dY^T X)"),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_quant_sweep(stream, dev):
    """The quantize-only sweep (two BF16 tensors, 8192x5120 and 8192x20480,
    N(0,1) with 0.1 % heavy-tailed entries): each amax pass and each
    quantize mode alone -- the tensor amax already computed, as in the layer
    step -- with the L2 flushed before every launch.  Algorithmic bytes: an
    amax pass reads 2 B per element; a quantize reads 2 B and writes 0.5 B of
    codes and 1/16 B of scales per element for each output."""
    import torch

    from nvfp4_bit_numerics_gb300 import binding as B, workloads

    hbm_peak, _, src = measured_peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    seed = 2024
    for x_h in workloads.quant_sweep():
        x = x_h.to(dev)
        rows, cols = x.shape
        n = rows * cols
        amax = torch.zeros(3, dtype=torch.float32, device=dev)
        out = B.empty_qtensor(rows, cols, device=dev)
        out_t = B.empty_qtensor(cols, rows, device=dev)
        B.nvfp4_amax(x, 7, rht_seed=seed, out=amax)  # plain, Hadamard along rows, Hadamard along columns
        torch.cuda.synchronize()

        def q(kind, rounding, rht, a_row, a_t=None):
            """A quantize call whose outputs' amaxes (slots of `amax`) are set
            before it is timed."""
            def f():
                first = out_t if kind == B.NVFP4_Q_TRANSPOSE else out
                B.nvfp4_quantize(x, kind, rounding, rht=rht, seed=seed, sr_stream=0, sr_stream_t=1,
                                 compute_amax=False, out=first,
                                 out_t=out_t if kind in (B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, B.NVFP4_Q_2D) else None,
                                 stream=stream)
            f.amax_slots = (a_row, a_t)
            return f

        RNE, SR = B.NVFP4_ROUND_RNE, B.NVFP4_ROUND_SR
        modes = [
            ("amax_plain", lambda: B.nvfp4_amax(x, B.NVFP4_AMAX_PLAIN, out=amax, stream=stream), 2.0),
            ("amax_plain_and_rht_cols", lambda: B.nvfp4_amax(x, B.NVFP4_AMAX_PLAIN | B.NVFP4_AMAX_RHT_COLS,
                                                             rht_seed=seed, out=amax, stream=stream), 2.0),
            ("rowwise_1x16_rne", q(B.NVFP4_Q_ROWWISE, RNE, False, 0), 2.5625),
            ("rowwise_1x16_sr", q(B.NVFP4_Q_ROWWISE, SR, False, 0), 2.5625),
            ("rowwise_1x16_rht_rne", q(B.NVFP4_Q_ROWWISE, RNE, True, 1), 2.5625),
            ("2d_16x16_rne_w_and_wt", q(B.NVFP4_Q_2D, RNE, False, 0), 3.125),
            ("transpose_1x16_rht_rne", q(B.NVFP4_Q_TRANSPOSE, RNE, True, None, 2), 2.5625),
            ("transpose_1x16_rht_sr", q(B.NVFP4_Q_TRANSPOSE, SR, True, None, 2), 2.5625),
            ("fused_rowwise_rne_and_transpose_rht_rne", q(B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, RNE, True, 0, 2), 3.125),
            ("fused_rowwise_sr_and_transpose_rht_sr", q(B.NVFP4_Q_ROWWISE_AND_TRANSPOSE, SR, True, 0, 2), 3.125),
        ]
        for name, fn, bpe in modes:
            a_row, a_t = getattr(fn, "amax_slots", (None, None))
            if a_row is not None:
                out.amax.copy_(amax[a_row:a_row + 1])
            if a_t is not None:
                out_t.amax.copy_(amax[a_t:a_t + 1])
            ms = time_ms_flushed(fn, stream, flush)
            gbs = n * bpe / (ms * 1e-3) / 1e9
            print(json.dumps({"sweep": "quantize", "workload": "%s_%dx%d" % (name, rows, cols), "ms": ms,
                              "value": gbs, "unit": "GB/s", "frac_hbm": gbs / hbm_peak,
                              "peak": hbm_peak, "peak_source": src, "bytes_per_element": bpe}), flush=True)
        if B.nvfp4_get_status() != B.NVFP4_OK:
            raise RuntimeError("device status in the quantize sweep")
        del x, out, out_t


def run_sweep(args, rank, world, local):
    """--sweep: one JSON line per further configured shape (the quantize-only
    sweep; the layer step for the MLP down-projection and the QKV projection;
    the GEMM alone for the M = 16384 shape sweep), with the library GEMMs for
    context."""
    import torch

    from nvfp4_bit_numerics_gb300 import binding as B, build as nbuild, workloads

    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    nbuild.build()
    B.load_library()
    stream = torch.cuda.current_stream(dev)
    fp4_peak = measured_peaks()[1] * FP4_OVER_BF16
    run_quant_sweep(stream, dev)
    for name, gen, (m, k, n) in [("mlp_down", workloads.mlp_down, (8192, 20480, 5120)),
                                 ("qkv", workloads.qkv, (8192, 5120, 7168))]:
        x, w, dy = (t.to(dev) for t in gen())
        ws = B.linear_workspace(m, k, n, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((n, k), dtype=torch.bfloat16, device=dev)

        def api():
            B.nvfp4_linear_fwd(x, w, SEED, ws, y=y, stream=stream)
            B.nvfp4_linear_bwd(dy, k, SEED, ws, dx=dx, dw=dw, stream=stream)

        ms = time_ms(api, stream, reps=args.steps, warm=args.warmup)
        if B.nvfp4_get_status() != B.NVFP4_OK:
            raise RuntimeError("device status in the sweep")
        print(json.dumps({"sweep": "layer", "workload": "%s_%dx%dx%d" % (name, m, k, n), "ms_per_step": ms,
                          "value": 6.0 * m * k * n / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "pct_fp4_peak": 100.0 * 6.0 * m * k * n / (ms * 1e-3) / 1e12 / fp4_peak}), flush=True)
        del x, w, dy, ws, y, dx, dw
    for (k, n) in [(4096, 4096), (5120, 5120), (8192, 8192), (5120, 20480), (20480, 5120)]:
        m = 16384
        x, w, _ = (t.to(dev) for t in workloads.gemm_sweep(k, n))
        qa = B.empty_qtensor(m, k, device=dev)
        qb = B.empty_qtensor(n, k, device=dev)
        B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, B.NVFP4_ROUND_RNE, out=qa)
        B.nvfp4_quantize(w, B.NVFP4_Q_2D, out=qb)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        ms = time_ms(lambda: B.nvfp4_gemm(qa, qb, out=y), stream, reps=args.steps, warm=args.warmup)
        if B.nvfp4_get_status() != B.NVFP4_OK:
            raise RuntimeError("device status in the sweep")
        tf = 2.0 * m * k * n / (ms * 1e-3) / 1e12
        ctx = library_gemms({"gemm": (x, w, y, qa, qb)}, stream)
        print(json.dumps({"sweep": "gemm", "workload": "gemm_%dx%dx%d" % (m, k, n), "ms": ms, "value": tf,
                          "unit": "TFLOP/s", "pct_fp4_peak": 100.0 * tf / fp4_peak,
                          "cublas_bf16_ms": ctx["cublas_bf16_ms"]["gemm"],
                          "cublaslt_nvfp4_ms": ctx["cublaslt_nvfp4_ms"]["gemm"]}), flush=True)
        del x, w, qa, qb, y
    return 0


def time_ms_flushed(fn, stream, flush, reps=5, warm=2):
    """Mean device time of fn() alone on `stream`, the L2 flushed before
    every launch: a write of the first half of `flush` (larger than L2), then
    a read of the second half, so that the write's dirty lines are written
    back before the timed launch rather than during it."""
    import torch

    half = flush.numel() // 2
    for _ in range(warm):
        fn()
    total = 0.0
    for _ in range(reps):
        flush[:half].add_(1)
        flush[half:].max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        total += e0.elapsed_time(e1)
    return total / reps


def run_next(args, rank, world, local):
    """--next: one JSON line per further path built on the same workload:
    (1) the GEMM epilogue's output amax (nvfp4_gemm_amax) against the plain
    GEMM plus a separate amax pass over its output; (2) the output quantized
    in the epilogue (nvfp4_gemm_quant) against the GEMM plus a separate
    quantize; (3) the MXFP4 variant of the layer step; (4) the layer step of
    a layer kept in BF16."""
    import torch

    from nvfp4_bit_numerics_gb300 import binding as B, build as nbuild, workloads

    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    nbuild.build()
    B.load_library()
    stream = torch.cuda.current_stream(dev)
    hbm_peak, bf16_peak, src = measured_peaks()
    fp4_peak = bf16_peak * FP4_OVER_BF16
    x, w, dy = (t.to(dev) for t in workloads.mlp_up())
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    # (1) NEXT-1: the output amax taken in the GEMM epilogue
    nqx = B.empty_qtensor(M, K, device=dev)
    nqw = B.empty_qtensor(N, K, device=dev)
    B.nvfp4_quantize(x, B.NVFP4_Q_ROWWISE, out=nqx)
    B.nvfp4_quantize(w, B.NVFP4_Q_2D, out=nqw)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    amax = torch.zeros(3, dtype=torch.float32, device=dev)
    g_ms = time_ms_flushed(lambda: B.nvfp4_gemm(nqx, nqw, out=y, stream=stream), stream, flush)
    ga_ms = time_ms_flushed(lambda: B.nvfp4_gemm_amax(nqx, nqw, out=y, amax=amax[:1], stream=stream), stream, flush)
    a_ms = time_ms_flushed(lambda: B.nvfp4_amax(y, B.NVFP4_AMAX_PLAIN, out=amax, stream=stream), stream, flush)
    if B.nvfp4_get_status() != B.NVFP4_OK:
        raise RuntimeError("device status in the amax-epilogue measurement")
    print(json.dumps({
        "next": "amax_epilogue", "workload": "fprop_gemm_%dx%dx%d_bf16_out" % (M, K, N),
        "gemm_ms": g_ms, "gemm_amax_ms": ga_ms, "separate_amax_pass_ms": a_ms,
        "saved_ms": g_ms + a_ms - ga_ms, "note": "each launch alone, L2 flushed before it"}), flush=True)

    # NEXT-2: Y quantized for the next layer in the GEMM epilogue (amax of the
    # previous, identical step) against the GEMM plus a separate quantize of Y
    yq = B.empty_qtensor(M, N, device=dev)
    yq.amax.copy_(amax[:1])
    q_ms = time_ms_flushed(lambda: B.nvfp4_quantize(y, B.NVFP4_Q_ROWWISE, compute_amax=False, out=yq,
                                                    stream=stream), stream, flush)
    gq_ms = time_ms_flushed(lambda: B.nvfp4_gemm_quant(nqx, nqw, yq, stream=stream), stream, flush)
    gqy_ms = time_ms_flushed(lambda: B.nvfp4_gemm_quant(nqx, nqw, yq, out=y, stream=stream), stream, flush)
    if B.nvfp4_get_status() != B.NVFP4_OK:
        raise RuntimeError("device status in the quantize-in-epilogue measurement")
    print(json.dumps({
        "next": "quantize_epilogue", "workload": "fprop_gemm_%dx%dx%d_nvfp4_out" % (M, K, N),
        "gemm_bf16_ms": g_ms, "separate_quantize_of_y_ms": q_ms, "gemm_quant_ms": gq_ms,
        "gemm_quant_plus_bf16_ms": gqy_ms, "saved_ms": g_ms + q_ms - gq_ms,
        "note": "each launch alone, L2 flushed before it; gemm_quant writes only the NVFP4 Y"}), flush=True)
    del yq

    # (2) NEXT-3: the MXFP4 layer step
    qx, qxt = B.empty_mx_qtensor(M, K, device=dev), B.empty_mx_qtensor(K, M, device=dev)
    qw, qwt = B.empty_mx_qtensor(N, K, device=dev), B.empty_mx_qtensor(K, N, device=dev)
    qdy, qdyt = B.empty_mx_qtensor(M, N, device=dev), B.empty_mx_qtensor(N, M, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    both = B.NVFP4_Q_ROWWISE_AND_TRANSPOSE
    parts = {
        "quant_x": lambda: B.nvfp4_quantize_mx(x, both, out=qx, out_t=qxt, stream=stream),
        "quant_w": lambda: B.nvfp4_quantize_mx(w, both, out=qw, out_t=qwt, stream=stream),
        "quant_dy": lambda: B.nvfp4_quantize_mx(dy, both, out=qdy, out_t=qdyt, stream=stream),
        "gemm_fprop": lambda: B.nvfp4_gemm(qx, qw, out=y, stream=stream),
        # Dgrad + Wgrad in one launch, as the NVFP4 layer's backward runs them
        "gemm_dgrad_wgrad": lambda: B.nvfp4_gemm2(qdy, qwt, qdyt, qxt, out0=dx, out1=dw, stream=stream),
    }

    def step():
        for f in parts.values():
            f()

    n0 = B.nvfp4_kernel_launch_count()
    step()
    launches = B.nvfp4_kernel_launch_count() - n0
    ms = time_ms(step, stream, reps=args.steps, warm=args.warmup)
    part_ms = {k: time_ms_flushed(f, stream, flush) for k, f in parts.items()}
    if B.nvfp4_get_status() != B.NVFP4_OK:
        raise RuntimeError("device status in the MXFP4 step")
    # NVFP4 GEMM of the same Fprop shape (operands from the NVFP4 quantizers)
    nv_ms = g_ms
    # algorithmic bytes of one fused MXFP4 quantization of an [r, c] tensor:
    # read 2 B, write two outputs of 0.5 B codes + 1/16 B scale words
    qbytes = lambda r, c: r * c * (2.0 + 2 * (0.5 + 1.0 / 16))  # noqa: E731
    dy_gbs = qbytes(M, N) / (part_ms["quant_dy"] * 1e-3) / 1e9
    gemm_tf = FLOPS_PER_GEMM / (part_ms["gemm_fprop"] * 1e-3) / 1e12
    print(json.dumps({
        "next": "mxfp4_layer", "workload": "mxfp4_linear_fwd_bwd_mlp_up_%dx%dx%d" % (M, K, N),
        "ms_per_step": ms, "value": FLOPS_PER_STEP / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
        "gpu_launches_per_step": launches, "parts_ms_l2_flushed": part_ms,
        "roofline_quant_dy": {"bound": "hbm", "achieved": dy_gbs, "peak": hbm_peak, "unit": "GB/s",
                              "frac": dy_gbs / hbm_peak, "peak_source": src},
        "roofline_gemm_fprop": {"bound": "tensor", "achieved": gemm_tf, "peak": fp4_peak, "unit": "TFLOP/s",
                                "frac": gemm_tf / fp4_peak, "peak_source": src + " bf16 x 6 (nominal fp4:bf16)"},
        "nvfp4_gemm_fprop_ms_l2_flushed": nv_ms,
    }), flush=True)
    del qx, qxt, qw, qwt, qdy, qdyt, nqx, nqw

    # (3) NEXT-4: a layer kept in BF16 (cuBLAS GEMMs inside the library)
    def bf16_step():
        B.nvfp4_linear_bf16_fwd(x, w, y=y, stream=stream)
        B.nvfp4_linear_bf16_bwd(dy, x, w, dx=dx, dw=dw, stream=stream)

    bms = time_ms(bf16_step, stream, reps=args.steps, warm=args.warmup)
    btf = FLOPS_PER_STEP / (bms * 1e-3) / 1e12
    print(json.dumps({
        "next": "bf16_layer", "workload": "bf16_linear_fwd_bwd_mlp_up_%dx%dx%d" % (M, K, N),
        "ms_per_step": bms, "value": btf, "unit": "TFLOP/s",
        "roofline": {"bound": "tensor", "achieved": btf, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": btf / bf16_peak, "peak_source": src + " bf16 burst"},
        "gemms": "cuBLAS (cublasGemmEx, BF16, FP32 accumulation)"}), flush=True)
    return 0


def run_profile_once(local):
    """One layer step through the public API on the benchmark's inputs (about
    1.6 GB on the device), for a profiler to capture single launches of it.
    The side stream of nvfp4_linear_fwd is joined before the GEMM, so the
    launch order is X amax, X quantize (or W's two on the side stream first),
    Fprop, dY amax, dY quantize, Dgrad + Wgrad (one launch)."""
    import torch

    from nvfp4_bit_numerics_gb300 import binding as B, build as nbuild, workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    nbuild.build()
    B.load_library()
    x, w, dy = (t.to(dev) for t in workloads.mlp_up())
    ws = B.linear_workspace(M, K, N, device=dev)
    B.nvfp4_linear_fwd(x, w, SEED, ws)
    B.nvfp4_linear_bwd(dy, K, SEED, ws)
    st = B.nvfp4_get_status()
    if st != B.NVFP4_OK:
        raise RuntimeError("device status %d" % st)
    print(json.dumps({"profile_once": WORKLOAD, "launches": int(B.nvfp4_kernel_launch_count())}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line, one line per further configured shape")
    ap.add_argument("--quant-sweep", action="store_true",
                    help="instead of the benchmark line, only the quantize-only sweep of --sweep")
    ap.add_argument("--profile-once", action="store_true",
                    help="for profiler captures: the layer step once (9 kernel launches: X amax, X quantize, "
                         "W amax, W 2D quantize, Fprop GEMM, dY amax, dY quantize, Dgrad GEMM, Wgrad GEMM) "
                         "on the benchmark's inputs, nothing else timed or launched after it")
    ap.add_argument("--next", action="store_true",
                    help="instead of the benchmark line, the further paths: GEMM-epilogue amax, the MXFP4 "
                         "layer step, a BF16 layer step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gpu":
        args.warmup = 3
    rank, world, local = dist_info()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.profile_once:
        return run_profile_once(local)
    if args.sweep:
        return run_sweep(args, rank, world, local)
    if args.next:
        return run_next(args, rank, world, local)
    if args.quant_sweep:
        if rank == 0:
            import torch

            from nvfp4_bit_numerics_gb300 import binding as B, build as nbuild

            dev = torch.device("cuda", local)
            nbuild.build()
            B.load_library()
            run_quant_sweep(torch.cuda.current_stream(dev), dev)
        return 0
    return run_gpu(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
