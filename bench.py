#!/usr/bin/env python
"""Benchmark of the LatentMoE layer forward pass: tokens/s per layer and roofline fraction.

Headline workload: the full Kimi K3 layer at prefill, the largest layer that fits one GPU (T=8192,
d=7168, l=3584, h=3072, E=896, k=16, N_s=2, MXFP4 routed experts, skewed router bias).  With one
GPU the same JSON line also carries a record for each other full-size workload: the K3-width bf16
prefill layer (E=128), K3 decode (T=32, MXFP4), the milder-skew MXFP4 prefill and the
routing/dispatch stress test (T=65536).  Synthetic seeded inputs and random-init weights are
resident in HBM; one step is one full forward pass; L2 is flushed (512 MiB write, untimed) before
every timed step.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload NAME] [--no-sub]

Under torchrun each rank runs an independent replica of the headline workload on its own GPU (the
layer's tokens are independent: no collective), timed between barriers; the slowest rank sets
the time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LatentMoE layer tokens/s; % of HBM (decode) / tensor (prefill) roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Dense FP4 : BF16 tensor rate by the datasheet (13.5 vs 2.25 PFLOP/s), used only when the MMA
# microbenchmark cannot run.
NOMINAL_FP4_RATIO = 6.0
HEADLINE = "k3_mxfp4_prefill_skew"
SUB_WORKLOADS = ("k3w_e128_bf16_prefill", "k3_mxfp4_decode", "k3_mxfp4_prefill_mild", "routing_dispatch_t65536")
# the same MXFP4 layers in K3's quantisation-aware numerics (MXFP8 activations, kind::mxf8f6f4)
MXFP8_SUB_WORKLOADS = ("k3_mxfp4_prefill_skew", "k3_mxfp4_decode")
NOMINAL_FP8_RATIO = 2.0
# token rows of the oracle's CPU baseline per workload (about 5-20 s of host work each: an MXFP4
# row decodes up to 16 experts of 6144 x 3584 + 3584 x 3072 values)
CPU_SAMPLE = {"k3_mxfp4_prefill_skew": 8, "k3w_e128_bf16_prefill": 8, "k3_mxfp4_decode": 4,
              "k3_mxfp4_prefill_mild": 4, "routing_dispatch_t65536": 64, "tiny_f32": 64}
ROUTED = ("routed_gate_up_glu", "routed_down")

# DRAM bytes per launch of the dominant kernel from one ncu capture, valid only while the kernel
# source is unchanged (sha256 of the file it lives in).  Filled from the committed profile.
# k3w_e128_bf16_prefill: an ncu capture of the same kernel on the 32-expert, 1024-token workload
# (k3w_e32_bf16_t1024) read 1.543810 GB and wrote 0.095298 GB; experts, rows and weight bytes all
# scale by 4 to the 128-expert, 4096-token workload.
TRAFFIC = {
    "k3w_e128_bf16_prefill": {
        "routed_gate_up_glu": {"bytes_per_launch": 4 * (1.543810e9 + 0.095298e9),
                               "src": "sparse_moe_layer_sigmoid_gb300/csrc/gemm_pair_swap.cu",
                               "sha256": "01bb6ec6eee881fa93642a6f02e244917e72cc9c4e61ae2398eb9c2ab6b281c9"},
    },
}
# Block-scaled kernels: DRAM bytes over algorithmic bytes (read: touched experts' E2M1 + E8M0
# bytes and the activation records read; write: records or fp16 rows written) from one ncu
# capture of a smaller case of the same kernel; a full launch's traffic is those ratios times its
# own algorithmic bytes (reads and writes each grow with experts touched and rows processed).
TRAFFIC_RATIOS = {
    # prefill tiles: k3_mxfp4_prefill_e32_t1024 (32 experts, 16384 rows): read 468150528 B of
    # 467927040 B, write 69632768 B of 80216064 B
    ("mxfp4_prefill", "routed_gate_up_glu"): {"read": 468150528 / 467927040, "write": 69632768 / 80216064,
                                              "src": "sparse_moe_layer_sigmoid_gb300/csrc/gemm_mx.cu",
                                              "sha256": "deb4f5de054232618e992038625d1a4be0f2f67fe858af5c8be67f51e92ae7c5"},
    # decode units: k3_mxfp4_decode_e128_t8 (85 experts, 128 rows): read 995229184 B of 995076096 B,
    # write 3851008 B of 626688 B (dirty lines of the untimed L2 flush written back meanwhile)
    ("mxfp4_decode", "routed_gate_up_glu"): {"read": 995229184 / 995076096, "write": 3851008 / 626688,
                                             "src": "sparse_moe_layer_sigmoid_gb300/csrc/gemm_mx.cu",
                                             "sha256": "deb4f5de054232618e992038625d1a4be0f2f67fe858af5c8be67f51e92ae7c5"},
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x, dist, device):
    """Largest ``x`` over all ranks: the slowest replica sets the job's step time."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, ms):
    """Whole-job throughput: every replica processes ``tokens_per_rank`` tokens per step."""
    return world * tokens_per_rank / (ms * 1e-3)


def rank_env():
    """(world, rank, local rank) from the launcher's environment (1, 0, 0 without one)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def expert_weight_bytes(cfg, rows, cols):
    """Stored bytes of one routed weight matrix [rows][cols] (MXFP4: E2M1 + one E8M0 per 32)."""
    if cfg.routed_w == "mxfp4":
        return rows * cols // 2 + rows * cols // 32
    return rows * cols * (4 if cfg.routed_w == "f32" else 2)


def expert_record_bytes(width):
    """Bytes of one three-term MXFP4 activation record of ``width`` values (block-scaled path)."""
    return 3 * width // 2 + 3 * width // 32


def traffic_alg_bytes(cfg, stage, experts_touched):
    """Algorithmic (read, write) bytes of one launch of a block-scaled routed stage."""
    l, h, rows = cfg.latent, cfg.hidden, cfg.tokens * cfg.top_k
    if stage == "routed_gate_up_glu":
        return (experts_touched * expert_weight_bytes(cfg, 2 * h, l) + rows * expert_record_bytes(l),
                rows * expert_record_bytes(h))
    return (experts_touched * expert_weight_bytes(cfg, l, h) + rows * expert_record_bytes(h), rows * 2 * l)


def stage_work(cfg, experts_touched, mx=None):
    """Algorithmic work of each stage: ('tensor', FLOPs) or ('hbm', bytes) or ('alu', FLOPs).

    Decode-shaped batches (T*k <= 32*E) are bound by streaming the touched experts' weights: their
    routed stages count those bytes plus the activations read and written.  ``mx``: MXFP4 experts
    on the block-scaled path (activations travel as three-term records); default: MXFP4 weights."""
    T, d, l, h, E, k = cfg.tokens, cfg.d, cfg.latent, cfg.hidden, cfg.experts, cfg.top_k
    ns, hs = cfg.n_shared, cfg.shared_hidden
    ab = 4 if cfg.act == "f32" else 2
    rows = T * k
    if mx is None:
        mx = cfg.routed_w == "mxfp4"
    mx = mx and not cfg.identity_experts
    zrow = expert_record_bytes(l) if mx else ab * l          # a gathered row of z
    arow = expert_record_bytes(h) if mx else ab * h          # a routed GLU activation row
    w = {
        # bf16 activations: tensor cores (over 3 bf16 terms of W_r); fp32: CUDA-core FMA
        "router_logits": ("tensor" if cfg.act == "bf16" else "alu", 2.0 * T * E * d),
        "topk": ("hbm", 4.0 * T * E + 8.0 * rows),
        "dispatch": ("hbm", 3 * 4.0 * rows),
        "w_down": ("tensor", 2.0 * T * d * l),
        "scatter_rows": ("hbm", float(ab * T * l + rows * zrow)),
        "combine_rmsnorm": ("hbm", float(ab) * (rows * l + T * l)),
    }
    if not cfg.identity_experts and rows <= 32 * E:
        w["routed_gate_up_glu"] = ("hbm", float(experts_touched * expert_weight_bytes(cfg, 2 * h, l)
                                                + rows * (zrow + arow)))
        w["routed_down"] = ("hbm", float(experts_touched * expert_weight_bytes(cfg, l, h) + rows * (arow + ab * l)))
    elif not cfg.identity_experts:
        w["routed_gate_up_glu"] = ("tensor", 2.0 * rows * l * 2 * h)
        w["routed_down"] = ("tensor", 2.0 * rows * h * l)
    if not cfg.identity_experts:
        w["shared_gate_up_glu"] = ("tensor", 2.0 * T * d * 2 * ns * hs)
        w["final_gemm"] = ("tensor", 2.0 * T * (ns * hs + l) * d)
    return w


def tensor_peak(stage, mx, peaks):
    """(peak TFLOP/s, name) a tensor stage is measured against: the routed stages of the
    block-scaled path run E2M1 x E2M1 MMAs (the FP4 peak; mx == "fp8": E2M1 x E4M3 on
    kind::mxf8f6f4, the FP8 peak), everything else bf16 MMAs."""
    if mx and stage in ROUTED:
        return (peaks["fp8_tflops"], "fp8") if mx == "fp8" else (peaks["fp4_tflops"], "fp4")
    return peaks["bf16_tflops"], "bf16"


def layer_roofline_ms(work, mx, peaks):
    """The layer's roofline time: every stage at its own bound (FLOPs at the tensor peak of the
    MMA kind that runs it, bytes at the HBM bandwidth), summed."""
    t = 0.0
    for stage, (kind, amount) in work.items():
        if kind == "tensor":
            t += amount / (tensor_peak(stage, mx, peaks)[0] * 1e12)
        elif kind == "hbm":
            t += amount / (peaks["hbm_gbs"] * 1e9)
        else:
            t += amount / (peaks["alu_tflops"] * 1e12)
    return 1e3 * t


def file_sha(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background; only samples time-stamped inside
    the timed region (mark_start/mark_stop) are kept."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.t0 = self.t1 = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_id), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.p = None

    def wait_first_sample(self, timeout=10.0):
        t = time.time()
        while self.p is not None and time.time() - t < timeout:
            if os.path.getsize(self.out.name) > 0:
                return
            time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()
        time.sleep(0.2)  # let the sampler flush the samples of the last interval

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.out.flush()
        self.out.seek(0)
        import datetime
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if self.t0 is not None and not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                    continue
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def blas_threads():
    """Threads numpy's BLAS runs with (read from the loaded OpenBLAS), else the CPU count."""
    try:
        with open("/proc/self/maps") as f:
            libs = {ln.split()[-1] for ln in f if "openblas" in ln.lower() and ln.rstrip().endswith(".so")}
        for path in libs:
            lib = ctypes.CDLL(path)
            for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                         "openblas_get_num_threads", "scipy_openblas_get_num_threads"):
                fn = getattr(lib, name, None)
                if fn is not None:
                    return int(fn())
    except OSError:
        pass
    return os.cpu_count()


def oracle_sample(cfg, host, n_tokens, seed):
    """Seconds the oracle takes on ``n_tokens`` seeded token rows of the workload (host cores).

    ``host`` is the host copy of the inputs (made once, outside the timing)."""
    import oracle
    from sparse_moe_layer_sigmoid_gb300 import inputs

    rows = inputs.sample_tokens(cfg.tokens, n_tokens, seed)
    t0 = time.perf_counter()
    oracle.layer_forward(host, cfg, tokens=rows)
    return time.perf_counter() - t0


def run_reference(args, cfg, rank, world):
    """Reference arm: the fp64 oracle, timed as it stands on this machine's host cores."""
    if rank != 0:
        return
    import torch

    from sparse_moe_layer_sigmoid_gb300 import inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    host = inputs.host_inputs(inputs.make_inputs(cfg, dev), lazy_experts=True)
    per_step = 1
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_sample(cfg, host, per_step, cfg.seed + 17 * i)
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = per_step / (ms / 1e3)
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} seeded token row(s) of the workload per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(cfg, args):
    return {"workload": cfg.name, "tokens": cfg.tokens, "d": cfg.d, "latent": cfg.latent, "hidden": cfg.hidden,
            "experts": cfg.experts, "top_k": cfg.top_k, "n_shared": cfg.n_shared,
            "shared_hidden": cfg.shared_hidden, "routed_w": cfg.routed_w, "bias": cfg.bias, "seed": cfg.seed,
            "global_batch": cfg.tokens * args.gpus, "parallelism": f"replicas x{args.gpus}",
            "l2": "flushed before every timed step (512 MiB write, untimed)"}


def measured_peaks(binding, device, src):
    """Roofline denominators: HBM and bf16 from MEASURED_PEAKS.json (else the fallback); the FP4
    tensor peak as the measured bf16 peak times the nominal dense FP4 / bf16 ratio (13.5 / 2.25 =
    6).  The rates of back-to-back kind::mxf4 and kind::f16 CTA-pair MMAs from the library's
    microbenchmark are reported beside it: kind::mxf4 reaches about 4x kind::f16 on this part, so
    the reachable block-scaled instruction rate sits below the nominal FP4 peak."""
    peaks, how = src
    out = {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
           "bf16_tflops_sustained": peaks.get("bf16_tflops_sustained"),
           "source": f"{how} (MEASURED_PEAKS.json)" if how == "measured" else "fallback"}
    props = __import__("torch").cuda.get_device_properties(device)
    clock = peaks.get("sm_max_mhz", 2070.0)
    out["alu_tflops"] = props.multi_processor_count * 128 * 2 * clock * 1e6 / 1e12
    try:
        f16 = binding.mma_peak_tflops("f16")
        fp4 = binding.mma_peak_tflops("mxf4")
        out["mma_f16_tflops"], out["mma_mxf4_tflops"] = f16, fp4
        out["mma_mxf4_over_f16"] = fp4 / f16
    except Exception as exc:  # noqa: BLE001 - reported in the line
        out["mma_rate_error"] = str(exc)
    out["fp4_over_bf16"] = NOMINAL_FP4_RATIO
    out["fp4_source"] = (f"{out['source']} bf16_tflops (burst) x nominal dense FP4/bf16 ratio "
                         f"{NOMINAL_FP4_RATIO:g} (13.5 / 2.25 PFLOP/s)")
    out["fp4_tflops"] = out["bf16_tflops"] * out["fp4_over_bf16"]
    out["fp8_tflops"] = out["bf16_tflops"] * NOMINAL_FP8_RATIO
    out["fp8_source"] = (f"{out['source']} bf16_tflops (burst) x nominal dense FP8/bf16 ratio "
                         f"{NOMINAL_FP8_RATIO:g} (4.5 / 2.25 PFLOP/s)")
    return out


def measure_workload(cfg, args, peaks, world, rank, dist, dev, flags, with_cpu):
    """One workload: warm-up, timed steps (device events), stage times, end-to-end through the
    host-memory entry point, roofline figures and (rank 0) the oracle's CPU baseline."""
    import torch

    from sparse_moe_layer_sigmoid_gb300 import binding, inputs
    from sparse_moe_layer_sigmoid_gb300.binding import LatentMoE

    inp = inputs.make_inputs(cfg, dev)
    layer = LatentMoE(cfg, flags=flags)
    mx = cfg.routed_w == "mxfp4" and not (flags & (binding.LMOE_FLAG_MXFP4_DEQUANT | binding.LMOE_FLAG_SINGLE_CTA_GEMM))
    f8 = mx and bool(flags & binding.LMOE_FLAG_MXFP8_ACT)
    mxk = ("fp8" if f8 else "fp4") if mx else None  # the MMA kind of the routed stages
    x = inp["x"]
    y = torch.empty((cfg.tokens, layer.out_width), dtype=x.dtype, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else dev.index
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    for _ in range(args.warmup):
        flush.zero_()
        layer.forward(x, inp, y)
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError(f"{cfg.name}: layer reported an error status during warm-up")
    if clocks:
        clocks.wait_first_sample()

    r = layer.route(x, inp)
    stats = layer.routing_stats()
    counts = (r["offsets"][1:] - r["offsets"][:-1]).cpu()
    route_stats = {"rows": int(counts.sum()), "experts_touched": int((counts > 0).sum()),
                   "load_max_over_mean": float(counts.max()) / max(1e-9, float(counts.float().mean())),
                   "refined_tokens": stats["refined_tokens"], "near_ties": stats["near_ties"],
                   "near_tie_rule": "exact k-th / (k+1)-th key gap below 1e-6, counted on the GPU"}
    del r

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    step_ms, stages, launches = [], {}, 0
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    for _ in range(args.steps):
        flush.zero_()
        ev0.record(stream)
        layer.forward(x, inp, y)
        ev1.record(stream)
        launches += layer.last_launch_count()
        ev1.synchronize()
        step_ms.append(ev0.elapsed_time(ev1))
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_stop()
    if dist:
        dist.barrier()
    # per-stage device times from separate steps with an event between stages (the library then
    # runs every stage on the caller's stream, one after another, so each stage is timed alone)
    layer.enable_stage_timing()
    for _ in range(max(3, min(args.steps, 10))):
        flush.zero_()
        layer.forward(x, inp, y)
        for k_, v in layer.stage_times_ms().items():
            stages.setdefault(k_, []).append(v)
    layer.disable_stage_timing()
    serial_ms = sum(sum(v) / len(v) for v in stages.values())
    graph_rec = graph_steps(layer, x, inp, y, flush, stream, args) if cfg.tokens <= GRAPH_MAX_TOKENS else None
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dist, dev)
    if layer.status() != 0:
        raise RuntimeError(f"{cfg.name}: layer reported an error status during the timed steps")

    # end to end through the public host-memory entry point (copies inside the timed region)
    x_host = x.cpu().pin_memory()
    y_host = torch.empty((cfg.tokens, layer.out_width), dtype=x.dtype, pin_memory=True)
    for _ in range(2):
        layer.forward_host(x_host, inp, y_host)
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.forward_host(x_host, inp, y_host)
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    e2e = max_over_ranks(sum(e2e_ms) / len(e2e_ms), dist, dev)
    elem = x.element_size()

    work = stage_work(cfg, route_stats["experts_touched"], mx)
    st_ms = {k_: sum(v) / len(v) for k_, v in stages.items()}
    dom = max((k_ for k_ in work if k_ in st_ms), key=st_ms.get)
    kind, amount = work[dom]
    roof = {"bound": kind, "kernel": dom}
    if kind == "tensor":
        peak, pname = tensor_peak(dom, mxk, peaks)
        achieved = amount / (st_ms[dom] * 1e-3) / 1e12
        roof.update({"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"{pname}: " + (peaks["fp4_source"] if pname == "fp4" else
                                                    peaks["fp8_source"] if pname == "fp8" else
                                                    peaks["source"] + " bf16_tflops (burst)")})
        if pname == "fp4":  # three E2M1 activation terms: three MMAs per algorithmic product
            roof["mma_work_per_flop"] = 3
            roof["mma_pipe_frac_of_nominal"] = 3 * achieved / peak
            if peaks.get("mma_mxf4_tflops"):  # against the kind::mxf4 rate this GPU reaches
                roof["mma_pipe_frac_of_mxf4_rate"] = 3 * achieved / peaks["mma_mxf4_tflops"]
    elif kind == "alu":
        achieved = amount / (st_ms[dom] * 1e-3) / 1e12
        roof.update({"achieved": achieved, "peak": peaks["alu_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["alu_tflops"],
                     "peak_source": "derived: SMs x 128 fp32 lanes x 2 x sm_max_mhz"})
    else:
        achieved = amount / (st_ms[dom] * 1e-3) / 1e9
        roof.update({"achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " hbm_gbs"})
    tr = TRAFFIC.get(cfg.name, {}).get(dom)
    roof["traffic"] = None
    if tr and tr["bytes_per_launch"] and tr["sha256"] == file_sha(tr["src"]):
        roof["traffic"] = tr["bytes_per_launch"]
    rt = (TRAFFIC_RATIOS.get(("mxfp4_decode" if work[dom][0] == "hbm" else "mxfp4_prefill", dom))
          if mx and not f8 else None)
    if rt and rt["sha256"] == file_sha(rt["src"]):
        rd, wr = traffic_alg_bytes(cfg, dom, route_stats["experts_touched"])
        roof["traffic"] = rt["read"] * rd + rt["write"] * wr
        roof["traffic_rule"] = ("ncu DRAM bytes / algorithmic bytes of a smaller capture of this kernel "
                                "x this launch's algorithmic reads and writes")
    total_flops = sum(a for kd, a in work.values() if kd in ("tensor", "alu"))
    total_bytes = sum(a for kd, a in work.values() if kd == "hbm")
    roof_ms = layer_roofline_ms(work, mxk, peaks)
    layer_rec = {"flops": total_flops, "hbm_bytes_counted": total_bytes,
                 "achieved_tflops": total_flops / (ms * 1e-3) / 1e12, "roofline_ms": roof_ms,
                 "roofline_frac": roof_ms / ms,
                 "roofline_rule": "each stage at its own bound: FLOPs at the peak of its MMA kind, bytes at HBM",
                 "stages_ms": st_ms, "stages_serial_sum_ms": serial_ms,
                 "stages_rule": ("stage times from separate steps run stage after stage on one stream; the "
                                 "timed steps overlap W_down and the shared GLU with the routing chain")}
    if f8 and work["routed_gate_up_glu"][0] == "tensor":
        routed = work["routed_gate_up_glu"][1] + work["routed_down"][1]
        dense = total_flops - routed
        r8 = 1e3 * (routed / (peaks["fp8_tflops"] * 1e12) + dense / (peaks["bf16_tflops"] * 1e12))
        layer_rec.update({"fp8_aware_roofline_ms": r8, "fp8_aware_frac": r8 / ms,
                          "fp8_aware_rule": "routed FLOPs at the FP8 peak (kind::mxf8f6f4) + the rest at the bf16 peak"})
    elif mx and work["routed_gate_up_glu"][0] == "tensor":
        routed = work["routed_gate_up_glu"][1] + work["routed_down"][1]
        dense = total_flops - routed
        fp4_roof = 1e3 * (routed / (peaks["fp4_tflops"] * 1e12) + dense / (peaks["bf16_tflops"] * 1e12))
        three = 1e3 * (3 * routed / (peaks["fp4_tflops"] * 1e12) + dense / (peaks["bf16_tflops"] * 1e12))
        layer_rec.update({"fp4_aware_roofline_ms": fp4_roof, "fp4_aware_frac": fp4_roof / ms,
                          "three_term_ceiling_frac": fp4_roof / three,
                          "fp4_aware_rule": "routed FLOPs at the FP4 peak + the rest at the bf16 peak"})
        if peaks.get("mma_mxf4_tflops"):  # the same with the kind::mxf4 rate this GPU reaches
            rate_roof = 1e3 * (routed / (peaks["mma_mxf4_tflops"] * 1e12) + dense / (peaks["bf16_tflops"] * 1e12))
            rate_three = 1e3 * (3 * routed / (peaks["mma_mxf4_tflops"] * 1e12)
                                + dense / (peaks["bf16_tflops"] * 1e12))
            layer_rec.update({"mxf4_rate_frac": rate_roof / ms, "mxf4_rate_three_term_ceiling_frac": rate_roof / rate_three})
    elif work.get("routed_gate_up_glu", ("", 0))[0] == "hbm":
        layer_rec.update({"achieved_gbs": total_bytes / (ms * 1e-3) / 1e9,
                          "hbm_frac": total_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]})
    else:
        layer_rec["frac_of_bf16_peak"] = total_flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]
    if cfg.identity_experts:
        layer_rec["achieved_gbs"] = total_bytes / (ms * 1e-3) / 1e9
    dtype = ("e2m1 x e4m3 experts (MXFP8 activations), bf16 dense" if f8 else
             "e2m1 x e2m1 experts (three-term MXFP4 activations), bf16 dense" if mx else
             "fp16 (MXFP4 experts decoded), bf16 dense" if cfg.routed_w == "mxfp4" else cfg.act)
    rec = {"value": job_tokens_per_s(world, cfg.tokens, ms), "unit": UNIT, "ms_per_step": ms, "dtype": dtype,
           "config": workload_config(cfg, args), "roofline": roof, "layer": layer_rec,
           "e2e": {"value": job_tokens_per_s(world, cfg.tokens, e2e), "unit": UNIT,
                   "h2d_bytes_per_step": cfg.tokens * cfg.d * elem,
                   "d2h_bytes_per_step": cfg.tokens * layer.out_width * elem},
           "gpu_launches": launches, "routing": route_stats, "clocks": clk}
    if graph_rec:
        graph_rec["value"] = job_tokens_per_s(world, cfg.tokens, graph_rec["ms_per_step"])
        rec["graph"] = graph_rec
    if f8:
        rec["config"]["activations"] = "mxfp8 (LMOE_FLAG_MXFP8_ACT; compared with the oracle's MXFP8 mode)"
    layer.close()
    y = flush = None
    if with_cpu and rank == 0 and world == 1:
        n = CPU_SAMPLE.get(cfg.name, 8) if args.cpu_sample is None else args.cpu_sample
        if n > 0:
            host = inputs.host_inputs(inp, lazy_experts=True)
            dt = oracle_sample(cfg, host, n, cfg.seed + 99)
            rec["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                                   "sample": f"{n} seeded token rows of the workload, fp64 oracle"}
            del host
    del inp
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


GRAPH_MAX_TOKENS = 256  # decode-sized batches: also time the forward replayed as one CUDA graph


def graph_steps(layer, x, inp, y, flush, stream, args):
    """The whole forward captured once into a CUDA graph (the library's launches, its second
    stream's fork and joins) and replayed: device time per step against the stream-launched
    steps, i.e. what launch gaps cost; plus host time per launch of the two forms."""
    import time

    import torch

    layer.forward(x, inp, y)  # the library's one-time setup (function attributes, occupancy) outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        layer.forward(x, inp, y, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dev_ms, host_graph, host_stream = [], [], []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        ev0.record(stream)
        h0 = time.perf_counter()
        g.replay()
        h1 = time.perf_counter()
        ev1.record(stream)
        ev1.synchronize()
        if it >= args.warmup:
            dev_ms.append(ev0.elapsed_time(ev1))
            host_graph.append((h1 - h0) * 1e3)
    for it in range(args.steps):
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        layer.forward(x, inp, y)
        host_stream.append((time.perf_counter() - h0) * 1e3)
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError("graph replay reported an error status")
    del g
    return {"ms_per_step": sum(dev_ms) / len(dev_ms), "host_ms_per_launch": sum(host_graph) / len(host_graph),
            "host_ms_per_stream_forward": sum(host_stream) / len(host_stream),
            "rule": "device time of a replay of the captured forward (events on the launching stream)"}


EP_WORKLOAD = "k3_mxfp4_prefill_mild"  # routing of the mildly skewed K3 prefill (T=8192, E=896, k=16)
EP_RANKS = 8


def measure_ep(args, dev):
    """Expert-parallel dispatch and combine emulated on one GPU (latentmoe_ep_emulate) at the
    latent width and at the full width: per token the all-to-all carries k rows of l (latent) or
    d (full) values each way.  Reports the rows crossing ranks, payload per token, and the
    device time and HBM rate of pack / exchange / return / combine."""
    import torch

    from sparse_moe_layer_sigmoid_gb300 import binding, configs, inputs

    cfg = configs.CONFIGS[EP_WORKLOAD]
    inp = inputs.make_inputs(cfg, dev)
    layer = binding.LatentMoE(cfg)
    x = inp["x"]
    rows = cfg.tokens * cfg.top_k
    out = {"workload": f"ep_dispatch_combine_{cfg.name}_r{EP_RANKS}", "ranks": EP_RANKS, "tokens": cfg.tokens,
           "experts": cfg.experts, "top_k": cfg.top_k, "rows": rows,
           "rule": ("rank r owns tokens [r T/R, (r+1) T/R) and experts [r E/R, (r+1) E/R); identity experts; "
                    "exchange = one HBM copy of every row per direction on this one GPU")}
    for name, full in (("latent", False), ("full_width", True)):
        width = cfg.d if full else cfg.latent
        dt = x.dtype if full else torch.float16
        send = torch.empty((rows, width), dtype=dt, device=dev)
        recv = torch.empty((rows, width), dtype=dt, device=dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for e in evs:
            e.record()
        times = []
        for it in range(args.warmup + args.steps):
            u, cells = layer.ep_emulate(x, inp, EP_RANKS, full, send=send, recv=recv, events=evs)
            evs[-1].synchronize()
            if it >= args.warmup:
                times.append([evs[i].elapsed_time(evs[i + 1]) for i in range(5)])
        if layer.status() != 0:
            raise RuntimeError("ep emulation reported an error status")
        t = [sum(c) / len(c) for c in zip(*times)]
        cells = cells.cpu()
        cross = int(cells.sum() - cells.diag().sum())
        row_bytes = width * send.element_size()
        out[name] = {"width": width, "row_bytes": row_bytes,
                     "payload_values_per_token": cfg.top_k * width,
                     "payload_bytes_per_token_all_rows": cfg.top_k * row_bytes,
                     "cross_rank_rows": cross, "cross_rank_frac": cross / rows,
                     "payload_bytes_per_token_cross_rank": cross * row_bytes / cfg.tokens,
                     "ms": {"route_and_rows": t[0], "pack": t[1], "exchange": t[2], "return": t[3],
                            "combine": t[4]},
                     "exchange_gbs": 2 * rows * row_bytes / (t[2] * 1e-3) / 1e9}
        del send, recv, u
    out["payload_ratio_full_over_latent"] = (out["full_width"]["payload_bytes_per_token_all_rows"]
                                             / out["latent"]["payload_bytes_per_token_all_rows"])
    layer.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-sub", action="store_true", help="time the headline workload only")
    ap.add_argument("--cpu-sample", type=int, default=None, help="token rows for the oracle CPU baseline")
    ap.add_argument("--single-cta", action="store_true",
                    help="run every tensor-core GEMM on single CTAs (no CTA-pair GEMMs)")
    ap.add_argument("--mxfp8-act", action="store_true",
                    help="MXFP4 experts with MXFP8 activations (kind::mxf8f6f4; K3's QAT numerics)")
    ap.add_argument("--mxfp4-dequant", action="store_true",
                    help="MXFP4 experts through the dequantizing kernels instead of the block-scaled MMA")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch

    from sparse_moe_layer_sigmoid_gb300 import configs

    cfg = configs.CONFIGS[args.workload]
    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, cfg, rank, world)
        if dist:
            dist.destroy_process_group()
        return

    import __graft_entry__
    from sparse_moe_layer_sigmoid_gb300 import binding

    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flags = ((binding.LMOE_FLAG_SINGLE_CTA_GEMM if args.single_cta else 0) |
             (binding.LMOE_FLAG_MXFP4_DEQUANT if args.mxfp4_dequant else 0) |
             (binding.LMOE_FLAG_MXFP8_ACT if args.mxfp8_act else 0))
    peaks = measured_peaks(binding, dev, load_peaks())
    head = measure_workload(cfg, args, peaks, world, rank, dist, dev, flags, with_cpu=True)
    subs = {}
    if world == 1 and not args.no_sub and args.workload == HEADLINE:
        for name in SUB_WORKLOADS:
            subs[name] = measure_workload(configs.CONFIGS[name], args, peaks, world, rank, dist, dev, flags,
                                          with_cpu=True)
        for name in MXFP8_SUB_WORKLOADS:
            subs[name + "_mxfp8act"] = measure_workload(configs.CONFIGS[name], args, peaks, world, rank, dist, dev,
                                                        flags | binding.LMOE_FLAG_MXFP8_ACT, with_cpu=False)
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"], "roofline": head["roofline"], "layer": head["layer"],
            "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "routing": head["routing"],
            "clocks": head["clocks"], "peaks": peaks}
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if "graph" in head:
        line["graph"] = head["graph"]
    if subs:
        line["workloads"] = subs
        line["ep_emulation"] = measure_ep(args, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
