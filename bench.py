#!/usr/bin/env python
"""Benchmark of the LatentMoE layer forward pass: tokens/s per layer and roofline fraction.

Default workload: the K3-width bf16 prefill layer (T=4096, d=7168, l=3584, h=3072, E=128,
k=16, N_s=2), synthetic seeded inputs and random-init weights resident in HBM.  One step is
one full forward pass (router, top-k, dispatch, W_down, experts, combine + RMSNorm, shared
experts, W_up).  L2 is flushed (512 MiB write, untimed) before every timed step.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun each rank runs an independent replica on its own GPU (the layer's tokens
are independent: no collective), timed between barriers; the slowest rank sets the time.
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


def stage_work(cfg, experts_touched):
    """Algorithmic work of each stage: ('tensor', FLOPs) or ('hbm', bytes).

    Decode-shaped batches (T*k <= 32*E, the swapped-operand kernels) are bound by streaming the
    touched experts' weights: their routed stages count those bytes (plus activations)."""
    T, d, l, h, E, k = cfg.tokens, cfg.d, cfg.latent, cfg.hidden, cfg.experts, cfg.top_k
    ns, hs = cfg.n_shared, cfg.shared_hidden
    ab = 4 if cfg.act == "f32" else 2
    rows = T * k
    w = {
        # bf16 activations: tensor cores (over 3 bf16 terms of W_r); fp32: CUDA-core FMA
        "router_logits": ("tensor" if cfg.act == "bf16" else "alu", 2.0 * T * E * d),
        "topk": ("hbm", 4.0 * T * E + 8.0 * rows),
        "dispatch": ("hbm", 3 * 4.0 * rows),
        "w_down": ("tensor", 2.0 * T * d * l),
        "scatter_rows": ("hbm", float(ab) * (T * l + rows * l)),
        "combine_rmsnorm": ("hbm", float(ab) * (rows * l + T * l)),
    }
    if not cfg.identity_experts and rows <= 32 * E:
        w["routed_gate_up_glu"] = ("hbm", float(experts_touched * expert_weight_bytes(cfg, 2 * h, l)
                                                + ab * rows * (l + h)))
        w["routed_down"] = ("hbm", float(experts_touched * expert_weight_bytes(cfg, l, h) + ab * rows * (h + l)))
    elif not cfg.identity_experts:
        w["routed_gate_up_glu"] = ("tensor", 2.0 * rows * l * 2 * h)
        w["routed_down"] = ("tensor", 2.0 * rows * h * l)
    if not cfg.identity_experts:
        w["shared_gate_up_glu"] = ("tensor", 2.0 * T * d * 2 * ns * hs)
        w["final_gemm"] = ("tensor", 2.0 * T * (ns * hs + l) * d)
    return w


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
    host = inputs.host_inputs(inputs.make_inputs(cfg, dev))
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
            "shared_hidden": cfg.shared_hidden, "routed_w": cfg.routed_w, "seed": cfg.seed,
            "global_batch": cfg.tokens * args.gpus, "parallelism": f"replicas x{args.gpus}",
            "l2": "flushed before every timed step (512 MiB write, untimed)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="k3w_e128_bf16_prefill")
    ap.add_argument("--cpu-sample", type=int, default=8, help="token rows for the oracle CPU baseline")
    ap.add_argument("--single-cta", action="store_true",
                    help="run every tensor-core GEMM on single CTAs (no CTA-pair GEMMs)")
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
    from sparse_moe_layer_sigmoid_gb300 import inputs
    from sparse_moe_layer_sigmoid_gb300 import binding
    from sparse_moe_layer_sigmoid_gb300.binding import LatentMoE

    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = inputs.make_inputs(cfg, dev)
    layer = LatentMoE(cfg, flags=binding.LMOE_FLAG_SINGLE_CTA_GEMM if args.single_cta else 0)
    layer.enable_stage_timing()
    x = inp["x"]
    y = torch.empty((cfg.tokens, layer.out_width), dtype=x.dtype, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else local
    clocks = ClockSampler(gpu_id) if rank == 0 else None
    for _ in range(args.warmup):
        flush.zero_()
        layer.forward(x, inp, y)
    torch.cuda.synchronize()
    st = layer.status()
    if st != 0:
        raise RuntimeError(f"layer reported status {st} during warm-up")
    if clocks:
        clocks.wait_first_sample()

    # grouped-GEMM M-tile utilisation of this routing (rows / (128-row tiles * 128))
    r = layer.route(x, inp)
    counts = (r["offsets"][1:] - r["offsets"][:-1]).cpu()
    m_tiles = int(((counts + 127) // 128).sum())
    route_stats = {"rows": int(counts.sum()), "m_tiles_128": m_tiles,
                   "m_tile_utilization": float(counts.sum()) / max(1, 128 * m_tiles),
                   "experts_touched": int((counts > 0).sum()),
                   "load_max_over_mean": float(counts.max()) / max(1e-9, float(counts.float().mean()))}
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
        for k_, v in layer.stage_times_ms().items():
            stages.setdefault(k_, []).append(v)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_stop()
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dist, dev)
    if layer.status() != 0:
        raise RuntimeError("layer reported an error status during the timed steps")

    # end to end through the public host-memory entry point
    x_host = x.cpu().pin_memory()
    y_host = torch.empty((cfg.tokens, layer.out_width), dtype=x.dtype, pin_memory=True)
    layer.enable_stage_timing()
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

    peaks, src = load_peaks()
    work = stage_work(cfg, route_stats["experts_touched"])
    st_ms = {k_: sum(v) / len(v) for k_, v in stages.items()}
    dom = max((k_ for k_ in work if k_ in st_ms), key=st_ms.get)
    kind, amount = work[dom]
    if kind == "tensor":
        achieved = amount / (st_ms[dom] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    elif kind == "alu":
        # fp32 FMA on CUDA cores: 152 SMs x 128 lanes x 2 FLOP x max SM clock
        achieved = amount / (st_ms[dom] * 1e-3) / 1e12
        peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        unit = "TFLOP/s"
    else:
        achieved = amount / (st_ms[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    tr = TRAFFIC.get(cfg.name, {}).get(dom)
    traffic = None
    if tr and tr["bytes_per_launch"] and tr["sha256"] == file_sha(tr["src"]):
        traffic = tr["bytes_per_launch"]
    total_flops = sum(a for kd, a in work.values() if kd in ("tensor", "alu"))

    line = {"metric": METRIC, "value": job_tokens_per_s(world, cfg.tokens, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg.act, "data": "synthetic",
            "config": workload_config(cfg, args),
            "roofline": {"bound": kind, "kernel": dom, "achieved": achieved,
                         "peak": peak, "unit": unit, "frac": achieved / peak, "traffic": traffic,
                         "peak_source": {"tensor": f"{src} bf16_tflops (burst)", "hbm": f"{src} hbm_gbs",
                                         "alu": "derived: 152 SMs x 128 fp32 lanes x 2 x sm_max_mhz"}[kind]},
            "layer": {"flops": total_flops, "achieved_tflops": total_flops / (ms * 1e-3) / 1e12,
                      "frac_of_bf16_peak": total_flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                      "stages_ms": st_ms},
            "e2e": {"value": job_tokens_per_s(world, cfg.tokens, e2e), "unit": UNIT,
                    "h2d_bytes_per_step": cfg.tokens * cfg.d * elem,
                    "d2h_bytes_per_step": cfg.tokens * layer.out_width * elem},
            "gpu_launches": launches,
            "routing": route_stats,
            "clocks": clk}
    if rank == 0 and world == 1 and args.cpu_sample > 0:
        layer.close()
        y = flush = None
        host = inputs.host_inputs(inp)
        dt = oracle_sample(cfg, host, args.cpu_sample, cfg.seed + 99)
        line["cpu_baseline"] = {"value": args.cpu_sample / dt, "unit": UNIT, "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"{args.cpu_sample} seeded token rows of the workload, fp64 oracle"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
