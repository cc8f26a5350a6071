"""Benchmark: one optimizer step = global gradient norm (fp64-accurate, clip
1.0) + fused AdamW over the Llama-3-8B-shaped list (291 tensors,
8,030,261,248 fp32 parameters, BF16 gradients, FP32 m and v), through the C
ABI of libpsopt.so.

Prints ONE JSON line (rank 0).  ``value`` is whole-job Gparams/s with inputs
resident in HBM; ``e2e`` is the same metric with each step's gradients copied
from pinned host memory through opt_grads_upload and the norm result read
back; ``roofline`` is the fused step kernel's achieved HBM bandwidth (its
algorithmic bytes / its CUDA-event time) against the measured copy bandwidth;
``cpu_baseline`` is the CPU oracle timed on a bounded sample.

Multi-GPU: one process per GPU under torchrun, each an independent replica
over its own copy of the list (the step shards with no data-path exchange;
see the design doc); value = all ranks' parameters / max-over-ranks time.

``--impl reference`` times the CPU oracle instead (bounded sample per step).
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
sys.path.insert(0, ROOT)

METRIC = "optimizer-step Gparams/s and HBM GB/s (% of ~8 TB/s peak), 1×GB300"
UNIT = "Gparams/s"
# algorithmic bytes per parameter: step = p r+w (8) + g r (2) + m r+w (8) + v r+w (8)
STEP_BYTES_PER_PARAM = {"bf16": 26, "f32": 28}
NORM_BYTES_PER_PARAM = {"bf16": 2, "f32": 4}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-seconds", type=float, default=12.0)
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (profiling recipe)"


def traffic_for(kernel_key: str, params: int):
    """DRAM bytes per launch from the committed ncu summary, scaled to this
    launch by parameters, if the kernel source is unchanged since capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel_key]
    except (OSError, KeyError, ValueError):
        return None
    from precision_states_gb300 import build as b
    if d.get("source_stamp") != b._stamp():
        return None
    return d["dram_bytes_per_param"] * params


# ----------------------------------------------------------- cpu baseline
def cpu_baseline(w, seconds: float):
    """Time the CPU oracle (as it stands, single-threaded) on a bounded sample
    of the workload: norm + AdamW step over a growing prefix of the list's
    sampled tensors until about `seconds` of CPU time."""
    import numpy as np
    import torch

    import oracle
    import workloads as W

    order = sorted(range(len(w.sizes)), key=lambda i: (w.sizes[i] > 50_000_000, i))
    # deterministic sample: tensors in list order, skipping the embedding and
    # head, cut to a budget measured on a first small tensor
    ohp = oracle.hparams(**{k: v for k, v in {**dict(beta1=0.9, beta2=0.999), **w.hp}.items()})
    probe = order[1]
    n_probe = min(w.sizes[probe], 2_000_000)
    p = np.zeros(n_probe, np.float32)
    g = W.make_grads(W.Workload("probe", [n_probe], w.grad_dtype), "cpu", 1, 0)[0]
    g = W.to_numpy_codes(g)
    t0 = time.perf_counter()
    oracle.grad_norm([g], w.max_norm)
    oracle.adam_tensor(oracle.ADAMW, p, g, np.zeros(n_probe, np.float32), np.zeros(n_probe, np.float32),
                       ohp, 1)
    per_elem = (time.perf_counter() - t0) / n_probe
    budget = int(seconds / max(per_elem, 1e-10))
    idx, total = [], 0
    for i in order:
        if total + w.sizes[i] > budget and idx:
            break
        idx.append(i)
        total += w.sizes[i]
    grads = [W.to_numpy_codes(t) for t in W.make_grads(w, "cpu", 1, 0, idx)]
    params = [W.to_numpy_codes(t) for t in W.make_params(w, "cpu", 0, idx)]
    ms = [np.zeros(w.sizes[i], np.float32) for i in idx]
    vs = [np.zeros(w.sizes[i], np.float32) for i in idx]
    t0 = time.perf_counter()
    r = oracle.grad_norm(grads, w.max_norm)
    for k in range(len(idx)):
        oracle.adam_tensor(oracle.ADAMW, params[k], grads[k], ms[k], vs[k], ohp, 1, coef=r["clip_coef"])
    dt = time.perf_counter() - t0
    return {"value": total / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(idx)} of {len(w.sizes)} tensors ({total:,} params, {total / w.numel:.2%} of the "
                      f"list): norm + one AdamW step, single-threaded C oracle, {dt:.1f} s"}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, local_rank, world):
    import torch

    import precision_states_gb300 as ps
    import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    w = W.workload(args.workload)
    params = W.make_params(w, dev, seed=rank)
    grads = W.make_grads(w, dev, step=1, seed=rank)
    m = [W.state_storage(w.m_dtype, n, dev) for n in w.sizes]
    v = [W.state_storage(w.v_dtype, n, dev) for n in w.sizes]
    m2 = [W.state_storage(w.m_dtype, n, dev) for n in w.sizes] if w.algo == "ademamix" else None
    plan = ps.Plan(params, grads, m, v, m2, m_dtype=w.m_dtype, v_dtype=w.v_dtype)
    hp = ps.hparams(**{**dict(beta1=0.9, beta2=0.999), **w.hp})
    stream = torch.cuda.current_stream(dev)
    clip = w.max_norm > 0
    d_norm = plan.norm_buffer() if clip else None
    step_fn = plan.ademamix_step if w.algo == "ademamix" else plan.adamw_step
    launches_per_step = (2 if clip else 0) + 1   # norm partials + finish, fused step (one dtype bucket)

    def one_step(t, ev=None):
        if ev is not None:
            ev[0].record(stream)
        if clip:
            plan.grad_norm(w.max_norm, sync=False, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        step_fn(hp, t, d_norm, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    t = 0
    for _ in range(args.warmup):
        t += 1
        one_step(t)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for k in range(args.steps):
        t += 1
        one_step(t, evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    norm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    step_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if pg:
        tt = torch.tensor([total_ms], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        total_ms = float(tt.item())
    params_per_step = w.numel
    value = params_per_step * world * args.steps / (total_ms / 1e3) / 1e9

    # end-to-end through the C ABI with host buffers: per step, H2D of the
    # gradients from pinned memory, norm + step, D2H of the norm result
    e2e = None
    if not args.no_e2e:
        host = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
        for h, g in zip(host, grads):
            h.copy_(g)
        ke = args.e2e_steps or args.steps
        h2d = sum(g.numel() * g.element_size() for g in grads)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ke):
            t += 1
            plan.grads_upload(host, stream=stream)
            r = plan.grad_norm(w.max_norm, sync=True, stream=stream)   # D2H of the 48-byte result
            step_fn(hp, t, d_norm, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1)
        if pg:
            tt = torch.tensor([e_ms], device=dev)
            pg.all_reduce(tt, op=pg.ReduceOp.MAX)
            e_ms = float(tt.item())
        e2e = {"value": params_per_step * world * ke / (e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 48, "steps": ke,
               "note": "per step: opt_grads_upload from pinned host memory (one cudaMemcpyAsync per "
                       "tensor), opt_grad_norm with a host copy of the result, opt_adamw_step"}
        del host

    peak, peak_src = measured_peak()
    step_bytes = STEP_BYTES_PER_PARAM[w.grad_dtype] * params_per_step
    norm_bytes = NORM_BYTES_PER_PARAM[w.grad_dtype] * params_per_step
    step_avg = sum(step_ms) / len(step_ms)
    norm_avg = sum(norm_ms) / len(norm_ms)
    achieved = step_bytes / (step_avg / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "step_kernel<bf16 grads, f32 states, AdamW>",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic_for("adamw_step_f32_bf16grad",
                                                                          params_per_step),
                "peak_source": peak_src, "bytes_per_launch": step_bytes,
                "bytes_per_param": STEP_BYTES_PER_PARAM[w.grad_dtype], "ms_per_launch": round(step_avg, 4),
                "norm": {"achieved": round(norm_bytes / (norm_avg / 1e3) / 1e9, 1), "ms_per_launch_pair":
                         round(norm_avg, 4), "bytes_per_launch": norm_bytes,
                         "frac": round(norm_bytes / (norm_avg / 1e3) / 1e9 / peak, 4)}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del params, grads, m, v, m2
        plan.close()
        torch.cuda.empty_cache()
        cpu = cpu_baseline(w, args.cpu_sample_seconds)

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "tensors": len(w.sizes), "params_per_gpu": params_per_step,
                       "grad_dtype": w.grad_dtype, "m_dtype": w.m_dtype, "v_dtype": w.v_dtype,
                       "clip_max_norm": w.max_norm, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (%.0f GB streamed per step)" % ((step_bytes + norm_bytes) / 1e9)},
            "hbm_gbs": round((step_bytes + norm_bytes) / (total_ms / args.steps / 1e3) / 1e9, 1),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches_per_step * args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# ---------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload (norm + AdamW step over the sampled tensors)."""
    if rank != 0:
        return
    import workloads as W
    w = W.workload(args.workload)
    per_step = max(1.0, min(6.0, 90.0 / max(1, args.steps + args.warmup)))
    vals = []
    cb = None
    for k in range(args.warmup + args.steps):
        cb = cpu_baseline(w, per_step)
        if k >= args.warmup:
            vals.append(cb["value"])
    value = statistics.median(vals)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tensors": len(w.sizes), "params_per_gpu": w.numel,
                       "grad_dtype": w.grad_dtype, "m_dtype": w.m_dtype, "v_dtype": w.v_dtype,
                       "clip_max_norm": w.max_norm, "parallelism": "replicas1"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
