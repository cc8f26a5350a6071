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
over its own copy of the list (the step is elementwise per tensor, so a
sharded list needs no data-path exchange; the only cross-rank quantity, the
norm, combines on the host with opt_norm_combine); value = all ranks'
parameters / max-over-ranks time.

``--impl reference`` times the CPU oracle instead (bounded sample per step).
``--graph`` (FP32 states) takes the step number from the plan's device
counter and replays the norm and the step from CUDA graphs captured once.
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
ELEM_BYTES = {"f32": 4, "bf16": 2, "e4m3": 1, "e2m2": 0.5}
L2_BYTES = 129 * 10**6           # GB300's L2
FLUSH_BYTES = 256 * 2**20        # each of the two L2 flush buffers


def step_bytes_per_param(w) -> float:
    """Algorithmic bytes per parameter of one fused step: p read + write,
    g read, m (and m2) read + write, v read + write."""
    b = 8 + ELEM_BYTES[w.grad_dtype] + 2 * ELEM_BYTES[w.m_dtype] + 2 * ELEM_BYTES[w.v_dtype]
    if w.algo == "ademamix":
        b += 2 * ELEM_BYTES[w.m_dtype]
    if w.algo == "lamb":      # second pass: p read + write, m and v read again
        b += 4 + ELEM_BYTES[w.m_dtype] + ELEM_BYTES[w.v_dtype]
    return b


def resident_bytes(w) -> float:
    """Bytes one step's inputs occupy: p, g, m, v (and m2)."""
    per = (4 + ELEM_BYTES[w.grad_dtype] + ELEM_BYTES[w.m_dtype] + ELEM_BYTES[w.v_dtype]
           + (ELEM_BYTES[w.m_dtype] if w.algo == "ademamix" else 0))
    return per * w.numel


def needs_l2_flush(w) -> bool:
    """A list whose inputs come to less than four times L2 is flushed from L2
    before every timed step; larger ones stream from HBM anyway."""
    return resident_bytes(w) < 4 * L2_BYTES


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b")
    ap.add_argument("--v-dtype", default=None, choices=["f32", "bf16", "e4m3", "e2m2"],
                    help="override the state dtypes: f32 = f32 m and v; otherwise bf16 m and this v")
    ap.add_argument("--rounding", default="nearest", choices=["nearest", "stochastic"])
    ap.add_argument("--lamb", type=float, default=None, metavar="MAX_UNORM",
                    help="time the update-norm clipping (LAMB) step with this bound instead of AdamW")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: same as --steps")
    ap.add_argument("--graph", action="store_true",
                    help="FP32 states: device step counter, norm and step replayed from CUDA graphs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-companions", action="store_true",
                    help="default run only: skip the short device-timed runs of the other workloads")
    ap.add_argument("--companion-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="cpu_baseline: time oracle steps over the sample for at least this long")
    ap.add_argument("--oracle-sample-elems", type=int, default=120_000_000,
                    help="elements of the fixed tensor sample the oracle steps (both arms)")
    ap.add_argument("--stall-curve", action="store_true",
                    help="instead of timing: the fraction of v codes left unchanged per step, every state "
                         "mode, over the low-precision workload's steps (one JSON line per mode)")
    ap.add_argument("--curve-steps", type=int, default=1000)
    ap.add_argument("--constant-sigma", action="store_true", help="stall curve with a fixed gradient scale")
    ap.add_argument("--reset-every", type=int, default=0, help="stall curve with periodic state resets")
    ap.add_argument("--cast", action="store_true",
                    help="instead of the step: the standalone fp32 -> state-format cast (opt_encode) in every "
                         "format and rounding mode beside torch's builtin RNE casts (one JSON line per mode)")
    ap.add_argument("--cast-elems", type=int, default=(1 << 28) + 12)
    return ap.parse_args()


def apply_overrides(w, args):
    """The state dtypes and the algorithm the flags select, on workload w."""
    if args.v_dtype:
        w.m_dtype, w.v_dtype = ("f32", "f32") if args.v_dtype == "f32" else ("bf16", args.v_dtype)
    if args.lamb is not None:
        w.algo = "lamb"
    return w


def sample_indices(w, max_elems: int):
    """The oracle's tensor sample, from sizes alone: tensors in list order,
    those above 50M elements (embedding, head, MLP matrices) last, while they
    fit in max_elems (at least one)."""
    order = sorted(range(len(w.sizes)), key=lambda i: (w.sizes[i] > 50_000_000, i))
    idx, total = [], 0
    for i in order:
        if total + w.sizes[i] > max_elems and idx:
            break
        idx.append(i)
        total += w.sizes[i]
    return idx, total


def run_config(w, args, replicas: int) -> dict:
    """The benchmark's configuration, identical in both arms: the workload,
    the timing protocol of the GPU arm, and the oracle's tensor sample."""
    clip = w.max_norm > 0
    per_step = (step_bytes_per_param(w) + (ELEM_BYTES[w.grad_dtype] if clip else 0)) * w.numel
    idx, total = sample_indices(w, args.oracle_sample_elems)
    return {"workload": w.name, "tensors": len(w.sizes), "params_per_gpu": w.numel,
            "grad_dtype": w.grad_dtype, "m_dtype": w.m_dtype, "v_dtype": w.v_dtype,
            "rounding": args.rounding, "algo": w.algo, "clip_max_norm": w.max_norm,
            "parallelism": f"replicas{replicas}",
            "launch": "cuda-graph replay, device step counter" if args.graph else "direct",
            "l2": ("L2 flushed before every timed step (256 MiB written, 256 MiB read); steps "
                   "timed by their own events; e2e steps not flushed" if needs_l2_flush(w) else
                   "inputs larger than L2 (%.0f GB streamed per step)" % (per_step / 1e9)),
            "oracle_sample": {"tensors": len(idx), "params": total,
                              "rule": "list order, tensors above 50M elements last, up to %d elements"
                                      % args.oracle_sample_elems}}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, tag: str = ""):
        self.idx = gpu_index
        self.proc = None
        # the raw samples, beside the summary the JSON line carries
        out_dir = os.environ.get("BENCH_OUT_DIR", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks{tag}_rank{gpu_index}.csv")

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


def step_kernel_name(w, rounding: str) -> str:
    """The step's kernel as the library dispatches it (the roofline's label
    and the key of its traffic record): LAMB's three passes; the short-list
    kernel for at most 8 tensors and 4,096 tiles of 2,048 elements (its
    four-elements-per-thread form with FP32 states); the
    warp-dynamic kernel for FP32 states (AdamW, AdEMAMix); the staged kernel for
    low-precision states with stochastic rounding and for BF16 v; else the
    register-pipelined kernel."""
    args = f"{w.grad_dtype} grads, {w.m_dtype} m, {w.v_dtype} v, {w.algo}, {rounding}"
    nonempty = [n for n in w.sizes if n > 0]
    tiles = sum((n + 2047) // 2048 for n in nonempty)
    if w.algo == "lamb":
        return f"lamb_stats_kernel + lamb_ratio_kernel + lamb_apply_kernel<{args}>"
    if len(nonempty) <= 8 and tiles <= 4096:
        return f"step_small4_kernel<{args}>" if w.m_dtype == "f32" else f"step_small_kernel<{args}>"
    if w.m_dtype == "f32":
        return f"step_dyn_kernel<{args}>"
    if w.m_dtype != "f32" and w.algo == "adamw" and (rounding == "stochastic" or w.v_dtype == "bf16"):
        return f"step_bulk_kernel<{args}>"
    return f"step_kernel<{args}>"


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
    if d.get("source_stamp") != b.source_stamp(b.STEP_KERNEL_SOURCES):
        return None
    return d["dram_bytes_per_param"] * params


# ----------------------------------------------------------- cpu baseline
class OracleSample:
    """A bounded, deterministic sample of the workload for the CPU oracle:
    the tensors sample_indices picks, from sizes alone, so that both arms
    (and every box) time the oracle on the same tensors."""

    def __init__(self, w, max_elems: int, stochastic: bool = False, max_unorm: float = 0.0):
        import oracle
        import workloads as W

        self.w = w
        self.ohp = oracle.hparams(**{**dict(beta1=0.9, beta2=0.999), **w.hp})
        self.idx, self.numel = sample_indices(w, max_elems)
        self.grads = [W.to_numpy_codes(t) for t in W.make_grads(w, "cpu", 1, 0, self.idx)]
        self.params = [W.to_numpy_codes(t) for t in W.make_params(w, "cpu", 0, self.idx)]
        self.m = [W.to_numpy_codes(W.state_storage(w.m_dtype, w.sizes[i], "cpu")) for i in self.idx]
        self.v = [W.to_numpy_codes(W.state_storage(w.v_dtype, w.sizes[i], "cpu")) for i in self.idx]
        self.m2 = ([W.to_numpy_codes(W.state_storage(w.m_dtype, w.sizes[i], "cpu")) for i in self.idx]
                   if w.algo == "ademamix" else None)
        self.stochastic = stochastic
        self.max_unorm = max_unorm
        self.t = 0

    def step(self) -> float:
        """One oracle step over the sample (norm + update); returns seconds."""
        import oracle
        self.t += 1
        algo = oracle.ADEMAMIX if self.w.algo == "ademamix" else oracle.ADAMW
        t0 = time.perf_counter()
        coef = 1.0
        if self.w.max_norm > 0:
            coef = oracle.grad_norm(self.grads, self.w.max_norm)["clip_coef"]
        for k in range(len(self.idx)):
            if self.w.algo == "lamb":
                oracle.lamb_tensor(self.params[k], self.grads[k], self.m[k], self.v[k], self.ohp, self.t,
                                   self.max_unorm, coef)
                continue
            oracle.adam_tensor(algo, self.params[k], self.grads[k], self.m[k], self.v[k], self.ohp, self.t,
                               m2=None if self.m2 is None else self.m2[k], m_dtype=self.w.m_dtype,
                               v_dtype=self.w.v_dtype, coef=coef, stochastic=self.stochastic, seed=1234,
                               tensor_index=self.idx[k])
        return time.perf_counter() - t0

    def describe(self, dt: float, steps: int) -> str:
        return (f"{len(self.idx)} of {len(self.w.sizes)} tensors ({self.numel:,} params, "
                f"{self.numel / self.w.numel:.2%} of the list): norm + one step per timed step, "
                f"{steps} timed steps, single-threaded C oracle, {dt:.2f} s per step")


def cpu_baseline(w, args):
    """The CPU oracle as it stands, timed on the machine's host cores (one
    thread) over the fixed sample of the same workload: steps until at
    least --cpu-seconds have passed (two at least), after one untimed."""
    smp = OracleSample(w, args.oracle_sample_elems, args.rounding == "stochastic",
                       args.lamb if args.lamb is not None else 0.0)
    smp.step()
    times = []
    while len(times) < 2 or sum(times) < args.cpu_seconds:
        times.append(smp.step())
    dt = sum(times) / len(times)
    return {"value": smp.numel / dt / 1e9, "unit": UNIT, "cores": 1, "cpu_model": cpu_model(),
            "kind": "oracle", "sample": smp.describe(dt, len(times))}


# ---------------------------------------------------------------- our arm
class Case:
    """One workload on one device: its seeded tensors, the plan over them,
    the hyperparameters and the step call the flags select."""

    def __init__(self, w, rounding: str, lamb, dev, seed: int):
        import torch

        import precision_states_gb300 as ps
        import workloads as W

        self.w, self.lamb, self.dev = w, lamb, dev
        self.params = W.make_params(w, dev, seed=seed)
        self.grads = W.make_grads(w, dev, step=1, seed=seed)
        self.m = [W.state_storage(w.m_dtype, n, dev) for n in w.sizes]
        self.v = [W.state_storage(w.v_dtype, n, dev) for n in w.sizes]
        self.m2 = [W.state_storage(w.m_dtype, n, dev) for n in w.sizes] if w.algo == "ademamix" else None
        self.plan = ps.Plan(self.params, self.grads, self.m, self.v, self.m2, m_dtype=w.m_dtype,
                            v_dtype=w.v_dtype)
        self.hp = ps.hparams(rounding=rounding, seed=1234, **{**dict(beta1=0.9, beta2=0.999), **w.hp})
        self.clip = w.max_norm > 0
        self.d_norm = self.plan.norm_buffer() if self.clip else None
        self.step_fn = self.stepper(self.plan)
        # The timed steps must not find their inputs in L2 (129 MB on GB300).
        # A list whose per-step bytes are under four times that is flushed
        # before every step: a 256 MiB buffer is written, then another 256 MiB
        # read, so that L2 holds neither the step's data nor dirty lines of
        # the flush.  Such steps are timed by their own events (norm start to
        # step end), so the flush stays out of the figure.
        self.flush = needs_l2_flush(w)
        if self.flush:
            self.flush_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
            self.flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def stepper(self, pl):
        """The step call on plan pl: AdamW, AdEMAMix, or LAMB with the bound."""
        if self.lamb is not None:
            return lambda hp_, t_, dn_, stream=None: pl.lamb_step(hp_, t_, self.lamb, dn_, stream=stream)
        return pl.ademamix_step if self.w.algo == "ademamix" else pl.adamw_step

    def launches_per_step(self) -> int:
        """The norm is one launch per gradient dtype (one here; its last CTA
        finishes), the step one launch (LAMB: three passes)."""
        return (1 if self.clip else 0) + (3 if self.lamb is not None else 1)

    def one_step(self, t, hp, stream, ev=None, graphs=None):
        """Norm + step number t on stream; ev = three events (start, after
        the norm, after the step) or None; graphs replace the launches."""
        graphs = graphs or {}
        if self.flush:
            self.flush_w.fill_(float(t))
            self.flush_r.sum()
        if ev is not None:
            ev[0].record(stream)
        if self.clip:
            if "norm" in graphs:
                graphs["norm"].replay()
            else:
                self.plan.grad_norm(self.w.max_norm, sync=False, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if "step" in graphs:
            graphs["step"].replay()
        else:
            self.step_fn(hp, t, self.d_norm, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def time_steps(self, hp, stream, t, steps, graphs=None, step_arg=None):
        """steps timed steps after step t: (last t, per-step event triples,
        total ms).  A flushed list's total is the sum of its steps' own
        intervals; otherwise the span of the loop."""
        import torch

        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(steps):
            t += 1
            self.one_step(t if step_arg is None else step_arg, hp, stream, evs[k], graphs)
        end.record(stream)
        torch.cuda.synchronize()
        total = start.elapsed_time(end)
        if self.flush:
            total = sum(e[0].elapsed_time(e[2]) for e in evs)
        return t, evs, total

    def norm_clean_ms(self, stream, n: int) -> float:
        """The norm alone with L2 clean: in the step loop each norm follows a
        step, and the write-back of the step's dirty L2 lines lands in the
        norm's interval.  Here a 512 MiB read (untimed) evicts them first, so
        the norm's events time the kernel's own traffic."""
        import torch

        rd = torch.ones(2 * FLUSH_BYTES // 4, dtype=torch.float32, device=self.dev)
        cl = []
        for k in range(n + 2):
            rd.sum()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            self.plan.grad_norm(self.w.max_norm, sync=False, stream=stream)
            a1.record(stream)
            torch.cuda.synchronize()
            if k >= 2:
                cl.append(a0.elapsed_time(a1))
        del rd
        return sum(cl) / len(cl)

    def close(self):
        import torch

        self.plan.close()
        for k in ("plan", "d_norm", "step_fn", "params", "grads", "m", "v", "m2", "flush_w", "flush_r"):
            self.__dict__.pop(k, None)
        torch.cuda.empty_cache()


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

    w = apply_overrides(W.workload(args.workload), args)
    case = Case(w, args.rounding, args.lamb, dev, seed=rank)
    params, grads, m, v, m2 = case.params, case.grads, case.m, case.v, case.m2
    plan, hp, clip, d_norm = case.plan, case.hp, case.clip, case.d_norm
    stream = torch.cuda.current_stream(dev)
    # with --graph the device step counter adds one launch
    launches_per_step = case.launches_per_step() + (1 if args.graph else 0)
    if args.graph and (w.m_dtype != "f32" or args.lamb is not None):
        raise SystemExit("--graph needs FP32 states and the AdamW or AdEMAMix step")
    hp_step = hp
    if args.graph:
        hp_step = ps.opt_hparams.from_buffer_copy(hp)
        hp_step.flags |= ps.OPT_STEP_DEVICE_COUNTER
    graphs = {}
    step_arg = 0 if args.graph else None

    t = 0
    for _ in range(args.warmup):
        t += 1
        case.one_step(t if step_arg is None else step_arg, hp_step, stream)
    torch.cuda.synchronize()
    if args.graph:
        # capture once (nothing runs); each replay is the counter's next step
        side = torch.cuda.Stream(dev)
        if clip:
            graphs["norm"] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graphs["norm"], stream=side):
                plan.grad_norm(w.max_norm, sync=False, stream=side)
        graphs["step"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs["step"], stream=side):
            case.step_fn(hp_step, 0, d_norm, stream=side)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    t, evs, total_ms = case.time_steps(hp_step, stream, t, args.steps, graphs, step_arg)
    clk = clocks.stop()
    norm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    step_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if pg:
        tt = torch.tensor([total_ms], device=dev)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        total_ms = float(tt.item())
    params_per_step = w.numel
    value = params_per_step * world * args.steps / (total_ms / 1e3) / 1e9
    norm_clean_ms = case.norm_clean_ms(stream, min(args.steps, 20)) if clip else None

    # end-to-end through the C ABI with host buffers.  Every step copies its
    # gradients from pinned host memory (opt_grads_upload) and reads its norm
    # result back to pinned host memory.  Two device gradient buffers, each
    # with a plan over the same p, m, v, let step k+1's copy (copy stream)
    # overlap step k (compute stream); events order the reuse of a buffer.
    e2e = None
    if not args.no_e2e:
        host = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
        for h, g in zip(host, grads):
            h.copy_(g)
        ke = args.e2e_steps or args.steps
        grads_b = [torch.empty_like(g) for g in grads]
        plan_b = ps.Plan(params, grads_b, m, v, m2, m_dtype=w.m_dtype, v_dtype=w.v_dtype)
        plans = [plan, plan_b]
        steps_of = [case.stepper(plan), case.stepper(plan_b)]
        copy_stream = torch.cuda.Stream(dev)
        res_dev = torch.zeros((max(ke, 2), 6), dtype=torch.float64, device=dev)   # 48 B per step
        res_host = torch.zeros((max(ke, 2), 6), dtype=torch.float64, pin_memory=True)
        up_done = [torch.cuda.Event(), torch.cuda.Event()]
        step_done = [torch.cuda.Event(), torch.cuda.Event()]
        h2d = sum(g.numel() * g.element_size() for g in grads)

        def timing_event():
            return torch.cuda.Event(enable_timing=True)

        def e2e_loop(nsteps, t):
            """nsteps uploads + norms + steps; returns (elapsed ms, last step,
            mean upload ms, mean compute ms), the means from events around
            each upload (copy stream) and each norm + step (compute stream)."""
            e0, e1 = timing_event(), timing_event()
            ups, comps = [], []
            e0.record(stream)
            copy_stream.wait_event(e0)
            u = (timing_event(), timing_event())
            u[0].record(copy_stream)
            plans[0].grads_upload(host, stream=copy_stream)
            u[1].record(copy_stream)
            ups.append(u)
            up_done[0].record(copy_stream)
            for k in range(nsteps):
                b = k % 2
                stream.wait_event(up_done[b])
                t += 1
                d_res = res_dev[k].data_ptr()
                c = (timing_event(), timing_event())
                c[0].record(stream)
                plans[b].grad_norm(w.max_norm, d_out=d_res, sync=False, stream=stream)
                steps_of[b](hp, t, d_res if clip else None, stream=stream)
                c[1].record(stream)
                comps.append(c)
                res_host[k].copy_(res_dev[k], non_blocking=True)             # D2H of the result
                step_done[b].record(stream)
                # prefetch the next step's gradients into the other buffer once
                # the step that last read it (k - 1) is done.  Issued after
                # step k so that a host call that blocks on the copy queue
                # cannot hold back step k's launch.
                if k + 1 < nsteps:
                    if k >= 1:
                        copy_stream.wait_event(step_done[1 - b])
                    u = (timing_event(), timing_event())
                    u[0].record(copy_stream)
                    plans[1 - b].grads_upload(host, stream=copy_stream)
                    u[1].record(copy_stream)
                    ups.append(u)
                    up_done[1 - b].record(copy_stream)
            e1.record(stream)
            torch.cuda.synchronize()
            mean = lambda pairs: sum(x.elapsed_time(y) for x, y in pairs) / max(len(pairs), 1)
            return e0.elapsed_time(e1), t, mean(ups), mean(comps)

        _, t, _, _ = e2e_loop(2, t)                     # untimed: both buffers and plans warm
        torch.cuda.synchronize()

        def uploads_alone(n):
            """Mean ms of n uploads with nothing else on the GPU."""
            out = []
            for _ in range(n):
                u0, u1 = timing_event(), timing_event()
                u0.record(copy_stream)
                plans[0].grads_upload(host, stream=copy_stream)
                u1.record(copy_stream)
                torch.cuda.synchronize()
                out.append(u0.elapsed_time(u1))
            return sum(out) / len(out)

        def uploads_beside_copies(n):
            """Mean ms of n uploads while the compute stream runs plain device
            copies that keep HBM busy for the whole upload (no optimizer work)."""
            out = []
            for _ in range(n):
                u0, u1 = timing_event(), timing_event()
                done = torch.cuda.Event()
                u0.record(copy_stream)
                plans[0].grads_upload(host, stream=copy_stream)
                u1.record(copy_stream)
                done.record(copy_stream)
                while not done.query():
                    for _ in range(16):
                        hbm_b.copy_(hbm_a)
                torch.cuda.synchronize()
                out.append(u0.elapsed_time(u1))
            return sum(out) / len(out)

        # A/B/C, interleaved three times: uploads alone (A), the overlapped
        # loop (B: its uploads, its compute, its time per step), uploads
        # beside HBM-saturating copies (C).  Whether the loop's uploads run
        # slower than uploads alone, and whether plain HBM traffic does the
        # same to them, separates the link's own variation from contention
        # with the compute.
        hbm_a = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
        hbm_b = torch.empty_like(hbm_a)
        ab = {"upload_alone_ms": [], "loop_upload_ms": [], "loop_compute_ms": [], "loop_ms_per_step": [],
              "upload_beside_hbm_copies_ms": []}
        kab = max(3, min(5, ke))
        for _ in range(3):
            ab["upload_alone_ms"].append(round(uploads_alone(2), 3))
            l_ms, t, l_up, l_comp = e2e_loop(kab, t)
            ab["loop_upload_ms"].append(round(l_up, 3))
            ab["loop_compute_ms"].append(round(l_comp, 3))
            ab["loop_ms_per_step"].append(round(l_ms / kab, 3))
            ab["upload_beside_hbm_copies_ms"].append(round(uploads_beside_copies(2), 3))
        del hbm_a, hbm_b
        torch.cuda.synchronize()
        upload_alone_ms = sum(ab["upload_alone_ms"]) / len(ab["upload_alone_ms"])
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e_ms, t, upload_ms, compute_ms = e2e_loop(ke, t)
        finite = all(int(res_host[k].view(torch.int32)[11]) == 0 for k in range(ke))
        if pg:
            tt = torch.tensor([e_ms], device=dev)
            pg.all_reduce(tt, op=pg.ReduceOp.MAX)
            e_ms = float(tt.item())
        e2e = {"value": params_per_step * world * ke / (e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 48, "steps": ke,
               "ms_per_step": round(e_ms / ke, 3), "all_norms_finite": finite,
               "upload_alone_ms": round(upload_alone_ms, 3),
               "h2d_gbs_alone": round(h2d / (upload_alone_ms / 1e3) / 1e9, 1),
               "upload_ms_in_loop": round(upload_ms, 3), "compute_ms_in_loop": round(compute_ms, 3),
               "h2d_gbs_in_loop": round(h2d / (upload_ms / 1e3) / 1e9, 1),
               "ab": {**ab, "steps_per_loop": kab,
                      "how": "three rounds of: two uploads alone; the overlapped loop (uploads, norm + "
                             "step); two uploads beside device copies that keep HBM busy"},
               "note": "per step: opt_grads_upload of the step's gradients from pinned host memory (one "
                       "cudaMemcpyAsync per tensor, copy stream, double-buffered), opt_grad_norm, the step, "
                       "and a copy of the 48-byte norm result to pinned host memory"}
        plan_b.close()
        del host, grads_b

    # per-step distribution (norm + step, CUDA events on the launching stream);
    # every sample goes to a JSONL file beside the clock samples
    out_dir = os.environ.get("BENCH_OUT_DIR", os.path.join(ROOT, "bench_out"))
    os.makedirs(out_dir, exist_ok=True)
    with open(os.path.join(out_dir, f"steps_rank{rank}.jsonl"), "w") as fh:
        for k, e in enumerate(evs):
            fh.write(json.dumps({"workload": w.name, "timed_step": k, "norm_ms": round(norm_ms[k], 5),
                                 "step_ms": round(step_ms[k], 5),
                                 "total_ms": round(e[0].elapsed_time(e[2]), 5)}) + "\n")
    per_step = sorted(e[0].elapsed_time(e[2]) for e in evs)

    def pct(q):
        k = (len(per_step) - 1) * q
        lo, hi = int(k), min(int(k) + 1, len(per_step) - 1)
        return per_step[lo] + (per_step[hi] - per_step[lo]) * (k - lo)
    per_step_stats = {"median": round(pct(0.5), 4), "p10": round(pct(0.1), 4), "p90": round(pct(0.9), 4),
                      "min": round(per_step[0], 4), "max": round(per_step[-1], 4), "n": len(per_step)}

    peak, peak_src = measured_peak()
    bpp = step_bytes_per_param(w)
    step_bytes = int(bpp * params_per_step)
    norm_bytes = int(ELEM_BYTES[w.grad_dtype] * params_per_step) if clip else 0
    step_avg = sum(step_ms) / len(step_ms)
    norm_avg = sum(norm_ms) / len(norm_ms)
    achieved = step_bytes / (step_avg / 1e3) / 1e9
    kname = step_kernel_name(w, args.rounding)
    roofline = {"bound": "hbm", "kernel": kname,
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic_for(kname, params_per_step),
                "peak_source": peak_src, "bytes_per_launch": step_bytes,
                "bytes_per_param": bpp, "ms_per_launch": round(step_avg, 4)}
    if clip:
        roofline["norm"] = {"achieved": round(norm_bytes / (norm_avg / 1e3) / 1e9, 1),
                            "ms_per_norm": round(norm_avg, 4), "bytes_per_launch": norm_bytes,
                            "frac": round(norm_bytes / (norm_avg / 1e3) / 1e9 / peak, 4),
                            "clean_l2": {"ms_per_norm": round(norm_clean_ms, 4),
                                         "achieved": round(norm_bytes / (norm_clean_ms / 1e3) / 1e9, 1),
                                         "frac": round(norm_bytes / (norm_clean_ms / 1e3) / 1e9 / peak, 4),
                                         "how": "each norm after an untimed 512 MiB read that evicts the "
                                                "step's dirty L2 lines (in the loop, their write-back lands "
                                                "in the norm's interval)"}}

    # the main list's tensors are not needed past this point
    del params, grads, m, v, m2, plan, d_norm
    case.close()
    companions = None
    if companions_wanted(args, world):
        companions = run_companions(args, dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args)

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": run_config(w, args, world),
            "hbm_gbs": round((step_bytes + norm_bytes) / (total_ms / args.steps / 1e3) / 1e9, 1),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
            "per_step_ms": per_step_stats}
    if companions is not None:
        line["companions"] = companions
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


# ------------------------------------------------------------- companions
# The default run also times, briefly and by device events only, every other
# workload the benchmark covers, so that one invocation records them all:
# (workload, state override as for --v-dtype, rounding, LAMB bound).
COMPANIONS = (
    ("adamw_1m", None, "nearest", None),
    ("clip_740", None, "nearest", None),
    ("ademamix_gpt2", None, "nearest", None),
    ("lowp_gpt2", "f32", "nearest", None),
    ("lowp_gpt2", "bf16", "nearest", None),
    ("lowp_gpt2", "bf16", "stochastic", None),
    ("lowp_gpt2", "e4m3", "nearest", None),
    ("lowp_gpt2", "e4m3", "stochastic", None),
    ("lowp_gpt2", "e2m2", "nearest", None),
    ("lowp_gpt2", "e2m2", "stochastic", None),
    ("llama3_8b", None, "nearest", 1.0),
)


def companions_wanted(args, world: int) -> bool:
    """Only the default invocation on one GPU: the Llama-3-8B list with its
    own states, AdamW, direct launches."""
    return (world == 1 and not args.no_companions and args.workload == "llama3_8b" and args.v_dtype is None
            and args.lamb is None and not args.graph)


def run_companions(args, dev, stream, peak) -> dict:
    """Each COMPANIONS entry: a fresh seeded list, --warmup untimed steps,
    --companion-steps timed ones (events as in the main loop, L2 flushed
    where the list is small), then freed; plus the standalone cast in every
    format and rounding.  One clock record covers all of them."""
    import torch

    import workloads as W

    clocks = ClockSampler(dev.index, tag="_companions")
    clocks.start()
    time.sleep(0.3)
    runs = []
    for name, vdt, rnd, lamb in COMPANIONS:
        w = apply_overrides(W.workload(name), argparse.Namespace(v_dtype=vdt, lamb=lamb))
        case = Case(w, rnd, lamb, dev, seed=0)
        t = 0
        for _ in range(args.warmup):
            t += 1
            case.one_step(t, case.hp, stream)
        torch.cuda.synchronize()
        t, evs, total = case.time_steps(case.hp, stream, t, args.companion_steps)
        k = len(evs)
        step_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / k
        step_bytes = step_bytes_per_param(w) * w.numel
        rec = {"workload": name, "tensors": len(w.sizes), "params": w.numel, "grad_dtype": w.grad_dtype,
               "m_dtype": w.m_dtype, "v_dtype": w.v_dtype, "rounding": rnd, "algo": w.algo,
               "value": round(w.numel * k / (total / 1e3) / 1e9, 3), "ms_per_step": round(total / k, 4),
               "step_kernel": {"ms_per_launch": round(step_ms, 4), "bytes_per_launch": int(step_bytes),
                               "frac": round(step_bytes / (step_ms / 1e3) / 1e9 / peak, 4)},
               "l2": "flushed before every step" if case.flush else "inputs larger than L2"}
        if lamb is not None:
            rec["lamb_max_unorm"] = lamb
        if case.clip:
            nb = ELEM_BYTES[w.grad_dtype] * w.numel
            norm_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / k
            clean = case.norm_clean_ms(stream, k)
            rec["norm"] = {"ms": round(norm_ms, 4), "frac": round(nb / (norm_ms / 1e3) / 1e9 / peak, 4),
                           "clean_l2_ms": round(clean, 4),
                           "clean_l2_frac": round(nb / (clean / 1e3) / 1e9 / peak, 4)}
        runs.append(rec)
        case.close()
        del case
    casts = cast_rows(args.cast_elems, 50, args.warmup, dev, stream, peak)
    clk = clocks.stop()
    return {"how": "each workload seeded afresh, %d warm-up and %d timed steps, CUDA events on the launching "
                   "stream; fractions of the measured copy bandwidth" % (args.warmup, args.companion_steps),
            "runs": runs, "cast": casts, "clocks": clk}


# ---------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is the oracle's norm +
    step over the same fixed sample of the workload as the GPU arm's
    cpu_baseline.  Rank 0 alone runs it, so its line reports one replica
    (parallelism replicas1, oracle_rank 0) whatever the launch's world size;
    the other ranks exit without work."""
    if rank != 0:
        return
    import workloads as W
    w = apply_overrides(W.workload(args.workload), args)
    smp = OracleSample(w, args.oracle_sample_elems, args.rounding == "stochastic",
                       args.lamb if args.lamb is not None else 0.0)
    for _ in range(args.warmup):
        smp.step()
    times = [smp.step() for _ in range(args.steps)]
    total = sum(times)
    value = smp.numel * args.steps / total / 1e9
    cb = {"value": round(value, 6), "unit": UNIT, "cores": 1, "cpu_model": cpu_model(), "kind": "oracle",
          "sample": smp.describe(total / args.steps, args.steps)}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "oracle_rank": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": run_config(w, args, 1),
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_stall_curve(args):
    """The low-precision workload's report: for each state mode, the fraction
    of v coordinates whose stored code a step left unchanged ("When Small
    Updates Disappear", sec. 1.1 and 4), every step, over the whole GPT-2
    list.  Gradients are drawn fresh every step with the workload's scale
    schedule (or a fixed scale), optionally with periodic resets (sec. 5).
    The model's stationary prediction is printed beside each mode."""
    import torch

    import precision_states_gb300 as ps
    import workloads as W
    from oracle import stall_model

    dev = torch.device("cuda", 0)
    modes = [("f32", "nearest"), ("bf16", "nearest"), ("bf16", "stochastic"), ("e4m3", "nearest"),
             ("e4m3", "stochastic"), ("e2m2", "nearest"), ("e2m2", "stochastic")]
    T = args.curve_steps
    for vd, rnd in modes:
        w = W.workload("lowp_gpt2", sigma_decay_steps=0 if args.constant_sigma else T)
        w.m_dtype, w.v_dtype = ("f32", "f32") if vd == "f32" else ("bf16", vd)
        params = W.make_params(w, dev, 0)
        grads = [torch.empty(n, dtype=torch.bfloat16, device=dev) for n in w.sizes]
        m = [W.state_storage(w.m_dtype, n, dev) for n in w.sizes]
        v = [W.state_storage(w.v_dtype, n, dev) for n in w.sizes]
        plan = ps.Plan(params, grads, m, v, m_dtype=w.m_dtype, v_dtype=w.v_dtype)
        frac, t_local = [], 0
        for t in range(1, T + 1):
            W.fill_grads(w, grads, t, 0)
            reset = args.reset_every > 0 and t > 1 and (t - 1) % args.reset_every == 0
            t_local = 1 if reset else t_local + 1
            hp = ps.hparams(rounding=rnd, seed=99, count_unchanged=True, reset_states=reset,
                            **{**dict(beta1=0.9, beta2=0.999), **w.hp})
            plan.adamw_step(hp, t_local)
            frac.append(plan.unchanged_count() / w.numel)
        plan.close()
        del params, grads, m, v
        torch.cuda.empty_cache()
        p = stall_model.FRACTION_BITS.get(vd)
        model = None if p is None else {
            "nearest": round(stall_model.stall_nearest(0.999, p), 4) if rnd == "nearest" else None,
            "stochastic": round(stall_model.stall_stochastic(0.999, p), 4) if rnd == "stochastic" else None}
        pick = [s for s in (1, 2, 5, 10, 20, 50, 100, 200, 300, 500, 700, 1000) if s <= T]
        print(json.dumps({"report": "unchanged-v fraction per step", "workload": w.name, "params": w.numel,
                          "v_dtype": vd, "m_dtype": w.m_dtype, "rounding": rnd, "beta2": 0.999, "steps": T,
                          "grad_scale": "constant 1" if args.constant_sigma else f"1 -> 0.1 linearly over {T}",
                          "reset_every": args.reset_every or None,
                          "at_step": {str(s): round(frac[s - 1], 5) for s in pick},
                          "mean_last_100": round(sum(frac[-100:]) / min(100, T), 5),
                          "model_stationary": model}), flush=True)


def cast_rows(n: int, launches: int, warmup: int, dev, stream, peak, clocks=None) -> list:
    """The standalone cast ("When Small Updates Disappear", sec. 6-8: an fp32
    tensor rounded to BF16, nearest or stochastic, one read and one write
    per element) for BF16, E4M3 and E2M2 through opt_encode, timed with CUDA
    events over `launches` launches after `warmup`, beside torch's builtin
    round-to-nearest conversions (copy_ into a preallocated BF16 / E4M3
    tensor), which are the hardware-cast yardstick.  The input (4 B per
    element) is larger than L2, so every launch streams from HBM.  With a
    ClockSampler, each row carries the clocks of its own launches."""
    import torch

    import precision_states_gb300 as ps

    gen = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn(n, generator=gen, device=dev, dtype=torch.float32) * 1e-3
    out_bytes = {"bf16": 2, "e4m3": 1, "e2m2": 0.5}
    outs = {"bf16": torch.empty(n, dtype=torch.int16, device=dev),
            "e4m3": torch.empty(n, dtype=torch.uint8, device=dev),
            "e2m2": torch.empty((n + 1) // 2, dtype=torch.uint8, device=dev)}
    builtin = {"bf16": torch.empty(n, dtype=torch.bfloat16, device=dev)}
    if hasattr(torch, "float8_e4m3fn"):
        builtin["e4m3"] = torch.empty(n, dtype=torch.float8_e4m3fn, device=dev)

    def timed(fn):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(launches):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / launches

    ref_ms = {dt: timed(lambda t=t: t.copy_(x)) for dt, t in builtin.items()}
    rows = []
    for dt in ("bf16", "e4m3", "e2m2"):
        for rnd in ("nearest", "stochastic"):
            if clocks is not None:
                clocks.start()
                time.sleep(0.2)
            ms = timed(lambda: ps.opt_encode(x, outs[dt], dt, rnd, seed=11, tensor_index=0, step=1,
                                             stream=stream))
            nbytes = n * (4 + out_bytes[dt])
            gbs = nbytes / (ms / 1e3) / 1e9
            row = {"elements": n, "format": dt, "rounding": rnd, "ms_per_launch": round(ms, 4),
                   "gelem_per_s": round(n / (ms / 1e3) / 1e9, 2), "hbm_gbs": round(gbs, 1),
                   "frac": round(gbs / peak, 4), "bytes_per_elem": 4 + out_bytes[dt], "launches": launches}
            if clocks is not None:
                row["clocks"] = clocks.stop()
            if dt in ref_ms:
                row["builtin_rne_ms"] = round(ref_ms[dt], 4)
                row["vs_builtin_rne"] = round(ref_ms[dt] / ms, 4)
            rows.append(row)
    del x, outs, builtin
    torch.cuda.empty_cache()
    return rows


def run_cast(args):
    """One JSON line per format and rounding of the standalone cast."""
    import torch

    dev = torch.device("cuda", 0)
    peak, peak_src = measured_peak()
    launches = max(args.steps, 100)       # ~0.2 ms each: enough launches for a stable mean
    rows = cast_rows(args.cast_elems, launches, args.warmup, dev, torch.cuda.current_stream(dev), peak,
                     clocks=ClockSampler(0))
    for row in rows:
        line = {"report": "standalone cast", **row, "peak_gbs": peak, "peak_source": peak_src,
                "warmup": max(3, args.warmup), "l2": "input larger than L2 (%.2f GB)" % (4 * row["elements"] / 1e9)}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.cast:
        if rank == 0:
            run_cast(args)
        return
    if args.stall_curve:
        if rank == 0:
            run_stall_curve(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
