"""CPU test of bench.py's reference arm (the CPU oracle timed on a bounded
sample of the workload): it runs without a GPU and prints one JSON line with
the fields the bench contract names for it."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "sweep", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["config"]["workload"] == "sweep"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the multi-GPU bench is (torch.distributed.run, two ranks,
    127.0.0.1), only rank 0 runs the oracle and prints; the other rank exits
    0 without work."""
    import socket
    with socket.socket() as sock:              # a free port for the rendezvous
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "sweep", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    # rank 0 alone ran the oracle: one replica, whatever the launch's size
    assert d["config"]["parallelism"] == "replicas1" and d["oracle_rank"] == 0


def run_reference_line(*extra):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", *extra],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])


def test_both_arms_share_config_and_oracle_sample():
    """The reference arm's config is the GPU arm's, key for key (the GPU
    arm's is built by the same run_config for one replica), and both time
    the oracle on one sample fixed by the tensor sizes alone."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    argv = ["--workload", "sweep", "--v-dtype", "e4m3", "--rounding", "stochastic",
            "--oracle-sample-elems", "200000"]
    d = run_reference_line(*argv)
    old = sys.argv
    try:
        sys.argv = ["bench.py", "--steps", "1", "--warmup", "0", *argv]
        args = bench.parse()
    finally:
        sys.argv = old
    w = bench.apply_overrides(W.workload("sweep"), args)
    assert d["config"] == json.loads(json.dumps(bench.run_config(w, args, 1)))
    idx, total = bench.sample_indices(w, 200000)
    assert d["config"]["oracle_sample"]["tensors"] == len(idx)
    assert d["config"]["oracle_sample"]["params"] == total
    assert total <= 200000 and idx == sorted(idx)
    smp = bench.OracleSample(w, 200000, True)
    assert smp.idx == idx and smp.numel == total
    assert d["cpu_baseline"]["cpu_model"] and d["cpu_baseline"]["cores"] == 1


def test_oracle_sample_is_fixed_by_sizes():
    """Llama-3-8B list: the sample is the same set every time and on every
    box (no timing calibration), the attention and norm tensors of the first
    layers, the matrices above 50M elements left for last."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.workload("llama3_8b")
    a = bench.sample_indices(w, 120_000_000)
    assert a == bench.sample_indices(w, 120_000_000)
    idx, total = a
    assert all(w.sizes[i] <= 50_000_000 for i in idx) and 100_000_000 < total <= 120_000_000


def test_l2_flush_only_for_lists_that_fit():
    """bench.py flushes L2 before each timed step only where the step's
    inputs would otherwise stay in it: the 1M-parameter list (16.8 MB), not
    the 740-tensor, GPT-2 or Llama-3-8B lists."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    assert bench.resident_bytes(W.workload("adamw_1m")) == 16 * (1 << 20)
    assert bench.needs_l2_flush(W.workload("adamw_1m"))
    for name in ("clip_740", "ademamix_gpt2", "lowp_gpt2", "llama3_8b"):
        assert not bench.needs_l2_flush(W.workload(name)), name
    w = W.workload("lowp_gpt2")
    w.v_dtype = "e2m2"
    assert not bench.needs_l2_flush(w)
