"""The N > 1 host logic on CPU with two gloo ranks: each rank holds a shard of
the tensor list and its own norm result; the ranks all-gather the 48-byte
results and combine them in rank order with the library's opt_norm_combine
("perf(training): fused multi-tensor gradient-norm reduction", 'Correctness
properties': the caller owns the cross-rank scalar reduction).  Both ranks
must get the same bits, equal to the oracle's global norm within 1e-12, and
a NaN on one rank must make both see a non-finite norm.

Each rank's own result comes from the oracle here (there is no GPU in this
test); on a GPU it would come from opt_grad_norm over the rank's shard."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _shard(rank, world, poison):
    rng = np.random.default_rng(1234)
    arrays = [(rng.standard_normal(int(n)) * s).astype(np.float32)
              for n, s in zip(rng.integers(1, 50000, 37), np.exp(rng.uniform(-5, 3, 37)))]
    if poison:
        arrays[5][7] = np.nan
    return arrays, arrays[rank::world]


def _worker(rank, world, port, poison, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import precision_states_gb300 as ps
    everything, mine = _shard(rank, world, poison)
    local = oracle.grad_norm(mine, 0.0)
    r = ps.opt_norm_result()
    for k in ("sumsq", "norm2", "norm_inf", "nan_count", "inf_count", "clip_coef", "status"):
        setattr(r, k, local[k])
    gathered = [None] * world
    dist.all_gather_object(gathered, bytes(r))
    parts = [ps.opt_norm_result.from_buffer_copy(b) for b in gathered]
    combined = ps.opt_norm_combine(parts, 1.0)
    want = oracle.grad_norm(everything, 1.0)
    out_q.put((rank, bytes(combined), want))
    dist.barrier()
    dist.destroy_process_group()


def _run(poison):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, poison, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_ranks_combine_deterministically():
    import precision_states_gb300 as ps
    (r0, b0, want), (r1, b1, _) = _run(poison=False)
    assert b0 == b1, "ranks disagree"
    got = ps.opt_norm_result.from_buffer_copy(b0)
    assert got.status == 0
    assert abs(got.norm2 - want["norm2"]) <= 1e-12 * want["norm2"]
    assert got.norm_inf == want["norm_inf"]
    assert got.clip_coef == want["clip_coef"]


def test_nan_on_one_rank_reaches_both():
    import precision_states_gb300 as ps
    (_, b0, want), (_, b1, _) = _run(poison=True)
    assert b0 == b1
    got = ps.opt_norm_result.from_buffer_copy(b0)
    assert got.status == ps.OPT_ENONFINITE and got.nan_count == 1
    assert math.isnan(got.norm2) and math.isnan(want["norm2"])
