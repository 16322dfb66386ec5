"""Multi-process host logic on the CPU: gloo ranks (world sizes 2 and 4).

Covers what the multi-process benchmark and driver rely on: the global skip
decision (a one-word OR over the group), the max-over-ranks timing, the
process-to-rank mapping, and the whole ZeRO-DP choreography of one step
("ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
section "ZeRO-DP": gradients reduce-scattered, each rank steps only its 1/Nd,
parameters all-gathered) with the oracle standing in for the GPU kernel on
each rank; the assembled result must equal the oracle's unsharded step.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _checks(rank, world)
    finally:
        dist.destroy_process_group()


def _checks(rank: int, world: int):
    import dataclasses

    import oracle
    import synth
    import zero_sharded_optimizer_02_gb300 as z
    from zero_sharded_optimizer_02_gb300.step import (data_parallel_rank, global_skip,
                                                      max_over_ranks, sum_over_ranks)
    g = dist.group.WORLD
    # skip decision: one rank's overflow skips everyone; clean everywhere commits
    assert global_skip(False, g) is False
    assert global_skip(rank == 1, g) is True
    assert global_skip(rank == 0, g) is True
    assert max_over_ranks(rank + 1.5, g) == world - 1 + 1.5
    assert sum_over_ranks(rank + 5, g) == sum(r + 5 for r in range(world))
    assert data_parallel_rank(0, rank, 64) == rank
    assert data_parallel_rank(64 - world, rank, 64) == 64 - world + rank
    with pytest.raises(ValueError):
        data_parallel_rank(65 - world, world - 1, 64)

    # one ZeRO-DP step, Nd = world, rank r owns shard r
    w = dataclasses.replace(synth.WORKLOADS["c0"], psi=1001, nd=world, bucket=64)
    L = z.zero_partition_layout(w.psi, w.nd, rank, 8)
    s, pitch, n, begin = int(L.shard_elems), int(L.row_pitch), int(L.length), int(L.begin)
    idx = torch.arange(w.psi, dtype=torch.int64)
    h = w.hparams
    state0 = [synth.state_values(w, k, idx).numpy() for k in ("master", "m", "v")]
    for step, plant in ((0, False), (1, True)):
        # this rank's own full gradient (its contribution), padded partitions
        mine = np.zeros(world * pitch, np.uint16)
        flat = synth.grad_values(w, step, rank, idx).view(torch.int16).numpy().view(np.uint16)
        if plant and rank == 1:
            flat = flat.copy()
            flat[s // 2] = 0x7C00               # +inf into rank 0's shard
        for r in range(world):
            b = r * s
            k = max(0, min(s, w.psi - b))
            mine[r * pitch:r * pitch + k] = flat[b:b + k]
        # reduce-scatter data movement: every rank pulls every contribution row
        # (16-bit payloads travel widened to int32: gloo has no int16 all-gather)
        rows = [torch.zeros(world * pitch, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(rows, torch.from_numpy(mine.astype(np.int32)))
        grads = np.stack([r.numpy().astype(np.uint16) for r in rows])
        # this rank's shard step (the oracle stands in for the GPU kernel)
        params = np.zeros(world * s, np.uint16)
        p, m, v = (a[begin:begin + n].copy() for a in state0)
        f, p1, m1, v1 = oracle.step_rank(np.ascontiguousarray(grads.reshape(-1)),
                                         world * pitch, rank * pitch, n, world, oracle.F16,
                                         w.bucket, w.loss_scale, h, 1, p, m, v, params, begin)
        skipped = global_skip(bool(f), g)
        assert skipped == plant
        if skipped:
            continue
        # all-gather of the cast parameters
        slot = torch.from_numpy(params[begin:begin + s].astype(np.int32))
        slots = [torch.zeros(s, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(slots, slot)
        gathered = torch.cat(slots).numpy().astype(np.uint16)[:w.psi]
        # ... equals the unsharded data-parallel step
        full = np.stack([synth.grad_values(w, step, j, idx).view(torch.int16).numpy().view(
            np.uint16) for j in range(world)])
        sk, rp, rm, rv, rparams = oracle.step_unsharded(full, oracle.F16, w.loss_scale, h, 1,
                                                        *state0)
        assert not sk
        assert np.array_equal(gathered, rparams)
        assert np.array_equal(p1.view(np.uint32), rp[begin:begin + n].view(np.uint32))
        assert np.array_equal(v1.view(np.uint32), rv[begin:begin + n].view(np.uint32))


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks(world):
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    import oracle
    oracle.build()
    mp.spawn(_worker, args=(world, _free_port()), nprocs=world, join=True)


def _worker_leaves(rank: int, world: int, port: int, result_path: str):
    import datetime
    import sys
    import time
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=3))
    from zero_sharded_optimizer_02_gb300.step import global_skip
    g = dist.group.WORLD
    assert global_skip(False, g) is False          # one step with both ranks
    if rank == 1:
        os._exit(0)                                # rank 1 leaves between steps
    t0 = time.monotonic()
    try:
        global_skip(False, g)                      # the survivor's next skip exchange
        outcome = "completed"
    except Exception as e:                         # the process group reports the loss
        outcome = f"error:{type(e).__name__}"
    with open(result_path, "w") as f:
        f.write(f"{outcome} {time.monotonic() - t0:.2f}")
    os._exit(0)


def test_a_rank_that_leaves_is_detected(tmp_path):
    """A rank leaving between steps: the survivor's next skip exchange ends
    with an error within the process group's timeout instead of hanging."""
    result = tmp_path / "result.txt"
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker_leaves, args=(r, 2, port, str(result))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=60)
        assert not p.is_alive(), "a rank hung"
    outcome, seconds = result.read_text().split()
    assert outcome.startswith("error:"), outcome
    assert float(seconds) < 30
