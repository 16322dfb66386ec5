"""Full-size workloads on the GPU in the launch configuration the benchmark
times, checked against the oracle on sampled elements (the oracle computes
any element on its own from the seeded generator) and through properties that
hold at any size (padding untouched, skip decisions, step count).

Samples include the 16 elements on each side of every cut between two launch
windows of the fused step (the 7.5B shard runs as 12 windows).

Workloads: GPT-2-small-sized ZeRO-2 shard (psi = 124,439,808, Nd = 8, bf16,
10 steps); padding and overflow (psi = 350,000,017, Nd = 16, fp16 x 1024,
all 16 ranks, +inf planted at step 5); GPT-2 1.5B shard view (Nd = 64, fp16,
20 steps); 7.5B shard view (Nd = 64, bf16, bucket 5e8, 20 steps), and its
bucket-ready step in 16 launch groups, its unfused step and its nonfinite
pre-check; the end-to-end forms (rows in pinned host memory) on the 1.5B
shard view.
"""
import dataclasses
import gc

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (assert_params_close, assert_state_close, f32, full_rows, make_group,
                      oracle_trajectory, sample_indices, shard_rows, u16)
from window_rule import inner_cuts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(autouse=True)
def free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _sampled_state(dps, idx, with_params=True):
    """Current state and gathered params of the group at flat indices idx."""
    s = int(dps.layouts[dps.ranks[0]].shard_elems)
    out = [np.empty(idx.size, np.float32) for _ in range(3)]
    params = u16(dps.gathered_view()[torch.from_numpy(idx).to(dps.device)]) if with_params \
        else None
    for r in dps.ranks:
        sel = (idx // s) == r
        if not sel.any():
            continue
        local = torch.from_numpy(idx[sel] - r * s).to(dps.device)
        for i, t in enumerate(dps.state[r].tensors("cur")):
            out[i][sel] = f32(t[local])
    return out, params


def _check(dps, idx, entry, what):
    p, m, v, params, t = entry
    (gp, gm, gv), gparams = _sampled_state(dps, idx)
    assert_state_close(gp, p, 1e-12, f"{what} master")
    assert_state_close(gm, m, 1e-20, f"{what} m")
    assert_state_close(gv, v, 1e-20, f"{what} v")
    if params is not None:
        assert_params_close(gparams, params, f"{what} params")
    assert dps.t == t, what


def _bench_driver(w, rank):
    """The driver configuration bench.py times: PipelinedStep, slot buffers,
    the benchmark's row pitch."""
    from bench import ROW_ALIGN
    from zero_sharded_optimizer_02_gb300.step import PipelinedStep
    dps = PipelinedStep(w.psi, w.nd, [rank], w.grad_dtype, w.hparams, w.loss_scale, w.bucket,
                        "cuda", gathered="slot", row_align=ROW_ALIGN)
    st = dps.state[rank]
    for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
        synth.fill_shard_state(w, rank, which, row)
    return dps


def _slot_params(dps, rank, idx):
    s = int(dps.layouts[rank].shard_elems)
    slot = dps.gathered_view(rank)
    local = torch.from_numpy(idx - rank * s).to(slot.device)
    return u16(slot[local])


@pytest.mark.parametrize("key,rank,bench_cfg", [("c1", 0, False), ("c1", 5, False),
                                                ("c3", 0, False), ("c3", 1, False),
                                                ("c4", 0, True), ("c4", 63, False)])
def test_shard_view_sampled(key, rank, bench_cfg):
    w = synth.WORKLOADS[key]
    dps = _bench_driver(w, rank) if bench_cfg else make_group(w, ranks=[rank])
    idx = sample_indices(w.psi, w.nd, [rank], 2048, seed=rank + 17)
    # every cut between two launch windows of the step is sampled on both sides
    s, b, n = synth.shard_of(w.psi, w.nd, rank)
    cuts = inner_cuts(n)
    assert len(cuts) == z.fused_launch_count(n, w.bucket) - 1
    assert all(np.isin(b + c + np.arange(-16, 16), idx).all() for c in cuts)
    _, hist = oracle_trajectory(w, idx, w.steps)
    buf = None
    for k in range(w.steps):
        if buf is None or w.fresh_grads:
            buf, desc = shard_rows(w, dps, rank, k, buf)
        assert not dps.step(desc)
        if k in (0, w.steps - 1) or w.fresh_grads:
            if bench_cfg:   # slot buffers: the parameters sit at their local index
                p, m, v, params, t = hist[k]
                (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
                assert_state_close(gp, p, 1e-12, f"{key} master step {k}")
                assert_state_close(gm, m, 1e-20, f"{key} m step {k}")
                assert_state_close(gv, v, 1e-20, f"{key} v step {k}")
                assert_params_close(_slot_params(dps, rank, idx), params, f"{key} params")
                assert dps.t == t
            else:
                _check(dps, idx, hist[k], f"{key} rank {rank} step {k}")
    L = dps.layouts[rank]
    n = int(L.length)
    for b in dps.state[rank].bufs:
        assert not b[:, n:].any()


def test_c2_padding_and_overflow_all_ranks():
    w = synth.WORKLOADS["c2"]
    step_plant, j_plant, flat_plant = w.plant
    dps = make_group(w)
    idx = sample_indices(w.psi, w.nd, range(w.nd), 512, seed=2, extra=[flat_plant])
    _, hist = oracle_trajectory(w, idx, w.steps)
    s = int(dps.layouts[0].shard_elems)
    pitch = int(dps.layouts[0].row_pitch)
    buf, desc = full_rows(w, dps, 0)
    for k in range(w.steps):
        if k == step_plant:
            buf[j_plant, (flat_plant // s) * pitch + flat_plant % s] = float("inf")
        skipped = dps.step(desc)
        assert skipped == (k == step_plant), k
        _check(dps, idx, hist[k], f"c2 step {k}")
    assert dps.t == step_plant and dps.skipped_steps == [False] * step_plant + [True]
    # the 15 padding parameters of the last shard are never written
    for g in dps.gathered:
        assert not g[w.psi:].view(torch.int16).any()
    last = dps.layouts[w.nd - 1]
    assert int(last.length) == 21_874_987 and w.nd * s - w.psi == 15


@pytest.mark.parametrize("form", ["zero_copy", "zero_copy_device_params", "fed"])
def test_c3_end_to_end_forms_sampled(form):
    """The benchmark's end-to-end forms on the GPT-2 1.5B shard view (Nd = 64
    fp16 rows, 3 GB): the rows stay in pinned host memory and are either read
    in place by the step (zero-copy, with the new parameters written in place
    to pinned host memory or to device memory) or landed bucket by bucket by
    the feeder while the bucket-ready step consumes them (16 buckets).  Two
    steps, checked on sampled elements against the oracle."""
    w = synth.WORKLOADS["c3"]
    rank = 0
    dps = make_group(w, ranks=[rank], gathered="slot", gathered_on_host=form == "zero_copy")
    if form == "zero_copy":
        assert dps.gathered_view(rank).device.type == "cpu"
        assert dps.gathered_view(rank).is_pinned()
    idx = sample_indices(w.psi, w.nd, [rank], 2048, seed=33)
    _, hist = oracle_trajectory(w, idx, 2)
    buf, desc = shard_rows(w, dps, rank, 0)
    host = torch.empty(buf.shape, dtype=buf.dtype, pin_memory=True)
    host.copy_(buf)
    pitch = int(dps.layouts[rank].row_pitch)
    n = int(dps.layouts[rank].length)
    copy = torch.cuda.Stream()
    bucket = -(-(-(-n // 16)) // 8) * 8
    if form == "fed":
        buf.zero_()                       # the device rows fill as the buckets land
    for k in range(2):
        if form.startswith("zero_copy"):
            assert not dps.step({rank: z.grads(host, pitch, 0, w.nd, w.grad_dtype)})
        else:
            dps.launch_host_fed(rank, host, desc[rank], bucket, copy)
            assert not dps.decide()
            dps.commit(False)
            assert dps.host_fed_status() == 0
        p, m, v, params, t = hist[k]
        (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
        assert_state_close(gp, p, 1e-12, f"{form} master step {k}")
        assert_state_close(gm, m, 1e-20, f"{form} m step {k}")
        assert_state_close(gv, v, 1e-20, f"{form} v step {k}")
        assert_params_close(_slot_params(dps, rank, idx), params, f"{form} params step {k}")
        assert dps.t == t


def test_shard_past_the_int32_range():
    """Rank 1 of two holds 2,147,483,657 elements (2^31 + 9, bf16): every
    element index of the second half is past the int32 range and its flat
    indices pass 2^32; the fused step runs it as 205 launch windows.  Two
    steps, sampled against the oracle at both ends, around every window cut
    and at random points; the state past the shard stays zero.  About 70 GB
    on the device."""
    n = 2 ** 31 + 9
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=2 * n, nd=2, plant=None,
                            bucket=1 << 30, fresh_grads=False, steps=2)
    rank = 1
    dps = make_group(w, ranks=[rank], gathered="slot")
    assert int(dps.layouts[rank].length) == n
    assert z.fused_launch_count(n, w.bucket) == 205
    idx = sample_indices(w.psi, w.nd, [rank], 4096, seed=31,
                         extra=[n + 2 ** 31 - 1, n + 2 ** 31, n + 2 ** 32 - n])
    _, hist = oracle_trajectory(w, idx, 2)
    buf, desc = shard_rows(w, dps, rank, 0)
    for k in range(2):
        assert not dps.step(desc)
        p, m, v, params, t = hist[k]
        (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
        assert_state_close(gp, p, 1e-12, f"master step {k}")
        assert_state_close(gm, m, 1e-20, f"m step {k}")
        assert_state_close(gv, v, 1e-20, f"v step {k}")
        assert_params_close(_slot_params(dps, rank, idx), params, f"params step {k}")
        assert dps.t == t
    for b in dps.state[rank].bufs:
        assert not b[:, n:].any()


def test_7p5b_shard_at_nd_1024():
    """The 7.5B model at Nd = 1,024 (the largest data-parallel degree of the
    pages' Stage-3 memory table): rank 517's shard of 7,324,219 parameters
    folds 1,024 bf16 rows (15 GB).  One step, sampled against the oracle."""
    w = dataclasses.replace(synth.WORKLOADS["c4"], nd=1024, plant=None, steps=1)
    rank = 517
    dps = make_group(w, ranks=[rank], gathered="slot")
    n = int(dps.layouts[rank].length)
    assert n == 7_324_219
    idx = sample_indices(w.psi, w.nd, [rank], 1024, seed=1024)
    _, hist = oracle_trajectory(w, idx, 1)
    buf, desc = shard_rows(w, dps, rank, 0)
    assert not dps.step(desc)
    p, m, v, params, t = hist[0]
    (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
    assert_state_close(gp, p, 1e-12, "master")
    assert_state_close(gm, m, 1e-20, "m")
    assert_state_close(gv, v, 1e-20, "v")
    assert_params_close(_slot_params(dps, rank, idx), params, "params")


def test_7p5b_bucket_ready_step_sampled():
    """The bucket-ready step on the 7.5B shard view (rank 0, Nd = 64 bf16
    rows resident, 15 GB) in the configuration `bench.py --op streamed` times:
    16 transfer buckets, every ready word already set, dealt into launch
    groups of about 1 GB of step traffic, each group behind its own wait
    kernel.  Two steps, sampled against the oracle, with the 16 elements on
    each side of every group boundary in the sample."""
    w = synth.WORKLOADS["c4"]
    rank = 0
    dps = make_group(w, ranks=[rank], gathered="slot")
    L = dps.layouts[rank]
    n, pitch = int(L.length), int(L.row_pitch)
    sb = max(8, -(-(-(-n // 16)) // 8) * 8)            # bench.py's transfer bucket
    groups = z._abi.stream_groups(n, sb, w.nd)
    assert len(groups) == 16 and groups[-1][0] + groups[-1][1] == n
    s, b, _ = synth.shard_of(w.psi, w.nd, rank)
    edges = [b + g0 + d for g0, _ in groups[1:] for d in range(-16, 16)]
    idx = sample_indices(w.psi, w.nd, [rank], 1024, seed=77, extra=edges)
    _, hist = oracle_trajectory(w, idx, 2)
    buf, desc = shard_rows(w, dps, rank, 0)
    ready = torch.ones(-(-n // sb), dtype=torch.int32, device=dps.device)
    status = torch.zeros(1, dtype=torch.int32, device=dps.device)
    st = dps.state[rank]
    for k in range(2):
        gbuf, goff = dps._gathered_target(rank, 1 - dps.gcur)
        dps.h.step = dps.t + 1
        z.zero_step_shard_streamed(desc[rank], L, st.states[st.cur], st.states[1 - st.cur], gbuf,
                                   goff, sb, dps.loss_scale, dps.h, ready, 1, 10 ** 10, dps.flag,
                                   status, dps.stream)
        assert not dps.decide()
        dps.commit(False)
        assert int(status.item()) == 0
        p, m, v, params, t = hist[k]
        (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
        assert_state_close(gp, p, 1e-12, f"master step {k}")
        assert_state_close(gm, m, 1e-20, f"m step {k}")
        assert_state_close(gv, v, 1e-20, f"v step {k}")
        assert_params_close(_slot_params(dps, rank, idx), params, f"params step {k}")
        assert dps.t == t


def test_7p5b_unfused_step_sampled():
    """The unfused step on the 7.5B shard view (rank 0, Nd = 64 bf16 rows) in
    the configuration `bench.py --op unfused` times: one bucket of the whole
    shard through the fusion buffer (469 MB), reduced in 12 launch windows,
    then AdamW and the cast.  Two steps, sampled against the oracle (every
    window cut in the sample)."""
    w = synth.WORKLOADS["c4"]
    rank = 0
    dps = make_group(w, ranks=[rank], gathered="slot", fused=False)
    n = int(dps.layouts[rank].length)
    assert z._abi.unfused_launch_count(n, w.bucket, 0) == 12 + 2
    idx = sample_indices(w.psi, w.nd, [rank], 1024, seed=78)
    _, hist = oracle_trajectory(w, idx, 2)
    buf, desc = shard_rows(w, dps, rank, 0)
    for k in range(2):
        assert not dps.step(desc)
        p, m, v, params, t = hist[k]
        (gp, gm, gv), _ = _sampled_state(dps, idx, with_params=False)
        assert_state_close(gp, p, 1e-12, f"master step {k}")
        assert_state_close(gm, m, 1e-20, f"m step {k}")
        assert_state_close(gv, v, 1e-20, f"v step {k}")
        assert_params_close(_slot_params(dps, rank, idx), params, f"params step {k}")
        assert dps.t == t


def test_7p5b_precheck_flags_a_single_nonfinite_anywhere():
    """The nonfinite pre-check (the read-only pass the benchmark's read
    ceiling times) over the 7.5B shard view's 64 bf16 rows, in its 12 launch
    windows: clean rows leave the flag 0; one +inf, -inf or NaN in any row, at
    a window cut, the first or the last element, sets it."""
    w = synth.WORKLOADS["c4"]
    rank = 0
    dps = make_group(w, ranks=[rank], gathered="slot")
    n = int(dps.layouts[rank].length)
    cuts = inner_cuts(n)
    assert len(cuts) == 11
    buf, desc = shard_rows(w, dps, rank, 0)
    flag = dps.flag

    def check() -> int:
        flag.zero_()
        z.zero_check_nonfinite(desc[rank], 0, n, flag)
        torch.cuda.synchronize()
        return int(flag.item())
    assert check() == 0
    bad = {"+inf": 0x7F80, "-inf": 0xFF80, "nan": 0x7FC1}
    places = [(0, 0), (63, n - 1), (31, cuts[0] - 1), (32, cuts[0]), (17, cuts[5] + 3),
              (63, cuts[-1])]
    for k, (row, e) in enumerate(places):
        code = list(bad.values())[k % 3]
        old = buf[row, e].clone()
        val = torch.from_numpy(np.array([code], np.uint16).view(np.int16)).view(torch.bfloat16)
        buf[row, e] = val[0]
        assert check() == 1, (row, e, hex(code))
        buf[row, e] = old
    assert check() == 0
