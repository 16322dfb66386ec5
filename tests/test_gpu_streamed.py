"""Bucket-ready stepping (zero_step_shard_streamed) on the GPU.

"ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
section "ZeRO-DP", Stage 2: gradients are reduce-scattered bucket by bucket
during backward, so the optimizer can start on a bucket once it is complete.
A copy stream lands each bucket's contributions and then writes its ready
word; on the compute stream a one-thread kernel waits for each word
(bounded) before the bucket's step launches.  Results must equal the fused
step bit for bit.  A ready word that nothing writes makes the bounded wait
run out: ZERO_ERR_TIMEOUT lands in the status word, the late buckets stay
untouched, and the context stays usable.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, TORCH_DT, f32, make_group, shard_rows, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _setup(psi, nd, rank, dt):
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=psi, nd=nd, grad_dtype=dt,
                            loss_scale=1024.0 if dt == "f16" else 1.0, plant=None)
    dps = make_group(w, ranks=[rank], gathered="full")
    rows, desc = shard_rows(w, dps, rank, 0)
    return w, dps, rows, desc[rank]


def _fused_reference(w, dps, rank, g, bucket):
    L = dps.layouts[rank]
    st = dps.state[rank]
    out = torch.full_like(st.bufs[0], -1.0)
    gath = torch.zeros_like(dps.gathered[0])
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    z.zero_step_shard(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                      w.loss_scale, h, flag)
    torch.cuda.synchronize()
    return out, gath


@pytest.mark.parametrize("group_bytes", [None, "0"])
@pytest.mark.parametrize("psi,nd,rank,dt,bucket", [(400_003, 8, 3, "bf16", 7_000),
                                                   (250_000, 64, 1, "f16", 1_001),
                                                   (90_001, 5, 4, "f16", 90_001)])
def test_streamed_matches_fused(psi, nd, rank, dt, bucket, group_bytes, monkeypatch):
    # default launch groups (here one group of all buckets), and one group a bucket
    if group_bytes is None:
        monkeypatch.delenv("ZERO_STREAM_GROUP_BYTES", raising=False)
    else:
        monkeypatch.setenv("ZERO_STREAM_GROUP_BYTES", group_bytes)
    w, dps, rows, g = _setup(psi, nd, rank, dt)
    out_ref, gath_ref = _fused_reference(w, dps, rank, g, bucket)
    L = dps.layouts[rank]
    n = int(L.length)
    nb = -(-n // bucket)
    host = rows.cpu().pin_memory()
    rows.zero_()                                   # the data arrives bucket by bucket
    ready = torch.zeros(nb, dtype=torch.int32, device=DEV)
    epoch = torch.ones(1, dtype=torch.int32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = dps.state[rank]
    out = torch.full_like(st.bufs[0], -1.0)
    gath = torch.zeros_like(dps.gathered[0])
    compute, copy = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    torch.cuda.synchronize()
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    # consumer first, so it really waits for the producer
    z.zero_step_shard_streamed(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                               w.loss_scale, h, ready, 1, 5_000_000_000, flag, status, compute)
    with torch.cuda.stream(copy):
        for b in range(nb):
            b0, b1 = b * bucket, min(n, (b + 1) * bucket)
            for j in range(nd):
                rows[j, b0:b1].copy_(host[j, b0:b1], non_blocking=True)
            ready[b:b + 1].copy_(epoch, non_blocking=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(flag.item()) == 0
    assert torch.equal(out[:, :n].view(torch.int32), out_ref[:, :n].view(torch.int32))
    b = int(L.begin)
    assert np.array_equal(u16(gath[b:b + n]), u16(gath_ref[b:b + n]))


@pytest.mark.parametrize("bucket", [2 ** 64 - 1, 2 ** 63 + 5])
def test_bucket_near_the_top_of_the_range(bucket):
    """A bucket size near 2^64 is one bucket of the whole shard: the feeder
    lands it with one copy and its ready word, and the bucket-ready step waits
    for that word and steps everything (its bucket count must not wrap)."""
    w, dps, rows, g = _setup(200_003, 4, 2, "bf16")
    out_ref, gath_ref = _fused_reference(w, dps, rank=2, g=g, bucket=64)
    L = dps.layouts[2]
    n = int(L.length)
    host = rows.cpu().pin_memory()
    rows.zero_()
    ready = torch.zeros(1, dtype=torch.int32, device=DEV)
    epoch = torch.ones(1, dtype=torch.int32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = dps.state[2]
    out = torch.full_like(st.bufs[0], -1.0)
    gath = torch.zeros_like(dps.gathered[0])
    compute, copy = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    torch.cuda.synchronize()
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    z.zero_step_shard_streamed(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                               w.loss_scale, h, ready, 1, 5_000_000_000, flag, status, compute)
    z.zero_feed_buckets(host, int(L.row_pitch), g, n, bucket, ready, epoch, copy)
    torch.cuda.synchronize()
    assert int(ready.item()) == 1 and int(status.item()) == 0 and int(flag.item()) == 0
    assert torch.equal(out[:, :n].view(torch.int32), out_ref[:, :n].view(torch.int32))
    b = int(L.begin)
    assert np.array_equal(u16(gath[b:b + n]), u16(gath_ref[b:b + n]))


def test_wait_that_nothing_satisfies_times_out(monkeypatch):
    monkeypatch.setenv("ZERO_STREAM_GROUP_BYTES", "0")     # every bucket its own group
    psi, nd, rank, bucket = 300_000, 4, 0, 10_000
    w, dps, rows, g = _setup(psi, nd, rank, "bf16")
    out_ref, _ = _fused_reference(w, dps, rank, g, bucket)
    L = dps.layouts[rank]
    n = int(L.length)
    nb = -(-n // bucket)
    ready = torch.zeros(nb, dtype=torch.int32, device=DEV)
    ready[:2] = 1                                   # only the first two buckets arrive
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = dps.state[rank]
    out = torch.full_like(st.bufs[0], -1.0)
    gath = torch.zeros_like(dps.gathered[0])
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    torch.cuda.synchronize()
    z.zero_step_shard_streamed(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                               w.loss_scale, h, ready, 1, 20_000_000, flag, status, None)
    torch.cuda.synchronize()
    assert int(status.item()) == z.ZERO_ERR_TIMEOUT
    done = 2 * bucket
    assert torch.equal(out[:, :done].view(torch.int32), out_ref[:, :done].view(torch.int32))
    assert bool((out[:, done:n] == -1.0).all()), "a late bucket was touched"
    # the context is still usable: the same step completes once the words are set
    ready.fill_(1)
    status.zero_()
    z.zero_step_shard_streamed(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                               w.loss_scale, h, ready, 1, 20_000_000, flag, status, None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out[:, :n].view(torch.int32), out_ref[:, :n].view(torch.int32))


def test_streamed_rejects_unbounded_waits():
    psi, nd, rank = 1000, 2, 0
    w, dps, rows, g = _setup(psi, nd, rank, "bf16")
    L = dps.layouts[rank]
    st = dps.state[rank]
    ready = torch.ones(1, dtype=torch.int32, device=DEV)
    h = z.adamw(1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    for timeout in (0, 61_000_000_000):
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_shard_streamed(g, L, st.states[0], st.states[1], dps.gathered[1], 0,
                                       1000, 1.0, h, ready, 1, timeout, dps.flag, dps.flag)
        assert e.value.status == z.ZERO_ERR_INVALID_ARG


def test_host_fed_step_matches_fused():
    """The driver's host-fed step (feeder + bucket-ready kernel) gives the
    fused step's result; two steps in a row reuse the ready words (epochs)."""
    psi, nd, rank, bucket = 500_001, 16, 5, 4_096
    w, dps, rows, g = _setup(psi, nd, rank, "bf16")
    ref = make_group(w, ranks=[rank], gathered="full")
    host = rows.cpu().pin_memory()
    rows.zero_()
    copy = torch.cuda.Stream(DEV)
    for step in range(2):
        rrows, rdesc = shard_rows(w, ref, rank, 0)
        assert not ref.step(rdesc)
        dps.launch_host_fed(rank, host, g, bucket, copy)
        assert not dps.decide()
        dps.commit(False)
        assert dps.host_fed_status() == 0
        for a, b in zip(dps.state[rank].tensors(), ref.state[rank].tensors()):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), step
        L = dps.layouts[rank]
        lo, hi = int(L.begin), int(L.begin) + int(L.length)
        assert torch.equal(dps.gathered_view()[lo:hi].view(torch.int16),
                           ref.gathered_view()[lo:hi].view(torch.int16))


def test_feeder_rejects_short_rows():
    psi, nd, rank = 1000, 2, 0
    w, dps, rows, g = _setup(psi, nd, rank, "bf16")
    host = torch.zeros(nd, 10, dtype=torch.bfloat16).pin_memory()
    ready = torch.zeros(4, dtype=torch.int32, device=DEV)
    ep = torch.ones(1, dtype=torch.int32).pin_memory()
    with pytest.raises(z.ZeroError) as e:
        z.zero_feed_buckets(host, 10, g, 500, 128, ready, ep, None)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG


def test_a_group_waits_for_all_its_buckets(monkeypatch):
    """With the default grouping the 8 small buckets form one launch group:
    one bucket that never lands keeps the whole group untouched."""
    monkeypatch.delenv("ZERO_STREAM_GROUP_BYTES", raising=False)
    psi, nd, rank, bucket = 300_000, 4, 0, 10_000
    w, dps, rows, g = _setup(psi, nd, rank, "bf16")
    L = dps.layouts[rank]
    n = int(L.length)
    assert len(z._abi.stream_groups(n, bucket, nd)) == 1
    ready = torch.ones(-(-n // bucket), dtype=torch.int32, device=DEV)
    ready[-1] = 0                                   # the last bucket never arrives
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = dps.state[rank]
    out = torch.full_like(st.bufs[0], -1.0)
    gath = torch.zeros_like(dps.gathered[0])
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    torch.cuda.synchronize()
    z.zero_step_shard_streamed(g, L, st.states[st.cur], z.state(*out), gath, L.begin, bucket,
                               w.loss_scale, h, ready, 1, 20_000_000, flag, status, None)
    torch.cuda.synchronize()
    assert int(status.item()) == z.ZERO_ERR_TIMEOUT
    assert bool((out[:, :n] == -1.0).all()), "a bucket of an incomplete group was touched"

