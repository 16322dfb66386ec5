"""The step drivers when a bounded device wait expires.

A bucket-ready step whose copies have not landed when its wait runs out
(ZERO_ERR_TIMEOUT in the status word), and a step kernel that reports an
expired pipeline wait (the ZERO_STEP_FLAG_WAIT_TIMEOUT bit of the flag):
the driver raises ZeroError(ZERO_ERR_TIMEOUT) after the skip decision, the
committed state stays, and the next steps run as if the failed one had
never been launched.  The waits here expire for real (the copies are held
behind a sleeping kernel on another stream) or are reported by a wrapper
that sets the flag bit after the real kernels: no GPU is faulted or hung.
"""
import dataclasses
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, make_group, shard_rows
from zero_sharded_optimizer_02_gb300 import _abi, step as step_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _w(psi=200_003, nd=8):
    return dataclasses.replace(synth.WORKLOADS["c1"], psi=psi, nd=nd, plant=None)


def _equal_state(a, b, rank):
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32))
               for x, y in zip(a.state[rank].tensors(), b.state[rank].tensors()))


def test_host_fed_wait_expiry_raises_and_keeps_the_state():
    w, rank, bucket = _w(), 1, 4096
    dps = make_group(w, ranks=[rank], gathered="full")
    rows, desc = shard_rows(w, dps, rank, 0)
    host = rows.cpu().pin_memory()
    rows.zero_()
    copy, blocker = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    # one ordinary host-fed step first: it also loads every kernel the step
    # uses, since loading a kernel on first launch can wait for the kernels
    # already running (the sleeping one below) and delay the wait kernel
    dps.launch_host_fed(rank, host, desc[rank], bucket, copy)
    assert not dps.decide()
    dps.commit(False)
    before = [t.clone() for t in dps.state[rank].tensors()]
    torch.cuda._sleep(1000)
    torch.cuda.synchronize()
    with torch.cuda.stream(blocker):
        torch.cuda._sleep(200_000_000)          # ~0.1 s; the copies queue behind it
    held = torch.cuda.Event()
    held.record(blocker)
    copy.wait_event(held)
    dps.launch_host_fed(rank, host, desc[rank], bucket, copy, timeout_ns=1_000_000)
    with pytest.raises(z.ZeroError) as e:
        dps.decide()
    assert e.value.status == z.ZERO_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert dps.t == 1 and int(dps.flag.item()) == 0 and dps.host_fed_status() == 0
    for a, b in zip(before, dps.state[rank].tensors()):
        assert torch.equal(a, b)
    # the next step runs normally: two committed steps, as the fused driver's
    dps.launch_host_fed(rank, host, desc[rank], bucket, copy)
    assert not dps.decide()
    dps.commit(False)
    ref = make_group(w, ranks=[rank], gathered="full")
    _, rdesc = shard_rows(w, ref, rank, 0)
    for _ in range(2):
        assert not ref.step(rdesc)
    assert dps.t == ref.t == 2 and _equal_state(dps, ref, rank)


def _flag_timeout_on(calls: set, monkeypatch):
    """zero_step_shard as usual, then the wait-expired bit set in the flag
    word on the same stream for the call numbers in `calls` (0-based)."""
    real = _abi.zero_step_shard
    count = [0]

    def wrapper(g, L, s_in, s_out, gathered, goff, bucket, ls, h, flag, stream=None):
        real(g, L, s_in, s_out, gathered, goff, bucket, ls, h, flag, stream)
        if count[0] in calls:
            with torch.cuda.stream(stream):
                flag.fill_(_abi.ZERO_STEP_FLAG_WAIT_TIMEOUT - (1 << 32))   # as int32
        count[0] += 1
    monkeypatch.setattr(_abi, "zero_step_shard", wrapper)


def test_step_kernel_wait_expiry_in_the_synchronous_driver(monkeypatch):
    w, rank = _w(), 2
    dps = make_group(w, ranks=[rank], gathered="slot")
    ref = make_group(w, ranks=[rank], gathered="slot")
    _, desc = shard_rows(w, dps, rank, 0)
    _, rdesc = shard_rows(w, ref, rank, 0)
    _flag_timeout_on({1}, monkeypatch)
    assert not dps.step(desc)
    with pytest.raises(z.ZeroError) as e:
        dps.step(desc)
    assert e.value.status == z.ZERO_ERR_TIMEOUT
    assert dps.t == 1 and int(dps.flag.item()) == 0
    assert not dps.step(desc)
    monkeypatch.undo()
    for _ in range(2):
        assert not ref.step(rdesc)
    assert dps.t == ref.t == 2 and _equal_state(dps, ref, rank)


def test_step_kernel_wait_expiry_in_the_pipelined_driver(monkeypatch):
    w, rank = _w(), 3
    dps = step_mod.PipelinedStep(w.psi, w.nd, [rank], w.grad_dtype, w.hparams, w.loss_scale,
                                 w.bucket, DEV, gathered="slot", depth=2)
    ref = make_group(w, ranks=[rank], gathered="slot")
    for d in (dps, ref):
        st = d.state[rank]
        for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
            synth.fill_shard_state(w, rank, which, row)
    _, desc = shard_rows(w, dps, rank, 0)
    _, rdesc = shard_rows(w, ref, rank, 0)
    _flag_timeout_on({1}, monkeypatch)        # the second launched step
    # depth 2: the third launch decides step 1, the fourth decides step 2
    decided = dps.launch(desc) + dps.launch(desc) + dps.launch(desc)
    assert decided == [False] and dps.t == 1
    with pytest.raises(z.ZeroError) as e:
        dps.launch(desc)
    assert e.value.status == z.ZERO_ERR_TIMEOUT
    assert dps.t == 1 and dps.pending == []
    assert not dps.step(desc)                 # the driver carries on from step 1
    monkeypatch.undo()
    for _ in range(2):
        assert not ref.step(rdesc)
    assert dps.t == ref.t == 2
    assert all(torch.equal(a.view(torch.int32), b.view(torch.int32))
               for a, b in zip(dps.state[rank].tensors(), ref.state[rank].tensors()))
    assert int(dps.flags.abs().sum().item()) == 0


def test_first_host_fed_step_of_a_process_completes():
    """The first bucket-ready step of a fresh process, whose kernels are not
    loaded yet (CUDA's lazy loading), lands within its wait limit: the
    library loads every kernel it will launch before the first wait starts,
    so loading cannot wait for that wait while the copies it needs are not
    yet issued."""
    tests = os.path.dirname(os.path.abspath(__file__))
    script = textwrap.dedent(f"""
        import dataclasses, sys, time
        sys.path[:0] = [{os.path.dirname(tests)!r}, {tests!r}]
        import torch
        import synth
        from gpu_util import make_group, shard_rows
        w = dataclasses.replace(synth.WORKLOADS["c1"], psi=200_003, nd=8, plant=None)
        dps = make_group(w, ranks=[1], gathered="full")
        rows, desc = shard_rows(w, dps, 1, 0)
        host = rows.cpu().pin_memory()
        rows.zero_()
        copy = torch.cuda.Stream()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dps.launch_host_fed(1, host, desc[1], 4096, copy, timeout_ns=3_000_000_000)
        assert not dps.decide()
        print("elapsed", time.perf_counter() - t0)
    """)
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    out = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                         timeout=300, env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    elapsed = float(out.stdout.split("elapsed")[-1])
    assert elapsed < 2.0, elapsed
