"""Concurrent calls: the C ABI is thread-safe and stream-ordered.

include/zero.h promises that every call is thread-safe and that the library
keeps no state a call could trip over.  Here four host threads each own one
rank of an 8-rank group and one CUDA stream, and step their ranks at the same
time, three steps each, on every path that takes no shared workspace: the
fused step on each of its kernels (one kernel per test: the variant is read
from the environment, so all threads share it), the unfused step with its
own fusion buffer per thread, and the reduction primitive.  The binding's
foreign calls release the GIL, so the threads' host code (argument checks,
pointer queries, launches) really runs concurrently.  Every rank's state and
parameters must equal the oracle's, bit for bit.
"""
import dataclasses
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, f32,
                      oracle_trajectory, u16)
from zero_sharded_optimizer_02_gb300.step import DataParallelStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_threads(fn, args_list):
    errors = []
    barrier = threading.Barrier(len(args_list))

    def body(*a):
        try:
            barrier.wait()
            fn(*a)
        except BaseException as e:          # reported on the main thread
            errors.append(e)
    ts = [threading.Thread(target=body, args=a) for a in args_list]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]


@pytest.mark.parametrize("path", ["ring", "tma", "registers", "small", "unfused"])
def test_threads_step_their_own_ranks(path, monkeypatch):
    if path != "unfused":
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=2_000_003, nd=8, plant=None,
                            bucket=100_000)
    steps = 3
    _, hist = oracle_trajectory(w, np.arange(w.psi), steps)
    ranks = [1, 2, 5, 7]
    groups, rows = {}, {}
    for r in ranks:
        dps = DataParallelStep(w.psi, w.nd, [r], w.grad_dtype, w.hparams, w.loss_scale,
                               w.bucket, DEV, gathered="slot", fused=path != "unfused",
                               stream=torch.cuda.Stream())
        st = dps.state[r]
        for row, which in zip(st.bufs[st.cur], ("master", "m", "v")):
            synth.fill_shard_state(w, r, which, row)
        pitch = int(dps.layouts[r].row_pitch)
        bufs = []
        for k in range(steps):
            b = torch.empty(w.nd, pitch, dtype=TORCH_DT[w.grad_dtype], device=DEV)
            synth.fill_shard_rows(w, k, r, b)
            bufs.append(b)
        groups[r], rows[r] = dps, bufs
    torch.cuda.synchronize()

    def run(r):
        dps = groups[r]
        pitch = int(dps.layouts[r].row_pitch)
        for k in range(steps):
            desc = {r: z.grads(rows[r][k], pitch, 0, w.nd, w.grad_dtype)}
            assert not dps.step(desc)
    _run_threads(run, [(r,) for r in ranks])
    torch.cuda.synchronize()
    p, m, v, params, t = hist[-1]
    s = -(-w.psi // w.nd)
    for r in ranks:
        dps = groups[r]
        n = int(dps.layouts[r].length)
        b = r * s
        got = [f32(x) for x in dps.state[r].tensors("cur")]
        for g, ref, name, tau in zip(got, (p, m, v), ("master", "m", "v"),
                                     (1e-12, 1e-20, 1e-20)):
            assert_state_close(g, ref[b:b + n], tau, f"{path} rank {r} {name}")
        assert_params_close(u16(dps.gathered_view(r)[:n]), params[b:b + n],
                            f"{path} rank {r} params")
        assert dps.t == t


def test_threads_reduce_buckets_concurrently():
    """zero_reduce_scatter_bucket from four threads on their own streams, each
    reducing its own buckets of one shard into its own fusion buffer."""
    w = dataclasses.replace(synth.WORKLOADS["c0"], psi=4 * 300_007, nd=4, plant=None)
    r = 1
    s, begin, n = synth.shard_of(w.psi, w.nd, r)
    pitch = synth.pitch_of(s)
    buf = torch.empty(w.nd, pitch, dtype=TORCH_DT[w.grad_dtype], device=DEV)
    synth.fill_shard_rows(w, 0, r, buf)
    host = u16(buf).reshape(-1)
    inv = float(np.float32(1.0 / (w.nd * w.loss_scale)))
    g = z.grads(buf, pitch, 0, w.nd, w.grad_dtype)
    cuts = [0, 70_001, 150_000, 222_223, n]
    outs = [torch.full((cuts[i + 1] - cuts[i],), -1.0, dtype=torch.float32, device=DEV)
            for i in range(4)]
    flags = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in range(4)]
    torch.cuda.synchronize()

    def run(i):
        stream = torch.cuda.Stream()
        for _ in range(5):
            z.zero_reduce_scatter_bucket(g, cuts[i], cuts[i + 1] - cuts[i], inv, outs[i],
                                         flags[i], stream)
        stream.synchronize()
    _run_threads(run, [(i,) for i in range(4)])
    for i in range(4):
        f, ref = oracle.reduce_scaled(host, oracle.dtype_code(w.grad_dtype), pitch, cuts[i],
                                      cuts[i + 1] - cuts[i], w.nd, inv)
        assert np.array_equal(f32(outs[i]).view(np.uint32), ref.view(np.uint32)), i
        assert int(flags[i].item()) == f == 0
