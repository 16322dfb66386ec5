"""Gradient contributions read, and cast parameters written, in place in
page-locked host memory.

On a Grace-Blackwell node the GPU reads and writes page-locked host memory
over the host link at the link's bandwidth, so a rank's step can take its Nd
contributions straight from host memory, and return its new parameters
there, without device copies of either.  The results must be those of the
same step in device memory, and a pointer the GPU cannot use (pageable host
memory) must be refused before anything is launched.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, flat_state,
                      full_rows, make_group, oracle_shard_step, oracle_trajectory, shard_rows,
                      u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _pinned_copy(buf: torch.Tensor) -> torch.Tensor:
    host = torch.empty(buf.shape, dtype=buf.dtype, pin_memory=True)
    host.copy_(buf)
    return host


@pytest.mark.parametrize("fused", [True, False])
def test_host_rows_match_the_oracle(fused):
    """The 4-rank fp16 workload, every rank's contributions in pinned host
    memory (full emulation: rank r reads its slice of every row)."""
    w = synth.WORKLOADS["c0"]
    dps = make_group(w, fused=fused)
    idx = np.arange(w.psi)
    _, hist = oracle_trajectory(w, idx, 2)
    pitch = int(dps.layouts[0].row_pitch)
    buf = None
    for k in range(2):
        buf, _ = full_rows(w, dps, k, buf)
        host = _pinned_copy(buf)
        desc = {r: z.grads(host, w.nd * pitch, r * pitch, w.nd, w.grad_dtype)
                for r in dps.ranks}
        assert not dps.step(desc)
        p, m, v, params, t = hist[k]
        gp, gm, gv = flat_state(dps)
        assert_state_close(gp, p, 1e-12, f"step {k} master")
        assert_state_close(gm, m, 1e-20, f"step {k} m")
        assert_state_close(gv, v, 1e-20, f"step {k} v")
        assert_params_close(u16(dps.gathered_view()[:w.psi]), params, f"step {k} params")
        assert dps.t == t


def test_host_rows_over_several_launch_windows_match_oracle():
    """A 30,000,003-element shard (three launch windows of the fused step),
    Nd = 2 bf16: host-resident and device-resident contributions each give
    the oracle's state and parameters over the whole shard."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=60_000_005, nd=2, plant=None,
                            bucket=1 << 30)
    assert z.fused_launch_count(30_000_003, 1 << 30) == 3
    f, rp, rm, rv, rparams = oracle_shard_step(w, 0)
    assert f == 0
    for where in ("device", "host"):
        dps = make_group(w, ranks=[0], gathered="slot")
        buf, desc = shard_rows(w, dps, 0, 0)
        if where == "host":
            host = _pinned_copy(buf)
            del buf
            desc = {0: z.grads(host, int(dps.layouts[0].row_pitch), 0, w.nd, w.grad_dtype)}
        assert not dps.step(desc)
        n = int(dps.layouts[0].length)
        got = [t.cpu().numpy() for t in dps.state[0].tensors("cur")]
        for g, ref, name, tau in zip(got, (rp, rm, rv), ("master", "m", "v"),
                                     (1e-12, 1e-20, 1e-20)):
            assert_state_close(g, ref, tau, f"{where} rows {name}")
        assert_params_close(u16(dps.gathered_view(0)[:n]), rparams, f"{where} rows params")
        del dps
        torch.cuda.empty_cache()


def test_primitives_read_host_rows():
    """zero_reduce_scatter_bucket and zero_check_nonfinite on host rows: the
    same fp32 bucket as from device rows, and a planted +inf is seen."""
    w = synth.WORKLOADS["c0"]
    dps = make_group(w, ranks=[2], gathered="slot")
    buf, desc = shard_rows(w, dps, 2, 0)
    host = _pinned_copy(buf)
    pitch = int(dps.layouts[2].row_pitch)
    gd = desc[2]
    gh = z.grads(host, pitch, 0, w.nd, w.grad_dtype)
    n = int(dps.layouts[2].length)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    cb_d = torch.empty(n, dtype=torch.float32, device=DEV)
    cb_h = torch.empty(n, dtype=torch.float32, device=DEV)
    inv = 1.0 / (w.nd * w.loss_scale)
    z.zero_reduce_scatter_bucket(gd, 0, n, inv, cb_d, flag)
    z.zero_reduce_scatter_bucket(gh, 0, n, inv, cb_h, flag)
    torch.cuda.synchronize()
    assert torch.equal(cb_d.view(torch.int32), cb_h.view(torch.int32))
    assert int(flag.item()) == 0
    host[3, n // 2] = float("inf")
    z.zero_check_nonfinite(gh, 0, n, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) != 0


def test_pageable_host_rows_are_refused():
    w = synth.WORKLOADS["c0"]
    dps = make_group(w, ranks=[1], gathered="slot")
    pitch = int(dps.layouts[1].row_pitch)
    pageable = torch.zeros(w.nd, pitch, dtype=TORCH_DT[w.grad_dtype])
    assert not pageable.is_pinned()
    before = [t.clone() for t in dps.state[1].tensors("cur")]
    desc = {1: z.grads(pageable, pitch, 0, w.nd, w.grad_dtype)}
    for fused in (True, False):
        dps.fused = fused
        if not fused:
            dps.cb_elems = pitch + 4
            dps.cb = torch.empty(dps.cb_elems, dtype=torch.float32, device=DEV)
        with pytest.raises(z.ZeroError) as e:
            dps.launch(desc)
        assert e.value.status == z.ZERO_ERR_INVALID_ARG
    with pytest.raises(z.ZeroError) as e:
        z.zero_check_nonfinite(desc[1], 0, 16, dps.flag)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(dps.flag.item()) == 0
    for a, b in zip(before, dps.state[1].tensors("cur")):
        assert torch.equal(a, b)


@pytest.mark.parametrize("path", ["ring", "registers", "tma", "small", "unfused"])
def test_host_params_equal_device_params(path, monkeypatch):
    """Every rank's cast parameters written into one flat gathered buffer in
    pinned host memory (16 ranks, S mod 8 = 3: every slot phase; buckets of
    7), contributions in device or host memory: the same state and
    parameters, bit for bit, as with the buffer in device memory."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=70_001, nd=16, grad_dtype="f16",
                            loss_scale=1024.0, plant=None)
    if path != "unfused":
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    out = {}
    for params_on_host in (False, True):
        for rows_on_host in (False, True):
            dps = make_group(w, fused=path != "unfused", bucket=7,
                             gathered_on_host=params_on_host)
            assert dps.gathered_view().is_pinned() == params_on_host
            pitch = int(dps.layouts[0].row_pitch)
            buf = None
            for k in range(2):
                buf, desc = full_rows(w, dps, k, buf)
                if rows_on_host:
                    host = _pinned_copy(buf)
                    desc = {r: z.grads(host, w.nd * pitch, r * pitch, w.nd, w.grad_dtype)
                            for r in dps.ranks}
                assert not dps.step(desc)
            got = [a.tobytes() for a in flat_state(dps)] + \
                [u16(dps.gathered_view()).tobytes()]
            out[params_on_host, rows_on_host] = got
    first = out[False, False]
    for key, got in out.items():
        assert got == first, key


def test_host_params_streamed_and_cast():
    """The bucket-ready step and the standalone cast write a pinned host slot
    at an odd element phase: the bytes of the device-memory results, and the
    guard elements on either side untouched."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=8 * 30_001 + 3, nd=8, plant=None)
    rank = 5
    dps = make_group(w, ranks=[rank], gathered="slot")
    buf, desc = shard_rows(w, dps, rank, 0)
    L = dps.layouts[rank]
    n = int(L.length)
    st = dps.state[rank]
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    bucket = 6_001
    ready = torch.ones(-(-n // bucket), dtype=torch.int32, device=DEV)
    results = []
    for on_host in (False, True):
        slot = torch.full((n + 10,), 0x5A5A, dtype=torch.int16,
                          **({"pin_memory": True} if on_host else {"device": DEV}))
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        s_out = z.state(*(torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(3)))
        z.zero_step_shard_streamed(desc[rank], L, st.states[st.cur], s_out, slot, 3, bucket,
                                   w.loss_scale, h, ready, 1, 10 ** 9, flag, status)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0 and int(status.item()) == 0
        cast = torch.full((n + 10,), 0x5A5A, dtype=torch.int16,
                          **({"pin_memory": True} if on_host else {"device": DEV}))
        master = dps.state[rank].tensors("cur")[0]
        z.zero_gather_params_shard(master, n, cast, 5, w.grad_dtype)
        torch.cuda.synchronize()
        results.append((slot.cpu().numpy().tobytes(), cast.cpu().numpy().tobytes()))
        for t, off in ((slot, 3), (cast, 5)):
            c = t.cpu()
            assert (c[:off] == 0x5A5A).all() and (c[off + n:] == 0x5A5A).all()
    assert results[0] == results[1]


def test_pageable_params_are_refused():
    """A gathered buffer in pageable host memory: every entry point that writes
    parameters returns ZERO_ERR_INVALID_ARG and launches nothing."""
    w = synth.WORKLOADS["c0"]
    rank = 1
    dps = make_group(w, ranks=[rank], gathered="slot")
    buf, desc = shard_rows(w, dps, rank, 0)
    L = dps.layouts[rank]
    n = int(L.length)
    st = dps.state[rank]
    before = [t.clone() for t in st.tensors("cur")]
    pageable = torch.zeros(n + 8, dtype=TORCH_DT[w.grad_dtype])
    assert not pageable.is_pinned()
    s_out = st.states[1 - st.cur]
    out_before = [t.clone() for t in st.tensors("next")]
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    cb = torch.empty(n + 4, dtype=torch.float32, device=DEV)
    ready = torch.ones(1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    calls = [
        lambda: z.zero_step_shard(desc[rank], L, st.states[st.cur], s_out, pageable, 0, w.bucket,
                                  w.loss_scale, h, dps.flag),
        lambda: z.zero_step_shard_unfused(desc[rank], L, st.states[st.cur], s_out, pageable, 0,
                                          w.bucket, w.loss_scale, h, cb, n + 4, dps.flag),
        lambda: z.zero_step_shard_unfused_static(desc[rank], L, st.states[st.cur], s_out,
                                                 pageable, 0, w.bucket, w.loss_scale, h,
                                                 dps.flag),
        lambda: z.zero_step_shard_streamed(desc[rank], L, st.states[st.cur], s_out, pageable, 0,
                                           n, w.loss_scale, h, ready, 1, 10 ** 9, dps.flag,
                                           status),
        lambda: z.zero_gather_params_shard(st.tensors("cur")[0], n, pageable, 0, w.grad_dtype),
    ]
    for call in calls:
        with pytest.raises(z.ZeroError) as e:
            call()
        assert e.value.status == z.ZERO_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(dps.flag.item()) == 0 and int(status.item()) == 0
    assert not pageable.any()
    for a, b in zip(before, st.tensors("cur")):
        assert torch.equal(a, b)
    for a, b in zip(out_before, st.tensors("next")):
        assert torch.equal(a, b)
