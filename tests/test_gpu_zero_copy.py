"""Gradient contributions read in place from page-locked host memory.

On a Grace-Blackwell node the GPU reads page-locked host memory over the
host link at the link's bandwidth, so a rank's step can take its Nd
contributions straight from host memory without a device copy of them.  The
results must be those of the same contributions in device memory, and a
pointer the GPU cannot read (pageable host memory) must be refused before
anything is launched.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, flat_state,
                      full_rows, make_group, oracle_trajectory, shard_rows, u16)

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


def test_host_rows_over_several_launch_windows_equal_device_rows():
    """A 30,000,003-element shard (two launch windows of the fused step),
    Nd = 2 bf16: host-resident and device-resident contributions give
    bitwise the same state and parameters."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=60_000_005, nd=2, plant=None,
                            bucket=1 << 30)
    assert z.fused_launch_count(30_000_003, 1 << 30) == 2
    out = []
    for where in ("device", "host"):
        dps = make_group(w, ranks=[0], gathered="slot")
        buf, desc = shard_rows(w, dps, 0, 0)
        if where == "host":
            host = _pinned_copy(buf)
            del buf
            desc = {0: z.grads(host, int(dps.layouts[0].row_pitch), 0, w.nd, w.grad_dtype)}
        assert not dps.step(desc)
        n = int(dps.layouts[0].length)
        out.append([t.cpu().numpy().tobytes() for t in dps.state[0].tensors("cur")] +
                   [u16(dps.gathered_view(0)[:n]).tobytes()])
        del dps
        torch.cuda.empty_cache()
    assert out[0] == out[1]


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
