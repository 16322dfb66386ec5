"""Stage variants on the GPU, against the oracle.

"ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
section "ZeRO-DP": Stage 1 partitions only the optimizer state -- every rank
holds the whole gradient after a data-parallel all-reduce and steps its own
shard from it; Stage 2 reduce-scatters, so each owner folds the Nd
contributions to its shard only.  The ZeRO summary's DeepSpeed note says its
Stage 2 all-reduces by default: with the fixed rank-order fold, reducing the
whole row (all-reduce) gives every owner exactly its reduce-scatter result.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, f32, full_rows,
                      make_group, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_stage1_prereduced_gradient(dt):
    """Every rank steps its shard from the one all-reduced gradient row."""
    nd, psi = 8, 300_001
    ls = 1024.0 if dt == "f16" else 1.0
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=psi, nd=nd, grad_dtype=dt,
                            loss_scale=ls, plant=None)
    dps = make_group(w, gathered="full", bucket=50_000)
    s, pitch = int(dps.layouts[0].shard_elems), int(dps.layouts[0].row_pitch)
    # the all-reduced gradient: one row in padded-partition layout
    row = torch.zeros(1, nd * pitch, dtype=TORCH_DT[dt], device=DEV)
    w1 = dataclasses.replace(w, nd=1)
    for r in range(nd):
        n = int(dps.layouts[r].length)
        idx = torch.arange(r * s, r * s + n, dtype=torch.int64, device=DEV)
        row[0, r * pitch:r * pitch + n] = synth.grad_values(w1, 0, 0, idx)
    desc = {r: z.grads(row, nd * pitch, r * pitch, 1, dt) for r in range(nd)}
    dps.loss_scale = ls * nd            # keeps the 1/Nd averaging of the summed gradient
    assert not dps.step(desc)
    host = u16(row).reshape(-1)
    flat_params = np.zeros(nd * s, np.uint16)
    for r in range(nd):
        L = dps.layouts[r]
        n, b = int(L.length), int(L.begin)
        idx = torch.arange(b, b + n, dtype=torch.int64)
        p0, m0, v0 = (synth.state_values(w, k, idx).numpy() for k in ("master", "m", "v"))
        f, p1, m1, v1 = oracle.step_rank(host, nd * pitch, r * pitch, n, 1, oracle.dtype_code(dt),
                                         50_000, ls * nd, w.hparams, 1, p0, m0, v0, flat_params, b)
        assert f == 0
        gp, gm, gv = (f32(t) for t in dps.state[r].tensors())
        assert_state_close(gp, p1, 1e-12, f"stage1 rank {r} master")
        assert_state_close(gm, m1, 1e-20, f"stage1 rank {r} m")
        assert_state_close(gv, v1, 1e-20, f"stage1 rank {r} v")
    assert_params_close(u16(dps.gathered_view()[:psi]), flat_params[:psi], "stage1 params")


def test_all_reduce_gives_every_owner_its_reduce_scatter():
    nd, psi = 16, 500_003
    w = dataclasses.replace(synth.WORKLOADS["c2"], psi=psi, nd=nd, plant=None)
    dps = make_group(w, gathered="full")
    buf, _ = full_rows(w, dps, 0)
    s, pitch = int(dps.layouts[0].shard_elems), int(dps.layouts[0].row_pitch)
    inv = float(np.float32(1.0 / (nd * w.loss_scale)))
    g = z.grads(buf, nd * pitch, 0, nd, w.grad_dtype)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    allred = [torch.empty(nd * pitch, dtype=torch.float32, device=DEV) for _ in range(2)]
    for a in allred:                       # the whole row, twice (two "ranks")
        z.zero_reduce_scatter_bucket(g, 0, nd * pitch, inv, a, flag)
    torch.cuda.synchronize()
    assert torch.equal(allred[0].view(torch.int32), allred[1].view(torch.int32))
    host = u16(buf).reshape(-1)
    for r in range(nd):
        n = int(dps.layouts[r].length)
        cb = torch.empty(max(n, 1), dtype=torch.float32, device=DEV)
        z.zero_reduce_scatter_bucket(z.grads(buf, nd * pitch, r * pitch, nd, w.grad_dtype), 0, n,
                                     inv, cb, flag)
        torch.cuda.synchronize()
        seg = allred[0][r * pitch:r * pitch + n]
        assert torch.equal(seg.view(torch.int32), cb[:n].view(torch.int32)), r
        f, ref = oracle.reduce_scaled(host, oracle.F16, nd * pitch, r * pitch, n, nd, inv)
        assert np.array_equal(f32(cb[:n]).view(np.uint32), ref.view(np.uint32))
    assert int(flag.item()) == 0
