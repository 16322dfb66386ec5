"""GPU parity of the whole shard step (zero_step_shard, zero_step_shard_unfused)
against the oracle's unsharded data-parallel step, element by element.

The invariant checked is the one ZeRO-DP rests on ("ZeRO: Memory Optimizations
Toward Training Trillion Parameter Models", section "ZeRO-DP", Stage 1: each
rank updates only its 1/Nd): running every rank's shard step on the GPU and
concatenating the shards gives the unsharded step of the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, DT_CODE, EDGE_CASES, TORCH_DT, assert_params_close,
                      assert_state_close, check_against_oracle, f32, flat_state, full_rows,
                      make_group, oracle_trajectory, shard_rows, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_generator_identical_on_device():
    for key in ("c0", "c2", "c4"):
        w = synth.WORKLOADS[key]
        idx = torch.tensor([0, 1, 5, 1 << 20, w.psi - 1, w.psi // 3], dtype=torch.int64)
        for j in (0, w.nd - 1):
            a = synth.grad_values(w, 0, j, idx)
            b = synth.grad_values(w, 0, j, idx.to(DEV)).cpu()
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        for which in ("master", "m", "v"):
            assert torch.equal(synth.state_values(w, which, idx),
                               synth.state_values(w, which, idx.to(DEV)).cpu())


@pytest.mark.parametrize("fused", [True, False])
def test_c0_full_emulation_matches_unsharded_oracle(fused):
    """Tiny ZeRO-2 step: psi = 1,048,576, Nd = 4, fp16 grads with loss scale
    1024, bucket 65,536 (4 buckets a shard), 3 steps, fresh grads a step."""
    w = synth.WORKLOADS["c0"]
    dps = make_group(w, fused=fused)
    _, hist = oracle_trajectory(w, np.arange(w.psi), w.steps)
    buf = None
    for k in range(w.steps):
        buf, desc = full_rows(w, dps, k, buf)
        assert not dps.step(desc)
        check_against_oracle(w, dps, hist[k], f"c0 step {k} fused={fused}")




@pytest.mark.parametrize("psi,nd,dt,bucket", EDGE_CASES)
@pytest.mark.parametrize("fused", [True, False])
def test_edge_shapes(psi, nd, dt, bucket, fused):
    w = dataclasses.replace(synth.WORKLOADS["c1"], grad_dtype=dt,
                            loss_scale=1024.0 if dt == "f16" else 1.0, plant=None)
    dps = make_group(w, fused=fused, bucket=bucket, psi=psi, nd=nd)
    _, hist = oracle_trajectory(w, np.arange(psi), 2, psi=psi, nd=nd)
    buf = None
    for k in range(2):
        buf, desc = full_rows(w, dps, k, buf)
        assert not dps.step(desc)
        check_against_oracle(dataclasses.replace(w, psi=psi, nd=nd), dps, hist[k],
                              f"psi={psi} nd={nd} step {k}")


def test_bucket_size_invariance():
    w = synth.WORKLOADS["c0"]
    ref = None
    for bucket, fused in ((65_536, True), (7, True), (1 << 30, True), (1000, False),
                          (262_144, False)):
        dps = make_group(w, fused=fused, bucket=bucket)
        buf, desc = full_rows(w, dps, 0)
        dps.step(desc)
        cur = [a.tobytes() for a in flat_state(dps)] + [u16(dps.gathered_view()).tobytes()]
        ref = ref or cur
        assert cur == ref, (bucket, fused)


@pytest.mark.parametrize("fused", [True, False])
def test_global_skip_keeps_everything(fused):
    """A single +inf in one rank's contribution skips the step on every shard:
    state, gathered parameters and t stay bitwise unchanged."""
    w = dataclasses.replace(synth.WORKLOADS["c2"], psi=100_003, nd=16, plant=None,
                            fresh_grads=True)
    dps = make_group(w, fused=fused, bucket=4096)
    buf, desc = full_rows(w, dps, 0)
    assert not dps.step(desc)
    before = [a.copy() for a in flat_state(dps)] + [u16(dps.gathered_view()).copy()]
    s = int(dps.layouts[0].shard_elems)
    pitch = int(dps.layouts[0].row_pitch)
    buf, desc = full_rows(w, dps, 1, buf)
    buf[7, 7 * pitch + s // 2] = float("inf")       # rank 7's contribution, rank 7's chunk
    assert dps.step(desc)
    after = [a.copy() for a in flat_state(dps)] + [u16(dps.gathered_view()).copy()]
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
    assert dps.t == 1 and dps.skipped_steps == [False, True]
    assert int(dps.flag.item()) == 0                 # cleared after the skip
    # the next clean step commits and matches the oracle run that skipped too
    buf, desc = full_rows(w, dps, 2, buf)
    assert not dps.step(desc)
    idx = np.arange(w.psi)
    I = torch.from_numpy(idx)
    tr = oracle.Trajectory(DT_CODE[w.grad_dtype], w.loss_scale, w.hparams,
                           *(synth.state_values(w, k, I).numpy() for k in ("master", "m", "v")))
    for k in (0, 1, 2):
        rows = np.stack([u16(synth.grad_values(w, k, j, I)) for j in range(w.nd)])
        if k == 1:
            rows[7, 7 * s + s // 2] = 0x7C00
        tr.step(rows)
    assert tr.skipped == [False, True, False]
    check_against_oracle(w, dps, (tr.p, tr.m, tr.v, tr.params, tr.t), "after skip")


def test_in_place_with_precheck():
    """out == in updates in place; zero_check_nonfinite decides first."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=50_001, nd=8, plant=None)
    dps = make_group(w, ranks=[3], gathered="slot")
    L = dps.layouts[3]
    buf, desc = shard_rows(w, dps, 3, 0)
    st = dps.state[3]
    s_cur = st.states[st.cur]
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    z.zero_check_nonfinite(desc[3], 0, int(L.length), flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    gath = torch.zeros(int(L.shard_elems) + 8, dtype=TORCH_DT[w.grad_dtype], device=DEV)
    z.zero_step_shard(desc[3], L, s_cur, s_cur, gath, 0, 4096, w.loss_scale,
                      z.adamw(1e-4, 0.9, 0.999, 1e-8, 0.01, 1), flag)
    torch.cuda.synchronize()
    n = int(L.length)
    idx = np.arange(int(L.begin), int(L.begin) + n)
    _, hist = oracle_trajectory(w, idx, 1)
    p, m, v = (f32(t) for t in st.tensors("cur"))
    assert_state_close(p, hist[0][0], 1e-12, "in-place master")
    assert_state_close(m, hist[0][1], 1e-20, "in-place m")
    assert_state_close(v, hist[0][2], 1e-20, "in-place v")
    assert_params_close(u16(gath[:n]), hist[0][3], "in-place params")


@pytest.mark.parametrize("where", ["pageable", "pinned"])
@pytest.mark.parametrize("what", ["state_in", "state_out", "flag", "cb", "adam_grad",
                                  "cast_master"])
def test_host_memory_is_refused_where_device_memory_is_required(what, where):
    """The fp32 state, the flag word, the fusion buffer and the primitives'
    fp32 inputs must be device memory: a host pointer there is
    ZERO_ERR_INVALID_ARG before anything is launched, and nothing is written."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=80_003, nd=4, plant=None)
    dps = make_group(w, ranks=[1], gathered="slot")
    buf, desc = shard_rows(w, dps, 1, 0)
    L = dps.layouts[1]
    n = int(L.length)
    st = dps.state[1]

    def host_like(t):
        h = torch.full(t.shape, 3.0, dtype=t.dtype)
        return h.pin_memory() if where == "pinned" else h
    s_in, s_out = st.states[st.cur], st.states[1 - st.cur]
    flag = dps.flag
    cb = torch.zeros(n + 4, dtype=torch.float32, device=DEV)
    gath = dps.gathered_view(1)
    out_dev = torch.full((3, n), 5.0, device=DEV)
    keep = []
    if what == "state_in":
        keep = [host_like(st.bufs[st.cur])]
        s_in = z.state(*keep[0])
    elif what == "state_out":
        keep = [host_like(st.bufs[1 - st.cur])]
        s_out = z.state(*keep[0])
    elif what == "flag":
        keep = [host_like(dps.flag)]
        flag = keep[0]
    elif what == "cb":
        keep = [host_like(cb)]
        cb = keep[0]
    before = [t.clone() for t in st.bufs] + [gath.clone(), out_dev.clone()]
    h = z.adamw(1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    with pytest.raises(z.ZeroError) as e:
        if what == "adam_grad":
            z.zero_adam_step_shard(host_like(cb)[:n], z.state(*st.bufs[st.cur][:, :n]),
                                   z.state(*out_dev), n, h)
        elif what == "cast_master":
            z.zero_gather_params_shard(host_like(out_dev)[0], n, gath, 0, w.grad_dtype)
        elif what == "cb":
            z.zero_step_shard_unfused(desc[1], L, s_in, s_out, gath, 0, 4096, w.loss_scale, h,
                                      cb, cb.numel(), flag)
        else:
            z.zero_step_shard(desc[1], L, s_in, s_out, gath, 0, 4096, w.loss_scale, h, flag)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    torch.cuda.synchronize()
    after = [t for t in st.bufs] + [gath, out_dev]
    assert all(torch.equal(a, b) for a, b in zip(before, after)), "a refused call wrote"
    assert all(bool((k == 3.0).all()) for k in keep)
