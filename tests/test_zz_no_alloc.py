"""The allocation-free shard step, zero_step_shard_unfused_static.

Some callers cannot call cudaMalloc: a framework whose memory pool owns the
whole device and forbids allocations from outside it, or code that must not
take the device-wide synchronisation that cudaMalloc/cudaFree can imply.  For
them the library keeps its own 16 MiB fusion buffer in device memory, so the
step needs no workspace from the caller.  This file checks, through the C ABI,
that it gives bit for bit the results of zero_step_shard_unfused with a
caller-provided workspace, and the oracle's, on two calls in a row (the
second call finds the first call's data in the shared buffer), including
buckets that fill the buffer to within 2 floats of its end, and that a bucket
larger than the buffer is refused before anything runs.  It is collected last
and passes both on its own in a fresh process and after the other tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, f32, full_rows,
                      make_group, oracle_shard_step, oracle_trajectory, shard_rows, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _h(w, t):
    return z.adamw(w.hparams["lr"], w.hparams["beta1"], w.hparams["beta2"], w.hparams["eps"],
                   w.hparams["weight_decay"], t)


def test_static_matches_workspace_version_and_oracle_on_two_calls():
    """Every rank of an 8-rank group, two calls in a row: the static form's
    state and parameters equal the workspace form's bit for bit (the same
    kernels in the same order), and the oracle's unsharded steps."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=600_011, nd=8, plant=None)
    bucket = 65_536
    dps = make_group(w, bucket=bucket)
    _, hist = oracle_trajectory(w, np.arange(w.psi), 2)
    buf, desc = full_rows(w, dps, 0)
    s = int(dps.layouts[0].shard_elems)
    tdt = TORCH_DT[w.grad_dtype]
    for call in range(2):
        if call == 1:   # fresh gradients for the second call
            buf, desc = full_rows(w, dps, 1, buf)
        h = _h(w, call + 1)
        ref_p, ref_m, ref_v, ref_params, _ = hist[call]
        for r in dps.ranks:
            L = dps.layouts[r]
            n, b = int(L.length), int(L.begin)
            src = dps.state[r].bufs[dps.state[r].cur]
            s_in = z.state(src[0], src[1], src[2])
            out_ref = torch.zeros_like(src)
            out_new = torch.zeros_like(src)
            g_ref = torch.zeros(w.nd * s + 8, dtype=tdt, device=DEV)
            g_new = torch.zeros(w.nd * s + 8, dtype=tdt, device=DEV)
            cb = torch.empty(min(bucket, n) + 4, dtype=torch.float32, device=DEV)
            f_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
            f_new = torch.zeros(1, dtype=torch.int32, device=DEV)
            z.zero_step_shard_unfused(desc[r], L, s_in, z.state(*out_ref), g_ref, L.begin,
                                      bucket, w.loss_scale, h, cb, cb.numel(), f_ref)
            z.zero_step_shard_unfused_static(desc[r], L, s_in, z.state(*out_new), g_new,
                                             L.begin, bucket, w.loss_scale, h, f_new)
            torch.cuda.synchronize()
            what = f"call {call} rank {r}"
            assert torch.equal(out_new, out_ref), f"{what}: state differs from the workspace form"
            assert torch.equal(g_new, g_ref), f"{what}: parameters differ from the workspace form"
            for i, (ref, name, tau) in enumerate(((ref_p, "master", 1e-12), (ref_m, "m", 1e-20),
                                                  (ref_v, "v", 1e-20))):
                assert_state_close(f32(out_new[i, :n]), ref[b:b + n], tau, f"{what} {name}")
            assert_params_close(u16(g_new[b:b + n]), ref_params[b:b + n], f"{what} params")
            assert int(f_new.item()) == int(f_ref.item()) == 0
            src.copy_(out_new)     # the next call starts from this call's result


@pytest.mark.parametrize("bucket", [z.ZERO_STATIC_CB_MAX_BUCKET, z.ZERO_STATIC_CB_MAX_BUCKET - 1])
def test_static_buffer_filled_to_its_end(bucket):
    """Buckets as large as the library's buffer allows, on a shard of three
    and a bit buckets: with 4,194,299-element buckets the second, third and
    fourth start at 16-byte phases 3, 2 and 1 of the buffer, so the last
    element of the second lands 2 floats from the buffer's end.  Equal to the
    workspace form bit for bit and to the oracle's shard step, twice."""
    n = 3 * (z.ZERO_STATIC_CB_MAX_BUCKET - 1) + 5
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=2 * n, nd=2, plant=None, bucket=bucket,
                            fresh_grads=False)
    rank = 1
    f, rp, rm, rv, rparams = oracle_shard_step(w, rank)
    assert f == 0
    dps = make_group(w, ranks=[rank], gathered="slot")
    L = dps.layouts[rank]
    assert int(L.length) == n
    buf, desc = shard_rows(w, dps, rank, 0)
    src = dps.state[rank].bufs[dps.state[rank].cur]
    h = _h(w, 1)
    tdt = TORCH_DT[w.grad_dtype]
    cb = torch.empty(bucket + 4, dtype=torch.float32, device=DEV)
    for call in range(2):
        out_ref, out_new = torch.zeros_like(src), torch.zeros_like(src)
        g_ref = torch.zeros(n + 8, dtype=tdt, device=DEV)
        g_new = torch.zeros(n + 8, dtype=tdt, device=DEV)
        f_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        f_new = torch.zeros(1, dtype=torch.int32, device=DEV)
        z.zero_step_shard_unfused(desc[rank], L, z.state(*src), z.state(*out_ref), g_ref, 0,
                                  bucket, w.loss_scale, h, cb, cb.numel(), f_ref)
        z.zero_step_shard_unfused_static(desc[rank], L, z.state(*src), z.state(*out_new), g_new,
                                         0, bucket, w.loss_scale, h, f_new)
        torch.cuda.synchronize()
        assert torch.equal(out_new, out_ref) and torch.equal(g_new, g_ref), f"call {call}"
        for i, (ref, name, tau) in enumerate(((rp, "master", 1e-12), (rm, "m", 1e-20),
                                              (rv, "v", 1e-20))):
            assert_state_close(f32(out_new[i, :n]), ref, tau, f"call {call} {name}")
        assert_params_close(u16(g_new[:n]), rparams, f"call {call} params")
        assert int(f_new.item()) == int(f_ref.item()) == 0


def test_static_refuses_buckets_beyond_its_buffer():
    """A bucket one element larger than the buffer holds is refused before
    anything is launched, through the binding and through the raw C call; the
    descriptor points at real rows, so a regression would give a wrong status,
    not a stray read."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=9_000_000, nd=2, plant=None)
    dps = make_group(w, ranks=[0], gathered="slot")
    L = dps.layouts[0]
    st = dps.state[0]
    buf, desc = shard_rows(w, dps, 0, 0)
    g = desc[0]
    h = _h(w, 1)
    too_big = z.ZERO_STATIC_CB_MAX_BUCKET + 1
    assert int(L.length) >= too_big
    before = [t.clone() for t in st.bufs] + [dps.gathered_view(0).clone()]
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_shard_unfused_static(g, L, st.states[0], st.states[1],
                                         dps.gathered_view(0), 0, too_big, 1.0, h, dps.flag)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    raw = z.lib().zero_step_shard_unfused_static
    import ctypes as C
    rc = raw(C.byref(g), C.byref(L), C.byref(st.states[0]), C.byref(st.states[1]),
             dps.gathered_view(0).data_ptr(), 0, too_big, 1.0, C.byref(h),
             dps.flag.data_ptr(), None)
    assert rc == z.ZERO_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(dps.flag.item()) == 0
    after = [t for t in st.bufs] + [dps.gathered_view(0)]
    assert all(torch.equal(a, b) for a, b in zip(before, after)), "a refused call wrote"
