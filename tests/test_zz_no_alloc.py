"""The allocation-free shard step, zero_step_shard_unfused_static.

Some callers cannot call cudaMalloc: a framework whose memory pool owns the
whole device and forbids allocations from outside it, or code that must not
take the device-wide synchronisation that cudaMalloc/cudaFree can imply.  For
them the library keeps its own 16 MiB fusion buffer in device memory, so the
step needs no workspace from the caller.  This file checks, through the C ABI,
that it gives the same results as zero_step_shard_unfused with a
caller-provided workspace, on two calls in a row (the second call finds the
first call's data in the shared buffer), and that a bucket larger than the
buffer is refused before anything runs.  It is collected last and passes both
on its own in a fresh process and after the other tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (DEV, TORCH_DT, assert_params_close, assert_state_close, f32, full_rows,
                      make_group, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _clone_state(st):
    """A second, independent copy of a rank's current state block."""
    return st.bufs[st.cur].clone()


def test_static_matches_workspace_version_on_two_calls():
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=600_011, nd=8, plant=None)
    bucket = 65_536
    dps = make_group(w, bucket=bucket)
    buf, desc = full_rows(w, dps, 0)
    s = int(dps.layouts[0].shard_elems)
    tdt = TORCH_DT[w.grad_dtype]
    for call in range(2):
        if call == 1:   # fresh gradients for the second call
            buf, desc = full_rows(w, dps, 1, buf)
        h = z.adamw(w.hparams["lr"], w.hparams["beta1"], w.hparams["beta2"], w.hparams["eps"],
                    w.hparams["weight_decay"], call + 1)
        for r in dps.ranks:
            L = dps.layouts[r]
            n = int(L.length)
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
            for i, (name, tau) in enumerate((("master", 1e-12), ("m", 1e-20), ("v", 1e-20))):
                assert_state_close(f32(out_new[i, :n]), f32(out_ref[i, :n]), tau,
                                   f"call {call} rank {r} {name}")
            b = int(L.begin)
            assert_params_close(u16(g_new[b:b + n]), u16(g_ref[b:b + n]),
                                f"call {call} rank {r} params")
            assert int(f_new.item()) == int(f_ref.item()) == 0
            src.copy_(out_new)     # the next call starts from this call's result


def test_static_refuses_buckets_beyond_its_buffer():
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=9_000_000, nd=2, plant=None)
    dps = make_group(w, ranks=[0], gathered="slot")
    L = dps.layouts[0]
    st = dps.state[0]
    g = z.grads(0x100000, int(L.row_pitch), 0, 2, w.grad_dtype)
    h = z.adamw(1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_shard_unfused_static(g, L, st.states[0], st.states[1],
                                         dps.gathered_view(0), 0, z.ZERO_STATIC_CB_MAX_BUCKET + 1,
                                         1.0, h, dps.flag)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    raw = z.lib().zero_step_shard_unfused_static
    import ctypes as C
    rc = raw(C.byref(g), C.byref(L), C.byref(st.states[0]), C.byref(st.states[1]),
             dps.gathered_view(0).data_ptr(), 0, z.ZERO_STATIC_CB_MAX_BUCKET + 1, 1.0,
             C.byref(h), dps.flag.data_ptr(), None)
    assert rc == z.ZERO_ERR_INVALID_ARG
    assert int(dps.flag.item()) == 0
