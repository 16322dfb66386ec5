"""Save the GPU state as a sharded checkpoint, reload it on a different
number of ranks and keep stepping: the trajectory equals the oracle's
uninterrupted unsharded run bit for bit ("ZeRO" (process-cxr ai-library),
checkpointing and recovery: resuming with a different number of GPUs)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (assert_params_close, assert_state_close, flat_state, full_rows, make_group,
                      oracle_trajectory, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("nd_old,nd_new", [(4, 3), (4, 4), (8, 5)])
def test_resume_on_other_rank_count(tmp_path, nd_old, nd_new):
    psi = 200_003
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=psi, nd=nd_old, plant=None)
    a = make_group(w, bucket=30_000)
    for k in range(2):
        _, desc = full_rows(w, a, k)
        assert not a.step(desc)
    paths = a.save_checkpoint(str(tmp_path))
    # the resumed group: nd_new ranks; contributions now come from nd_new ranks
    w2 = dataclasses.replace(w, nd=nd_new)
    b = make_group(w2, bucket=30_000)
    b.load_checkpoint(paths)
    assert b.t == 2
    got = flat_state(b)
    ref = flat_state(a)
    for x, y in zip(got, ref):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    # one more step on nd_new ranks, against the oracle: two steps with nd_old
    # contributions, then one with nd_new
    _, desc = full_rows(w2, b, 2)
    assert not b.step(desc)
    idx = np.arange(psi)
    tr, _ = oracle_trajectory(w, idx, 2)
    I = torch.from_numpy(idx)
    rows = np.stack([u16(synth.grad_values(w2, 2, j, I)) for j in range(nd_new)])
    tr.loss_scale = w2.loss_scale
    tr.step(rows)
    p, m, v = flat_state(b)
    assert_state_close(p, tr.p, 1e-12, "master")
    assert_state_close(m, tr.m, 1e-20, "m")
    assert_state_close(v, tr.v, 1e-20, "v")
    assert_params_close(u16(b.gathered_view()[:psi]), tr.params, "params")
    assert b.t == tr.t == 3
