"""Seeded random shapes against the oracle, on every path of the step.

Each case draws a flat size, a data-parallel degree, a bucket size, a
gradient type, the ranks held and the path (fused with each kernel variant or
the default choice among them, unfused, bucket-ready, or fused with the rows and the gathered parameters in
pinned host memory), runs two steps on the GPU with every rank's whole
gradient resident, and compares every element of state and parameters with
the oracle's unsharded step.  The draws favour the awkward: sizes not
multiple of 8, shards that are short or empty, buckets of 1 to a few
thousand elements, odd slot phases.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, check_against_oracle, full_rows, make_group, oracle_trajectory

pytestmark = pytest.mark.gpu

PATHS = ["ring", "registers", "tma", "small", "auto", "unfused", "streamed", "host"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _draw(seed: int):
    rng = np.random.default_rng(1000 + seed)
    nd = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 31, 64, 67]))
    psi = int(rng.integers(1, 200_000))
    if rng.random() < 0.25:
        psi = int(rng.integers(1, 3 * nd + 2))          # shards of 0 or a few elements
    bucket = int(rng.choice([1, 7, 8, 63, 1000, 4096, 65_536, 1 << 30]))
    if bucket == 1 and psi > 20_000:
        bucket = 7                                      # keep the launch count modest
    dt = "f16" if rng.random() < 0.5 else "bf16"
    path = PATHS[seed % len(PATHS)]
    return psi, nd, bucket, dt, path


def _streamed_step(w, dps, buf, step_bucket):
    """One bucket-ready step of every held rank, all ready words already set."""
    nd = dps.nd
    pitch = int(dps.layouts[dps.ranks[0]].row_pitch)
    dps.h.step = dps.t + 1
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for r in dps.ranks:
        L = dps.layouts[r]
        n = int(L.length)
        nb = max(1, -(-n // step_bucket))
        ready = torch.ones(nb, dtype=torch.int32, device=DEV)
        st = dps.state[r]
        gbuf, goff = dps._gathered_target(r, 1 - dps.gcur)
        g = z.grads(buf, nd * pitch, r * pitch, nd, w.grad_dtype)
        z.zero_step_shard_streamed(g, L, st.states[st.cur], st.states[1 - st.cur], gbuf, goff,
                                   step_bucket, dps.loss_scale, dps.h, ready, 1, 10 ** 9,
                                   dps.flag, status, dps.stream)
    skipped = dps.decide()
    dps.commit(skipped)
    assert int(status.item()) == 0
    return skipped


@pytest.mark.parametrize("seed", range(30))
def test_random_shape(seed, monkeypatch):
    psi, nd, bucket, dt, path = _draw(seed)
    w = dataclasses.replace(synth.WORKLOADS["c1"], grad_dtype=dt,
                            loss_scale=1024.0 if dt == "f16" else 1.0, plant=None,
                            fresh_grads=True)
    if path in ("ring", "registers", "tma", "small"):
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    if path == "streamed":
        monkeypatch.setenv("ZERO_STREAM_GROUP_BYTES", "0")
    dps = make_group(w, fused=path != "unfused", bucket=bucket, psi=psi, nd=nd,
                     gathered_on_host=path == "host")
    _, hist = oracle_trajectory(w, np.arange(psi), 2, psi=psi, nd=nd)
    buf = None
    for k in range(2):
        buf, desc = full_rows(w, dps, k, buf)
        if path == "host":
            host = torch.empty(buf.shape, dtype=buf.dtype, pin_memory=True)
            host.copy_(buf)
            pitch = int(dps.layouts[0].row_pitch)
            desc = {r: z.grads(host, nd * pitch, r * pitch, nd, w.grad_dtype)
                    for r in dps.ranks}
        if path == "streamed":
            skipped = _streamed_step(w, dps, buf, bucket)
        else:
            skipped = dps.step(desc)
        assert not skipped
        check_against_oracle(dataclasses.replace(w, psi=psi, nd=nd), dps, hist[k],
                             f"seed {seed}: psi={psi} nd={nd} bucket={bucket} {dt} {path} "
                             f"step {k}")
