"""Helpers for the GPU parity tests: device buffers from the seeded generator,
oracle trajectories on the same inputs, and the comparison rules.

Tolerances (stated for the step): reduced gradient sums bit-exact in fp32;
master weights and moments within 1e-6 relative error (|a-b| <= 1e-6 *
max(|b|, tau), tau = 1e-12 for master and 1e-20 for the moments); cast
parameters within 1 ulp.  The kernels use the oracle's exact operation
sequence, so the tests also require bitwise equality.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from zero_sharded_optimizer_02_gb300.step import DataParallelStep
from window_rule import inner_cuts

DEV = "cuda"
DT_CODE = {"f16": oracle.F16, "bf16": oracle.BF16}
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def ulp_dist16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(x):
        x = x.astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def assert_state_close(got: np.ndarray, ref: np.ndarray, tau: float, what: str):
    assert got.shape == ref.shape, what
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    lim = 1e-6 * np.maximum(np.abs(ref.astype(np.float64)), tau)
    bad = ~(err <= lim)
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1e-6 rel, first {np.argmax(bad)}"
    nb = (got.view(np.uint32) != ref.view(np.uint32)).sum()
    assert nb == 0, f"{what}: {nb} elements differ bitwise (within tolerance)"


def assert_params_close(got: np.ndarray, ref: np.ndarray, what: str):
    d = ulp_dist16(got, ref)
    assert d.max(initial=0) <= 1, f"{what}: max ulp distance {d.max()}"
    assert np.array_equal(got, ref), f"{what}: {(got != ref).sum()} params differ by 1 ulp"


# -- workloads on the device -------------------------------------------------

def make_group(w: synth.Workload, ranks=None, fused=True, bucket=None, gathered="full",
               psi=None, nd=None, gathered_on_host=False):
    """A DataParallelStep over `ranks` with the workload's initial state."""
    psi = psi or w.psi
    nd = nd or w.nd
    ranks = list(range(nd)) if ranks is None else list(ranks)
    dps = DataParallelStep(psi, nd, ranks, w.grad_dtype, w.hparams, w.loss_scale,
                           bucket or w.bucket, DEV, gathered=gathered, fused=fused,
                           gathered_on_host=gathered_on_host)
    for r in ranks:
        st = dps.state[r]
        buf = st.bufs[st.cur]
        for row, which in zip(buf, ("master", "m", "v")):
            synth.fill_shard_state(_resized(w, psi, nd), r, which, row)
    return dps


def _resized(w, psi, nd):
    if psi == w.psi and nd == w.nd:
        return w
    import dataclasses
    return dataclasses.replace(w, psi=psi, nd=nd, plant=None)


def full_rows(w, dps: DataParallelStep, step: int, buf=None):
    """All ranks' gradients in padded-partition layout and their descriptors."""
    pitch = int(dps.layouts[dps.ranks[0]].row_pitch)
    nd = dps.nd
    if buf is None:
        buf = torch.empty(nd, nd * pitch, dtype=TORCH_DT[w.grad_dtype], device=DEV)
    synth.fill_full_rows(_resized(w, dps.psi, nd), step, buf)
    desc = {r: z.grads(buf, nd * pitch, r * pitch, nd, w.grad_dtype) for r in dps.ranks}
    return buf, desc


def shard_rows(w, dps: DataParallelStep, rank: int, step: int, buf=None):
    pitch = int(dps.layouts[rank].row_pitch)
    if buf is None:
        buf = torch.empty(dps.nd, pitch, dtype=TORCH_DT[w.grad_dtype], device=DEV)
    synth.fill_shard_rows(_resized(w, dps.psi, dps.nd), step, rank, buf)
    return buf, {rank: z.grads(buf, pitch, 0, dps.nd, w.grad_dtype)}


def flat_state(dps: DataParallelStep):
    """Concatenate the ranks' current state into flat arrays (rank order)."""
    parts = [dps.state[r].tensors("cur") for r in sorted(dps.ranks)]
    return tuple(np.concatenate([f32(p[i]) for p in parts]) for i in range(3))


# -- oracle on the same inputs ----------------------------------------------

def oracle_trajectory(w, idx: np.ndarray, steps: int, psi=None, nd=None):
    """Oracle run over flat indices ``idx`` (the whole vector or a sample):
    returns the Trajectory after ``steps`` steps and the per-step states."""
    ww = _resized(w, psi or w.psi, nd or w.nd)
    I = torch.from_numpy(np.asarray(idx, np.int64))
    p0, m0, v0 = (synth.state_values(ww, k, I).numpy() for k in ("master", "m", "v"))
    tr = oracle.Trajectory(DT_CODE[w.grad_dtype], w.loss_scale, w.hparams, p0, m0, v0)
    history = []
    for k in range(steps):
        rows = np.stack([u16(synth.grad_values(ww, k, j, I)) for j in range(ww.nd)])
        tr.step(rows)
        history.append((tr.p.copy(), tr.m.copy(), tr.v.copy(),
                        None if tr.params is None else tr.params.copy(), tr.t))
    return tr, history


def oracle_shard_step(w, rank: int, step: int = 0):
    """The oracle's step t = 1 of one rank's whole shard from the workload's
    initial state, on the contributions of generator step ``step``:
    (flag, master, m, v, params), params being the cast into the rank's slot."""
    s, b, n = synth.shard_of(w.psi, w.nd, rank)
    I = torch.arange(b, b + n, dtype=torch.int64)
    p0, m0, v0 = (synth.state_values(w, k, I).numpy() for k in ("master", "m", "v"))
    rows = np.stack([u16(synth.grad_values(w, step, j, I)) for j in range(w.nd)])
    params = np.zeros(max(n, 1), np.uint16)
    f, p, m, v = oracle.step_rank(rows, n, 0, n, w.nd, DT_CODE[w.grad_dtype], w.bucket,
                                  w.loss_scale, w.hparams, 1, p0, m0, v0, params, 0)
    return f, p, m, v, params[:n]


def sample_indices(psi: int, nd: int, ranks, per_rank: int, seed: int, extra=()):
    """Flat indices: each rank's first/last elements, neighbours of every
    8-element boundary near the ends, the 16 elements on each side of every
    cut between two launch windows of the fused step (shards longer than one
    window, rows starting on a 32-byte boundary as in every sampled test),
    random interior points, and ``extra``."""
    rng = np.random.default_rng(seed)
    s = -(-psi // nd)
    out = set(int(e) for e in extra)
    for r in ranks:
        b = r * s
        n = max(0, min(s, psi - b))
        if n == 0:
            continue
        for d in range(min(n, 17)):
            out.add(b + d)
            out.add(b + n - 1 - d)
        for c in inner_cuts(n, 0):
            out.update(b + c + d for d in range(-16, 16) if 0 <= c + d < n)
        out.update(int(x) for x in b + rng.integers(0, n, per_rank))
    return np.array(sorted(out), np.int64)


# -- whole-group checks ------------------------------------------------------

EDGE_CASES = [
    # (psi, nd, dtype, bucket): ragged tails, psi < nd, nd = 1, odd slot phases
    (1000, 3, "bf16", 64),
    (1001, 7, "f16", 1),         # one launch per element
    (3, 5, "f16", 7),            # psi < nd: empty shards
    (4099, 1, "bf16", 1000),     # one rank: plain data parallel
    (70_001, 16, "f16", 7),      # S mod 8 = 3: every slot phase
    (130_003, 64, "bf16", 2049), # 64 ranks, S mod 8 = 4
    (250_000, 2, "f16", 250_000),
    (102_407, 1024, "bf16", 4099),   # the pages' largest Nd: 1,024 rows folded, S mod 8 = 5
]


def check_against_oracle(w, dps, history_entry, what):
    """The group's whole state, gathered parameters and t against one oracle
    step, and nothing written outside the shards."""
    p, m, v, params, t = history_entry
    gp, gm, gv = flat_state(dps)
    assert_state_close(gp, p, 1e-12, f"{what} master")
    assert_state_close(gm, m, 1e-20, f"{what} m")
    assert_state_close(gv, v, 1e-20, f"{what} v")
    if params is not None:
        got = u16(dps.gathered_view()[:dps.psi])
        assert_params_close(got, params, f"{what} params")
    assert dps.t == t
    # nothing written outside the shards: padding of the gathered buffer and
    # the state rows past each shard's length stay zero
    s = int(dps.layouts[0].shard_elems)
    assert not dps.gathered_view()[dps.psi:].view(torch.int16).any(), f"{what} gathered pad"
    for r in dps.ranks:
        st = dps.state[r]
        n = int(dps.layouts[r].length)
        for b in st.bufs:
            assert not b[:, n:].any(), f"{what} state pad rank {r}"
