"""The seeded counter-based input generator (shared by oracle and CUDA tests)."""
import numpy as np
import torch

import synth
from synth import WORKLOADS


def _py_centred(key, i):
    z = synth.splitmix64_int(key + (i + 1) * synth.GAMMA)
    s = sum((z >> sh) & 0xFFFF for sh in (0, 16, 32, 48))
    return 2 * s - synth.CENTRE


def test_hash_matches_scalar_definition():
    key = synth.stream_key(3, synth.T_GRAD, 0, 17)
    idx = torch.tensor([0, 1, 2, 12345, 2 ** 33 + 7, 7_499_999_999], dtype=torch.int64)
    got = synth.centred_int(key, idx).tolist()
    assert got == [_py_centred(key, int(i)) for i in idx]


def test_distribution_and_bounds():
    idx = torch.arange(1 << 20, dtype=torch.int64)
    x = synth.normal_f32(0, synth.T_MASTER, 0, 0, idx, 0.02).double()
    assert abs(x.mean().item()) < 1e-4
    assert abs(x.std().item() / 0.02 - 1) < 0.01
    assert x.abs().max().item() <= 0.02 * 3.47


def test_grads_are_exact_roundings_and_deterministic():
    w = WORKLOADS["c0"]
    idx = torch.arange(4096, dtype=torch.int64)
    a = synth.grad_values(w, 1, 2, idx)
    b = synth.grad_values(w, 1, 2, idx)
    assert a.dtype == torch.float16 and torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = synth.grad_values(w, 2, 2, idx)          # fresh gradients per step
    assert not torch.equal(a, c)
    # value = fp16(fp32(c) * fp32(sigma * LS / STD)): one fp32 multiply, one rounding
    key = synth.stream_key(w.seed, synth.T_GRAD, 1, 2)
    ci = np.array([_py_centred(key, i) for i in range(4096)], np.float32)
    ref = (ci * np.float32(w.grad_sigma * w.loss_scale / synth.STD)).astype(np.float16)
    assert np.array_equal(a.numpy().view(np.uint16), ref.view(np.uint16))


def test_fixed_grads_and_plant():
    w = WORKLOADS["c2"]
    step, j, flat = w.plant
    idx = torch.tensor([flat - 1, flat, flat + 1], dtype=torch.int64)
    clean = synth.grad_values(w, 0, j, idx)
    assert torch.equal(synth.grad_values(w, 3, j, idx), clean)   # fixed across steps
    planted = synth.grad_values(w, step, j, idx)
    assert torch.isinf(planted[1]) and planted[1] > 0
    assert torch.equal(planted[[0, 2]], clean[[0, 2]])
    assert not torch.isinf(synth.grad_values(w, step, j + 1, idx)).any()
    s, begin, n = synth.shard_of(w.psi, w.nd, 7)
    assert begin <= flat < begin + n


def test_shard_fill_matches_flat_index():
    w = WORKLOADS["c0"]
    s, begin, n = synth.shard_of(w.psi, w.nd, 2)
    rows = torch.zeros(w.nd, synth.pitch_of(s) + 8, dtype=torch.float16)
    synth.fill_shard_rows(w, 0, 2, rows, chunk=1 << 16)
    idx = torch.arange(begin, begin + n, dtype=torch.int64)
    for j in range(w.nd):
        assert torch.equal(rows[j, :n], synth.grad_values(w, 0, j, idx))
    assert not rows[:, n:].any()
    st = torch.empty(s + 8)
    synth.fill_shard_state(w, 2, "master", st, chunk=1 << 16)
    assert torch.equal(st[:n], synth.state_values(w, "master", idx)) and not st[n:].any()


def test_workload_table():
    assert [WORKLOADS[k].shard for k in ("c0", "c1", "c2", "c3", "c4")] == \
        [262_144, 15_554_976, 21_875_002, 23_437_500, 117_187_500]
    assert WORKLOADS["c4"].bytes_per_param == 154 and WORKLOADS["c1"].bytes_per_param == 42


def test_full_rows_placements_agree():
    """The one-call-per-contributor placement of small vectors gives the same
    bytes as the shard-by-shard one (padding zero, a planted +inf kept)."""
    import dataclasses
    for psi, nd in [(1000, 3), (3, 5), (70_001, 16), (102_407, 64)]:
        w = dataclasses.replace(synth.WORKLOADS["c2"], psi=psi, nd=nd, plant=(0, 1, psi // 2))
        s = -(-psi // nd)
        pitch = synth.pitch_of(s)
        a = torch.full((nd, nd * pitch), 7, dtype=torch.float16)
        b = torch.full((nd, nd * pitch), 7, dtype=torch.float16)
        synth.fill_full_rows(w, 0, a)
        synth.fill_full_rows(w, 0, b, chunk=nd * s - 1)    # below nd*S: shard by shard
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (psi, nd)
        assert bool(torch.isinf(a).any())
