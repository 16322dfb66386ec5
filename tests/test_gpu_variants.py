"""Every variant of the fused step kernel gives the oracle's step bit for bit.

zero_step_shard runs the cp.async-ring kernel by default, and the
short-window kernel for windows that one wave of it covers (SMs x 3,072
elements); the environment variable ZERO_FUSED_VARIANT selects one kernel for every window:
the ring ("ring"), the short-window kernel ("small": 4 elements a thread),
the register kernel ("registers", also the kernel for host-resident rows) or
the bulk-copy kernel ("tma": a producer warp, mbarrier-tracked cp.async.bulk
copies of rows and state).  Each is checked here on the same cases as the
default: the 4-rank workload against the oracle, ragged shapes and every slot
phase, a global skip, and whole shards of several launch windows against the
oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import (EDGE_CASES, assert_params_close, assert_state_close,
                      check_against_oracle, flat_state, full_rows, make_group, oracle_shard_step,
                      oracle_trajectory, shard_rows, u16)

pytestmark = pytest.mark.gpu

VARIANTS = ["registers", "ring", "tma", "small"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture
def variant(request, monkeypatch):
    monkeypatch.setenv("ZERO_FUSED_VARIANT", request.param)
    return request.param


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("variant", VARIANTS, indirect=True)
def test_c0_matches_oracle(variant, fused):
    """Fused, and unfused (whose reduction follows the variant: the ring's
    reduction mode, or the register kernel)."""
    w = synth.WORKLOADS["c0"]
    dps = make_group(w, fused=fused)
    _, hist = oracle_trajectory(w, np.arange(w.psi), w.steps)
    buf = None
    for k in range(w.steps):
        buf, desc = full_rows(w, dps, k, buf)
        assert not dps.step(desc)
        check_against_oracle(w, dps, hist[k], f"{variant} fused={fused} c0 step {k}")


@pytest.mark.parametrize("psi,nd,dt,bucket", EDGE_CASES)
@pytest.mark.parametrize("variant", ["registers", "tma", "ring", "small"], indirect=True)
def test_edge_shapes(variant, psi, nd, dt, bucket):
    w = dataclasses.replace(synth.WORKLOADS["c1"], grad_dtype=dt,
                            loss_scale=1024.0 if dt == "f16" else 1.0, plant=None)
    dps = make_group(w, bucket=bucket, psi=psi, nd=nd)
    _, hist = oracle_trajectory(w, np.arange(psi), 2, psi=psi, nd=nd)
    buf = None
    for k in range(2):
        buf, desc = full_rows(w, dps, k, buf)
        assert not dps.step(desc)
        check_against_oracle(dataclasses.replace(w, psi=psi, nd=nd), dps, hist[k],
                             f"{variant} psi={psi} nd={nd} step {k}")


@pytest.mark.parametrize("variant", ["registers", "tma", "ring", "small"], indirect=True)
def test_global_skip(variant):
    w = dataclasses.replace(synth.WORKLOADS["c2"], psi=100_003, nd=16, plant=None)
    dps = make_group(w, bucket=4096)
    buf, desc = full_rows(w, dps, 0)
    assert not dps.step(desc)
    before = [a.copy() for a in flat_state(dps)] + [u16(dps.gathered_view()).copy()]
    s = int(dps.layouts[0].shard_elems)
    pitch = int(dps.layouts[0].row_pitch)
    buf[7, 7 * pitch + s // 2] = float("inf")
    assert dps.step(desc)
    after = [a.copy() for a in flat_state(dps)] + [u16(dps.gathered_view()).copy()]
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
    assert dps.t == 1 and int(dps.flag.item()) == 0


def test_several_launch_windows_match_oracle_on_every_variant(monkeypatch):
    """Whole shards against the oracle, element by element, on every variant:
    rank 1 of psi = 60,000,005 over 2 bf16 rows (30,000,002 elements, three
    launch windows cut at elements 10,000,016 and 20,000,032) and rank 5 of a
    64-row fp16 shard of 1,000,003 elements.  The bulk-copy kernel runs twice (a race
    would vary between runs)."""
    from window_rule import inner_cuts
    cases = [(dataclasses.replace(synth.WORKLOADS["c1"], psi=60_000_005, nd=2, plant=None,
                                  bucket=1 << 30), 1),
             (dataclasses.replace(synth.WORKLOADS["c3"], psi=64 * 1_000_003, plant=None,
                                  bucket=1 << 30), 5)]
    assert z.fused_launch_count(30_000_002, 1 << 30) == 3
    assert inner_cuts(30_000_002) == [10_000_016, 20_000_032]
    for w, rank in cases:
        f, rp, rm, rv, rparams = oracle_shard_step(w, rank)
        assert f == 0
        for v in VARIANTS + ["tma"]:
            monkeypatch.setenv("ZERO_FUSED_VARIANT", v)
            dps = make_group(w, ranks=[rank], gathered="slot")
            buf, desc = shard_rows(w, dps, rank, 0)
            assert not dps.step(desc)
            n = int(dps.layouts[rank].length)
            got = [t.cpu().numpy() for t in dps.state[rank].tensors("cur")]
            for g, ref, name, tau in zip(got, (rp, rm, rv), ("master", "m", "v"),
                                         (1e-12, 1e-20, 1e-20)):
                assert_state_close(g, ref, tau, f"{v} psi={w.psi} {name}")
            assert_params_close(u16(dps.gathered_view(rank)[:n]), rparams,
                                f"{v} psi={w.psi} params")
            del dps, buf, desc
            torch.cuda.empty_cache()


@pytest.mark.parametrize("fused", [True, False])
def test_plain_and_programmatic_launches_agree(fused, monkeypatch):
    """Every step kernel runs as a programmatic dependent launch by default;
    ZERO_PDL=0 launches them plainly.  Both give the oracle's result (the
    4-rank workload, 3 steps: consecutive launches of the same stream)."""
    w = synth.WORKLOADS["c0"]
    _, hist = oracle_trajectory(w, np.arange(w.psi), w.steps)
    for pdl in ("0", "1"):
        monkeypatch.setenv("ZERO_PDL", pdl)
        dps = make_group(w, fused=fused)
        buf = None
        for k in range(w.steps):
            buf, desc = full_rows(w, dps, k, buf)
            assert not dps.step(desc)
            check_against_oracle(w, dps, hist[k], f"ZERO_PDL={pdl} fused={fused} step {k}")


@pytest.mark.parametrize("variant", ["ring", "registers"], indirect=True)
def test_reductions_over_several_launch_windows_match_oracle(variant):
    """The reductions cut a long range into launch windows like the fused step
    (each after the first starting as its predecessor drains):
    zero_reduce_scatter_bucket over 30,000,002 elements of 2 bf16 rows (three
    windows), bit for bit against the oracle; the pre-check over the same
    range with a +inf planted in the second window; and the unfused step with
    one bucket of the whole shard (three reduction windows, then AdamW and
    cast) against the oracle's shard step."""
    from window_rule import inner_cuts
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=60_000_005, nd=2, plant=None,
                            bucket=1 << 30)
    rank = 1
    dps = make_group(w, ranks=[rank], gathered="slot", fused=False)
    buf, desc = shard_rows(w, dps, rank, 0)
    L = dps.layouts[rank]
    n = int(L.length)
    pitch = int(L.row_pitch)
    assert inner_cuts(n) == [10_000_016, 20_000_032]
    inv = float(np.float32(1.0 / w.nd))
    cb = torch.empty(n, dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    z.zero_reduce_scatter_bucket(desc[rank], 0, n, inv, cb, flag)
    torch.cuda.synchronize()
    host = u16(buf).reshape(-1)
    f, ref = oracle.reduce_scaled(host, oracle.BF16, pitch, 0, n, w.nd, inv)
    assert f == 0 and int(flag.item()) == 0
    assert np.array_equal(cb.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # the unfused step: two reduction windows into the fusion buffer
    f, rp, rm, rv, rparams = oracle_shard_step(w, rank)
    assert not dps.step(desc)
    got = [t.cpu().numpy() for t in dps.state[rank].tensors("cur")]
    for g, r, name, tau in zip(got, (rp, rm, rv), ("master", "m", "v"), (1e-12, 1e-20, 1e-20)):
        assert_state_close(g, r, tau, f"unfused {name}")
    assert_params_close(u16(dps.gathered_view(rank)[:n]), rparams, "unfused params")
    # the pre-check sees a +inf that only the second window reads
    buf[1, 20_000_001] = float("inf")
    flag.zero_()
    z.zero_check_nonfinite(desc[rank], 0, n, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1


def _boundary_cases():
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    wave = sms * 3 * 256 * 4          # one wave of the short-window kernel's wide shape
    light = sms * 2 * 256 * 4         # the light shape's limit: 2 CTAs a SM
    # (rows, shard elements): each side of the ring / short-window cut (by
    # elements), of the light / wide cut (by CTAs: 4-element groups, hence
    # + 4) and of the light shape's 16-row limit
    return [(3, wave), (3, wave + 1), (4, light), (4, light + 4), (16, 5_003), (17, 5_003)]


@pytest.mark.parametrize("case", range(6))
def test_default_choice_at_its_boundaries(case, monkeypatch):
    """By default a shard that one wave of the short-window kernel covers
    (SMs x 3 x 256 x 4 elements) runs on that kernel and one element more on
    the ring, and within it shards of up to 16 rows that need at most 2 CTAs
    a SM run on the kernel's light shape.  Both sides of each boundary, and
    the same shards on the short-window and ring kernels named explicitly,
    against the oracle element by element (fp16 rows; rank 1 writes its slot
    of the flat gathered buffer, whose 16-byte phase moves with the shard's
    length)."""
    nd, s = _boundary_cases()[case]
    w = dataclasses.replace(synth.WORKLOADS["c2"], psi=nd * s - 1, nd=nd, plant=None,
                            bucket=1 << 30)
    f, rp, rm, rv, rparams = oracle_shard_step(w, 1)
    assert f == 0
    for v in (None, "small", "ring"):
        if v is None:
            monkeypatch.delenv("ZERO_FUSED_VARIANT", raising=False)
        else:
            monkeypatch.setenv("ZERO_FUSED_VARIANT", v)
        dps = make_group(w, ranks=[1], gathered="full")
        buf, desc = shard_rows(w, dps, 1, 0)
        assert not dps.step(desc)
        n = int(dps.layouts[1].length)
        assert n == s
        got = [t.cpu().numpy() for t in dps.state[1].tensors("cur")]
        for g, ref, name, tau in zip(got, (rp, rm, rv), ("master", "m", "v"),
                                     (1e-12, 1e-20, 1e-20)):
            assert_state_close(g, ref, tau, f"{v} nd={nd} n={n} {name}")
        b = int(dps.layouts[1].begin)
        assert_params_close(u16(dps.gathered_view(1)[b:b + n]), rparams,
                            f"{v} nd={nd} n={n} params")
        del dps, buf, desc
