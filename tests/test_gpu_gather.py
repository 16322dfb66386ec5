"""GPU parity of zero_gather_range (ZeRO-3 on-demand parameter gather and
fp32 resharding) against the oracle, bit for bit.

"ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
section "ZeRO-DP", Stage 3: each rank keeps only its shard of the parameters;
a layer's parameters are collected from the owners before use.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, full_rows, make_group, oracle_trajectory, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _ranges(rng, psi, s, count):
    out = [(0, psi), (0, 0), (psi, 0), (0, 1), (psi - 1, 1)] if psi else [(0, 0)]
    for r in range(0, psi, max(s, 1)):
        out += [(r, min(s, psi - r)), (max(0, r - 3), min(psi - max(0, r - 3), 11))]
    for _ in range(count):
        b = int(rng.integers(0, psi + 1))
        out.append((b, int(rng.integers(0, psi - b + 1))))
    return out


@pytest.mark.parametrize("psi,nd,pad", [(1000, 3, 0), (100_003, 7, 5), (64, 64, 0),
                                        (2_000_001, 16, 13), (5, 8, 3), (300_000, 1, 0)])
@pytest.mark.parametrize("dtype", [np.uint16, np.float32])
def test_gather_range_matches_oracle(psi, nd, pad, dtype):
    rng = np.random.default_rng(psi + nd)
    s = -(-psi // nd)
    pitch = s + pad
    host = rng.integers(0, 1 << 16, size=(nd, pitch)).astype(dtype)
    if dtype == np.float32:
        host = rng.standard_normal((nd, pitch)).astype(np.float32)
    tdt = torch.int16 if dtype == np.uint16 else torch.float32
    dev = torch.from_numpy(host.view(np.int16) if dtype == np.uint16 else host).to(DEV)
    eb = host.itemsize
    for b, ln in _ranges(rng, psi, s, 12):
        for shift in (0, 1, 3):             # destination phases
            out = torch.full((ln + shift + 16,), 7, dtype=tdt, device=DEV)
            z.zero_gather_range(dev, pitch, psi, nd, b, ln, eb, out[shift:])
            torch.cuda.synchronize()
            got = out[shift:shift + ln].cpu().numpy()
            ref = oracle.gather_range(host, psi, nd, b, ln)
            assert np.array_equal(got.view(dtype), ref), (b, ln, shift)
            rest = torch.cat([out[:shift], out[shift + ln:]])
            assert bool((rest == 7).all()), "write outside the destination range"


def test_gather_rejects_bad_ranges():
    buf = torch.zeros(4, 16, dtype=torch.int16, device=DEV)
    out = torch.zeros(64, dtype=torch.int16, device=DEV)
    for args in ((buf, 16, 60, 4, 50, 11, 2, out), (buf, 14, 60, 4, 0, 1, 2, out),
                 (buf, 16, 60, 0, 0, 1, 2, out), (buf, 16, 60, 4, 0, 1, 3, out),
                 (buf, 16, 60, 4, 0, 8, 2, buf[1])):
        with pytest.raises(z.ZeroError) as e:
            z.zero_gather_range(*args)
        assert e.value.status == z.ZERO_ERR_INVALID_ARG


def test_zero3_layer_gather_after_step():
    """ZeRO-3 flow: every rank steps its shard into its own parameter row,
    then each "layer" (a flat range) is gathered from the rows and equals the
    oracle's unsharded parameters over that range."""
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=1_000_003, nd=16, plant=None)
    dps = make_group(w, gathered="pitched", bucket=50_000)
    buf, desc = full_rows(w, dps, 0)
    assert not dps.step(desc)
    _, hist = oracle_trajectory(w, np.arange(w.psi), 1)
    params_ref = hist[0][3]
    rows = dps.gathered_view()
    pitch = rows.shape[1]
    bounds = np.sort(np.random.default_rng(3).choice(np.arange(1, w.psi), 6, replace=False))
    layers = list(zip(np.r_[0, bounds], np.r_[bounds, w.psi]))
    for a, b in layers:
        out = torch.empty(int(b - a), dtype=rows.dtype, device=DEV)
        z.zero_gather_range(rows, pitch, w.psi, w.nd, int(a), int(b - a), 2, out)
        torch.cuda.synchronize()
        assert np.array_equal(u16(out), params_ref[a:b]), (a, b)


def test_gather_from_and_into_host_memory():
    """Shards and destination in page-locked host memory are accessed in
    place at their device mapping and give the oracle's range; a pageable host
    pointer is refused with ZERO_ERR_INVALID_ARG before anything is launched
    (the destination is left untouched)."""
    psi, nd = 100_003, 7
    s = -(-psi // nd)
    pitch = -(-s // 8) * 8 + 8
    rng = np.random.default_rng(5)
    host = rng.integers(0, 1 << 16, (nd, pitch), dtype=np.uint64).astype(np.uint16)
    begin, length = s - 77, 3 * s + 5
    ref = oracle.gather_range(host, psi, nd, begin, length)
    shards_dev = torch.from_numpy(host.view(np.int16)).to(DEV)
    shards_pin = torch.from_numpy(host.view(np.int16)).pin_memory()
    out_pin = torch.zeros(length, dtype=torch.int16).pin_memory()
    out_dev = torch.zeros(length, dtype=torch.int16, device=DEV)
    for src, dst in ((shards_pin, out_dev), (shards_dev, out_pin), (shards_pin, out_pin)):
        dst.zero_()
        z.zero_gather_range(src, pitch, psi, nd, begin, length, 2, dst)
        torch.cuda.synchronize()
        assert np.array_equal(dst.cpu().numpy().view(np.uint16), ref)
    pageable_out = torch.full((length,), 7, dtype=torch.int16)
    pageable_src = torch.from_numpy(host.view(np.int16).copy())
    for src, dst in ((shards_dev, pageable_out), (pageable_src, out_dev)):
        out_dev.fill_(7)
        with pytest.raises(z.ZeroError) as e:
            z.zero_gather_range(src, pitch, psi, nd, begin, length, 2, dst)
        assert e.value.status == z.ZERO_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert bool((dst == 7).all()), "a refused gather wrote"


def test_gather_ranges_of_the_7p5b_model():
    """The ZeRO-3 range gather at the 7.5B model's full size: 64 shards of
    117,187,500 fp16 parameters (15 GB, slots 8-element pitched), each slot
    holding a closed-form function of the flat parameter index.  Ranges past
    2^32 elements, across four shard boundaries, and ending on the model's
    last parameter come back as exactly that function of their flat
    indices."""
    psi, nd = 7_500_000_000, 64
    s = -(-psi // nd)
    pitch = -(-s // 8) * 8
    dev = torch.device("cuda")

    def f(flat):   # the parameter at flat index `flat`, as 16 bits (no int64 overflow)
        return ((flat * 331_804_481) >> 7) & 0xFFFF

    shards = torch.zeros(nd * pitch, dtype=torch.int16, device=dev)
    for r in range(nd):
        n = min(s, psi - r * s)
        idx = torch.arange(r * s, r * s + n, dtype=torch.int64, device=dev)
        shards[r * pitch:r * pitch + n] = f(idx).to(torch.int32).to(torch.int16)
        del idx
    for begin, length in [(60 * s - 12_345, 3 * s + 77), (psi - 1_000, 1_000),
                          ((1 << 32) + 13, 5_000_000), (s - 1, 2)]:
        out = torch.empty(length, dtype=torch.int16, device=dev)
        z.zero_gather_range(shards, pitch, psi, nd, begin, length, 2, out)
        want = f(torch.arange(begin, begin + length, dtype=torch.int64, device=dev))
        torch.cuda.synchronize()
        assert torch.equal(out.to(torch.int64) & 0xFFFF, want), (begin, length)
        del out, want
