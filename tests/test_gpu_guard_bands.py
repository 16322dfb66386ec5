"""Guard bands: no entry point writes a byte outside the buffers it is given.

Every output buffer (new state, gathered parameters, fusion buffer, flag,
gather destination) is carved out of a larger allocation with 4 KiB canary
bands of a fixed byte pattern before and after it.  The entry points run on
ragged shards (lengths not a multiple of 8, slots off a 16-byte boundary):
one of 20,004 elements in buckets of 6,001, and one of 25,165,890 elements,
which the fused step runs as three launch windows whose rows start half a
32-byte sector in (the cuts move by that phase).  The bands must come back
byte for byte.
"""
import dataclasses

import pytest
import torch

import oracle
import synth
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, full_rows, make_group

pytestmark = pytest.mark.gpu

BAND = 4096          # bytes
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


class Guarded:
    """A device buffer of `count` elements of `dtype` between two canary bands
    (its start 16-byte aligned, plus `phase` elements)."""

    def __init__(self, count: int, dtype: torch.dtype, phase: int = 0):
        esize = torch.empty(0, dtype=dtype).element_size()
        self.lead = BAND + phase * esize
        self.nbytes = count * esize
        self.raw = torch.full((self.lead + self.nbytes + BAND,), PATTERN, dtype=torch.uint8,
                              device=DEV)
        self.view = self.raw[self.lead:self.lead + self.nbytes].view(dtype)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head = self.raw[:self.lead]
        tail = self.raw[self.lead + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _guarded_state(n):
    bufs = [Guarded(n, torch.float32) for _ in range(3)]
    return bufs, z.state(*(b.view for b in bufs))


# (psi, nd, rank, bucket):
#  - psi = 64 * 20003 + 5: shards of 20,004 (S mod 8 = 4); rank 3's slot in a
#    flat buffer starts 8 bytes past a 16-byte boundary; buckets of 6,001;
#  - S = 25,165,893 over 2 ranks: rank 1 holds 25,165,890 elements (three launch
#    windows of the fused step); the row pitch is 8 elements past a multiple of
#    16, so rank 1's rows start 16 bytes into a 32-byte sector and the window
#    cuts shift by 8 elements; its slot starts 10 bytes past a 16-byte
#    boundary; buckets of 4,194,304.
SHAPES = [(64 * 20_003 + 5, 64, 3, 6_001), (2 * 25_165_893 - 3, 2, 1, 1 << 22)]


@pytest.mark.parametrize("shape", SHAPES, ids=["64 ranks", "three launch windows"])
@pytest.mark.parametrize("path", ["ring", "registers", "tma", "small", "unfused", "streamed"])
def test_step_paths_stay_inside_their_buffers(path, shape, monkeypatch):
    psi, nd, rank, bucket = shape
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=psi, nd=nd, plant=None)
    if path in ("ring", "registers", "tma", "small"):
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    monkeypatch.setenv("ZERO_STREAM_GROUP_BYTES", "0")
    dps = make_group(w, ranks=[rank], gathered="full")
    buf, desc = full_rows(w, dps, 0)
    L = dps.layouts[rank]
    n = int(L.length)
    assert z.fused_launch_count(n, bucket) == (3 if nd == 2 else 1)
    st = dps.state[rank]
    outs, s_out = _guarded_state(n)
    gath = Guarded(n, torch.bfloat16, phase=int(L.begin) % 8)
    flag = Guarded(1, torch.int32)
    flag.view.zero_()
    h = z.adamw(w.hparams["lr"], 0.9, 0.999, 1e-8, 0.01, 1)
    if path == "unfused":
        cb = Guarded(bucket + 4, torch.float32)
        z.zero_step_shard_unfused(desc[rank], L, st.states[st.cur], s_out, gath.view, 0, bucket,
                                  w.loss_scale, h, cb.view, bucket + 4, flag.view)
        assert cb.intact(), "fusion buffer bands"
    elif path == "streamed":
        ready = torch.ones(-(-n // bucket), dtype=torch.int32, device=DEV)
        status = Guarded(1, torch.int32)
        status.view.zero_()
        z.zero_step_shard_streamed(desc[rank], L, st.states[st.cur], s_out, gath.view, 0,
                                   bucket, w.loss_scale, h, ready, 1, 10 ** 9, flag.view,
                                   status.view)
        assert status.intact() and int(status.view.item()) == 0
    else:
        z.zero_step_shard(desc[rank], L, st.states[st.cur], s_out, gath.view, 0, bucket,
                          w.loss_scale, h, flag.view)
    for i, b in enumerate(outs):
        assert b.intact(), f"state array {i} bands"
    assert gath.intact(), "gathered slot bands"
    assert flag.intact() and int(flag.view.item()) == 0
    # and the outputs match the library's own step into plain buffers
    ref = make_group(w, ranks=[rank], gathered="full")
    assert not ref.step(desc)
    for a, b in zip(ref.state[rank].tensors(), outs):
        assert torch.equal(a.view(torch.int32), b.view.view(torch.int32))
    lo = int(L.begin)
    assert torch.equal(ref.gathered_view()[lo:lo + n].view(torch.int16),
                       gath.view.view(torch.int16))


def test_primitives_and_gather_stay_inside_their_buffers():
    w = dataclasses.replace(synth.WORKLOADS["c1"], psi=8 * 30_001 + 3, nd=8, plant=None)
    rank = 5
    dps = make_group(w, ranks=[rank], gathered="full")
    buf, desc = full_rows(w, dps, 0)
    L = dps.layouts[rank]
    n = int(L.length)
    flag = Guarded(1, torch.int32)
    flag.view.zero_()
    cb = Guarded(n, torch.float32, phase=1)
    z.zero_reduce_scatter_bucket(desc[rank], 0, n, 0.125, cb.view, flag.view)
    assert cb.intact() and flag.intact()
    z.zero_check_nonfinite(desc[rank], 0, n, flag.view)
    assert flag.intact() and int(flag.view.item()) == 0
    st = dps.state[rank]
    outs, s_out = _guarded_state(n)
    grad = torch.zeros(n, dtype=torch.float32, device=DEV)
    z.zero_adam_step_shard(grad, st.states[st.cur], s_out, n, z.adamw(1e-4, 0.9, 0.999, 1e-8,
                                                                        0.01, 1))
    assert all(b.intact() for b in outs)
    slot = Guarded(n, torch.float16, phase=3)
    z.zero_gather_params_shard(outs[0].view, n, slot.view, 0, "f16")
    assert slot.intact()
    # a ZeRO-3 range gather across three shards into an odd-phase destination
    psi, nd = 1_000_003, 7
    s = -(-psi // nd)
    pitch = -(-s // 8) * 8
    shards = torch.randint(-30000, 30000, (nd, pitch), dtype=torch.int16, device=DEV)
    begin, length = s - 1001, 2 * s + 77
    dst = Guarded(length, torch.int16, phase=5)
    z.zero_gather_range(shards, pitch, psi, nd, begin, length, 2, dst.view)
    assert dst.intact()
    flat = torch.cat([shards[r, :min(s, psi - r * s)] for r in range(nd)])
    assert torch.equal(dst.view, flat[begin:begin + length])
