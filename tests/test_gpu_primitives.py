"""GPU parity of the unfused primitives against the oracle, through the C ABI.

zero_reduce_scatter_bucket (bit-exact sums), zero_check_nonfinite,
zero_adam_step_shard and zero_gather_params_shard, on sizes that span many
CTAs with ragged heads and tails, unaligned windows and every slot phase, with
canary bands around every output to catch stray writes.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, TORCH_DT, assert_params_close, assert_state_close, f32, u16

pytestmark = pytest.mark.gpu

H = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
CANARY = 4096          # guard elements on each side of an output buffer


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rand_grads(rng, nd, row_stride, dt, ls):
    x = rng.standard_normal((nd, row_stride)) * 1e-3 * ls
    t = torch.from_numpy(x).to(torch.float32).to(TORCH_DT[dt])
    return t


def _guarded(n, dtype, fill):
    t = torch.full((n + 2 * CANARY,), fill, dtype=dtype, device=DEV)
    return t, t[CANARY:CANARY + n]


@pytest.mark.parametrize("dt,nd,n,begin,cb_shift", [
    ("f16", 1, 1000, 0, 0), ("bf16", 3, 300_001, 0, 0), ("f16", 8, 123_457, 5, 0),
    ("bf16", 64, 40_003, 3, 1), ("f16", 16, 7, 1, 0), ("bf16", 5, 65_536, 8, 2),
    ("f16", 2, 1, 7, 3),
])
def test_reduce_scatter_bucket_bit_exact(orc, dt, nd, n, begin, cb_shift):
    rng = np.random.default_rng(n + nd)
    ls = 1024.0 if dt == "f16" else 1.0
    row_stride = -(-(begin + n + 16) // 8) * 8
    host = _rand_grads(rng, nd, row_stride, dt, ls)
    dev = host.to(DEV)
    offset = 8 if begin + n + 8 <= row_stride else 0
    g = z.grads(dev, row_stride, offset, nd, dt)
    inv = float(np.float32(1.0 / (nd * ls)))
    buf = torch.full((n + cb_shift + 2 * CANARY,), -7.0, dtype=torch.float32, device=DEV)
    cb = buf[CANARY + cb_shift:CANARY + cb_shift + n]
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    z.zero_reduce_scatter_bucket(g, begin, n, inv, cb, flag)
    torch.cuda.synchronize()
    f, ref = orc.reduce_scaled(u16(host).reshape(-1), orc.dtype_code(dt), row_stride,
                               offset + begin, n, nd, inv)
    got = f32(cb)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert int(flag.item()) == f == 0
    b = f32(buf)
    assert (b[:CANARY + cb_shift] == -7.0).all() and (b[CANARY + cb_shift + n:] == -7.0).all()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_nonfinite_flag_and_precheck(orc, dt):
    rng = np.random.default_rng(1)
    nd, n = 6, 50_001
    row_stride = -(-n // 8) * 8 + 8
    host = _rand_grads(rng, nd, row_stride, dt, 1.0)
    cases = {"clean": None, "inf": (3, 41_000, float("inf")), "nan": (0, 17, float("nan")),
             "ninf": (5, n - 1, float("-inf"))}
    for name, plant in cases.items():
        h = host.clone()
        if plant:
            h[plant[0], plant[1]] = plant[2]
        dev = h.to(DEV)
        g = z.grads(dev, row_stride, 0, nd, dt)
        for fn in ("reduce", "check"):
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            if fn == "reduce":
                cb = torch.empty(n, dtype=torch.float32, device=DEV)
                z.zero_reduce_scatter_bucket(g, 0, n, 1.0, cb, flag)
            else:
                z.zero_check_nonfinite(g, 0, n, flag)
            torch.cuda.synchronize()
            assert int(flag.item()) == (0 if plant is None else 1), (name, fn)
    if dt == "bf16":   # finite contributions whose fp32 sum overflows
        h = torch.zeros(2, 16, dtype=torch.bfloat16)
        h[:, 9] = 3.0e38
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        z.zero_check_nonfinite(z.grads(h.to(DEV), 16, 0, 2, dt), 0, 16, flag)
        torch.cuda.synchronize()
        assert int(flag.item()) == 1
        f, _ = orc.reduce_scaled(u16(h).reshape(-1), orc.BF16, 16, 0, 16, 2, 1.0)
        assert f == 1


@pytest.mark.parametrize("n,shift,inplace", [(1, 0, False), (1001, 0, False), (250_003, 1, False),
                                             (77_777, 2, True), (64, 3, False)])
def test_adam_step_shard(orc, n, shift, inplace):
    rng = np.random.default_rng(n)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[:3] = 0.0
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    t = 9
    # state buffers 16-byte aligned; the gradient possibly at another phase
    gdev = torch.zeros(n + 8, dtype=torch.float32, device=DEV)[shift:shift + n]
    gdev.copy_(torch.from_numpy(g))
    ins = [torch.from_numpy(a).to(DEV) for a in (p, m, v)]
    outs = ins if inplace else [torch.full((n,), 5.0, device=DEV) for _ in range(3)]
    z.zero_adam_step_shard(gdev, z.state(*ins), z.state(*outs), n,
                           z.adamw(H["lr"], H["beta1"], H["beta2"], H["eps"],
                                   H["weight_decay"], t))
    torch.cuda.synchronize()
    rp, rm, rv = orc.adamw_from_grad(g, H, t, p, m, v)
    assert_state_close(f32(outs[0]), rp, 1e-12, "master")
    assert_state_close(f32(outs[1]), rm, 1e-20, "m")
    assert_state_close(f32(outs[2]), rv, 1e-20, "v")


def _special_floats(rng, n):
    x = (rng.standard_normal(n) * 0.02).astype(np.float32)
    sp = np.float32([0.0, -0.0, np.inf, -np.inf, np.nan, 65504, 65519.99, 65520, 1e6, -1e6,
                     1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -24, 2 ** -25, 3 * 2 ** -26, 1e-40,
                     3.4e38, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -133, -2 ** -134])
    x[:sp.size] = sp
    bits = rng.integers(0, 1 << 32, n // 4, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x[sp.size:sp.size + bits.size] = bits
    return x


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("master_shift", [0, 1, 3])
def test_gather_params_shard_all_phases(orc, dt, master_shift):
    rng = np.random.default_rng(master_shift)
    n = 100_003
    x = _special_floats(rng, n)
    mdev = torch.zeros(n + 4, dtype=torch.float32, device=DEV)[master_shift:master_shift + n]
    mdev.copy_(torch.from_numpy(x))
    ref = orc.encode(x, orc.dtype_code(dt))
    fill = -3.0
    for slot in range(8):
        buf, _ = _guarded(n + 8, TORCH_DT[dt], fill)
        z.zero_gather_params_shard(mdev, n, buf[CANARY:], slot, dt)
        torch.cuda.synchronize()
        got = u16(buf[CANARY + slot:CANARY + slot + n])
        nan = np.isnan(x)
        assert_params_close(got[~nan], ref[~nan], f"{dt} slot {slot}")
        assert np.isnan(orc.decode(got[nan], orc.dtype_code(dt))).all()
        fill_bits = torch.tensor([fill], dtype=TORCH_DT[dt]).view(torch.int16).item()
        rest = torch.cat([buf[:CANARY + slot], buf[CANARY + slot + n:]]).view(torch.int16)
        assert bool((rest == fill_bits).all()), "write outside the slot"
