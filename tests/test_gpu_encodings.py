"""Every fp16 and bf16 encoding through the GPU fold, against the oracle.

The gradient contributions of the step are 2-byte floats ("ZeRO: Memory
Optimizations Toward Training Trillion Parameter Models", section
"Quantifying memory consumption": fp16 gradients, reduced in fp32).  Here each
of the 65,536 encodings of the gradient type -- zeros of both signs,
subnormals, the largest finite values, infinities and NaNs -- goes through the
kernels' decode and rank-ordered fp32 fold:

* one row (nd = 1): the decode alone;
* two rows, the second rotated against the first (every encoding meets many
  partners; a rotation by 32,768 pairs each value with its negation, an exact
  cancellation);
* three rows with a +max / -max pair around the encodings (rounding of a large
  intermediate, then cancellation).

The reduced, scaled sums must equal the oracle's bit for bit, except that a
NaN may carry any payload (the GPU's arithmetic returns its canonical NaN);
the nonfinite flag must agree.  The scale is 1 and 1/(nd * 1024), so scaled
subnormal sums are rounded too.  The same runs through the kernels'
one-element path (a window's ragged head), which decodes separately.  Then
the step runs over rows that hold subnormals and +-max finite values (and no
nonfinite sum) on every kernel variant and on the unfused path, against the
oracle's shard step: once as one shard (the 8-element path) and once with
every 7-element block as a shard of its own (the one-element path).
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_optimizer_02_gb300 as z
from gpu_util import DEV, assert_params_close, assert_state_close, f32, u16

pytestmark = pytest.mark.gpu

MAX_FINITE = {"f16": 0x7BFF, "bf16": 0x7F7F}
EXP_MASK = {"f16": 0x7C00, "bf16": 0x7F80}
H = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _all_encodings():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _row_cases(dt):
    """name -> [nd, 65536] uint16 contribution rows."""
    e = _all_encodings()
    mx = np.full_like(e, MAX_FINITE[dt])
    neg = mx | np.uint16(0x8000)
    return {
        "one row": e[None, :],
        "rotated by 1": np.stack([e, np.roll(e, 1)]),
        "rotated by 12,345": np.stack([e, np.roll(e, 12_345)]),
        "rotated by 32,768 (negations)": np.stack([e, np.roll(e, 32_768)]),
        "+max, encodings, -max": np.stack([mx, e, neg]),
        "encodings, +max, -max": np.stack([e, mx, neg]),
    }


def _device_rows(rows: np.ndarray, pad: int = 8):
    """rows [nd, n] uint16 into a device buffer with a 16-byte aligned pitch;
    returns (tensor, row_stride)."""
    nd, n = rows.shape
    stride = -(-(n + pad) // 8) * 8
    host = np.zeros((nd, stride), np.uint16)
    host[:, :n] = rows
    return torch.from_numpy(host.view(np.int16)).to(DEV), stride, host


def _same_bits_or_both_nan(got: np.ndarray, ref: np.ndarray, what: str):
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ ({(gn != rn).sum()})"
    diff = (got.view(np.uint32) != ref.view(np.uint32)) & ~rn
    assert not diff.any(), (f"{what}: {diff.sum()} sums differ, first at {np.argmax(diff)}: "
                            f"{got[np.argmax(diff)]!r} vs {ref[np.argmax(diff)]!r}")


@pytest.mark.parametrize("variant", ["ring", "registers", "small"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_every_encoding_folds_like_the_oracle(dt, variant, monkeypatch):
    """zero_reduce_scatter_bucket (the ring's reduction mode, or the register
    kernel) and zero_check_nonfinite over all 65,536 encodings."""
    monkeypatch.setenv("ZERO_FUSED_VARIANT", variant)
    code = oracle.dtype_code(dt)
    for name, rows in _row_cases(dt).items():
        nd, n = rows.shape
        dev, stride, host = _device_rows(rows)
        g = z.grads(dev, stride, 0, nd, dt)
        for inv in (1.0, float(np.float32(1.0 / (nd * 1024.0)))):
            cb = torch.full((n,), -7.0, dtype=torch.float32, device=DEV)
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            check = torch.zeros(1, dtype=torch.int32, device=DEV)
            z.zero_reduce_scatter_bucket(g, 0, n, inv, cb, flag)
            z.zero_check_nonfinite(g, 0, n, check)
            torch.cuda.synchronize()
            f, ref = orc_reduce(host, code, stride, n, nd, inv)
            what = f"{dt} {variant} {name} inv={inv}"
            _same_bits_or_both_nan(f32(cb), ref, what)
            assert int(flag.item()) == int(check.item()) == f, what


def orc_reduce(host, code, stride, n, nd, inv):
    return oracle.reduce_scaled(host.reshape(-1), code, stride, 0, n, nd, inv)


def _extreme_rows(dt):
    """Three contribution rows whose sums are finite but cover subnormals,
    exact cancellations and values next to +-max: row 0 holds every finite
    encoding, row 1 the negation of its neighbour (so the first add cancels to
    a few ulps, a subnormal for bf16), row 2 is +max or -max on every fourth
    element (unless the first two rows are too large to take a max without
    overflowing fp32) and 0 elsewhere."""
    e = _all_encodings()
    finite = e[(e & EXP_MASK[dt]) != EXP_MASK[dt]]
    a = finite
    b = np.roll(finite, 1) ^ np.uint16(0x8000)
    code = oracle.dtype_code(dt)
    big = np.maximum(np.abs(oracle.decode(a, code)), np.abs(oracle.decode(b, code))) >= 2.0 ** 100
    i = np.arange(a.size)
    c = np.where(i % 8 == 1, MAX_FINITE[dt], MAX_FINITE[dt] | 0x8000).astype(np.uint16)
    c[(i % 4 != 1) | big] = 0
    return np.stack([a, b, c])


@pytest.mark.parametrize("path", ["ring", "registers", "tma", "small", "unfused"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_step_over_extreme_rows(dt, path, monkeypatch):
    """zero_step_shard (each kernel) and zero_step_shard_unfused on rows of
    subnormals, cancellations and +-max finite values, against the oracle's
    shard step, element by element, into a slot at an odd phase."""
    if path != "unfused":
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    rows = _extreme_rows(dt)
    nd, n = rows.shape
    ls = 1024.0 if dt == "f16" else 1.0
    t = 3
    code = oracle.dtype_code(dt)
    rng = np.random.default_rng(n)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    dev, stride, host = _device_rows(rows)
    params = np.zeros(n, np.uint16)
    bucket = 4096
    f, rp, rm, rv = oracle.step_rank(host.reshape(-1), stride, 0, n, nd, code, bucket, ls, H, t,
                                     p, m, v, params, 0)
    assert f == 0, "the rows were built to give finite sums"
    L = z.zero_partition_layout(n, 1, 0, 8)
    pitch = int(L.row_pitch)
    st_in = torch.zeros(3, pitch, dtype=torch.float32, device=DEV)
    for k, a in enumerate((p, m, v)):
        st_in[k, :n] = torch.from_numpy(a)
    st_out = torch.zeros_like(st_in)
    slot = 3
    gath = torch.zeros(n + 16, dtype=torch.int16, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    g = z.grads(dev, stride, 0, nd, dt)
    h = z.adamw(H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], t)
    if path == "unfused":
        cb = torch.empty(bucket + 4, dtype=torch.float32, device=DEV)
        z.zero_step_shard_unfused(g, L, z.state(*st_in), z.state(*st_out), gath, slot, bucket,
                                  ls, h, cb, cb.numel(), flag)
    else:
        z.zero_step_shard(g, L, z.state(*st_in), z.state(*st_out), gath, slot, bucket, ls, h,
                          flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    for k, (ref, name, tau) in enumerate(((rp, "master", 1e-12), (rm, "m", 1e-20),
                                          (rv, "v", 1e-20))):
        got = f32(st_out[k, :n])
        if name == "v":        # g*g overflows to +inf where |g| is near the bf16 maximum
            inf = np.isinf(ref)
            assert np.array_equal(np.isinf(got), inf), f"{dt} {path} v: inf positions"
            got, ref = got[~inf], ref[~inf]
        assert_state_close(got, ref, tau, f"{dt} {path} {name}")
    assert_params_close(u16(gath[slot:slot + n]), params, f"{dt} {path} params")
    rest = torch.cat([gath[:slot], gath[slot + n:]])
    assert not rest.any(), "write outside the slot"


@pytest.mark.parametrize("variant", ["ring", "registers", "small"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_every_encoding_through_the_scalar_path(dt, variant, monkeypatch):
    """Ragged heads and tails of a window are folded one element at a time
    (widen1 / fold1), not in 8-element vectors.  Encoding i sits at element
    8*(i // 7) + 1 + i % 7 of its row, so every 7-element block starts one
    element past a 16-byte line; one call per block reduces the block alone,
    all of it as the window's scalar head.  One row (the decode alone) and
    two rows (the second rotated by 12,345), scale 1 and 1/(nd * 1024), bit
    for bit against the oracle (NaN payloads aside)."""
    monkeypatch.setenv("ZERO_FUSED_VARIANT", variant)
    code = oracle.dtype_code(dt)
    e = _all_encodings()
    nblk = -(-e.size // 7)
    pos = 8 * (np.arange(e.size) // 7) + 1 + np.arange(e.size) % 7
    stride = 8 * nblk + 8
    for nd in (1, 2):
        host = np.zeros((nd, stride), np.uint16)
        host[0, pos] = e
        if nd == 2:
            host[1, pos] = np.roll(e, 12_345)
        dev = torch.from_numpy(host.view(np.int16)).to(DEV)
        g = z.grads(dev, stride, 0, nd, dt)
        for inv in (1.0, float(np.float32(1.0 / (nd * 1024.0)))):
            cb = torch.full((stride,), -7.0, dtype=torch.float32, device=DEV)
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            for k in range(nblk):
                b0 = 8 * k + 1
                cnt = min(7, e.size - 7 * k)
                z.zero_reduce_scatter_bucket(g, b0, cnt, inv, cb[b0:b0 + cnt], flag)
            torch.cuda.synchronize()
            f, ref = oracle.reduce_scaled(host.reshape(-1), code, stride, 0, stride, nd, inv)
            what = f"{dt} {variant} nd={nd} inv={inv} scalar path"
            _same_bits_or_both_nan(f32(cb)[pos], ref[pos], what)
            assert int(flag.item()) == f == 1, what
            gaps = np.setdiff1d(np.arange(stride), pos)
            assert bool((f32(cb)[gaps] == -7.0).all()), f"{what}: a gap was written"


@pytest.mark.parametrize("path", ["ring", "registers", "tma", "small", "unfused"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_step_scalar_path_over_extreme_rows(dt, path, monkeypatch):
    """The step's scalar path (a shard's last n mod 8 elements) over the
    extreme rows: each 7-element block of them is stepped as a shard of its
    own, so every element goes through the one-element fold, AdamW and cast.
    Against the oracle's step of the same elements, bit for bit; the element
    after each block is never written."""
    if path != "unfused":
        monkeypatch.setenv("ZERO_FUSED_VARIANT", path)
    rows = _extreme_rows(dt)
    nd, cnt_all = rows.shape
    nblk = -(-cnt_all // 7)
    stride = 8 * nblk
    i = np.arange(cnt_all)
    pos = 8 * (i // 7) + i % 7
    host = np.zeros((nd, stride), np.uint16)
    host[:, pos] = rows
    ls = 1024.0 if dt == "f16" else 1.0
    t = 3
    code = oracle.dtype_code(dt)
    rng = np.random.default_rng(cnt_all + 1)
    p = (rng.standard_normal(stride) * 0.02).astype(np.float32)
    m = (rng.standard_normal(stride) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(stride) * 1e-6).astype(np.float32)
    params = np.zeros(stride, np.uint16)
    f, rp, rm, rv = oracle.step_rank(host.reshape(-1), stride, 0, stride, nd, code, 4096, ls, H,
                                     t, p, m, v, params, 0)
    assert f == 0
    dev = torch.from_numpy(host.view(np.int16)).to(DEV)
    st_in = torch.from_numpy(np.stack([p, m, v])).to(DEV)
    st_out = torch.full((3, stride), -5.0, dtype=torch.float32, device=DEV)
    gath = torch.zeros(stride + 8, dtype=torch.int16, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    cb = torch.empty(16, dtype=torch.float32, device=DEV)
    h = z.adamw(H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], t)
    for k in range(nblk):
        b0 = 8 * k
        cnt = min(7, cnt_all - 7 * k)
        L = z.zero_partition_layout(cnt, 1, 0, 8)
        g = z.grads(dev, stride, b0, nd, dt)
        s_in = z.state(st_in[0, b0:], st_in[1, b0:], st_in[2, b0:])
        s_out = z.state(st_out[0, b0:], st_out[1, b0:], st_out[2, b0:])
        if path == "unfused":
            z.zero_step_shard_unfused(g, L, s_in, s_out, gath, b0, 4096, ls, h, cb, cb.numel(),
                                      flag)
        else:
            z.zero_step_shard(g, L, s_in, s_out, gath, b0, 4096, ls, h, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    for k, (ref, name, tau) in enumerate(((rp, "master", 1e-12), (rm, "m", 1e-20),
                                          (rv, "v", 1e-20))):
        got = f32(st_out[k])[pos]
        r = ref[pos]
        if name == "v":
            inf = np.isinf(r)
            assert np.array_equal(np.isinf(got), inf), f"{dt} {path} v: inf positions"
            got, r = got[~inf], r[~inf]
        assert_state_close(got, r, tau, f"{dt} {path} {name} (scalar path)")
    assert_params_close(u16(gath[:stride])[pos], params[pos], f"{dt} {path} params (scalar path)")
    gaps = np.setdiff1d(np.arange(stride), pos)
    assert bool((f32(st_out)[:, gaps] == -5.0).all()), "an element after a block was written"
