"""Pins of the oracle's fp16 / bf16 codecs against library routines.

The mixed-precision step stores fp16 (or bf16) parameters and gradients next to
fp32 master state ("ZeRO: Memory Optimizations Toward Training Trillion
Parameter Models", section on quantifying memory consumption).  The oracle
encodes and decodes them with its own code written from the IEEE 754 binary16
and bfloat16 definitions; these tests pin that code to numpy's float16 and
torch's bfloat16 conversions, exhaustively where the domain allows.
"""
import numpy as np
import pytest
import torch

F16, BF16 = 0, 1


def _all16():
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def test_decode_f16_exhaustive(orc):
    h = _all16()
    got = orc.decode(h, F16)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_decode_bf16_exhaustive(orc):
    h = _all16()
    got = orc.decode(h, BF16)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _probe_floats(rng):
    """Random bit patterns over every exponent, exact midpoints between
    adjacent 16-bit values (ties), and the format boundaries."""
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    return x


def _midpoints(decoded: np.ndarray) -> np.ndarray:
    """Midpoints of adjacent finite values (exact in fp32 for both formats)."""
    d = decoded[np.isfinite(decoded)].astype(np.float64)
    d = np.unique(d)
    mids = (d[1:] + d[:-1]) / 2
    f = mids.astype(np.float32)
    return f[f.astype(np.float64) == mids]   # keep the exactly representable ones


def test_encode_f16_vs_numpy(orc):
    rng = np.random.default_rng(0)
    h = _all16()
    x = np.concatenate([_probe_floats(rng), _midpoints(orc.decode(h, F16)),
                        orc.decode(h, F16),
                        np.array([65504, 65519.996, 65520, 65536, 1e-8, 2.0 ** -25,
                                  2.0 ** -24 * 1.5, 2.0 ** -14 - 2.0 ** -25, -0.0, np.inf,
                                  -np.inf], np.float32)])
    got = orc.encode(x, F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(orc.decode(got[nan], F16)))


def test_encode_bf16_vs_torch(orc):
    rng = np.random.default_rng(1)
    h = _all16()
    x = np.concatenate([_probe_floats(rng), _midpoints(orc.decode(h, BF16)),
                        orc.decode(h, BF16),
                        np.array([3.3895314e38, 3.4e38, np.finfo(np.float32).max, 1e-40,
                                  -0.0, np.inf, -np.inf], np.float32)])
    got = orc.encode(x, BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(orc.decode(got[nan], BF16)))


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2.0 ** -11, 0x3C00),        # tie between 1 and 1+2^-10: to even (1.0)
    (1.0 + 3 * 2.0 ** -11, 0x3C02),    # tie between odd 0x3C01 and even 0x3C02
    (65504.0, 0x7BFF),                 # largest finite
    (65520.0, 0x7C00),                 # tie with 2^16 rounds to even -> inf
    (2.0 ** -24, 0x0001),              # smallest subnormal
    (2.0 ** -25, 0x0000),              # tie with 0 -> even (0)
    (-(2.0 ** -14), 0x8400),           # smallest normal, negative
])
def test_encode_f16_hand_cases(orc, x, bits):
    assert int(orc.encode(np.array([x], np.float32), F16)[0]) == bits


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2.0 ** -8, 0x3F80),         # tie -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),     # tie -> even (0x3F82)
    (2.0 ** -133, 0x0001),             # smallest bf16 subnormal
])
def test_encode_bf16_hand_cases(orc, x, bits):
    assert int(orc.encode(np.array([x], np.float32), BF16)[0]) == bits


def test_roundtrip(orc):
    h = _all16()
    for dt in (F16, BF16):
        d = orc.decode(h, dt)
        ok = ~np.isnan(d)
        assert np.array_equal(orc.encode(d[ok], dt), h[ok])
