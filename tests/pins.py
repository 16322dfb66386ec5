"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` takes the ``oracle`` module and raises AssertionError on a
mismatch.  The pins are: library routines (numpy float16, torch bfloat16,
``math.fsum``, ``torch.optim.AdamW`` in float64), closed forms, values the
pages print (see ``golden/``), hand-derived values and structural invariants
the method implies (ZeRO-DP: each rank updates only its 1/Nd, so the
concatenation of every shard's update is the unsharded data-parallel update).
The same checks run against mutated copies of the oracle in
``test_oracle_mutations.py`` to show that plausible mistakes fail them.
"""
from __future__ import annotations

import math

import numpy as np
import torch

F16, BF16 = 0, 1
U = 2.0 ** -24
H = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


# -- codecs ----------------------------------------------------------------

def check_codec(orc, n_random: int = 1 << 16):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref16 = h.view(np.float16).astype(np.float32)
    refbf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    for dt, ref in ((F16, ref16), (BF16, refbf)):
        got = orc.decode(h, dt)
        ok = ~np.isnan(ref)
        assert np.array_equal(np.isnan(got), ~ok)
        assert np.array_equal(got[ok].view(np.uint32), ref[ok].view(np.uint32)), "decode"
    rng = np.random.default_rng(7)
    x = rng.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = np.concatenate([x, ref16[np.isfinite(ref16)], (ref16[1:1024] + ref16[2:1025]) / 2,
                        np.float32([65520, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11])])
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        assert np.array_equal(orc.encode(x, F16), x.astype(np.float16).view(np.uint16)), "f16"
    refb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.encode(x, BF16), refb), "bf16"


# -- layout / accounting ----------------------------------------------------

def check_layout(orc):
    for psi in range(0, 70):
        for nd in range(1, 10):
            cov = []
            for r in range(nd):
                s, b, n = orc.layout(psi, nd, r)
                assert s == -(-psi // nd) and b == r * s
                cov.extend(range(b, b + n))
            assert cov == list(range(psi)), (psi, nd)


def check_accounting(orc):
    psi = 7_500_000_000
    table = {1: ("120", "120", "120", "120"), 64: ("120", "31.4", "16.6", "1.88"),
             1024: ("120", "30.1", "15.1", "0.12")}
    for nd, row in table.items():
        for st, printed in enumerate(row):
            dec = len(printed.split(".")[1]) if "." in printed else 0
            got = orc.model_state_bytes(psi, nd, st, 12) / 1e9
            assert round(got, dec) == float(printed), (nd, st, got)
    assert orc.model_state_bytes(1_500_000_000, 1, 0, 12) == 24 * 10 ** 9


# -- reduction -------------------------------------------------------------

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def check_fold(orc):
    rng = np.random.default_rng(3)
    # 1) Coarse grid: every partial sum is exact in fp32, so the fold equals
    #    the exact integer sum.
    for dt, lim in ((F16, 2000), (BF16, 255)):
        for nd in (1, 2, 5, 64):
            k = rng.integers(-lim, lim + 1, size=(nd, 257))
            vals = (k * 2.0 ** -4).astype(np.float32)
            bits = vals.astype(np.float16).view(np.uint16) if dt == F16 else _bf16_bits(vals)
            got = orc.fold(bits, dt)
            assert np.array_equal(got.astype(np.float64), k.sum(0) * 2.0 ** -4), (dt, nd)
    # 2) Order probes with hand-derived results.  [1, 2^25, -2^25, 1]:
    #    (1 + 2^25) rounds to 2^25, minus 2^25 is 0, plus 1 is 1; a pairwise
    #    tree gives (1 + 2^25) + (-2^25 + 1) = 2^25 - 2^25 = 0.
    probe = _bf16_bits(np.float32([1, 2 ** 25, -(2 ** 25), 1])).reshape(4, 1)
    assert orc.fold(probe, BF16)[0] == 1.0
    #    [2^25, 1, 1, 1, 1]: each +1 is lost (2^25 + 1 rounds to 2^25); the
    #    reverse order gives 2^25 + 4.
    probe = _bf16_bits(np.float32([2 ** 25, 1, 1, 1, 1])).reshape(5, 1)
    assert orc.fold(probe, BF16)[0] == 2.0 ** 25
    # 3) Random data: within the recursive-summation bound of the exactly
    #    rounded sum (math.fsum).
    nd = 64
    x = (rng.standard_normal((nd, 300)) * 1024e-3).astype(np.float16)
    got = orc.fold(x.view(np.uint16), F16).astype(np.float64)
    xs = x.astype(np.float64)
    for i in range(xs.shape[1]):
        exact = math.fsum(xs[:, i])
        gamma = (nd - 1) * U / (1 - (nd - 1) * U)
        assert abs(got[i] - exact) <= gamma * np.abs(xs[:, i]).sum() + 1e-30, i


# -- AdamW -------------------------------------------------------------------

def torch_adamw_f64(p, m, v, g, h, t):
    """One AdamW step of torch.optim.AdamW in float64 from state (m, v, t-1)."""
    param = torch.nn.Parameter(torch.from_numpy(np.asarray(p, np.float64).copy()))
    opt = torch.optim.AdamW([param], lr=h["lr"], betas=(h["beta1"], h["beta2"]), eps=h["eps"],
                            weight_decay=h["weight_decay"], foreach=False)
    opt.state[param] = {"step": torch.tensor(float(t - 1)),
                        "exp_avg": torch.from_numpy(np.asarray(m, np.float64).copy()),
                        "exp_avg_sq": torch.from_numpy(np.asarray(v, np.float64).copy())}
    param.grad = torch.from_numpy(np.asarray(g, np.float64).copy())
    opt.step()
    st = opt.state[param]
    return param.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def adamw_bounds(p, m, v, g, sum_abs_g, nd, h, t):
    """Per-element error bounds of the fp32 step (every operation correctly
    rounded, scalars rounded once) against the exact result, derived from the
    standard model |fl(x op y) - x op y| <= u |x op y|, times a safety of 2."""
    b1, b2, lr, eps = h["beta1"], h["beta2"], h["lr"], h["eps"]
    c1, c2 = 1 - b1, 1 - b2
    bc1, bc2 = 1 - b1 ** t, 1 - b2 ** t
    gamma = (nd - 1) * U / (1 - (nd - 1) * U)
    e_g = gamma * sum_abs_g + U * np.abs(g)
    m1 = b1 * m + c1 * g
    v1 = b2 * v + c2 * g * g
    e_m = 4 * U * (np.abs(b1 * m) + np.abs(c1 * g)) + c1 * e_g
    e_v = 4 * U * (np.abs(b2 * v) + c2 * g * g) + c2 * (2 * np.abs(g) * e_g + e_g ** 2)
    mh, vh = m1 / bc1, v1 / bc2
    e_mh = e_m / bc1 + 2 * U * np.abs(mh)
    e_vh = e_v / bc2 + 2 * U * np.abs(vh)
    sq = np.sqrt(vh)
    with np.errstate(divide="ignore", invalid="ignore"):
        e_sq = np.where(sq > 0, np.minimum(e_vh / (2 * sq), np.sqrt(e_vh)), np.sqrt(e_vh))
    e_sq = e_sq + U * sq
    den = sq + eps
    e_den = e_sq + U * den + U * eps
    upd = mh / den
    e_upd = e_mh / den + np.abs(upd) * e_den / den + 2 * U * np.abs(upd)
    p1 = p * (1 - lr * h["weight_decay"]) - lr * upd
    e_p = 3 * U * np.abs(p) + lr * e_upd + 3 * U * lr * np.abs(upd) + U * np.abs(p1)
    return 2 * e_p, 2 * e_m, 2 * e_v


def _random_case(rng, nd, n, dt, ls, zero_state=False):
    c = rng.standard_normal((nd, n)) * 1e-3 * ls
    c[:, :5] = 0.0                                   # zero-gradient elements
    bits = c.astype(np.float16).view(np.uint16) if dt == F16 else _bf16_bits(c)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    if zero_state:
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
    else:
        m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
        v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    return bits, p, m, v


def check_adamw_vs_torch(orc, n: int = 2000):
    rng = np.random.default_rng(11)
    for dt, ls, nd, zero_state, t in ((F16, 1024.0, 4, True, 1), (BF16, 1.0, 8, False, 1),
                                      (F16, 1024.0, 16, False, 5), (BF16, 1.0, 64, False, 20)):
        bits, p, m, v = _random_case(rng, nd, n, dt, ls, zero_state)
        skipped, p1, m1, v1, params = orc.step_unsharded(bits, dt, ls, H, t, p, m, v)
        assert not skipped
        c = orc.decode(bits, dt).astype(np.float64)
        g = np.array([math.fsum(c[:, i]) for i in range(n)]) / (nd * ls)
        sum_abs = np.abs(c).sum(0) / (nd * ls)
        rp, rm, rv = torch_adamw_f64(p, m, v, g, H, t)
        ep, em, ev = adamw_bounds(p.astype(np.float64), m.astype(np.float64),
                                  v.astype(np.float64), g, sum_abs, nd, H, t)
        assert np.all(np.abs(m1 - rm) <= em), ("m", dt, nd, t)
        assert np.all(np.abs(v1 - rv) <= ev), ("v", dt, nd, t)
        assert np.all(np.abs(p1 - rp) <= ep), ("p", dt, nd, t)
        # the cast is round-to-nearest-even of the new master weight
        if dt == F16:
            assert np.array_equal(params, p1.astype(np.float16).view(np.uint16))
        else:
            assert np.array_equal(params, _bf16_bits(p1))


def check_closed_forms(orc):
    rng = np.random.default_rng(5)
    n, nd = 64, 4
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    wdf = np.float32(1 - H["lr"] * H["weight_decay"])
    # Zero gradient from zero moments: only decoupled weight decay acts.
    skipped, p1, m1, v1, _ = orc.step_unsharded(np.zeros((nd, n), np.uint16), F16, 1024.0, H, 1,
                                                p, z, z)
    assert not skipped
    assert np.array_equal(p1, p * wdf) and not m1.any() and not v1.any()
    # First step from m = v = 0: the bias-corrected moments are g and g^2, so
    # the update is lr * g / (|g| + eps), about lr * sign(g).
    bits, p, m, v = _random_case(rng, nd, n, F16, 1024.0, zero_state=True)
    _, p1, m1, v1, _ = orc.step_unsharded(bits, F16, 1024.0, H, 1, p, m, v)
    c = orc.decode(bits, F16).astype(np.float64)
    g = np.array([math.fsum(c[:, i]) for i in range(n)]) / (nd * 1024.0)
    closed = p.astype(np.float64) * (1 - H["lr"] * H["weight_decay"]) - H["lr"] * g / (
        np.abs(g) + H["eps"])
    ep, em, ev = adamw_bounds(p.astype(np.float64), 0.0 * g, 0.0 * g, g,
                              np.abs(c).sum(0) / (nd * 1024.0), nd, H, 1)
    assert np.all(np.abs(p1 - closed) <= ep)
    assert np.all(np.abs(m1 - 0.1 * g) <= em) and np.all(np.abs(v1 - 0.001 * g * g) <= ev)
    # Scalars: at t = 1 the bias correction 1 - b1 equals c1; power-of-two scaling.
    s = orc.scalars(H, 1, 4, 1024.0)
    assert s.bc1 == s.c1 and s.inv == 2.0 ** -12
    assert s.wdf == np.float32(1 - 1e-6)


# -- structure ---------------------------------------------------------------

def padded_grads(full_rows: np.ndarray, psi: int, nd: int, pitch: int) -> np.ndarray:
    """Place [nd, psi] flat gradients into the padded-partition layout [nd, nd*pitch]."""
    s = -(-psi // nd)
    out = np.zeros((nd, nd * pitch), np.uint16)
    for r in range(nd):
        b = r * s
        n = max(0, min(s, psi - b))
        out[:, r * pitch:r * pitch + n] = full_rows[:, b:b + n]
    return out


def check_shard_invariant(orc):
    rng = np.random.default_rng(9)
    for psi, nd, dt, bucket in ((1000, 4, F16, 64), (1001, 7, BF16, 100), (3, 5, F16, 2),
                                (513, 1, BF16, 1000), (200, 16, F16, 7)):
        ls = 1024.0 if dt == F16 else 1.0
        bits, p, m, v = _random_case(rng, nd, psi, dt, ls)
        skipped, p1, m1, v1, params = orc.step_unsharded(bits, dt, ls, H, 3, p, m, v)
        s = -(-psi // nd)
        pitch = -(-s // 8) * 8
        gathered = np.full(nd * s + 8, 0xABCD, np.uint16)
        f, q1, n1, w1 = orc.step_sharded(padded_grads(bits, psi, nd, pitch), psi, nd, pitch, dt,
                                         bucket, ls, H, 3, p, m, v, gathered)
        assert f == 0 and not skipped
        for a, b in ((p1, q1), (m1, n1), (v1, w1)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (psi, nd)
        assert np.array_equal(gathered[:psi], params)
        assert np.all(gathered[psi:] == 0xABCD)   # padding slots are never written


def check_bucket_invariance(orc):
    rng = np.random.default_rng(13)
    n, nd = 300, 3
    bits, p, m, v = _random_case(rng, nd, n, BF16, 1.0)
    ref = None
    for bucket in (1, 7, 64, 300, 65536):
        out = np.zeros(n, np.uint16)
        f, q, mm, vv = orc.step_rank(bits, n, 0, n, nd, BF16, bucket, 1.0, H, 2, p, m, v, out, 0)
        cur = (q.tobytes(), mm.tobytes(), vv.tobytes(), out.tobytes())
        assert f == 0
        ref = ref or cur
        assert cur == ref, bucket


def check_skip(orc):
    rng = np.random.default_rng(17)
    psi, nd = 500, 4
    bits, p, m, v = _random_case(rng, nd, psi, F16, 1024.0)
    tr = orc.Trajectory(F16, 1024.0, H, p, m, v)
    assert not tr.step(bits)
    snap = (tr.p.copy(), tr.m.copy(), tr.v.copy(), tr.params.copy(), tr.t)
    bad = bits.copy()
    bad[2, 333] = 0x7C00                                  # +inf in one contribution
    assert tr.step(bad)
    assert tr.t == snap[4] == 1
    for a, b in zip((tr.p, tr.m, tr.v, tr.params), snap[:4]):
        assert np.array_equal(a, b)
    s = -(-psi // nd)
    pitch = -(-s // 8) * 8
    f, *_ = orc.step_sharded(padded_grads(bad, psi, nd, pitch), psi, nd, pitch, F16, 64, 1024.0,
                             H, 2, p, m, v, np.zeros(nd * s, np.uint16))
    assert f == 1
    # a sum that overflows fp32 from finite bf16 contributions also skips
    big = _bf16_bits(np.float32([3.0e38, 3.0e38])).reshape(2, 1)
    assert orc.step_unsharded(big, BF16, 1.0, H, 1, *(np.zeros(1, np.float32),) * 3)[0]


def check_f64_shadow(orc):
    rng = np.random.default_rng(19)
    for dt, ls, nd in ((F16, 1024.0, 16), (BF16, 1.0, 64)):
        n = 1000
        bits, p, m, v = _random_case(rng, nd, n, dt, ls)
        _, p1, m1, v1, _ = orc.step_unsharded(bits, dt, ls, H, 4, p, m, v)
        q, mm, vv = orc.step_unsharded_f64(bits, dt, ls, H, 4, p, m, v)
        c = orc.decode(bits, dt).astype(np.float64)
        ep, em, ev = adamw_bounds(p.astype(np.float64), m.astype(np.float64),
                                  v.astype(np.float64), c.sum(0) / (nd * ls),
                                  np.abs(c).sum(0) / (nd * ls), nd, H, 4)
        assert np.all(np.abs(p1 - q) <= ep) and np.all(np.abs(m1 - mm) <= em)
        assert np.all(np.abs(v1 - vv) <= ev)


def check_primitives_compose(orc):
    """The bucket reduce and AdamW-from-gradient primitives compose to the
    unsharded step (which the pins above tie to the library references)."""
    rng = np.random.default_rng(23)
    for dt, ls, nd in ((F16, 1024.0, 5), (BF16, 1.0, 64)):
        n = 777
        bits, p, m, v = _random_case(rng, nd, n, dt, ls)
        _, p1, m1, v1, _ = orc.step_unsharded(bits, dt, ls, H, 7, p, m, v)
        inv = orc.scalars(H, 7, nd, ls).inv
        f, g = orc.reduce_scaled(bits.reshape(-1), dt, n, 0, n, nd, inv)
        assert f == 0
        q, mm, vv = orc.adamw_from_grad(g, H, 7, p, m, v)
        for a, b in ((p1, q), (m1, mm), (v1, vv)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        # a window in the middle of the rows
        f, gw = orc.reduce_scaled(bits.reshape(-1), dt, n, 100, 50, nd, inv)
        assert np.array_equal(gw.view(np.uint32), g[100:150].view(np.uint32))


def check_comm_and_mp_accounting(orc):
    """Communication volumes 2/2/2/3 Psi and the ZeRO+MP example (1T params,
    16-way MP x 64-way DP fits a 32 GB GPU), both printed on the pages."""
    for stage, mult in ((0, 2), (1, 2), (2, 2), (3, 3)):
        assert orc.comm_volume_elems(10 ** 9, stage) == mult * 10 ** 9
    assert orc.comm_volume_elems(10, 4) == 2 ** 64 - 1
    per_gpu = orc.model_state_bytes_mp(10 ** 12, 64, 16, 3, 12)
    assert per_gpu == 16 * 10 ** 12 // 1024 and per_gpu < 32 * 10 ** 9
    # Nm = 1 is plain ZeRO-DP; the MP slice divides memory once more
    assert orc.model_state_bytes_mp(7_500_000_000, 64, 1, 2) == \
        orc.model_state_bytes(7_500_000_000, 64, 2)


def check_gather_range(orc):
    """The flat range of a partitioned buffer equals the same range of the
    concatenated shards (numpy concatenate), for every range on tiny cases."""
    rng = np.random.default_rng(29)
    for psi, nd in ((0, 3), (1, 1), (17, 4), (33, 5), (64, 8)):
        s = -(-psi // nd)
        pitch = -(-max(s, 1) // 8) * 8
        for dt in (np.uint16, np.float32):
            shards = rng.integers(0, 60000, size=(nd, pitch)).astype(dt)
            flat = np.concatenate([shards[r, :max(0, min(s, psi - r * s))] for r in range(nd)])
            for b in range(psi + 1):
                for ln in range(psi - b + 1):
                    got = orc.gather_range(shards, psi, nd, b, ln)
                    assert np.array_equal(got, flat[b:b + ln]), (psi, nd, b, ln)


ALL = [check_codec, check_layout, check_accounting, check_fold, check_adamw_vs_torch,
       check_closed_forms, check_shard_invariant, check_bucket_invariance, check_skip,
       check_f64_shadow, check_primitives_compose, check_comm_and_mp_accounting,
       check_gather_range]
