"""Seeded, counter-based synthetic inputs for the ZeRO shard step.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds none of the optimizer's arithmetic: it only turns
(seed, tensor, step, rank, flat index) into a value, so that any element of any
input can be regenerated on either side, on the CPU or on a GPU, bit for bit.

Recipe (the same on every device):

* ``h = splitmix64(key + (i + 1) * GAMMA)`` where ``key`` mixes
  (seed, tensor id, step, contributing rank) and ``i`` is the flat parameter
  index (the index into the unsharded Psi-element parameter vector).
* The four 16-bit fields of ``h`` are summed (Irwin-Hall, n = 4); the centred
  integer ``c = 2 * sum - 4 * 65535`` is exact in int32 and in fp32.
* ``value = fp32(c) * fp32(sigma / STD)`` -- one correctly rounded fp32
  multiply -- then, for gradients, one round-to-nearest-even conversion to
  fp16 or bf16 by the library (torch ``Tensor.to``).  Both steps are correctly
  rounded on the CPU and on CUDA, so both sides see the same bits.

The Irwin-Hall sum is bell-shaped with the stated standard deviation and
bounded at +-3.46 sigma, so no gradient overflows unless one is planted.
"""
from __future__ import annotations

import math

import torch

from .workloads import WORKLOADS, Workload  # noqa: F401

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# Tensor ids used in the key.
T_MASTER, T_M, T_V, T_GRAD = 1, 2, 3, 4

# Standard deviation of c = 2*(u0+u1+u2+u3) - 4*65535 with u_k uniform on
# [0, 65535]: Var(u) = (65536^2 - 1)/12, so Var(c) = 4 * 4 * (65536^2 - 1)/12.
STD = math.sqrt(16.0 * (65536.0 ** 2 - 1.0) / 12.0)
CENTRE = 4 * 65535


def _signed(x: int) -> int:
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def splitmix64_int(x: int) -> int:
    """Scalar splitmix64 finaliser on Python ints (mod 2^64)."""
    z = x & MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor: int, step: int, rank: int) -> int:
    """64-bit key of one (seed, tensor, step, rank) stream."""
    k = splitmix64_int(seed * GAMMA + 0x632BE59BD9B4E019)
    k = splitmix64_int(k ^ (tensor * 0xD1B54A32D192ED03))
    k = splitmix64_int(k ^ (step * 0xAEF17502108EF2D9))
    k = splitmix64_int(k ^ (rank * 0x8CB92BA72F3D8DD7))
    return k


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor viewed as uint64."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def hash_tensor(key: int, idx: torch.Tensor) -> torch.Tensor:
    """splitmix64(key + (idx + 1) * GAMMA) for an int64 index tensor (wraps mod 2^64)."""
    x = (idx + 1) * _signed(GAMMA) + _signed(key)
    z = (x ^ _lsr(x, 30)) * _signed(MIX1)
    z = (z ^ _lsr(z, 27)) * _signed(MIX2)
    return z ^ _lsr(z, 31)


def centred_int(key: int, idx: torch.Tensor) -> torch.Tensor:
    """The exact centred Irwin-Hall integer c in [-262140, 262140] (int32)."""
    z = hash_tensor(key, idx)
    s = (z & 0xFFFF) + ((z >> 16) & 0xFFFF) + ((z >> 32) & 0xFFFF) + _lsr(z, 48)
    return (2 * s - CENTRE).to(torch.int32)


def scale_f32(sigma: float) -> torch.Tensor:
    """fp32(sigma / STD) as a 0-dim float32 tensor (so the multiply is an fp32 one)."""
    return torch.tensor(sigma / STD, dtype=torch.float32)


def normal_f32(seed: int, tensor: int, step: int, rank: int, idx: torch.Tensor,
               sigma: float) -> torch.Tensor:
    """fp32 values ~ N(0, sigma) (Irwin-Hall, n=4) at flat indices ``idx``."""
    c = centred_int(stream_key(seed, tensor, step, rank), idx).to(torch.float32)
    return c * scale_f32(sigma).to(idx.device)


def grad_values(w: Workload, step: int, contributor: int, idx: torch.Tensor) -> torch.Tensor:
    """Gradient contribution of rank ``contributor`` at flat indices ``idx``.

    Returns fp16 or bf16 (``w.grad_dtype``); the static loss scale is folded
    into sigma (fp16 workloads store the loss-scaled gradient).
    """
    gstep = step if w.fresh_grads else 0
    v = normal_f32(w.seed, T_GRAD, gstep, contributor, idx, w.grad_sigma * w.loss_scale)
    out = v.to(w.torch_grad_dtype)
    if w.plant is not None and step == w.plant[0]:
        pj, pidx = w.plant[1], w.plant[2]
        if contributor == pj:
            hit = idx == pidx
            if bool(hit.any()):
                out = torch.where(hit, torch.tensor(float("inf"), dtype=out.dtype,
                                                    device=out.device), out)
    return out


def state_values(w: Workload, which: str, idx: torch.Tensor) -> torch.Tensor:
    """Initial fp32 master / m / v at flat indices ``idx`` (zeros where the workload says so)."""
    if which == "master":
        return normal_f32(w.seed, T_MASTER, 0, 0, idx, w.master_sigma)
    if which == "m":
        if w.m_sigma is None:
            return torch.zeros(idx.shape, dtype=torch.float32, device=idx.device)
        return normal_f32(w.seed, T_M, 0, 0, idx, w.m_sigma)
    if which == "v":
        if w.v_sigma is None:
            return torch.zeros(idx.shape, dtype=torch.float32, device=idx.device)
        return normal_f32(w.seed, T_V, 0, 0, idx, w.v_sigma).abs()
    raise ValueError(which)


# --------------------------------------------------------------------------
# Layout helpers: where flat index i lives in the emulated buffers.  These are
# placements of generated values, not part of the step's arithmetic.
# --------------------------------------------------------------------------

def shard_of(psi: int, nd: int, rank: int) -> tuple[int, int, int]:
    """(S, begin, n_r) of an equal partition with a zero-padded last shard."""
    s = -(-psi // nd)
    begin = rank * s
    n = max(0, min(s, psi - begin))
    return s, begin, n


def pitch_of(s: int, align: int = 8) -> int:
    return -(-s // align) * align


def fill_shard_rows(w: Workload, step: int, rank: int, out: torch.Tensor,
                    chunk: int = 1 << 26) -> None:
    """Write the Nd contribution rows of ``rank``'s shard into ``out`` [nd, pitch].

    Columns at or beyond the shard length are zero.
    """
    s, begin, n = shard_of(w.psi, w.nd, rank)
    nd, pitch = out.shape
    assert nd == w.nd
    dev = out.device
    out[:, n:].zero_()
    for j in range(nd):
        for c0 in range(0, n, chunk):
            c1 = min(n, c0 + chunk)
            idx = torch.arange(begin + c0, begin + c1, dtype=torch.int64, device=dev)
            out[j, c0:c1] = grad_values(w, step, j, idx)


def fill_full_rows(w: Workload, step: int, out: torch.Tensor, chunk: int = 1 << 26) -> None:
    """Write every rank's full gradient in the padded-partition layout.

    ``out`` is [nd, nd * pitch]: row j is contributor j's gradient of all Psi
    parameters, partition r at columns [r * pitch, r * pitch + S).
    """
    s = -(-w.psi // w.nd)
    pitch = out.shape[1] // w.nd
    if w.nd * s <= chunk:
        # small vectors: one generator call per contributor over all psi
        # indices, placed into the padded partitions (zero past each shard)
        idx = torch.arange(w.psi, dtype=torch.int64, device=out.device)
        for j in range(w.nd):
            vals = grad_values(w, step, j, idx)
            flat = torch.zeros(w.nd * s, dtype=vals.dtype, device=out.device)
            flat[:w.psi] = vals
            row = out[j].view(w.nd, pitch)
            row[:, :s] = flat.view(w.nd, s)
            row[:, s:].zero_()
        return
    for r in range(w.nd):
        fill_shard_rows(w, step, r, out[:, r * pitch:(r + 1) * pitch], chunk)


def fill_shard_state(w: Workload, rank: int, which: str, out: torch.Tensor,
                     chunk: int = 1 << 26) -> None:
    """Write rank's initial fp32 state shard (zero past the shard length)."""
    s, begin, n = shard_of(w.psi, w.nd, rank)
    out.zero_()
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        idx = torch.arange(begin + c0, begin + c1, dtype=torch.int64, device=out.device)
        out[c0:c1] = state_values(w, which, idx)
