"""Python access to the CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product path (the CUDA library and its binding)
never does.  ``build()`` compiles ``zero_oracle.c`` with gcc; every entry point
here is a thin ctypes marshaller over that plain C file, plus the multi-step
driver that applies the global skip/commit rule.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zero_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F16, BF16 = 0, 1


def _elf_matches_host(path: str) -> bool:
    import platform
    machine = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine(), -1)
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    return len(head) == 20 and head[:4] == b"\x7fELF" and \
        int.from_bytes(head[18:20], "little") == machine


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, IEEE fp32 with no FMA contraction)."""
    if (force or not os.path.exists(LIB) or not _elf_matches_host(LIB)
            or os.path.getmtime(LIB) < os.path.getmtime(SRC)):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", SRC, "-o", tmp, "-lm"])
        os.replace(tmp, LIB)
    return LIB


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double)]


class Scalars(C.Structure):
    _fields_ = [(n, C.c_float) for n in
                ("inv", "b1", "b2", "c1", "c2", "bc1", "bc2", "lr", "eps", "wdf")]


_lib = None


def _bind(L: C.CDLL) -> C.CDLL:
    """Declare the C signatures on a loaded oracle library."""
    u64, u32, i32, vp, dbl = C.c_uint64, C.c_uint32, C.c_int, C.c_void_p, C.c_double
    L.orc_half_to_float.argtypes = [C.c_uint16]
    L.orc_half_to_float.restype = C.c_float
    L.orc_bf16_to_float.argtypes = [C.c_uint16]
    L.orc_bf16_to_float.restype = C.c_float
    L.orc_float_to_half.argtypes = [C.c_float]
    L.orc_float_to_half.restype = C.c_uint16
    L.orc_float_to_bf16.argtypes = [C.c_float]
    L.orc_float_to_bf16.restype = C.c_uint16
    L.orc_decode_n.argtypes = [vp, vp, u64, i32]
    L.orc_encode_n.argtypes = [vp, vp, u64, i32]
    L.orc_layout.argtypes = [u64, u32, u32, C.POINTER(u64)]
    L.orc_layout.restype = i32
    L.orc_model_state_bytes.argtypes = [u64, u32, u32, u32]
    L.orc_model_state_bytes.restype = u64
    L.orc_model_state_bytes_formula.argtypes = [dbl, dbl, u32, dbl]
    L.orc_model_state_bytes_formula.restype = dbl
    L.orc_scalars.argtypes = [C.POINTER(Hparams), u64, u32, dbl, C.POINTER(Scalars)]
    L.orc_fold.argtypes = [vp, i32, u32, u64, u64]
    L.orc_fold.restype = C.c_float
    L.orc_step_unsharded.argtypes = [u64, u32, i32, vp, u64, dbl, C.POINTER(Hparams), u64,
                                     vp, vp, vp, vp, vp, vp, vp]
    L.orc_step_unsharded.restype = i32
    L.orc_step_rank.argtypes = [u64, u32, i32, vp, u64, u64, u64, vp, dbl,
                                C.POINTER(Hparams), u64, vp, vp, vp, vp, vp, vp, vp, u64]
    L.orc_step_rank.restype = i32
    L.orc_step_sharded.argtypes = [u64, u32, i32, vp, u64, u64, vp, dbl, C.POINTER(Hparams),
                                   u64, vp, vp, vp, vp, vp, vp, vp]
    L.orc_step_sharded.restype = i32
    L.orc_step_unsharded_f64.argtypes = [u64, u32, i32, vp, u64, dbl, C.POINTER(Hparams),
                                         u64, vp, vp, vp, vp, vp, vp]
    L.orc_comm_volume_elems.argtypes = [u64, u32]
    L.orc_comm_volume_elems.restype = u64
    L.orc_model_state_bytes_mp.argtypes = [u64, u32, u32, u32, u32]
    L.orc_model_state_bytes_mp.restype = u64
    L.orc_gather_range.argtypes = [vp, u64, u64, u32, u64, u64, u32, vp]
    L.orc_gather_range.restype = i32
    L.orc_reduce_scaled.argtypes = [vp, i32, u32, u64, u64, u64, C.c_float, vp]
    L.orc_reduce_scaled.restype = i32
    L.orc_adamw_from_grad.argtypes = [u64, vp, C.POINTER(Hparams), u64, vp, vp, vp, vp, vp, vp]
    return L


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(C.CDLL(build()))
    return _lib


class use_library:
    """Context manager that routes this module's calls to another build of
    the oracle (the tests use it to show that planted mistakes fail a pin)."""

    def __init__(self, path: str):
        self.L = _bind(C.CDLL(path))

    def __enter__(self):
        global _lib
        self.prev, _lib = lib(), self.L
        return self.L

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data_as(C.c_void_p)


def dtype_code(name: str) -> int:
    return {"f16": F16, "bf16": BF16}[name]


def hparams(d: dict) -> Hparams:
    return Hparams(d["lr"], d["beta1"], d["beta2"], d["eps"], d["weight_decay"])


# -- conversions -----------------------------------------------------------

def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    lib().orc_decode_n(_p(bits), _p(out), bits.size, dtype)
    return out


def encode(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_encode_n(_p(x), _p(out), x.size, dtype)
    return out


# -- layout and accounting -------------------------------------------------

def layout(psi: int, nd: int, rank: int) -> tuple[int, int, int]:
    out = (C.c_uint64 * 3)()
    if lib().orc_layout(psi, nd, rank, out) != 0:
        raise ValueError("invalid layout arguments")
    return int(out[0]), int(out[1]), int(out[2])


def model_state_bytes(psi: int, nd: int, stage: int, k: int = 12) -> int:
    return int(lib().orc_model_state_bytes(psi, nd, stage, k))


def model_state_bytes_formula(psi: float, nd: float, stage: int, k: float = 12.0) -> float:
    return float(lib().orc_model_state_bytes_formula(psi, nd, stage, k))


def comm_volume_elems(psi: int, stage: int) -> int:
    return int(lib().orc_comm_volume_elems(psi, stage))


def model_state_bytes_mp(psi: int, nd: int, nm: int, stage: int, k: int = 12) -> int:
    return int(lib().orc_model_state_bytes_mp(psi, nd, nm, stage, k))


def gather_range(shards: np.ndarray, psi: int, nd: int, begin: int, length: int) -> np.ndarray:
    """Flat range [begin, begin+length) of a partitioned buffer ``shards``
    ([nd, pitch], uint16 or float32)."""
    shards = np.ascontiguousarray(shards)
    assert shards.ndim == 2 and shards.shape[0] == nd
    out = np.empty(max(length, 1), shards.dtype)
    if lib().orc_gather_range(_p(shards), shards.shape[1], psi, nd, begin, length,
                              shards.itemsize, _p(out)) != 0:
        raise ValueError("invalid gather range")
    return out[:length]


def scalars(h: dict, t: int, nd: int, loss_scale: float) -> Scalars:
    s = Scalars()
    hp = hparams(h)
    lib().orc_scalars(C.byref(hp), t, nd, loss_scale, C.byref(s))
    return s


# -- the step --------------------------------------------------------------

def fold(grads: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 rank-ordered sums of a [nd, n] uint16 contribution array."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    nd, n = grads.shape
    L = lib()
    return np.array([L.orc_fold(_p(grads), dtype, nd, n, i) for i in range(n)],
                    dtype=np.float32)


def reduce_scaled(grads: np.ndarray, dtype: int, row_stride: int, offset: int, n: int,
                  nd: int, inv_scale: float):
    """(flag, out) of the reduce-scatter of shard window [offset, offset+n).
    ``grads`` is a flat uint16 array; contributor j's element i is at
    grads[j*row_stride + offset + i]."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    assert n == 0 or (nd - 1) * row_stride + offset + n <= grads.size
    out = np.empty(max(n, 1), np.float32)
    f = lib().orc_reduce_scaled(_p(grads), dtype, nd, row_stride, offset, n,
                                float(np.float32(inv_scale)), _p(out))
    return f, out[:n]


def adamw_from_grad(g: np.ndarray, h: dict, t: int, p, m, v):
    """(p', m', v') of AdamW from an fp32 reduced, scaled gradient."""
    g, p, m, v = (np.ascontiguousarray(a, np.float32) for a in (g, p, m, v))
    n = g.size
    po, mo, vo = (np.empty(n, np.float32) for _ in range(3))
    hp = hparams(h)
    lib().orc_adamw_from_grad(n, _p(g), C.byref(hp), t, _p(p), _p(m), _p(v), _p(po), _p(mo),
                              _p(vo))
    return po, mo, vo


def step_unsharded(grads: np.ndarray, dtype: int, loss_scale: float, h: dict, t: int,
                   p: np.ndarray, m: np.ndarray, v: np.ndarray):
    """One unsharded step.  grads: [nd, psi] uint16.  Returns
    (skipped, p', m', v', params) with None outputs when skipped."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    nd, psi = grads.shape
    po, mo, vo = (np.empty(psi, np.float32) for _ in range(3))
    params = np.empty(psi, np.uint16)
    hp = hparams(h)
    p, m, v = (np.ascontiguousarray(a, np.float32) for a in (p, m, v))
    skipped = lib().orc_step_unsharded(psi, nd, dtype, _p(grads), psi, loss_scale, C.byref(hp),
                                       t, _p(p), _p(m), _p(v), _p(po), _p(mo), _p(vo),
                                       _p(params))
    if skipped:
        return True, None, None, None, None
    return False, po, mo, vo, params


def step_unsharded_f64(grads: np.ndarray, dtype: int, loss_scale: float, h: dict, t: int,
                       p: np.ndarray, m: np.ndarray, v: np.ndarray):
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    nd, psi = grads.shape
    po, mo, vo = (np.empty(psi, np.float64) for _ in range(3))
    hp = hparams(h)
    lib().orc_step_unsharded_f64(psi, nd, dtype, _p(grads), psi, loss_scale, C.byref(hp), t,
                                 _p(np.ascontiguousarray(p, np.float32)),
                                 _p(np.ascontiguousarray(m, np.float32)),
                                 _p(np.ascontiguousarray(v, np.float32)), _p(po), _p(mo), _p(vo))
    return po, mo, vo


def step_rank(grads: np.ndarray, row_stride: int, offset: int, n: int, nd: int, dtype: int,
              bucket: int, loss_scale: float, h: dict, t: int, p, m, v, params_out, slot):
    """One rank's shard step; returns (flag, p', m', v') and writes params_out."""
    po, mo, vo = (np.empty(max(n, 1), np.float32) for _ in range(3))
    cb = np.empty(max(1, min(bucket, n)), np.float32)
    hp = hparams(h)
    f = lib().orc_step_rank(n, nd, dtype, _p(grads), row_stride, offset, bucket, _p(cb),
                            loss_scale, C.byref(hp), t, _p(p), _p(m), _p(v), _p(po), _p(mo),
                            _p(vo), _p(params_out), slot)
    if f < 0:
        raise ValueError("invalid oracle arguments")
    return f, po[:n], mo[:n], vo[:n]


def step_sharded(grads_padded: np.ndarray, psi: int, nd: int, pitch: int, dtype: int,
                 bucket: int, loss_scale: float, h: dict, t: int, p, m, v, params_out):
    """All ranks' shard steps.  grads_padded: [nd, nd*pitch] uint16.  Returns
    (flag, p', m', v'); params_out (flat, length >= nd*S) is written."""
    grads_padded = np.ascontiguousarray(grads_padded, dtype=np.uint16)
    po, mo, vo = (np.empty(psi, np.float32) for _ in range(3))
    s = -(-psi // nd)
    cb = np.empty(max(1, min(bucket, s)), np.float32)
    hp = hparams(h)
    f = lib().orc_step_sharded(psi, nd, dtype, _p(grads_padded), pitch, bucket, _p(cb),
                               loss_scale, C.byref(hp), t, _p(p), _p(m), _p(v), _p(po), _p(mo),
                               _p(vo), _p(params_out))
    if f < 0:
        raise ValueError("invalid oracle arguments")
    return f, po, mo, vo


class Trajectory:
    """Multi-step driver with the global skip/commit rule: a step whose
    reduced gradient holds a nonfinite value anywhere leaves the state, the
    cast parameters and the step counter unchanged; otherwise the new state is
    committed and t advances.  ``grads_at(step)`` returns [nd, n] uint16."""

    def __init__(self, dtype: int, loss_scale: float, h: dict, p, m, v, params=None):
        self.dtype, self.loss_scale, self.h = dtype, loss_scale, h
        self.p = np.array(p, np.float32)
        self.m = np.array(m, np.float32)
        self.v = np.array(v, np.float32)
        self.params = None if params is None else np.array(params, np.uint16)
        self.t = 0
        self.skipped = []

    def step(self, grads: np.ndarray) -> bool:
        skipped, po, mo, vo, params = step_unsharded(grads, self.dtype, self.loss_scale, self.h,
                                                     self.t + 1, self.p, self.m, self.v)
        self.skipped.append(skipped)
        if not skipped:
            self.p, self.m, self.v, self.params = po, mo, vo, params
            self.t += 1
        return skipped
