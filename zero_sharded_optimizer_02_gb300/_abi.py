"""ctypes binding of libzero.so: the C ABI of ``include/zero.h``, same names.

Argument marshalling only: every step of the optimizer runs in the library's
CUDA kernels.  Pointer arguments accept an int address or any object with a
``data_ptr()`` method (a torch tensor); ``stream`` accepts an int handle, a
``torch.cuda.Stream`` or None (the legacy default stream).  A non-OK status
raises ``ZeroError``.  There is no fallback: if the library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libzero.so")

ZERO_OK, ZERO_ERR_INVALID_ARG, ZERO_ERR_ALIGNMENT, ZERO_ERR_CUDA = 0, 1, 2, 3
ZERO_ERR_TIMEOUT, ZERO_ERR_UNSUPPORTED, ZERO_ERR_IO = 4, 5, 6
ZERO_F16, ZERO_BF16 = 0, 1
DTYPES = {"f16": ZERO_F16, "bf16": ZERO_BF16}
UINT64_MAX = (1 << 64) - 1

u64, u32, i32, vp, dbl = C.c_uint64, C.c_uint32, C.c_int32, C.c_void_p, C.c_double


class ZeroError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {zero_status_string(status)} ({status})")


class Layout(C.Structure):
    _fields_ = [("psi", u64), ("nd", u32), ("rank", u32), ("shard_elems", u64), ("begin", u64),
                ("length", u64), ("padded_elems", u64), ("row_pitch", u64)]


class Grads(C.Structure):
    _fields_ = [("base", vp), ("row_stride", u64), ("offset", u64), ("nd", u32), ("dtype", i32)]


class State(C.Structure):
    _fields_ = [("master", vp), ("m", vp), ("v", vp)]


class CkptHeader(C.Structure):
    _fields_ = [("magic", C.c_char * 8), ("version", u32), ("header_bytes", u32), ("psi", u64),
                ("nd", u32), ("rank", u32), ("shard_elems", u64), ("begin", u64),
                ("length", u64), ("step", u64), ("lr", dbl), ("beta1", dbl), ("beta2", dbl),
                ("eps", dbl), ("weight_decay", dbl), ("payload_checksum", u64)]


class AdamW(C.Structure):
    _fields_ = [("lr", dbl), ("beta1", dbl), ("beta2", dbl), ("eps", dbl),
                ("weight_decay", dbl), ("step", u64)]


_lib: C.CDLL | None = None

_SIGNATURES = {
    "zero_status_string": ([i32], C.c_char_p),
    "zero_partition_layout": ([u64, u32, u32, u32, C.POINTER(Layout)], i32),
    "zero_model_state_bytes": ([u64, u32, u32, u32], u64),
    "zero_reduce_scatter_bucket": ([C.POINTER(Grads), u64, u64, C.c_float, vp, vp, vp], i32),
    "zero_adam_step_shard": ([vp, C.POINTER(State), C.POINTER(State), u64, C.POINTER(AdamW),
                              vp], i32),
    "zero_gather_params_shard": ([vp, u64, vp, u64, i32, vp], i32),
    "zero_step_shard": ([C.POINTER(Grads), C.POINTER(Layout), C.POINTER(State),
                         C.POINTER(State), vp, u64, u64, dbl, C.POINTER(AdamW), vp, vp], i32),
    "zero_step_shard_unfused": ([C.POINTER(Grads), C.POINTER(Layout), C.POINTER(State),
                                 C.POINTER(State), vp, u64, u64, dbl, C.POINTER(AdamW), vp, u64,
                                 vp, vp], i32),
    "zero_check_nonfinite": ([C.POINTER(Grads), u64, u64, vp, vp], i32),
    "zero_step_shard_streamed": ([C.POINTER(Grads), C.POINTER(Layout), C.POINTER(State),
                                  C.POINTER(State), vp, u64, u64, dbl, C.POINTER(AdamW), vp, u32,
                                  u64, vp, vp, vp], i32),
    "zero_feed_buckets": ([vp, u64, C.POINTER(Grads), u64, u64, vp, vp, vp], i32),
    "zero_gather_range": ([vp, u64, u64, u32, u64, u64, u32, vp, vp], i32),
    "zero_checkpoint_save": ([C.c_char_p, C.POINTER(Layout), C.POINTER(AdamW), vp, vp, vp], i32),
    "zero_checkpoint_read_header": ([C.c_char_p, C.POINTER(CkptHeader)], i32),
    "zero_checkpoint_load": ([C.POINTER(C.c_char_p), u32, C.POINTER(Layout), vp, vp, vp,
                              C.POINTER(AdamW)], i32),
    "zero_comm_volume_elems": ([u64, u32], u64),
    "zero_model_state_bytes_mp": ([u64, u32, u32, u32, u32], u64),
    "zero_step_shard_unfused_static": ([C.POINTER(Grads), C.POINTER(Layout), C.POINTER(State),
                                        C.POINTER(State), vp, u64, u64, dbl, C.POINTER(AdamW),
                                        vp, vp], i32),
}

# Most contribution rows a gradient descriptor may name (include/zero.h).
ZERO_MAX_ND = 1 << 24

# Longest launch window of the fused step (include/zero.h).
ZERO_FUSED_WINDOW_ELEMS = 10485760


def _windows(length: int, phase: int) -> int:
    """Launch windows of one range (the library's split, see zero.h); `phase`
    is row 0's element offset past a 32-byte boundary (its element offset
    within the row when the rows' base is 32-byte aligned, as torch's are)."""
    nwin = -(-length // ZERO_FUSED_WINDOW_ELEMS)
    target = -(-(-(-length // nwin)) // 16) * 16
    cut, w0, count = target - (phase & 15), 0, 0
    while w0 < length:
        w1 = min(cut, length)
        if length - w1 < 64:
            w1 = length
        w0, cut = w1, cut + target
        count += 1
    return count


def fused_launch_count(n: int, bucket: int, offset: int = 0) -> int:
    """Kernel launches zero_step_shard issues for a shard of n elements whose
    rows start at element `offset`: the launch windows of the whole shard
    (the same split as the library).  The bucket size does not change them:
    the fused kernel never materialises a bucket."""
    if bucket <= 0:
        raise ValueError("bucket must be positive")
    return _windows(n, offset) if n > 0 else 0


# Least step traffic of a launch group of zero_step_shard_streamed (zero.h).
ZERO_STREAM_GROUP_BYTES = 1000000000


def stream_groups(n: int, bucket: int, nd: int) -> list:
    """The launch groups of zero_step_shard_streamed, as (first element,
    length): as many groups as the shard's step traffic holds
    ZERO_STREAM_GROUP_BYTES (0: one group a bucket), the buckets dealt as
    evenly as possible."""
    env = os.environ.get("ZERO_STREAM_GROUP_BYTES", "")
    group_bytes = int(env) if env.isdigit() else ZERO_STREAM_GROUP_BYTES
    nb = -(-n // bucket)
    if nb == 0:
        return []
    ngroups = n * (2 * nd + 26) // group_bytes if group_bytes else nb
    ngroups = min(max(ngroups, 1), nb)
    base, extra = divmod(nb, ngroups)
    groups, b = [], 0
    for grp in range(ngroups):
        b_end = b + base + (1 if grp < extra else 0)
        groups.append((b * bucket, min(b_end * bucket, n) - b * bucket))
        b = b_end
    return groups


def streamed_launch_count(n: int, bucket: int, nd: int, offset: int = 0) -> int:
    """Kernel launches zero_step_shard_streamed issues: per launch group, one
    wait and the fused step's launch windows."""
    return sum(1 + _windows(glen, offset + g0) for g0, glen in stream_groups(n, bucket, nd))


def unfused_launch_count(n: int, bucket: int, offset: int = 0) -> int:
    """Kernel launches zero_step_shard_unfused issues: per bucket, the
    reduction in the same launch windows, then the AdamW and cast passes."""
    return sum(_windows(min(bucket, n - b0), offset + b0) + 2 for b0 in range(0, n, bucket))


# Bit of the step flag word set when a step kernel gave up waiting on its own
# copy pipeline (include/zero.h).
ZERO_STEP_FLAG_WAIT_TIMEOUT = 0x80000000


def check_step_flag(word: int, where: str = "step kernel") -> bool:
    """The skip decision of one flag word (nonzero: skip); raises ZeroError
    (ZERO_ERR_TIMEOUT) if the kernel reported a pipeline wait that expired."""
    if int(word) & ZERO_STEP_FLAG_WAIT_TIMEOUT:
        raise ZeroError(ZERO_ERR_TIMEOUT, where)
    return int(word) != 0


# Shard segments that one zero_gather_range launch copies (include/zero.h).
ZERO_GATHER_SEGMENTS_PER_LAUNCH = 48


def gather_launch_count(psi: int, nd: int, begin: int, length: int) -> int:
    """Kernel launches zero_gather_range issues for the flat range
    [begin, begin + length): one per ZERO_GATHER_SEGMENTS_PER_LAUNCH shard
    segments the range spans."""
    if length == 0:
        return 0
    s = -(-psi // nd)
    segments = (begin + length - 1) // s - begin // s + 1
    return -(-segments // ZERO_GATHER_SEGMENTS_PER_LAUNCH)


# Capacity of the library's own fusion buffer (include/zero.h).
ZERO_STATIC_CB_ELEMS = 4194304
ZERO_STATIC_CB_MAX_BUCKET = ZERO_STATIC_CB_ELEMS - 4


def lib() -> C.CDLL:
    """The loaded library (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libzero.so not found at {LIB_PATH}; build it with "
                "zero_sharded_optimizer_02_gb300.build.build() (there is no CPU fallback)")
        L = C.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def exported_names() -> list[str]:
    return list(_SIGNATURES)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != ZERO_OK:
        raise ZeroError(status, where)


# -- descriptors -------------------------------------------------------------

def grads(base, row_stride: int, offset: int, nd: int, dtype) -> Grads:
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    return Grads(_ptr(base), row_stride, offset, nd, dt)


def state(master, m, v) -> State:
    return State(_ptr(master), _ptr(m), _ptr(v))


def adamw(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
          step: int) -> AdamW:
    return AdamW(lr, beta1, beta2, eps, weight_decay, step)


# -- entry points ------------------------------------------------------------

def zero_status_string(status: int) -> str:
    return lib().zero_status_string(status).decode()


def zero_partition_layout(psi: int, nd: int, rank: int, row_align_elems: int = 8) -> Layout:
    out = Layout()
    _check(lib().zero_partition_layout(psi, nd, rank, row_align_elems, C.byref(out)),
           "zero_partition_layout")
    return out


def zero_model_state_bytes(psi: int, nd: int, stage: int, k: int = 12) -> int:
    return int(lib().zero_model_state_bytes(psi, nd, stage, k))


def zero_step_shard_streamed(g: Grads, L: Layout, s_in: State, s_out: State, gathered,
                             gathered_offset_elems: int, bucket_elems: int, loss_scale: float,
                             h: AdamW, d_ready, epoch: int, timeout_ns: int, d_nonfinite,
                             d_status, stream=None) -> None:
    _check(lib().zero_step_shard_streamed(C.byref(g), C.byref(L), C.byref(s_in), C.byref(s_out),
                                          _ptr(gathered), gathered_offset_elems, bucket_elems,
                                          loss_scale, C.byref(h), _ptr(d_ready), epoch,
                                          timeout_ns, _ptr(d_nonfinite), _ptr(d_status),
                                          _stream(stream)), "zero_step_shard_streamed")


def zero_feed_buckets(host, host_row_stride: int, g: Grads, n: int, bucket_elems: int, d_ready,
                      h_epoch, copy_stream=None) -> None:
    _check(lib().zero_feed_buckets(_ptr(host), host_row_stride, C.byref(g), n, bucket_elems,
                                   _ptr(d_ready), _ptr(h_epoch), _stream(copy_stream)),
           "zero_feed_buckets")


def zero_gather_range(shards, pitch: int, psi: int, nd: int, begin: int, length: int,
                      elem_bytes: int, out, stream=None) -> None:
    _check(lib().zero_gather_range(_ptr(shards), pitch, psi, nd, begin, length, elem_bytes,
                                   _ptr(out), _stream(stream)), "zero_gather_range")


def zero_checkpoint_save(path: str, L: Layout, h: AdamW, master, m, v) -> None:
    """Host arrays (numpy float32, contiguous) of L.length elements."""
    _check(lib().zero_checkpoint_save(os.fsencode(path), C.byref(L), C.byref(h),
                                      _host_ptr(master), _host_ptr(m), _host_ptr(v)),
           "zero_checkpoint_save")


def zero_checkpoint_read_header(path: str) -> CkptHeader:
    out = CkptHeader()
    _check(lib().zero_checkpoint_read_header(os.fsencode(path), C.byref(out)),
           "zero_checkpoint_read_header")
    return out


def zero_checkpoint_load(paths, L: Layout, master, m, v) -> AdamW:
    """Fills host arrays master/m/v (L.length floats) of rank L.rank from the
    old ranks' files ``paths``; returns the saved hyperparameters and step."""
    arr = (C.c_char_p * len(paths))(*[os.fsencode(p) for p in paths])
    h = AdamW()
    _check(lib().zero_checkpoint_load(arr, len(paths), C.byref(L), _host_ptr(master),
                                      _host_ptr(m), _host_ptr(v), C.byref(h)),
           "zero_checkpoint_load")
    return h


def _host_ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "ctypes"):
        assert a.flags["C_CONTIGUOUS"] and a.dtype.itemsize == 4
        return a.ctypes.data
    return a.data_ptr()


def zero_comm_volume_elems(psi: int, stage: int) -> int:
    return int(lib().zero_comm_volume_elems(psi, stage))


def zero_model_state_bytes_mp(psi: int, nd: int, nm: int, stage: int, k: int = 12) -> int:
    return int(lib().zero_model_state_bytes_mp(psi, nd, nm, stage, k))


def zero_reduce_scatter_bucket(g: Grads, bucket_begin: int, bucket_len: int, inv_scale: float,
                               cb_out, d_nonfinite, stream=None) -> None:
    _check(lib().zero_reduce_scatter_bucket(C.byref(g), bucket_begin, bucket_len, inv_scale,
                                            _ptr(cb_out), _ptr(d_nonfinite), _stream(stream)),
           "zero_reduce_scatter_bucket")


def zero_adam_step_shard(grad, s_in: State, s_out: State, n: int, h: AdamW,
                         stream=None) -> None:
    _check(lib().zero_adam_step_shard(_ptr(grad), C.byref(s_in), C.byref(s_out), n, C.byref(h),
                                      _stream(stream)), "zero_adam_step_shard")


def zero_gather_params_shard(master, n: int, gathered, slot_offset_elems: int, dtype,
                             stream=None) -> None:
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    _check(lib().zero_gather_params_shard(_ptr(master), n, _ptr(gathered), slot_offset_elems,
                                          dt, _stream(stream)), "zero_gather_params_shard")


def zero_step_shard(g: Grads, L: Layout, s_in: State, s_out: State, gathered,
                    gathered_offset_elems: int, bucket_elems: int, loss_scale: float, h: AdamW,
                    d_nonfinite, stream=None) -> None:
    _check(lib().zero_step_shard(C.byref(g), C.byref(L), C.byref(s_in), C.byref(s_out),
                                 _ptr(gathered), gathered_offset_elems, bucket_elems, loss_scale,
                                 C.byref(h), _ptr(d_nonfinite), _stream(stream)),
           "zero_step_shard")


def zero_step_shard_unfused(g: Grads, L: Layout, s_in: State, s_out: State, gathered,
                            gathered_offset_elems: int, bucket_elems: int, loss_scale: float,
                            h: AdamW, cb, cb_elems: int, d_nonfinite, stream=None) -> None:
    _check(lib().zero_step_shard_unfused(C.byref(g), C.byref(L), C.byref(s_in), C.byref(s_out),
                                         _ptr(gathered), gathered_offset_elems, bucket_elems,
                                         loss_scale, C.byref(h), _ptr(cb), cb_elems,
                                         _ptr(d_nonfinite), _stream(stream)),
           "zero_step_shard_unfused")


def zero_check_nonfinite(g: Grads, begin: int, n: int, d_nonfinite, stream=None) -> None:
    _check(lib().zero_check_nonfinite(C.byref(g), begin, n, _ptr(d_nonfinite), _stream(stream)),
           "zero_check_nonfinite")


def zero_step_shard_unfused_static(g: Grads, L: Layout, s_in: State, s_out: State, gathered,
                                   gathered_offset_elems: int, bucket_elems: int,
                                   loss_scale: float, h: AdamW, d_nonfinite,
                                   stream=None) -> None:
    """zero_step_shard_unfused without a workspace argument: for callers that
    cannot allocate device memory (their framework's pool owns the device, or
    they must avoid the synchronisation cudaMalloc/cudaFree can cause).  The
    fusion buffer is the library's own 16 MiB device array, shared by every
    call on a device, so calls must not overlap on the GPU; buckets are limited
    to ZERO_STATIC_CB_MAX_BUCKET elements."""
    used = min(bucket_elems, int(L.length))
    if used > ZERO_STATIC_CB_MAX_BUCKET:
        raise ZeroError(ZERO_ERR_INVALID_ARG,
                        f"zero_step_shard_unfused_static: bucket of {used} elements exceeds the "
                        f"static fusion buffer ({ZERO_STATIC_CB_MAX_BUCKET} elements)")
    _check(lib().zero_step_shard_unfused_static(C.byref(g), C.byref(L), C.byref(s_in),
                                                C.byref(s_out), _ptr(gathered),
                                                gathered_offset_elems, bucket_elems, loss_scale,
                                                C.byref(h), _ptr(d_nonfinite), _stream(stream)),
           "zero_step_shard_unfused_static")
