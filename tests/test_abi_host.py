"""The C-ABI library without a GPU: it loads, exports every symbol declared in
include/zero.h, its host-only entry points agree with the oracle, and invalid
arguments are rejected on the host before anything is launched."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def z():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    import zero_sharded_optimizer_02_gb300 as z
    return z


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(z):
    names = declared_functions()
    assert len(names) >= 9
    raw = C.CDLL(z._abi.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(z.exported_names()) == set(names)


def test_layout_matches_oracle(z, orc):
    for psi in list(range(0, 60)) + [350_000_017, 7_500_000_000]:
        for nd in (1, 2, 3, 7, 16, 64):
            for r in sorted({0, nd // 2, nd - 1}):
                L = z.zero_partition_layout(psi, nd, r, 8)
                s, b, n = orc.layout(psi, nd, r)
                assert (L.shard_elems, L.begin, L.length) == (s, b, n)
                assert L.padded_elems == nd * s and L.row_pitch == -(-s // 8) * 8
                assert (L.psi, L.nd, L.rank) == (psi, nd, r)


def test_layout_invalid(z):
    for args in ((10, 0, 0, 8), (10, 4, 4, 8), (10, 4, 0, 0), (2 ** 64 - 1, 2, 0, 8)):
        with pytest.raises(z.ZeroError) as e:
            z.zero_partition_layout(*args)
        assert e.value.status == z.ZERO_ERR_INVALID_ARG


def test_accounting_matches_oracle_and_table(z, orc):
    for psi in (0, 1, 5, 1_000_003, 1_500_000_000, 7_500_000_000):
        for nd in (1, 3, 64, 1024):
            for st in range(4):
                for k in (12, 8):
                    assert z.zero_model_state_bytes(psi, nd, st, k) == \
                        orc.model_state_bytes(psi, nd, st, k)
    assert z.zero_model_state_bytes(1_500_000_000, 1, 0, 12) == 24 * 10 ** 9
    exp = {(64, 1): 31.4, (64, 2): 16.6, (64, 3): 1.88, (1024, 1): 30.1, (1024, 2): 15.1,
           (1024, 3): 0.12}
    for (nd, st), gb in exp.items():
        dec = len(str(gb).split(".")[1])
        assert round(z.zero_model_state_bytes(7_500_000_000, nd, st, 12) / 1e9, dec) == gb
    assert z.zero_model_state_bytes(1, 0, 0, 12) == 2 ** 64 - 1
    assert z.zero_model_state_bytes(1, 1, 4, 12) == 2 ** 64 - 1


def test_comm_volume_and_mp_accounting(z, orc):
    import os
    gold = os.path.join(ROOT, "tests", "golden")
    rows = [ln.split() for ln in open(os.path.join(gold, "stage_reductions.txt"))
            if ln.strip() and not ln.startswith("#")]
    for stage, _, comm in rows:
        assert z.zero_comm_volume_elems(10 ** 9, int(stage)) == int(comm) * 10 ** 9
    assert z.zero_comm_volume_elems(10 ** 9, 0) == 2 * 10 ** 9
    assert z.zero_comm_volume_elems(1, 4) == 2 ** 64 - 1
    kv = {r[0]: r[1] for r in (ln.split() for ln in open(os.path.join(
        gold, "model_state_examples.txt")) if ln.strip() and not ln.startswith("#"))}
    per_gpu = z.zero_model_state_bytes_mp(int(kv["mp_psi"]), int(kv["mp_nd"]), int(kv["mp_nm"]),
                                          3, int(kv["k"]))
    assert per_gpu < int(kv["mp_gpu_gb"]) * 10 ** 9
    for psi in (1, 999, 10 ** 12, 7_500_000_000):
        for nd, nm in ((64, 16), (1, 1), (7, 3)):
            for st in range(4):
                assert z.zero_model_state_bytes_mp(psi, nd, nm, st, 12) == \
                    orc.model_state_bytes_mp(psi, nd, nm, st, 12)
    assert z.zero_model_state_bytes_mp(10, 1, 0, 0, 12) == 2 ** 64 - 1


def test_status_strings(z):
    for code in range(6):
        assert z.zero_status_string(code).startswith("ZERO_")
    assert "UNKNOWN" in z.zero_status_string(99)


# Fake, never dereferenced device addresses: every call below fails host-side
# validation before any CUDA call.
A = 1 << 20   # 16-byte aligned


def test_valid_fake_arguments_reach_the_runtime(z):
    """The base case of the rejection tests below passes every host-side check
    and fails only where the library first asks the CUDA runtime about a
    pointer: ZERO_ERR_CUDA without a device, ZERO_ERR_INVALID_ARG for a
    pointer the runtime does not know.  So each rejection below comes from
    its own check, not from that question."""
    import torch
    L = z.zero_partition_layout(1000, 4, 1, 8)
    g = z.grads(A, 4 * 256, 256, 4, "f16")
    expect = z.ZERO_ERR_INVALID_ARG if torch.cuda.is_available() else z.ZERO_ERR_CUDA
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_shard(g, L, _state(z, 2 * A), _state(z, 4 * A), 8 * A, L.begin, 64, 1024.0,
                          _h(z), 9 * A)
    assert e.value.status == expect
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_shard_streamed(g, L, _state(z, 2 * A), _state(z, 4 * A), 8 * A, L.begin,
                                   64, 1024.0, _h(z), 10 * A, 1, 10 ** 9, 9 * A, 11 * A)
    assert e.value.status == expect


def _h(z, step=1):
    return z.adamw(1e-4, 0.9, 0.999, 1e-8, 0.01, step)


def _state(z, base):
    return z.state(base, base + (1 << 16), base + (2 << 16))


@pytest.mark.parametrize("case,status", [
    ("null_base", "ZERO_ERR_INVALID_ARG"), ("misaligned_base", "ZERO_ERR_ALIGNMENT"),
    ("odd_row_stride", "ZERO_ERR_ALIGNMENT"), ("odd_offset", "ZERO_ERR_ALIGNMENT"),
    ("bad_dtype", "ZERO_ERR_INVALID_ARG"), ("nd_zero", "ZERO_ERR_INVALID_ARG"),
    ("nd_too_large", "ZERO_ERR_INVALID_ARG"),
    ("shard_longer_than_s", "ZERO_ERR_INVALID_ARG"), ("misaligned_state", "ZERO_ERR_ALIGNMENT"),
    ("overlap_state", "ZERO_ERR_INVALID_ARG"), ("bucket_zero", "ZERO_ERR_INVALID_ARG"),
    ("step_zero", "ZERO_ERR_INVALID_ARG"), ("bad_beta", "ZERO_ERR_INVALID_ARG"),
    ("bad_loss_scale", "ZERO_ERR_INVALID_ARG"), ("odd_gathered", "ZERO_ERR_ALIGNMENT"),
    ("null_flag", "ZERO_ERR_INVALID_ARG"), ("row_overflow", "ZERO_ERR_INVALID_ARG"),
    ("slot_overlaps_state_in", "ZERO_ERR_INVALID_ARG"),
    ("slot_overlaps_state_out", "ZERO_ERR_INVALID_ARG"),
    ("slot_overlaps_rows", "ZERO_ERR_INVALID_ARG"),
    ("slot_offset_overflow", "ZERO_ERR_INVALID_ARG"),
])
def test_step_shard_rejects(z, case, status):
    L = z.zero_partition_layout(1000, 4, 1, 8)
    g = z.grads(A, 4 * 256, 256, 4, "f16")
    s_in, s_out = _state(z, 2 * A), _state(z, 4 * A)
    gathered, flag, bucket, ls, h = 8 * A, 9 * A, 64, 1024.0, _h(z)
    if case == "null_base":
        g.base = None
    elif case == "misaligned_base":
        g.base = A + 8
    elif case == "odd_row_stride":
        g.row_stride = 1020
    elif case == "odd_offset":
        g.offset = 252
    elif case == "bad_dtype":
        g.dtype = 7
    elif case == "nd_zero":
        g.nd = 0
    elif case == "nd_too_large":                 # past the kernels' row-count range
        g.nd = z._abi.ZERO_MAX_ND + 1
        g.row_stride = 8
    elif case == "shard_longer_than_s":
        L.length = L.shard_elems + 1
    elif case == "misaligned_state":
        s_out.m = s_out.m + 4
    elif case == "overlap_state":
        s_out.m = s_in.m + 16
    elif case == "bucket_zero":
        bucket = 0
    elif case == "step_zero":
        h = _h(z, 0)
    elif case == "bad_beta":
        h.beta1 = 1.0
    elif case == "bad_loss_scale":
        ls = 0.0
    elif case == "odd_gathered":
        gathered += 1
    elif case == "null_flag":
        flag = None
    elif case == "row_overflow":
        g.row_stride = 1 << 62
    goff = L.begin
    if case == "slot_overlaps_state_in":          # the slot's last element on master[0]
        gathered = s_in.master - 2 * (goff + L.length - 1)
    elif case == "slot_overlaps_state_out":       # the slot starts inside v'
        gathered = s_out.v + 4 * 100 - 2 * goff
    elif case == "slot_overlaps_rows":            # the slot lands in the last row
        gathered = A + 2 * (256 + 3 * 1024 + 10) - 2 * goff
    elif case == "slot_offset_overflow":
        goff = 1 << 62
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_shard(g, L, s_in, s_out, gathered, goff, bucket, ls, h, flag)
    assert e.value.status == getattr(z, status)
    if case.startswith("slot_"):                 # the bucket-ready step checks the same
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_shard_streamed(g, L, s_in, s_out, gathered, goff, bucket, ls, h,
                                       10 * A, 1, 10 ** 9, flag, 11 * A)
        assert e.value.status == getattr(z, status)
    # the unfused variant validates the same way, plus its workspace
    if case in ("misaligned_base", "overlap_state", "bucket_zero", "slot_overlaps_rows"):
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_shard_unfused(g, L, s_in, s_out, gathered, goff, bucket, ls, h,
                                      10 * A, 1 << 20, flag)
        assert e.value.status == getattr(z, status)


def test_primitives_reject(z):
    g = z.grads(A, 1024, 0, 4, "bf16")
    with pytest.raises(z.ZeroError) as e:
        z.zero_reduce_scatter_bucket(g, 0, 100, 1.0, A + 2, 9 * A)
    assert e.value.status == z.ZERO_ERR_ALIGNMENT
    with pytest.raises(z.ZeroError) as e:
        z.zero_reduce_scatter_bucket(g, 0, 100, 1.0, None, 9 * A)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    with pytest.raises(z.ZeroError) as e:
        z.zero_check_nonfinite(z.grads(A + 4, 1024, 0, 4, "bf16"), 0, 10, 9 * A)
    assert e.value.status == z.ZERO_ERR_ALIGNMENT
    with pytest.raises(z.ZeroError) as e:
        z.zero_adam_step_shard(A + 2, _state(z, 2 * A), _state(z, 4 * A), 10, _h(z))
    assert e.value.status == z.ZERO_ERR_ALIGNMENT
    with pytest.raises(z.ZeroError) as e:   # gradient overlapping an output
        z.zero_adam_step_shard(4 * A, _state(z, 2 * A), _state(z, 4 * A), 10, _h(z))
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    with pytest.raises(z.ZeroError) as e:
        z.zero_gather_params_shard(A, 10, A + 1, 0, "f16")
    assert e.value.status == z.ZERO_ERR_ALIGNMENT
    with pytest.raises(z.ZeroError) as e:
        z.zero_gather_params_shard(A, 10, 2 * A, 0, 5)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    with pytest.raises(z.ZeroError) as e:   # workspace too small
        L = z.zero_partition_layout(1000, 4, 1, 8)
        z.zero_step_shard_unfused(z.grads(A, 4 * 256, 256, 4, "f16"), L, _state(z, 2 * A),
                                  _state(z, 4 * A), 8 * A, L.begin, 64, 1024.0, _h(z), 10 * A,
                                  60, 9 * A)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import zero_sharded_optimizer_02_gb300._abi as abi
    monkeypatch.setattr(abi, "_lib", None)
    monkeypatch.setattr(abi, "LIB_PATH", str(tmp_path / "libzero.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        abi.lib()


def test_binding_constants_match_header(z):
    text = open(os.path.join(ROOT, "include", "zero.h")).read()
    for name in ("ZERO_FUSED_WINDOW_ELEMS", "ZERO_STATIC_CB_ELEMS",
                 "ZERO_GATHER_SEGMENTS_PER_LAUNCH", "ZERO_STREAM_GROUP_BYTES"):
        m = re.search(rf"#define {name} (\d+)ull", text)
        assert m and int(m.group(1)) == getattr(z._abi, name), name
    m = re.search(r"#define ZERO_MAX_ND (\d+)u", text)
    assert m and int(m.group(1)) == z._abi.ZERO_MAX_ND == 1 << 24
    m = re.search(r"#define ZERO_STEP_FLAG_WAIT_TIMEOUT (0x[0-9A-Fa-f]+)u", text)
    assert m and int(m.group(1), 16) == z._abi.ZERO_STEP_FLAG_WAIT_TIMEOUT
    # the flag word: zero commits, any nonfinite bit skips, the wait bit raises
    assert z._abi.check_step_flag(0) is False and z._abi.check_step_flag(1) is True
    with pytest.raises(z.ZeroError) as e:
        z._abi.check_step_flag(-(1 << 31) | 1)      # as an int32 read back from the device
    assert e.value.status == z.ZERO_ERR_TIMEOUT
    assert z._abi.fused_launch_count(117_187_500, 500_000_000) == 12
    assert z._abi.fused_launch_count(23_437_500, 50_000_000) == 3
    # the fused step plans its windows over the whole shard: the bucket size
    # does not add launches (the 4-rank workload's 4 buckets are one launch)
    assert z._abi.fused_launch_count(16, 1) == 1 and z._abi.fused_launch_count(0, 8) == 0
    assert z._abi.fused_launch_count(262_144, 65_536) == 1
    assert z._abi.fused_launch_count(117_187_500, 7) == 12
    # unfused: the reduction in the same windows, plus AdamW and cast, per bucket
    assert z._abi.unfused_launch_count(117_187_500, 500_000_000) == 12 + 2
    assert z._abi.unfused_launch_count(262_144, 65_536) == 4 * 3
    # bucket-ready groups: the 7.5B shard (18 GB of step traffic) keeps its 16
    # buckets apart; the 1.5B shard (3.6 GB) deals 16 buckets into 3 groups of
    # 6, 5 and 5; the 8-row shard (0.65 GB) is one group; the groups tile the shard
    g4 = z._abi.stream_groups(117_187_500, 7_324_224, 64)
    g3 = z._abi.stream_groups(23_437_500, 1_464_848, 64)
    g1 = z._abi.stream_groups(15_554_976, 972_192, 8)
    assert len(g4) == 16 and len(g1) == 1
    assert [round(x[1] / 1_464_848) for x in g3] == [6, 5, 5]
    for gs, n in ((g4, 117_187_500), (g3, 23_437_500), (g1, 15_554_976)):
        assert gs[0][0] == 0 and sum(x[1] for x in gs) == n
        assert all(a[0] + a[1] == b[0] for a, b in zip(gs, gs[1:]))
    assert z._abi.streamed_launch_count(117_187_500, 7_324_224, 64) == 16 * 2
    # a whole 64-shard vector is 64 segments: two gather launches; a layer
    # range inside one shard is one
    assert z._abi.gather_launch_count(1_500_000_000, 64, 0, 1_500_000_000) == 2
    assert z._abi.gather_launch_count(1000, 10, 95, 10) == 1
    assert z._abi.gather_launch_count(1000, 10, 0, 0) == 0
    assert z._abi.gather_launch_count(1000, 1000, 0, 1000) == 21


def _window_cuts(length: int, phase: int):
    from window_rule import window_cuts
    assert z_abi().ZERO_FUSED_WINDOW_ELEMS == 10485760
    return window_cuts(length, phase)


def z_abi():
    from zero_sharded_optimizer_02_gb300 import _abi
    return _abi


def test_launch_windows_properties():
    import random
    rng = random.Random(7)
    W = z_abi().ZERO_FUSED_WINDOW_ELEMS
    cases = [(117_187_500, 0), (23_437_500, 4), (10_485_760, 0), (10_485_761, 3),
             (25_165_824, 8), (25_165_825, 11), (2 ** 31 + 9, 0),
             (50_331_648 + 63, 5), (64, 7), (1, 0)]
    cases += [(rng.randrange(1, 400_000_000), rng.randrange(16)) for _ in range(300)]
    for length, phase in cases:
        cuts = _window_cuts(length, phase)
        # they tile the bucket in order
        assert cuts[0][0] == 0 and cuts[-1][1] == length
        assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:]))
        # every inner cut falls on a 32-byte (one L2 sector) boundary of the rows
        assert all((phase + c[0]) % 16 == 0 for c in cuts[1:])
        # ceil(length / W) windows (below 3.4e12 elements no remainder under
        # 64 is left after the last full window), none longer than W plus the
        # row phase (at most 15)
        nwin = -(-length // W)
        assert len(cuts) == nwin
        assert all(c[1] - c[0] <= W + 15 for c in cuts)
        # and the binding's launch count is exactly this split
        assert z_abi()._windows(length, phase) == len(cuts)


def test_header_is_plain_c_and_host_calls_work_from_c(z, tmp_path):
    """include/zero.h compiles as C99 with warnings as errors, and a C program
    linked against libzero.so gets the same layout and accounting as the
    binding (host-only calls: no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(z._abi.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe,
                           "-L", lib_dir, "-lzero", f"-Wl,-rpath,{lib_dir}"])
    out = subprocess.check_output([exe], text=True).splitlines()
    L = z.zero_partition_layout(350_000_017, 16, 15, 8)
    assert out[0] == (f"layout {L.shard_elems} {L.begin} {L.length} {L.padded_elems} "
                      f"{L.row_pitch}")
    for stage in range(4):
        expect = z.zero_model_state_bytes(7_500_000_000, 64, stage, 12)
        assert out[1 + stage] == f"bytes {stage} {expect}"
    assert out[5] == f"invalid {z.ZERO_ERR_INVALID_ARG}"
    assert out[6] == f"status {z.zero_status_string(z.ZERO_ERR_TIMEOUT)}"
    assert out[7] == f"window {z._abi.ZERO_FUSED_WINDOW_ELEMS}"


def test_launch_window_bounds_brute_force():
    """The split's bounds, brute force over small windows: with a window of
    W >= 1024 elements every range runs as ceil(n / W) windows, none longer
    than W + 15 (the row phase); with windows under 64 * 16 a remainder of
    under 64 elements may join a full window, the longest then W + 63."""
    from window_rule import window_cuts
    for W, lengths in ((1024, range(1, 12_000)), (4096, range(1, 40_000, 7)),
                       (64, range(1, 3_000)), (128, range(1, 3_000))):
        for length in lengths:
            for phase in range(16):
                cuts = window_cuts(length, phase, W)
                sizes = [b - a for a, b in cuts]
                assert max(sizes) <= W + (15 if W >= 1024 else 63), (W, length, phase)
                if W >= 1024:
                    assert len(cuts) == -(-length // W), (W, length, phase)
