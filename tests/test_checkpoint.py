"""Sharded checkpoints and resharding, on the CPU (host arrays only).

"ZeRO" (process-cxr ai-library), checkpointing and recovery: each rank saves
the state it owns; the metadata must be reliable and resuming on another
number of GPUs must be possible.  The step is elementwise over the flat
parameter vector, so a resharded load must reproduce the saved flat arrays
bit for bit.
"""
import os

import numpy as np
import pytest


@pytest.fixture(scope="module")
def z():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    import zero_sharded_optimizer_02_gb300 as z
    return z


H = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _save_all(z, tmp_path, flat, psi, nd, step=7, tag="ck"):
    paths = []
    for r in range(nd):
        L = z.zero_partition_layout(psi, nd, r, 8)
        b, n = int(L.begin), int(L.length)
        arrs = [np.ascontiguousarray(a[b:b + n]) for a in flat]
        p = str(tmp_path / f"{tag}_rank{r}.zck")
        z.zero_checkpoint_save(p, L, z.adamw(**H, step=step), *arrs)
        paths.append(p)
    return paths


def _load_flat(z, paths, psi, nd_new):
    out = [np.empty(psi, np.float32) for _ in range(3)]
    steps = set()
    for r in range(nd_new):
        L = z.zero_partition_layout(psi, nd_new, r, 8)
        b, n = int(L.begin), int(L.length)
        part = [np.empty(max(n, 1), np.float32) for _ in range(3)]
        h = z.zero_checkpoint_load(paths, L, *part)
        steps.add(int(h.step))
        assert (h.lr, h.beta1, h.beta2, h.eps, h.weight_decay) == tuple(H.values())
        for a, p in zip(out, part):
            a[b:b + n] = p[:n]
    return out, steps


@pytest.mark.parametrize("psi,nd_old,nd_new", [(1000, 4, 4), (1000, 4, 3), (1001, 4, 7),
                                                (10_007, 16, 1), (5, 8, 2), (257, 1, 64)])
def test_reshard_is_bit_exact(z, tmp_path, psi, nd_old, nd_new):
    rng = np.random.default_rng(psi + nd_old)
    flat = [rng.standard_normal(psi).astype(np.float32) for _ in range(3)]
    paths = _save_all(z, tmp_path, flat, psi, nd_old)
    got, steps = _load_flat(z, paths, psi, nd_new)
    assert steps == {7}
    for a, b in zip(got, flat):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_header_round_trip(z, tmp_path):
    flat = [np.arange(100, dtype=np.float32) * k for k in (1, 2, 3)]
    paths = _save_all(z, tmp_path, flat, 100, 3, step=42)
    hd = z.zero_checkpoint_read_header(paths[2])
    assert hd.magic == b"ZEROCKPT" and hd.version == 2 and hd.header_bytes == 112
    assert (hd.psi, hd.nd, hd.rank, hd.shard_elems, hd.begin, hd.length, hd.step) == \
        (100, 3, 2, 34, 68, 32, 42)
    assert os.path.getsize(paths[2]) == 112 + 3 * 32 * 4
    assert not any(p.endswith(".tmp") for p in os.listdir(tmp_path))


def test_detects_corruption_and_bad_sets(z, tmp_path):
    psi, nd = 999, 3
    flat = [np.ones(psi, np.float32) * k for k in (1, 2, 3)]
    paths = _save_all(z, tmp_path, flat, psi, nd)
    L = z.zero_partition_layout(psi, 2, 1, 8)
    buf = [np.empty(int(L.length), np.float32) for _ in range(3)]
    # a flipped payload byte
    with open(paths[1], "r+b") as f:
        f.seek(112 + 40)
        b = f.read(1)
        f.seek(112 + 40)
        f.write(bytes([b[0] ^ 0x10]))
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_load(paths, L, *buf)
    assert e.value.status == z.ZERO_ERR_IO
    paths = _save_all(z, tmp_path, flat, psi, nd, tag="ok")
    # a torn file
    torn = str(tmp_path / "torn.zck")
    with open(paths[2], "rb") as f, open(torn, "wb") as g:
        g.write(f.read()[:-8])
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_load([paths[0], paths[1], torn], z.zero_partition_layout(psi, 1, 0, 8),
                               *[np.empty(psi, np.float32) for _ in range(3)])
    assert e.value.status == z.ZERO_ERR_IO
    # missing file, ranks out of order, a different step, a bad header
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_load([paths[0], str(tmp_path / "nope"), paths[2]], L, *buf)
    assert e.value.status == z.ZERO_ERR_IO
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_load([paths[1], paths[0], paths[2]], L, *buf)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG
    other = _save_all(z, tmp_path, flat, psi, nd, step=8, tag="s8")
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_load([paths[0], other[1], paths[2]], L, *buf)
    assert e.value.status == z.ZERO_ERR_IO
    junk = str(tmp_path / "junk.zck")
    with open(junk, "wb") as f:
        f.write(b"not a checkpoint" * 10)
    with pytest.raises(z.ZeroError) as e:
        z.zero_checkpoint_read_header(junk)
    assert e.value.status == z.ZERO_ERR_IO
    with pytest.raises(z.ZeroError) as e:    # layout the partition would not produce
        bad = z.zero_partition_layout(psi, nd, 0, 8)
        bad.length = 5
        z.zero_checkpoint_save(str(tmp_path / "x"), bad, z.adamw(**H, step=1), *buf)
    assert e.value.status == z.ZERO_ERR_INVALID_ARG


def _checksum_by_definition(arrays) -> int:
    """The payload checksum as the header defines it, written out: 8 FNV-1a
    lanes over the little-endian 32-bit words (word k to lane k mod 8), then
    FNV-1a over the 64 bytes of the lane states."""
    mask, basis, prime = (1 << 64) - 1, 0xCBF29CE484222325, 0x100000001B3
    words = np.concatenate([np.asarray(a, "<f4").view("<u4") for a in arrays]).tolist()
    lanes = []
    for lane in range(8):
        h = basis
        for w in words[lane::8]:
            h = ((h ^ w) * prime) & mask
        lanes.append(h)
    x = basis
    for h in lanes:
        for k in range(8):
            x = ((x ^ ((h >> (8 * k)) & 0xFF)) * prime) & mask
    return x


@pytest.mark.parametrize("psi,nd", [(3001, 3), (40, 5), (7, 8)])
def test_payload_checksum_matches_its_definition(z, tmp_path, psi, nd):
    # lengths that are not multiples of 8 move the lane phase between the
    # three arrays and between the loader's chunks
    rng = np.random.default_rng(psi)
    flat = [rng.standard_normal(psi).astype(np.float32) for _ in range(3)]
    paths = _save_all(z, tmp_path, flat, psi, nd)
    for r, p in enumerate(paths):
        L = z.zero_partition_layout(psi, nd, r, 8)
        b, n = int(L.begin), int(L.length)
        h = z.zero_checkpoint_read_header(p)
        assert h.version == 2
        assert int(h.payload_checksum) == _checksum_by_definition([a[b:b + n] for a in flat])
