"""Pins of the oracle's partition layout and model-state accounting.

Values come from the golden fixtures (printed on the pages, cited there) and
from brute force over small partitions.
"""
import os

import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _kv(name):
    return {r[0]: r[1] for r in _rows(name)}


def _as_printed(x: float, printed: str) -> float:
    """Round x to the number of decimals the printed value shows."""
    decimals = len(printed.split(".")[1]) if "." in printed else 0
    return round(x, decimals)


def test_memory_table_7p5b(orc):
    rows = _rows("memory_table_7p5b.txt")
    psi = int(rows[0][1])
    k = int(rows[1][1])
    for r in rows[2:]:
        nd = int(r[0])
        for stage, printed in enumerate(r[1:]):
            got = orc.model_state_bytes(psi, nd, stage, k)
            assert _as_printed(got / 1e9, printed) == float(printed), (nd, stage, got)


def test_memory_table_exact_bytes(orc):
    # Exact bytes where Nd divides Psi (the pages' formula is then an integer).
    psi = 7_500_000_000
    exp = {(1, 0): 120e9, (64, 0): 120e9, (64, 1): 31_406_250_000, (64, 2): 16_640_625_000,
           (64, 3): 1_875_000_000}
    for (nd, st), b in exp.items():
        assert orc.model_state_bytes(psi, nd, st, 12) == b
        assert orc.model_state_bytes_formula(psi, nd, st, 12) == b
    # Nd = 1024 does not divide 7.5e9: a rank holds ceil(Psi/Nd) = 7,324,219 parameters.
    assert orc.model_state_bytes(psi, 1024, 1, 12) == 30_000_000_000 + 12 * 7_324_219
    assert orc.model_state_bytes(psi, 1024, 2, 12) == 15_000_000_000 + 14 * 7_324_219
    assert orc.model_state_bytes(psi, 1024, 3, 12) == 16 * 7_324_219
    assert orc.model_state_bytes_formula(psi, 1024, 2, 12) == 15_102_539_062.5


def test_sixteen_bytes_per_param(orc):
    kv = _kv("model_state_examples.txt")
    parts = [int(kv[k]) for k in ("bytes_fp16_param", "bytes_fp16_grad", "bytes_fp32_master",
                                  "bytes_fp32_momentum", "bytes_fp32_variance")]
    assert sum(parts) == int(kv["bytes_total"]) == 4 + int(kv["k"])
    for nd in (1, 3, 64):
        assert orc.model_state_bytes(1, nd, 0, 12) == int(kv["bytes_total"])
    # GPT-2 1.5B needs 24 GB of model states (stage 0 on one GPU).
    assert orc.model_state_bytes(int(kv["gpt2_psi"]), 1, 0, int(kv["k"])) == \
        int(kv["gpt2_min_gb"]) * 10 ** 9
    # CB example: a 3B model's fp32 buffer is 12 GB.
    assert int(kv["cb_psi"]) * 4 == int(kv["cb_fp32_gb"]) * 10 ** 9


def test_stage_reduction_limits(orc):
    # About 4x (P_os), 8x (P_os+g) and Nd x (P_os+g+p) for large Nd.
    psi = 10 ** 12
    nd = 1 << 20
    base = orc.model_state_bytes(psi, nd, 0)
    assert base / orc.model_state_bytes(psi, nd, 1) == pytest.approx(4.0, rel=1e-4)
    assert base / orc.model_state_bytes(psi, nd, 2) == pytest.approx(8.0, rel=1e-4)
    assert base / orc.model_state_bytes(psi, nd, 3) == pytest.approx(nd, rel=1e-4)
    for nd in (1, 2, 7):
        assert len({orc.model_state_bytes(psi, 1, s) for s in range(4)}) == 1


def test_invalid_accounting_args(orc):
    assert orc.model_state_bytes(10, 0, 0) == 2 ** 64 - 1
    assert orc.model_state_bytes(10, 1, 4) == 2 ** 64 - 1
    assert orc.model_state_bytes(2 ** 62, 1, 0) == 2 ** 64 - 1


def test_layout_brute_force(orc):
    for psi in range(0, 201):
        for nd in range(1, 18):
            covered = []
            s_expected = -(-psi // nd)
            for r in range(nd):
                s, begin, n = orc.layout(psi, nd, r)
                assert s == s_expected
                assert begin == r * s
                assert 0 <= n <= s
                covered.extend(range(begin, begin + n))
                if n < s:   # only trailing shards are short
                    assert all(orc.layout(psi, nd, q)[2] == 0 for q in range(r + 1, nd))
            assert covered == list(range(psi))


def test_layout_padding_case(orc):
    # 350,000,017 parameters over 16 ranks: shard 21,875,002, last one 15 short.
    s, begin, n = orc.layout(350_000_017, 16, 15)
    assert (s, begin, n) == (21_875_002, 15 * 21_875_002, 21_874_987)
    assert 16 * s - 350_000_017 == 15
    with pytest.raises(ValueError):
        orc.layout(10, 0, 0)
    with pytest.raises(ValueError):
        orc.layout(10, 4, 4)
