"""Planted mistakes in copies of the oracle must each fail a pin.

Each case edits one line of ``oracle/zero_oracle.c`` (a dropped term, a wrong
sign or index, a wrong convention), compiles the copy on the CPU into a
temporary directory and runs the pins of ``pins.py`` against it.  The real
oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle
import pins

MUTANTS = {
    "m_drops_gradient_term": ("float m1 = m_decay + m_new;", "float m1 = m_decay;"),
    "v_uses_g_not_g2": ("float g2 = g * g;", "float g2 = g;"),
    "step_sign_flipped": ("*p_out = p_decayed - step;", "*p_out = p_decayed + step;"),
    "eps_inside_sqrt": ("float denom = sqrtf(v_hat) + k->eps;",
                        "float denom = sqrtf(v_hat + k->eps);"),
    "bias_correction_off_by_one": ("o->bc1 = (float)(1.0 - pow(h->beta1, (double)t));",
                                   "o->bc1 = (float)(1.0 - pow(h->beta1, (double)(t + 1)));"),
    "no_bias_correction_v": ("float v_hat = v1 / k->bc2;", "float v_hat = v1;"),
    "weight_decay_not_times_lr": ("o->wdf = (float)(1.0 - h->lr * h->weight_decay);",
                                  "o->wdf = (float)(1.0 - h->weight_decay);"),
    "scale_missing_nd": ("o->inv = (float)(1.0 / ((double)nd * loss_scale));",
                         "o->inv = (float)(1.0 / loss_scale);"),
    "fold_reverse_order": (
        "    float s = grad_at(base, dtype, idx);\n    for (uint32_t j = 1; j < nd; ++j)\n"
        "        s = s + grad_at(base, dtype, (uint64_t)j * row_stride + idx);",
        "    float s = grad_at(base, dtype, (uint64_t)(nd - 1) * row_stride + idx);\n"
        "    for (uint32_t j = nd - 1; j-- > 0;)\n"
        "        s = s + grad_at(base, dtype, (uint64_t)j * row_stride + idx);"),
    "fold_skips_last_rank": ("for (uint32_t j = 1; j < nd; ++j)\n        s = s + grad_at(",
                             "for (uint32_t j = 1; j + 1 < nd; ++j)\n        s = s + grad_at("),
    "encode_truncates": ("nearbyint(ax / quantum)", "floor(ax / quantum)"),
    "encode_ties_away": ("nearbyint(ax / quantum)", "round(ax / quantum)"),
    "decode_subnormal_scale": ("ldexp((double)frac, f->emin - f->frac_bits)",
                               "ldexp((double)frac, f->emin - f->frac_bits - 1)"),
    "layout_floor_not_ceil": ("    uint64_t s = psi / nd + (psi % nd != 0);\n    uint64_t begin",
                              "    uint64_t s = psi / nd;\n    uint64_t begin"),
    "stage2_grads_not_partitioned": ("case 2: return 2 * psi + (2 + (uint64_t)k) * s;",
                                     "case 2: return 4 * psi + (uint64_t)k * s;"),
    "bucket_drops_scaling": ("cb[i] = s * k.inv;", "cb[i] = s;"),
    "shard_wrong_state_offset": ("adamw_elem(&k, cb[i], p[e], m[e], v[e]",
                                 "adamw_elem(&k, cb[i], p[i], m[i], v[i]"),
    "stage3_comm_like_stage2": ("uint64_t mult = stage == 3 ? 3 : 2;",
                                "uint64_t mult = 2;"),
    "mp_slice_floor": ("uint64_t slice = psi / nm + (psi % nm != 0);", "uint64_t slice = psi;"),
    "gather_wrong_owner": ("uint64_t r = flat / s;", "uint64_t r = flat / pitch;"),
    "skip_ignored": ("        if (!isfinite(orc_fold(grads, dtype, nd, row_stride, i)))\n"
                     "            return 1;", "        (void)0;"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(source, tmp_path, name):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation anchor not found: {name}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", str(src), "-o", str(so), "-lm"])
    failed = []
    with oracle.use_library(str(so)):
        for check in pins.ALL:
            try:
                check(oracle)
            except AssertionError:
                failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
