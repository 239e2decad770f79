"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/oracle.c (on the
CPU, never in the committed oracle), builds it, swaps it in for liboracle.so
and runs the pin battery of test_oracle_pins.py; at least one pin must fail.
The unmodified copy must pass the same battery.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "no_weight_decay": ("p0 - G->lr * G->weight_decay * p0 - ", "p0 - "),
    "decay_not_scaled_by_lr": ("G->lr * G->weight_decay * p0", "G->weight_decay * p0"),
    "update_sign": ("- G->lr * mhat", "+ G->lr * mhat"),
    "beta2_in_first_moment": ("(1.0 - G->beta1) * gc", "(1.0 - G->beta2) * gc"),
    "no_bias_correction_m": ("double mhat = m1 / bc1;", "double mhat = m1;"),
    "no_bias_correction_v": ("double vhat = v1 / bc2;", "double vhat = v1;"),
    "eps_inside_sqrt": ("(sqrt(vhat) + G->eps)", "sqrt(vhat + G->eps)"),
    "v_not_squared": ("(1.0 - G->beta2) * gc * gc", "(1.0 - G->beta2) * gc"),
    "bias_correction_t_minus_1": ("pow(G->beta1, (double)t)", "pow(G->beta1, (double)(t - 1))"),
    "clip_inverted": ("return max_norm / norm;", "return norm / max_norm;"),
    "norm_without_sqrt": ("double norm = sqrt(sumsq);", "double norm = sumsq;"),
    "bf16_truncation": ("(u + 0x7fffu + lsb) >> 16", "u >> 16"),
    "bf16_ties_away": ("(u + 0x7fffu + lsb) >> 16", "(u + 0x8000u) >> 16"),
    "accumulate_in_bf16": ("return (float)((double)a + gd);",
                           "return orc_bf16_to_f32(orc_f32_to_bf16((float)((double)a + gd)));"),
    "first_micro_batch_adds": ("if (first) return (float)gd;", "if (first) return (float)((double)a + gd);"),
    "grad_scale_ignored_in_norm": ("double x = (double)orc_effective(k->acc[i], k->gs);",
                                   "double x = (double)k->acc[i];"),
    "clip_not_applied": ("double gc = (double)e * c;", "double gc = (double)e;"),
    "lr_warmup_off_by_one": ("return lr * (double)t / (double)warmup;", "return lr * (double)(t - 1) / (double)warmup;"),
    "lr_cosine_sign": ("(1.0 + cos(3.14159265358979323846 * s))", "(1.0 - cos(3.14159265358979323846 * s))"),
    "lr_no_min_floor": ("return min_lr + (lr - min_lr) * (1.0 + cos", "return lr * (1.0 + cos"),
    "betas_swapped_in_bias_correction": ("*bc1 = 1.0 - pow(G->beta1, (double)t);",
                                         "*bc1 = 1.0 - pow(G->beta2, (double)t);"),
    "bias_correction_t_plus_1": ("pow(G->beta1, (double)t)", "pow(G->beta1, (double)(t + 1))"),
    "first_moment_unclipped": ("(1.0 - G->beta1) * gc;", "(1.0 - G->beta1) * (double)e;"),
    "second_moment_unclipped": ("(1.0 - G->beta2) * gc * gc", "(1.0 - G->beta2) * (double)e * e"),
    "grad_scale_ignored_in_update": ("orc_effective(k->acc[i], k->gs), k->c,", "k->acc[i], k->c,"),
    "later_micro_batches_overwrite": ("return (float)((double)a + gd);", "return (float)gd;"),
    "eps_scaled_by_bias_correction": ("(sqrt(vhat) + G->eps)", "(sqrt(vhat) + G->eps / sqrt(bc2))"),
}

import test_lr_schedule as lr_pins  # noqa: E402

BATTERY = [getattr(pins, name) for name in dir(pins) if name.startswith("test_") and "exhaustive" not in name]
BATTERY.append(lr_pins.test_oracle_schedule_closed_forms)


def _build(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace('#include "../synth/synth.h"',
                             '#include "' + os.path.join(ROOT, "synth", "synth.h") + '"'))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-I", os.path.join(ROOT, "oracle"), "-o", str(so), str(c), "-lm"], check=True)
    return str(so)


def _run_battery(so_path):
    saved = oracle._lib
    oracle._lib = None
    real_build = oracle._build.build
    real_path = oracle._build.LIB_PATH
    oracle._build.build = lambda force=False: so_path
    oracle._build.LIB_PATH = so_path
    failed = []
    try:
        oracle.lib()
        for fn in BATTERY:
            try:
                fn()
            except Exception:  # a pin failing is what we look for
                failed.append(fn.__name__)
    finally:
        oracle._lib = saved
        oracle._build.build = real_build
        oracle._build.LIB_PATH = real_path
    return failed


def test_unmodified_copy_passes(tmp_path):
    so = _build(tmp_path, "orig", open(SRC).read())
    assert _run_battery(so) == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, mutant):
    src = open(SRC).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation site for {mutant} not found"
    so = _build(tmp_path, mutant, src.replace(old, new))
    failed = _run_battery(so)
    assert failed, f"no pin caught {mutant}"
