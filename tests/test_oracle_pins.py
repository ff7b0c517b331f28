"""The CPU oracle against its pins, and the pins against planted mistakes.

The second half compiles copies of the oracle source with one plausible
mistake each (a sign, a dropped factor, a wrong operand, a wrong index, the
physical-growth offset bug that "Add request-owned eight-way MTP serving for
Qwen 35B", section 2, describes) and checks that at least one pin fails for
every one of them.
"""
import os

import numpy as np
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


MUTANTS = {
    "erase_sign": ("double e = beta * (v[j] - a * u);", "double e = beta * (v[j] + a * u);"),
    "erase_undecayed": ("double e = beta * (v[j] - a * u);", "double e = beta * (v[j] - u);"),
    "beta_dropped": ("double e = beta * (v[j] - a * u);", "double e = (v[j] - a * u);"),
    "output_reads_k": ("oj += row[i] * q[i];", "oj += row[i] * k[i];"),
    "output_before_update": (
        "    for (int i = 0; i < dk; ++i) row[i] = a * row[i] + e * k[i];\n"
        "    double oj = 0.0;\n"
        "    for (int i = 0; i < dk; ++i) oj += row[i] * q[i];\n",
        "    double oj = 0.0;\n"
        "    for (int i = 0; i < dk; ++i) oj += row[i] * q[i];\n"
        "    for (int i = 0; i < dk; ++i) row[i] = a * row[i] + e * k[i];\n"),
    "taps_reversed": ("acc += w[(size_t)c * OR_W + j] * v;", "acc += w[(size_t)c * OR_W + (OR_W - 1 - j)] * v;"),
    "q_unscaled": ("1.0 / sqrt((double)dk), qh);", "1.0, qh);"),
    "key_head_modulo": ("int hk = (int)(((long long)h * Hk) / Hv);", "int hk = h % Hk;"),
    "q_k_swapped": ("or_l2norm(dk, yt + (size_t)hk * dk, 1.0 / sqrt((double)dk), qh);",
                    "or_l2norm(dk, yt + (size_t)Hk * dk + (size_t)hk * dk, 1.0 / sqrt((double)dk), qh);"),
    "commit_first_state": ("const double *src = Sall + ((size_t)b * T + (kp - 1)) * nS;",
                           "const double *src = Sall + ((size_t)b * T + 0) * nS;"),
    "offset_physical_growth": ("    offsets[b] += kp;\n  }\n}", "    offsets[b] += T;\n  }\n}"),
    "inactive_commits": ("    if (active[b]) {\n      if (keep[b] >= 0", "    if (1) {\n      if (keep[b] >= 0"),
    "window_not_advanced": ("      for (int i = 0; i < OR_HIST; ++i) wc[i] = tail[i];", "      (void)tail;"),
    "decay_missing_on_state": ("row[i] = a * row[i] + e * k[i];", "row[i] = row[i] + e * k[i];"),
    "accept_ties_last": ("if (best < 0 || x > best_v) {", "if (best < 0 || x >= best_v) {"),
    "accept_wrong_target": ("draft[(size_t)b * T + k] == target[k - 1]", "draft[(size_t)b * T + k] == target[k]"),
    "accept_next_from_last": ("    next[b] = target[k - 1];", "    next[b] = target[T - 1];"),
    "accept_inactive_kept": ("    if (!active[b]) {\n      keep[b] = 0;", "    if (0) {\n      keep[b] = 0;"),
    "norm_sum_not_mean": ("const double inv = 1.0 / sqrt(ss / d + eps);", "const double inv = 1.0 / sqrt(ss + eps);"),
    "gate_sigmoid": ("const double gate = zrow[j] / (1.0 + exp(-zrow[j]));", "const double gate = 1.0 / (1.0 + exp(-zrow[j]));"),
    "norm_weight_dropped": ("y[(size_t)r * d + j] = orow[j] * inv * w[j] * gate;", "y[(size_t)r * d + j] = orow[j] * inv * gate;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    with np.errstate(all="ignore"):
        for pin in pins.ALL_PINS:
            try:
                pin(mutant)
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
