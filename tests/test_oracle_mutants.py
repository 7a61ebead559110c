"""The pins must catch plausible mistakes: each case plants one slip in a copy
of the oracle's C source (on the CPU, in a temporary directory), builds it,
swaps it in, and checks that at least one pin now fails."""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

ORACLE_C = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    # (replaced text, replacement)
    "silu_sign": ("g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
    "up_uses_gate": ("double u = q8_0_row_dot(wu, i, H, x);", "double u = q8_0_row_dot(wg, i, H, x);"),
    "down_index_swapped": ("y[o] = q8_0_row_dot(wd, o, I, a);",
                           "y[o] = q8_0_row_dot(wd, (o * 7) % H, I, a);"),
    "ties_to_higher_id": ("if (best < 0 || zt[e] > zt[best]) best = e;",
                          "if (best < 0 || zt[e] >= zt[best]) best = e;"),
    "bias_dropped": ("if (bias) acc += (double)bias[e];", "(void)bias;"),
    "round_half_down": ("double r = (a - fl >= 0.5) ? fl + 1.0 : fl;",
                        "double r = (a - fl > 0.5) ? fl + 1.0 : fl;"),
    "gates_not_renormalised": ("exp(zt[ids[t * k + j]] - zmax) / sum;",
                               "exp(zt[ids[t * k + j]] - zmax) / (sum + 1.0);"),
    "shared_dropped": ("for (int64_t h = 0; h < H; ++h) ot[h] += y[h];",
                       "for (int64_t h = 0; h < H; ++h) ot[h] += 0.0 * y[h];"),
    "scale_big_endian": ("return oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));",
                         "return oracle_half_to_double((uint16_t)(blk[1] | (blk[0] << 8)));"),
    "scale_rounded_before_division": ("q = round_half_away((double)x[i] / d);",
                                      "q = round_half_away((double)x[i] / oracle_half_to_double(dh));"),
    "perm_token_descending": ("for (int64_t t = 0; t < T; ++t)\n      for (int64_t j = 0; j < k; ++j)\n        if (ids",
                              "for (int64_t t = T - 1; t >= 0; --t)\n      for (int64_t j = 0; j < k; ++j)\n        if (ids"),
    "half_ties_away": ("return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "return fl + 1.0;"),
}

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and "generator" not in n]


def _run_pin(fn):
    import inspect
    params = inspect.signature(fn).parameters
    if "k" in params:
        for k in (1, 2, 5, 12):
            fn(k)
    else:
        fn()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(ORACLE_C).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(ORACLE_C[:-1] + "h").read())
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(mutated), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load(str(so)))
    failed = []
    for fn in PINS:
        try:
            _run_pin(fn)
        except AssertionError:
            failed.append(fn.__name__)
    assert failed, f"no pin caught mutant {name}"
