"""Each plausible mistake planted in a copy of the oracle (on the CPU) fails at least one pin.

The copies are compiled into a temporary directory from the real source with one textual
change each; the real oracle source is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "no_dt_on_B": ("const double bx = dt[t] * xt[p];", "const double bx = xt[p];"),
    "read_before_update": (
        "hp[n] = abar * hp[n] + bx * Bt[n];   /* h_t = Abar_t h_{t-1} + Bbar_t x_t */\n"
        "                acc += Ct[n] * hp[n];",
        "acc += Ct[n] * hp[n];\n"
        "                hp[n] = abar * hp[n] + bx * Bt[n];"),
    "sign_of_A": ("exp(dt[t] * A)", "exp(-dt[t] * A)"),
    "B_C_swapped": ("bx * Bt[n]", "bx * Ct[n]"),
    "no_skip": ("yt[p] = acc + D * xt[p];", "yt[p] = acc;"),
    "h0_ignored": ("if (h0) memcpy", "if (0) memcpy"),
    "decay_off_by_one": ("exp(dt[t] * A)", "exp(dt[t > 0 ? t - 1 : 0] * A)"),
    "decay_without_dt": ("exp(dt[t] * A)", "exp(A)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found in the oracle source"
    mpath = tmp_path / f"mutant_{name}.c"
    mpath.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mpath), out=str(tmp_path / f"libmutant_{name}.so"))
    lib = oracle.OracleLib(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
