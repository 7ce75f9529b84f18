"""The oracle's pins must catch plausible mistakes.  Each planted-mistake
build of the oracle (one bug each, compiled in from phs_oracle.c) is run
against the pin suite in a child process, which must fail; the clean build
must pass."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
MUTANTS = {
    1: "query head i uses KV head i % Hkv instead of i / G",
    2: "sliding window one token short",
    3: "softmax scale dropped",
    4: "ring slot walks the wrong way",
    5: "INT8 rounding half away from zero",
    6: "append writes the slot after the new token's",
    7: "INT8 dequantisation swaps the K and V scales",
    8: "page layout [page][slot][head] instead of [page][head][slot]",
    9: "softmax not normalised",
    10: "INT8 scale absmax / 128",
}


def _run_pins(lib_path):
    env = dict(os.environ)
    if lib_path:
        env["PHS_ORACLE_MUTANT_LIB"] = lib_path
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    so = oracle.build(mutant=mutant, out=str(tmp_path / f"libphs_oracle_m{mutant}.so"))
    rc, out = _run_pins(so)
    assert rc != 0, f"pins did not catch: {MUTANTS[mutant]}\n{out}"
