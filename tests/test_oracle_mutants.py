"""The oracle's pins must catch plausible mistakes.  Each planted mistake is
one textual change to a copy of oracle/phs_oracle.c (the committed source
holds none of them); the copy is compiled and the pin suite run against it
in a child process, which must fail.  Every change must apply to exactly
the places it names, so a mutant cannot silently stop applying when the
oracle is edited."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "phs_oracle.c")

# name -> list of (text in the clean source, replacement)
MUTANTS = {
    "query head i uses KV head i % Hkv instead of i / G": [
        ("        int h = i / G;\n", "        int h = i % Hkv;\n"),
        ("Hkv, D, i / G, ring_pos[b], n};", "Hkv, D, i % Hkv, ring_pos[b], n};")],
    "sliding window one token short": [
        ("int64_t t0 = n > W ? n - W : 0;", "int64_t t0 = n > W ? n - W + 1 : 0;")],
    "softmax scale dropped": [
        ("s[t - t0] = acc * scale;", "s[t - t0] = acc;")],
    "ring slot walks the wrong way": [
        ("pos_mod(c->newest_slot - (c->n - 1 - t), c->W)",
         "pos_mod(c->newest_slot + (c->n - 1 - t), c->W)")],
    "INT8 rounding half away from zero": [
        ("float r = rintf(x / s);", "float r = roundf(x / s);")],
    "append writes the slot after the new token's": [
        ("int64_t t = n - 1; /* the new token's position */", "int64_t t = n;")],
    "INT8 dequantisation swaps the K and V scales": [
        ("(is_v ? c->v_scale : c->k_scale)", "(is_v ? c->k_scale : c->v_scale)")],
    "page layout [page][slot][head] instead of [page][head][slot]": [
        ("int64_t dst = ((page * Hkv + h) * P + slot) * D + d;",
         "int64_t dst = ((page * P + slot) * Hkv + h) * D + d;"),
        ("pool + ((page * c->Hkv + c->h) * c->P + t % c->P) * c->D;",
         "pool + ((page * c->P + t % c->P) * c->Hkv + c->h) * c->D;")],
    "softmax not normalised": [
        ("    for (int d = 0; d < D; ++d) out[d] /= l;\n", "")],
    "INT8 scale absmax / 128": [
        ("return absmax / 127.0f;", "return absmax / 128.0f;")],
    "ring seed places token t at the mirrored slot": [
        ("pos_mod(pos - (n - 1 - t), W); /* seed: ring slot of token t */",
         "pos_mod(pos + (n - 1 - t), W);")],
    "ring seed takes the window's first page as n / P - W / P": [
        ("        int64_t first = lo / P;\n", "        int64_t first = n / P - W / P;\n")],
    "ring save copies a page shifted by one token": [
        ("int64_t dst = ((sp * Hkv + h) * P + t % P) * D + d;",
         "int64_t dst = ((sp * Hkv + h) * P + (t + 1) % P) * D + d;")],
}


def _run_pins(lib_path):
    env = dict(os.environ)
    if lib_path:
        env["PHS_ORACLE_MUTANT_LIB"] = lib_path
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def _planted(changes):
    with open(SRC) as f:
        text = f.read()
    for old, new in changes:
        assert text.count(old) == 1, f"mutant text not found exactly once: {old!r}"
        text = text.replace(old, new)
    return text


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = tmp_path / "phs_oracle_mutant.c"
    src.write_text(_planted(MUTANTS[name]))
    so = oracle.build(src=str(src), out=str(tmp_path / "libphs_oracle_mutant.so"))
    rc, out = _run_pins(so)
    assert rc != 0, f"pins did not catch: {name}\n{out}"


def test_committed_oracle_holds_no_planted_mistake():
    with open(SRC) as f:
        text = f.read()
    assert "MUTANT" not in text
    for changes in MUTANTS.values():
        for old, new in changes:
            if new:
                assert new not in text
