"""The oracle pins must reject plausible mistakes.

Each case copies oracle/mx_oracle.c, plants one slip (a swapped nibble order,
a gate/up swap, a wrong exponent bias, ...), builds the copy on the CPU and
runs tests/test_oracle_pins.py against it in a subprocess; the pins must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mx_oracle.c")

MUTANTS = {
    "nibble_order": ("(kk & 1) ? (byte >> 4) : (byte & 15u)", "(kk & 1) ? (byte & 15u) : (byte >> 4)"),
    "gate_up_swap": ("else { g = acc[i]; u = acc[I + i]; }", "else { g = acc[I + i]; u = acc[i]; }"),
    "interleave_parity": ("{ g = acc[2 * i]; u = acc[2 * i + 1]; }", "{ g = acc[2 * i + 1]; u = acc[2 * i]; }"),
    "clamp_gate_missing": ("    if (g > limit) g = limit;\n", ""),
    "clamp_gate_symmetric": ("    if (g > limit) g = limit;\n", "    if (g > limit) g = limit;\n    if (g < -limit) g = -limit;\n"),
    "clamp_up_missing": ("    if (u < -limit) u = -limit;\n", ""),
    "up_offset_missing": ("* (u + 1.0);", "* u;"),
    "alpha_missing": ("exp(-alpha * g)", "exp(-g)"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 8)"),
    "block_exponent_off_by_one": ("x = (e - 1) - emax_elem;", "x = e - emax_elem;"),
    "unstable_permutation": ("        perm[offsets[id] + fill[id]] = (int32_t)s;",
                             "        perm[offsets[id + 1] - 1 - fill[id]] = (int32_t)s;"),
    "dropped_routing_weight": ("sum[n] += wj * y;", "sum[n] += y;"),
    "route_tie_break": ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;"),
    "e2m1_subnormal": ("0.5 * (double)m : ldexp", "1.0 * (double)m : ldexp"),
    "dropped_weight_scale": ("acc += mxo_e8m0_value(sa[b]) * mxo_e8m0_value(sw[b]) * blk;",
                             "acc += mxo_e8m0_value(sa[b]) * blk;"),
    "silu_sign": ("if (act == 0) return g / (1.0 + exp(-g)) * u;", "if (act == 0) return g / (1.0 + exp(g)) * u;"),
    "bf16_truncation": ("q = ldexp(rne_nonneg(ldexp(a, 7 - e)), e - 7);", "q = ldexp(floor(ldexp(a, 7 - e)), e - 7);"),
    "renormalize_ignored": ("        if (renormalize) {", "        if (1) {"),
    "e4m3_no_saturation": ("if (a >= 448.0) return sign | 0x7Eu;", "if (a > 464.0) return sign | 0x7Fu;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mdir = tmp_path / name
    mdir.mkdir()
    msrc = mdir / "mx_oracle.c"
    msrc.write_text(src.replace(old, new))
    env = dict(os.environ, MXO_ORACLE_SRC=str(msrc))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins accepted the {name} mutant:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
