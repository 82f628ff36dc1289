"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is one textual edit of ``oracle/attention_oracle.c`` (a dropped
term, a wrong sign or index, a swapped operand), compiled on the CPU into a
temporary library.  A mutant that every pin accepts means the pins could not
tell that mistake from the truth, so the test fails.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_oracle.c")

MUTANTS = {
    "scale_dropped": ("s[kk] = scale * dot(qi, k + kk * d, d);", "s[kk] = dot(qi, k + kk * d, d);"),
    "mask_strict": ("return k <= i + (Nk - Nq);", "return k < i + (Nk - Nq);"),
    "mask_top_left": ("return k <= i + (Nk - Nq);", "return k <= i;"),
    "block_transposed": ("(i / m->bs) * m->nbc + k / m->bs]", "(k / m->bs) * m->nbc + i / m->bs]"),
    "block_head_ignored": ("m->block[g * m->head_stride +", "m->block[0 * m->head_stride +"),
    "block_ignored": ("if (m->block && !m->block[", "if (0 && m->block && !m->block["),
    "block_overrides_causal": ("        return 0;\n    if (!m->causal)", "        return 0;\n    if (m->block || !m->causal)"),
    "lse_log2": ("return m + log(l);", "return m + log2(l);"),
    "lse_no_max": ("return m + log(l);", "return log(l);"),
    "pv_wrong_operand": ("oi[c] += p * v[kk * d + c];", "oi[c] += p * k[kk * d + c];"),
    "delta_wrong_operand": ("D[r] = dot(dout + r * d, o + r * d, d);",
                            "D[r] = dot(dout + r * d, q + r * d, d);"),
    "dq_wrong_operand": ("dqi[c] += scale * ds * k[kk * d + c];", "dqi[c] += scale * ds * v[kk * d + c];"),
    "dq_scale_dropped": ("dqi[c] += scale * ds * k[kk * d + c];", "dqi[c] += ds * k[kk * d + c];"),
    "dk_scale_dropped": ("dkk[c] += scale * ds * qi[c];", "dkk[c] += ds * qi[c];"),
    "dv_uses_ds": ("dvk[c] += p * doi[c];", "dvk[c] += ds * doi[c];"),
    "ds_sign_flip_dk": ("double ds = p * (dp - D[r]);\n            for (long c = 0; c < d; ++c) {",
                        "double ds = p * (dp + D[r]);\n            for (long c = 0; c < d; ++c) {"),
    "ds_sign_flip_dq": ("double ds = p * (dp - D[r]);\n            for (long c = 0; c < d; ++c)\n                dqi",
                        "double ds = p * (D[r] - dp);\n            for (long c = 0; c < d; ++c)\n                dqi"),
    "dp_transposed": ("double dp = dot(doi, v + kk * d, d);\n            double ds = p * (dp - D[r]);\n            for (long c = 0; c < d; ++c) {",
                      "double dp = dot(doi, k + kk * d, d);\n            double ds = p * (dp - D[r]);\n            for (long c = 0; c < d; ++c) {"),
}


def _cases():
    src = open(SRC).read()
    for name in sorted(MUTANTS):
        n = src.count(MUTANTS[name][0])
        # each occurrence on its own, and all of them at once
        for which in ([0] if n == 1 else list(range(n)) + ["all"]):
            yield name, which


def _mutate(src, old, new, which):
    if which == "all":
        return src.replace(old, new)
    at = -1
    for _ in range(which + 1):
        at = src.index(old, at + 1)
    return src[:at] + new + src[at + len(old):]


@pytest.mark.parametrize("name,which", list(_cases()))
def test_pins_catch_mutant(name, which, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in the oracle source"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(_mutate(src, old, new, which))
    lib = oracle.load(oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmutant.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects the planted mistake {name} (occurrence {which})"
