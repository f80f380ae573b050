"""Mutation test of the oracle's pins (CPU only).

Plants one plausible mistake at a time in a copy of the oracle's C source
(oracle/gdr_oracle.c), builds the broken copy in a temporary directory and
checks that at least one pin rejects it.  This shows the pins are strong
enough to catch a dropped term, a wrong sign, a wrong operand or index, and a
wrong head mapping in the real oracle.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from oracle import build as obuild
from tests import oracle_pins as pins

MUTANTS = {
    "no_decay": ("S[i * dv + j] *= gamma;", ";"),
    "decay_sign": ("exp(gt[i])", "exp(-gt[i])"),
    "update_sign": ("(vt[j] - vhat[j])", "(vt[j] + vhat[j])"),
    "no_beta": ("+= bt * kt[i] *", "+= kt[i] *"),
    "output_reads_key": ("ot[j] += S[i * dv + j] * qt[i]", "ot[j] += S[i * dv + j] * kt[i]"),
    "predict_reads_query": ("vhat[j] += S[i * dv + j] * kt[i]", "vhat[j] += S[i * dv + j] * qt[i]"),
    "interleaved_heads": ("const long hk = hv / group;", "const long hk = hv % HK;"),
    "h0_ignored": ("if (a->h0) {", "if (0) {"),
    "previous_token_gate": ("const double *gt = a->g + ((b * T + t) * HV + hv) * dk;",
                            "const double *gt = a->g + ((b * T + (t ? t - 1 : 0)) * HV + hv) * dk;"),
    "previous_token_beta": ("const double bt = a->beta[(b * T + t) * HV + hv];",
                            "const double bt = a->beta[(b * T + (t ? t - 1 : 0)) * HV + hv];"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation site not found exactly once: %r" % old
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib_path = os.path.join(tmp_path, "libmutant.so")
    subprocess.run(["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O1", "-fPIC", "-shared",
                    "-pthread", "-o", lib_path, path, "-lm"], check=True)
    lib = oracle._open(lib_path)

    def rec(q, k, v, g, beta, h0):
        return oracle.recurrence(q, k, v, g, beta, h0, _lib_override=lib)

    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(rec)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
