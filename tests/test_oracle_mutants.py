"""Planted mistakes: each case copies oracle/conv_ref.c to a temporary
directory, plants one plausible bug (a dropped term, a wrong sign, index or
stride, a transposed operand, a wrong mask), builds it with gcc and checks that
at least one oracle pin rejects it.  The real oracle is never modified.  Every
mutant keeps all memory accesses in bounds."""
import os
import subprocess

import pytest

import oracle

from . import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "conv_ref.c")

# (name, text to find, replacement, which occurrence (0-based))
MUTANTS = [
    ("fwd: kh/kw swapped in the input row", "const int64_t h = oh * s->S + kh,",
     "const int64_t h = oh * s->S + kw,", 0),
    ("fwd: ReLU inverted", "j->out[o] = (s->relu && !(acc > 0.0)) ? 0.0 : acc;",
     "j->out[o] = (s->relu && (acc > 0.0)) ? 0.0 : acc;", 0),
    ("fwd: weight operand transposed (ic, oc)", "w[((oc * s->IC + ic) * s->K + kh) * s->K + kw]",
     "w[((ic * s->OC + oc) * s->K + kh) * s->K + kw]", 0),
    ("fwd: wrong sign of a term", "acc += t;", "acc -= t;", 0),
    ("fwd: denominator without abs", "den += fabs(t);", "den += t;", 0),
    ("dgrad: stride divisibility check dropped", "if (th < 0 || th % s->S != 0 || th / s->S >= OH)",
     "if (th < 0 || th / s->S >= OH)", 0),
    ("dgrad: kernel taps flipped", "w[((oc * s->IC + ic) * s->K + kh) * s->K + kw]",
     "w[((oc * s->IC + ic) * s->K + kw) * s->K + kh]", 1),
    ("dgrad: a term halved", "acc += t;", "acc += 0.5 * t;", 1),
    ("wgrad: stride ignored on the column", "ow * s->S + kw];", "ow + kw];", 0),
    ("wgrad: last sample dropped", "for (int64_t b = 0; b < s->B; ++b)",
     "for (int64_t b = 0; b + 1 < s->B; ++b)", 0),
    ("wgrad: denominator without abs", "den += fabs(t);", "den += t;", 2),
    ("mask: gradient passes at y == 0", "if (s->relu && !(y[i] > 0.0)) return 0.0;",
     "if (s->relu && !(y[i] >= 0.0)) return 0.0;", 0),
    ("mask: ignored", "if (s->relu && !(y[i] > 0.0)) return 0.0;", "", 0),
    ("fwd bias: one channel's bias for all", "const double bv = j->c[oc];",
     "const double bv = j->c[0];", 0),
    ("fwd bias: subtracted", "acc += bv;", "acc -= bv;", 0),
    ("fwd bias: denominator term dropped", "den += fabs(bv);", "", 0),
    ("fwd bias: added after the ReLU", "j->out[o] = (s->relu && !(acc > 0.0)) ? 0.0 : acc;",
     "j->out[o] = (s->relu && !(acc - (j->c ? j->c[oc] : 0.0) > 0.0)) ? (j->c ? j->c[oc] : 0.0) : acc;",
     0),
    ("bias grad: mask ignored", "const double t = ref_g(s, dy, y, ((b * s->OC + oc) * OH + oh) * OW + ow);",
     "const double t = dy[((b * s->OC + oc) * OH + oh) * OW + ow];", 0),
    ("bias grad: last sample dropped", "for (int64_t b = 0; b < s->B; ++b)",
     "for (int64_t b = 0; b + 1 < s->B; ++b)", 1),
]


def _replace_nth(text, old, new, n):
    pos = -1
    for _ in range(n + 1):
        pos = text.find(old, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {old!r} (occurrence {n})"
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    c = tmp_path / "conv_ref_mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-pthread", "-std=c11", "-o", str(so),
                    str(c), "-lm"], check=True)
    lib = oracle.bind(str(so))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {name}"
