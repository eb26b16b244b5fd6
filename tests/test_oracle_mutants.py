"""Plant plausible mistakes in a copy of the oracle and check a pin fails.

Each mutant is the oracle source with one textual edit (a dropped term, a
flipped sign, a wrong index or operand, a wrong mask alignment).  The copy
is executed as a fresh module on the CPU; the real oracle is untouched.  A
mutant that no pin in ``test_oracle_pins`` rejects would mean the pins leave
that part of the oracle unchecked.
"""

import os
import types

import numpy as np
import pytest

import test_oracle_pins as P

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "streamkl_oracle.py")

MUTANTS = {
    "kl weight P2 instead of P1": ("p1 * (logp1 - logp2), 0.0), axis=1)", "p2 * (logp1 - logp2), 0.0), axis=1)"),
    "kl log ratio flipped": ("p1 * (logp1 - logp2), 0.0), axis=1)", "p1 * (logp2 - logp1), 0.0), axis=1)"),
    "lse without max shift back": ("return m + np.log(", "return np.log("),
    "scale dropped on S2": ("s2 * (q2[rows] @ k2.T)", "(q2[rows] @ k2.T)"),
    "S2 takes the S1 scale": ("s2 * (q2[rows] @ k2.T)", "s1 * (q2[rows] @ k2.T)"),
    "online S2 takes the S1 scale": ("s2 = sc2 * (q2[rows] @ k2[keys].T)\n            t1", "s2 = sc1 * (q2[rows] @ k2[keys].T)\n            t1"),
    "gradient scale of the other side": ("sg = s2 if mode == MODE_P2 else s1\n    dq = np.zeros", "sg = s1 if mode == MODE_P2 else s2\n    dq = np.zeros"),
    "top-left causal alignment": ("return j <= rows[:, None] + (nk - nq)", "return j <= rows[:, None]"),
    "strict causal mask": ("return j <= rows[:, None] + (nk - nq)", "return j < rows[:, None] + (nk - nq)"),
    "online acc not rescaled": ("acc = a1 * acc + ", "acc = acc + "),
    "online l2 rescaled by m1": ("l2 = a2 * l2 + ", "l2 = a1 * l2 + "),
    "online diff sign": ("e1 * (s1 - s2), 0.0), axis=1)", "e1 * (s2 - s1), 0.0), axis=1)"),
    "two-pass final sign": ("kl[rows] = w - a + b", "kl[rows] = w + a - b"),
    "mode P2 sign": ('ds = dkl_rows[:, None] * (r["p2"] - r["p1"])', 'ds = dkl_rows[:, None] * (r["p1"] - r["p2"])'),
    "mode P1 drops KL": ('(ratio - r["kl"][:, None])', '(ratio)'),
    "mode P1 weight P2": ('ds = dkl_rows[:, None] * r["p1"] * (ratio', 'ds = dkl_rows[:, None] * r["p2"] * (ratio'),
    "dkl ignored": ('ds = dkl_rows[:, None] * (r["p2"] - r["p1"])', 'ds = (r["p2"] - r["p1"])'),
    "dq scale dropped": ("dq[rows] = sg * (ds @ kg)", "dq[rows] = (ds @ kg)"),
    "dk uses other side": ("dk += sg * (ds.T @ qg[rows])", "dk += sg * (ds.T @ (q1 if mode == MODE_P2 else q2)[rows][:, :qg.shape[1]])"),
    "sampled dq wrong side": ("kg, sg = (k2, s2) if mode == MODE_P2 else (k1, s1)", "kg, sg = (k1, s2) if mode == MODE_P2 else (k2, s1)"),
    "grouped key head by modulo": ("k1[b, h // g1], q2[b, h], k2[b, h // g2], scale, causal, row_block,\n",
                                   "k1[b, h % k1.shape[1]], q2[b, h], k2[b, h % k2.shape[1]], scale, causal, row_block,\n"),
    "grouped dK overwritten, not summed": ("dk[b, h // gg] += dk_h", "dk[b, h // gg] = dk_h"),
    "grouped dK into the other side's head": ("dk[b, h // gg] += dk_h", "dk[b, h // (g1 if gg == g2 else g2)] += dk_h"),
    "sampled forward rows taken as positions": ("causal, np.asarray(rows))\n    return r[\"kl\"]",
                                                "causal, np.arange(len(rows)))\n    return r[\"kl\"]"),
    "sampled forward ignores the second scale": ("r = _head_rows(q1, k1, q2, k2, *_scales(scale, scale2), causal, np.asarray(rows))",
                                                 "r = _head_rows(q1, k1, q2, k2, scale, scale, causal, np.asarray(rows))"),
    "sampled dk missing scale": ("dk += sg * (ds.T @ qg[rows])\n    return dk\n\n\ndef loss", "dk += (ds.T @ qg[rows])\n    return dk\n\n\ndef loss"),
}


def _load(src, name):
    mod = types.ModuleType(name)
    exec(compile(src, name, "exec"), mod.__dict__)
    return mod


def _failing_pins(mod):
    failed = []
    for pin in P.PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError, ZeroDivisionError):
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes():
    src = open(SRC_PATH).read()
    assert _failing_pins(_load(src, "oracle_copy")) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC_PATH).read()
    assert src.count(old) >= 1, f"mutation anchor for {name!r} not found"
    mutated = src.replace(old, new, 1)
    failed = _failing_pins(_load(mutated, "oracle_mutant"))
    assert failed, f"no pin caught mutant {name!r}"
