"""Shared helpers for the GPU parity tests: inputs from the seeded generator,
the oracle on the same bf16 values, and the tolerances the tests enforce.

Tolerances (stated for the method's outputs and applied element by element):
  KL   |gpu - oracle| <= 2e-3 + 1e-2 |oracle|   per row
  LSE  |gpu - oracle| <= 1e-3                   per row
  dQ, dK  ||gpu - oracle||_F <= 1e-2 ||oracle||_F  per tensor (and per head),
          plus an absolute floor of 1e-6 s max|dKL| (||Q_g||_F + ||K_g||_F) for the
          degenerate cases whose exact gradient is zero (a single visible key)
"""

import numpy as np
import torch

from attention_distillation_kl_gb300.workloads import generate, to_f64

KL_ATOL, KL_RTOL, LSE_ATOL, GRAD_RTOL = 2e-3, 1e-2, 1e-3, 1e-2


def inputs(w, heads=None):
    host = generate(w, heads)
    dev = [t.cuda() for t in host]
    return host, dev


def head64(host, b, h):
    return [to_f64(t[b, h]) for t in host]


def np_(t):
    return t.detach().float().cpu().double().numpy()


def assert_finite(*ts):
    for t in ts:
        a = np_(t) if isinstance(t, torch.Tensor) else t
        assert np.all(np.isfinite(a)), "non-finite output"


def assert_fwd_close(gkl, gl1, gl2, rkl, rl1, rl2, what=""):
    gkl, gl1, gl2 = (np.asarray(x, dtype=np.float64) for x in (gkl, gl1, gl2))
    assert np.all(np.isfinite(gkl)) and np.all(np.isfinite(gl1)) and np.all(np.isfinite(gl2)), what
    err = np.abs(gkl - rkl)
    bound = KL_ATOL + KL_RTOL * np.abs(rkl)
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"{what} KL: row {worst} gpu {gkl.flat[worst]} oracle {rkl.flat[worst]}"
    e1, e2 = np.abs(gl1 - rl1).max(), np.abs(gl2 - rl2).max()
    assert e1 <= LSE_ATOL and e2 <= LSE_ATOL, f"{what} LSE err {e1} {e2}"


def frob_rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite gradient"
    den = np.linalg.norm(want)
    return np.linalg.norm(got - want) / max(den, 1e-300)


def grad_close(got, want, floor):
    """||got - want||_F <= 1e-2 ||want||_F + floor; returns the relative error."""
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite gradient"
    err = np.linalg.norm(got - want)
    den = np.linalg.norm(want)
    assert err <= GRAD_RTOL * den + floor, f"gradient error {err} vs norm {den} (floor {floor})"
    return err / max(den, 1e-300)


def grad_floor(scale, dkl, qg, kg):
    return 1e-6 * scale * float(np.abs(dkl).max()) * (np.linalg.norm(qg) + np.linalg.norm(kg))
