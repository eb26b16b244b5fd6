"""The bound the deterministic backward scales its fixed-point dQ by, pinned
on the oracle's dS (article section "Backward" for dS of both modes):
  mode P2: sum_k |dS2_ik| <= |dKL_i| * 2                  (two distributions)
  mode P1: sum_k |dS1_ik| <= |dKL_i| (2 H(P1_i) + 2 KL_i) <= |dKL_i| (2 ln NK + 2 KL_i)
so |dQ_id| = s |sum_k dS_ik K_kd| <= s |dKL_i| max|K| C_i for every partial
sum over keys.  Checked on random heads, on pairs whose distributions share
almost no mass (KL of tens of nats), and on causal rows with one key."""

import numpy as np
import pytest

from oracle import streamkl_oracle as O


def heads(seed, nq, nk, d, sd1, sd2, causal):
    g = np.random.default_rng(seed)
    q1, k1 = g.normal(0, sd1, (nq, d)), g.normal(0, sd1, (nk, d))
    q2, k2 = g.normal(0, sd2, (nq, d)), g.normal(0, sd2, (nk, d))
    return q1, k1, q2, k2


CASES = [
    (1, 64, 200, 32, 1.0, 1.0, False),
    (2, 100, 100, 16, 3.0, 0.3, True),   # peaked teacher, flat student
    (5, 100, 100, 16, 6.0, 6.0, True),   # both peaked on different keys: KL of hundreds of nats
    (3, 50, 300, 8, 0.2, 4.0, False),    # flat teacher, peaked student
    (4, 1, 1, 16, 1.0, 1.0, True),       # one visible key: dS = 0
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"seed{c[0]}")
def test_row_sums_of_ds_within_the_fixed_point_bound(c):
    seed, nq, nk, d, sd1, sd2, causal = c
    q1, k1, q2, k2 = heads(seed, nq, nk, d, sd1, sd2, causal)
    s = 1.0 / np.sqrt(d)
    g = np.random.default_rng(seed + 100)
    dkl = g.uniform(-2.0, 2.0, nq)
    rows = np.arange(nq)
    r = O._head_rows(q1, k1, q2, k2, s, s, causal, rows)
    n_vis = r["vis"].sum(axis=1)
    with np.errstate(invalid="ignore"):  # 0 * -inf on masked or underflowed pairs
        h1 = -np.sum(np.where(r["p1"] > 0, r["p1"] * r["logp1"], 0.0), axis=1)
    assert np.all(h1 <= np.log(n_vis) + 1e-12)
    ds2 = O._grad_scores(r, dkl, O.MODE_P2)
    ds1 = O._grad_scores(r, dkl, O.MODE_P1)
    assert np.all(np.abs(ds2).sum(axis=1) <= 2.0 * np.abs(dkl) * (1 + 1e-12))
    c1 = 2.0 * h1 + 2.0 * r["kl"]
    assert np.all(np.abs(ds1).sum(axis=1) <= np.abs(dkl) * c1 * (1 + 1e-12) + 1e-300)
    assert np.all(c1 <= 2.0 * np.log(nk) + 2.0 * r["kl"] + 1e-12)
    # the dQ bound holds for every prefix of the key sum (any partial sum the kernel forms)
    for ds, kg, c in ((ds2, k2, 2.0), (ds1, k1, 2.0 * np.log(nk) + 2.0 * r["kl"])):
        partial = np.cumsum(s * ds[:, :, None] * kg[None, :, :], axis=1)
        bound = s * np.abs(dkl) * np.abs(kg).max() * c
        assert np.all(np.abs(partial).max(axis=(1, 2)) <= bound * (1 + 1e-12) + 1e-300)


def test_large_kl_case_is_large():
    # the second case does exercise the KL term of the mode-P1 bound
    q1, k1, q2, k2 = heads(5, 100, 100, 16, 6.0, 6.0, True)
    r = O._head_rows(q1, k1, q2, k2, 0.25, 0.25, True, np.arange(100))
    assert r["kl"].max() > 50.0
