"""The bound the deterministic backward takes its per-row dQ grid from,
pinned on the oracle's P1, P2 and dS (article section "Backward" for dS of
both modes).  With TV_i = sum_k max(P2_ik - P1_ik, 0), r = ln P1 - ln P2:
  Pinsker:  TV_i <= min(1, sqrt(KL_i / 2))
  mode P2:  sum_k |dS2_ik| = |dKL_i| 2 TV_i
  mode P1:  sum_k |dS1_ik| <= |dKL_i| (2 KL_i + 2 TV_i), because
            E_P1 |r - KL| <= E_P1 |r| + KL = 2 KL + 2 E_P1[max(-r, 0)] and
            E_P1[max(ln(P2 / P1), 0)] <= sum_k max(P2 - P1, 0) = TV
so every partial sum over keys of dQ_id = s sum_k dS_ik K_kd stays within
s |dKL_i| max|K| C_i.  Checked on random heads, on pairs that share almost
no mass (KL of hundreds of nats), near-identical pairs (KL ~ 1e-4) and
causal rows with one key."""

import numpy as np
import pytest

from oracle import streamkl_oracle as O


def heads(seed, nq, nk, d, sd1, sd2, causal, tie=0.0):
    g = np.random.default_rng(seed)
    q1, k1 = g.normal(0, sd1, (nq, d)), g.normal(0, sd1, (nk, d))
    q2, k2 = g.normal(0, sd2, (nq, d)), g.normal(0, sd2, (nk, d))
    if tie:  # student = teacher plus a little noise
        q2, k2 = q1 + tie * g.normal(0, 1, q1.shape), k1 + tie * g.normal(0, 1, k1.shape)
    return q1, k1, q2, k2


CASES = [
    (1, 64, 200, 32, 1.0, 1.0, False, 0.0),
    (2, 100, 100, 16, 3.0, 0.3, True, 0.0),    # peaked teacher, flat student
    (5, 100, 100, 16, 6.0, 6.0, True, 0.0),    # both peaked on different keys: KL of hundreds of nats
    (3, 50, 300, 8, 0.2, 4.0, False, 0.0),     # flat teacher, peaked student
    (6, 80, 160, 32, 1.0, 1.0, False, 0.01),   # near-identical pair
    (4, 1, 1, 16, 1.0, 1.0, True, 0.0),        # one visible key: dS = 0
]


def pieces(c):
    seed, nq, nk, d, sd1, sd2, causal, tie = c
    q1, k1, q2, k2 = heads(seed, nq, nk, d, sd1, sd2, causal, tie)
    s = 1.0 / np.sqrt(d)
    dkl = np.random.default_rng(seed + 100).uniform(-2.0, 2.0, nq)
    r = O._head_rows(q1, k1, q2, k2, s, s, causal, np.arange(nq))
    return s, dkl, r, k1, k2


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"seed{c[0]}")
def test_row_sums_of_ds_within_the_grid_bound(c):
    s, dkl, r, k1, k2 = pieces(c)
    p1, p2, kl = r["p1"], r["p2"], r["kl"]
    tv = np.maximum(p2 - p1, 0.0).sum(axis=1)
    pinsker = np.minimum(1.0, np.sqrt(np.maximum(kl, 0.0) / 2))
    assert np.all(tv <= pinsker * (1 + 1e-9) + 1e-12)
    ds2 = O._grad_scores(r, dkl, O.MODE_P2)
    ds1 = O._grad_scores(r, dkl, O.MODE_P1)
    assert np.allclose(np.abs(ds2).sum(axis=1), 2.0 * np.abs(dkl) * tv, rtol=1e-9, atol=1e-12)
    with np.errstate(invalid="ignore", divide="ignore"):
        rneg = np.where(r["vis"] & (p1 > 0), np.maximum(r["logp2"] - r["logp1"], 0.0), 0.0)
    assert np.all((p1 * rneg).sum(axis=1) <= tv * (1 + 1e-9) + 1e-12)
    c1 = 2.0 * kl + 2.0 * tv
    assert np.all(np.abs(ds1).sum(axis=1) <= np.abs(dkl) * c1 * (1 + 1e-9) + 1e-12)
    # the dQ bound, with Pinsker in place of TV, holds for every prefix of the key sum
    for ds, kg, c in ((ds2, k2, 2.0 * pinsker), (ds1, k1, 2.0 * kl + 2.0 * pinsker)):
        partial = np.cumsum(s * ds[:, :, None] * kg[None, :, :], axis=1)
        bound = s * np.abs(dkl) * np.abs(kg).max() * c
        assert np.all(np.abs(partial).max(axis=(1, 2)) <= bound * (1 + 1e-9) + 1e-12)


def test_cases_span_the_kl_range():
    kls = [pieces(c)[2]["kl"] for c in CASES[2:5:2]]
    assert kls[0].max() > 50.0 and kls[1].max() < 1e-2
