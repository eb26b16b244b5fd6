"""Pins for the float64 oracle, against things other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError on
a mismatch, so ``test_oracle_mutants.py`` can run the same pins against
copies of the oracle with planted mistakes.  What each pin rests on:

* closed forms: one key (KL = 0, LSE = S), zero student logits (uniform P2,
  KL = log|A| - H(P1) with H from scipy.stats.entropy), two keys (the
  Bernoulli KL), all-zero logits (LSE = log|A|);
* invariants: KL = 0 for identical inputs, Gibbs' inequality KL >= 0, key
  shift (KL unchanged, LSE shifted by s q.v), rows of dS summing to zero;
* brute force with pure-Python loops and ``math`` on tiny causal inputs;
* independent library routines: torch.nn.functional.kl_div / log_softmax,
  scipy.special.logsumexp, CPU float64 torch autograd;
* central finite differences of sum(dKL * KL) for both gradient modes;
* the online recurrence and the two-pass form agreeing with the direct one;
* a second softmax scale for the S2 side: s2 = 0 gives the uniform-student
  closed form, a power-of-two rescale of Q2 against s2 changes nothing, and
  per-side results equal single-scale results with Q2 pre-multiplied by
  s2/s1 (gradients by the chain rule), plus finite differences;
* grouped key heads: equal to every key head repeated over its group and run
  as independent heads (dK summed over the copies), plus finite differences
  w.r.t. a shared key head.
"""

import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle as O


def _rand(rng, *shape, sd=1.0):
    return rng.standard_normal(shape) * sd


def _head(rng, nq, nk, d1, d2, sd=1.0):
    return (_rand(rng, nq, d1, sd=sd), _rand(rng, nk, d1, sd=sd),
            _rand(rng, nq, d2, sd=sd), _rand(rng, nk, d2, sd=sd))


def _fwd_head(o, q1, k1, q2, k2, s, causal):
    kl, a, b = o.forward(q1[None, None], k1[None, None], q2[None, None], k2[None, None], s, causal)
    return kl[0, 0], a[0, 0], b[0, 0]


# ----------------------------------------------------------------------------- pins


def pin_identical_inputs_give_zero(o):
    rng = np.random.default_rng(1)
    for causal in (False, True):
        q, k, _, _ = _head(rng, 19, 23, 8, 8)
        kl, a, b = _fwd_head(o, q, k, q, k, 0.7, causal)
        assert np.all(kl == 0.0), kl
        assert np.array_equal(a, b)


def pin_gibbs(o):
    rng = np.random.default_rng(2)
    for causal in (False, True):
        q1, k1, q2, k2 = _head(rng, 31, 40, 8, 5, sd=1.5)
        kl, _, _ = _fwd_head(o, q1, k1, q2, k2, 0.9, causal)
        assert np.all(kl >= -1e-12), kl.min()
        assert np.all(kl > 0.0)


def pin_single_key(o):
    rng = np.random.default_rng(3)
    q1, k1, q2, k2 = _head(rng, 6, 1, 4, 4)
    kl, a, b = _fwd_head(o, q1, k1, q2, k2, 0.5, False)
    assert np.allclose(kl, 0.0, atol=1e-15)
    np.testing.assert_allclose(a, 0.5 * (q1 @ k1[0]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(b, 0.5 * (q2 @ k2[0]), rtol=0, atol=1e-14)
    # causal row 0 of a square problem sees exactly key 0
    q1, k1, q2, k2 = _head(rng, 9, 9, 4, 4)
    kl, a, b = _fwd_head(o, q1, k1, q2, k2, 0.5, True)
    assert abs(kl[0]) < 1e-15
    assert abs(a[0] - 0.5 * q1[0] @ k1[0]) < 1e-14
    assert abs(b[0] - 0.5 * q2[0] @ k2[0]) < 1e-14


def pin_uniform_student(o):
    """Q2 = 0 makes P2 uniform over the visible keys, so KL_i = log|A_i| - H(P1_i)."""
    rng = np.random.default_rng(4)
    nq, nk = 12, 17
    for causal in (False, True):
        q1, k1, _, k2 = _head(rng, nq, nk, 6, 3)
        q2 = np.zeros((nq, 3))
        kl, _, lse2 = _fwd_head(o, q1, k1, q2, k2, 0.8, causal)
        for i in range(nq):
            n_vis = nk if not causal else i + (nk - nq) + 1
            p1 = scipy.special.softmax(0.8 * (q1[i] @ k1[:n_vis].T))
            want = math.log(n_vis) - scipy.stats.entropy(p1)
            assert abs(kl[i] - want) < 1e-12, (i, kl[i], want)
            assert abs(lse2[i] - math.log(n_vis)) < 1e-12


def pin_zero_logits(o):
    rng = np.random.default_rng(5)
    nq, nk = 7, 11
    z1, z2 = np.zeros((nq, 4)), np.zeros((nq, 2))
    _, k1, _, k2 = _head(rng, nq, nk, 4, 2)
    kl, a, b = _fwd_head(o, z1, k1, z2, k2, 1.3, True)
    n_vis = np.arange(nq) + (nk - nq) + 1
    np.testing.assert_allclose(kl, 0.0, atol=1e-15)
    np.testing.assert_allclose(a, np.log(n_vis), rtol=0, atol=1e-14)
    np.testing.assert_allclose(b, np.log(n_vis), rtol=0, atol=1e-14)


def pin_two_keys_bernoulli(o):
    rng = np.random.default_rng(6)
    q1, k1, q2, k2 = _head(rng, 10, 2, 5, 5)
    s = 0.6
    kl, _, _ = _fwd_head(o, q1, k1, q2, k2, s, False)
    for i in range(10):
        p = 1.0 / (1.0 + math.exp(-s * (q1[i] @ (k1[0] - k1[1]))))
        q = 1.0 / (1.0 + math.exp(-s * (q2[i] @ (k2[0] - k2[1]))))
        want = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert abs(kl[i] - want) < 1e-13, (i, kl[i], want)


def pin_key_shift(o):
    rng = np.random.default_rng(7)
    q1, k1, q2, k2 = _head(rng, 14, 14, 6, 6)
    v1, v2 = rng.standard_normal(6), rng.standard_normal(6)
    s = 0.45
    for causal in (False, True):
        kl, a, b = _fwd_head(o, q1, k1, q2, k2, s, causal)
        kl2, a2, b2 = _fwd_head(o, q1, k1 + v1, q2, k2 + v2, s, causal)
        np.testing.assert_allclose(kl2, kl, rtol=0, atol=1e-12)
        np.testing.assert_allclose(a2, a + s * (q1 @ v1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(b2, b + s * (q2 @ v2), rtol=0, atol=1e-12)


def pin_brute_force_loops(o):
    """Pure-Python double loops with math.exp/math.log on a tiny causal case
    with NQ < NK, which fixes the bottom-right alignment of the mask."""
    rng = np.random.default_rng(8)
    nq, nk, s = 4, 7, 0.9
    q1, k1, q2, k2 = _head(rng, nq, nk, 3, 2)
    for causal in (False, True):
        kl, a, b = _fwd_head(o, q1, k1, q2, k2, s, causal)
        for i in range(nq):
            keys = [j for j in range(nk) if (not causal) or j <= i + (nk - nq)]
            z1 = [s * sum(q1[i, t] * k1[j, t] for t in range(3)) for j in keys]
            z2 = [s * sum(q2[i, t] * k2[j, t] for t in range(2)) for j in keys]
            l1 = math.log(sum(math.exp(x) for x in z1))
            l2 = math.log(sum(math.exp(x) for x in z2))
            want = sum(math.exp(x - l1) * ((x - l1) - (y - l2)) for x, y in zip(z1, z2))
            assert abs(kl[i] - want) < 1e-13, (causal, i)
            assert abs(a[i] - l1) < 1e-13 and abs(b[i] - l2) < 1e-13


def pin_causal_row_is_truncated_problem(o):
    rng = np.random.default_rng(9)
    nq, nk = 9, 13
    q1, k1, q2, k2 = _head(rng, nq, nk, 4, 4)
    kl, a, b = _fwd_head(o, q1, k1, q2, k2, 0.7, True)
    for i in range(nq):
        n_vis = i + (nk - nq) + 1
        kk, aa, bb = _fwd_head(o, q1[i:i + 1], k1[:n_vis], q2[i:i + 1], k2[:n_vis], 0.7, False)
        assert abs(kk[0] - kl[i]) < 1e-13 and abs(aa[0] - a[i]) < 1e-13 and abs(bb[0] - b[i]) < 1e-13


def pin_library_crosscheck(o):
    """torch log_softmax + kl_div(log_target=True) and scipy logsumexp, float64."""
    rng = np.random.default_rng(10)
    q1, k1, q2, k2 = _head(rng, 20, 33, 8, 4, sd=1.3)
    s = 0.55
    kl, a, b = _fwd_head(o, q1, k1, q2, k2, s, False)
    s1 = torch.from_numpy(s * (q1 @ k1.T))
    s2 = torch.from_numpy(s * (q2 @ k2.T))
    ref = torch.nn.functional.kl_div(torch.log_softmax(s2, -1), torch.log_softmax(s1, -1),
                                     reduction="none", log_target=True).sum(-1).numpy()
    np.testing.assert_allclose(kl, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a, scipy.special.logsumexp(s1.numpy(), axis=1), rtol=1e-14, atol=1e-13)
    np.testing.assert_allclose(b, scipy.special.logsumexp(s2.numpy(), axis=1), rtol=1e-14, atol=1e-13)


def pin_online_and_two_pass(o):
    rng = np.random.default_rng(11)
    for causal, nq, nk in ((False, 37, 53), (True, 37, 53), (True, 40, 40)):
        q1, k1, q2, k2 = _head(rng, nq, nk, 8, 6, sd=1.4)
        kl, a, b = o.forward_head(q1, k1, q2, k2, 0.8, causal)
        for tile in (1, 5, 16, 64):
            for fn in (o.forward_online, o.forward_two_pass):
                kl2, a2, b2 = fn(q1, k1, q2, k2, 0.8, causal, key_tile=tile, row_block=7)
                np.testing.assert_allclose(kl2, kl, rtol=1e-12, atol=1e-13)
                np.testing.assert_allclose(a2, a, rtol=1e-13, atol=1e-13)
                np.testing.assert_allclose(b2, b, rtol=1e-13, atol=1e-13)


def _fd_grad(o, q1, k1, q2, k2, s, causal, dkl, mode, h=1e-6, s2=None):
    """Central differences of L = sum(dkl * KL) w.r.t. the gradient side."""
    args = [q1.copy(), k1.copy(), q2.copy(), k2.copy()]
    iq, ik = (2, 3) if mode == O.MODE_P2 else (0, 1)

    def L():
        return o.loss(*(x[None, None] for x in args), s, causal, dkl[None, None], scale2=s2)

    out = []
    for idx in (iq, ik):
        g = np.zeros_like(args[idx])
        for e in np.ndindex(*g.shape):
            old = args[idx][e]
            args[idx][e] = old + h
            lp = L()
            args[idx][e] = old - h
            lm = L()
            args[idx][e] = old
            g[e] = (lp - lm) / (2 * h)
        out.append(g)
    return out


def pin_backward_finite_differences(o):
    rng = np.random.default_rng(12)
    for causal, nq, nk, d1, d2 in ((False, 5, 7, 4, 3), (True, 6, 6, 3, 3), (True, 4, 7, 2, 4)):
        q1, k1, q2, k2 = _head(rng, nq, nk, d1, d2, sd=1.2)
        dkl = rng.uniform(0.5, 1.5, nq)
        for mode in (O.MODE_P2, O.MODE_P1):
            dq, dk = o.backward(q1[None, None], k1[None, None], q2[None, None], k2[None, None],
                                0.9, causal, dkl[None, None], mode)
            gq, gk = _fd_grad(o, q1, k1, q2, k2, 0.9, causal, dkl, mode)
            for got, want in ((dq[0, 0], gq), (dk[0, 0], gk)):
                err = np.abs(got - want).max() / max(1e-12, np.abs(want).max())
                assert err < 1e-7, (causal, mode, err)


def pin_backward_autograd(o):
    """CPU float64 torch autograd of the direct formula (log_softmax, kl_div)."""
    rng = np.random.default_rng(13)
    nq, nk, s = 9, 12, 0.75
    q1, k1, q2, k2 = _head(rng, nq, nk, 5, 4, sd=1.3)
    dkl = rng.uniform(0.5, 1.5, nq)
    for causal in (False, True):
        mask = torch.from_numpy(np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)) \
            if causal else torch.ones(nq, nk, dtype=torch.bool)
        for mode in (O.MODE_P2, O.MODE_P1):
            t = [torch.from_numpy(x).requires_grad_(True) for x in (q1, k1, q2, k2)]
            ls1 = torch.log_softmax((s * t[0] @ t[1].T).masked_fill(~mask, -math.inf), -1)
            ls2 = torch.log_softmax((s * t[2] @ t[3].T).masked_fill(~mask, -math.inf), -1)
            zero = torch.zeros((), dtype=torch.float64)
            l1m, l2m = torch.where(mask, ls1, zero), torch.where(mask, ls2, zero)
            terms = torch.where(mask, l1m.exp() * (l1m - l2m), zero)
            (terms.sum(-1) * torch.from_numpy(dkl)).sum().backward()
            dq, dk = o.backward(q1[None, None], k1[None, None], q2[None, None], k2[None, None],
                                s, causal, dkl[None, None], mode)
            gq, gk = (t[2].grad, t[3].grad) if mode == O.MODE_P2 else (t[0].grad, t[1].grad)
            np.testing.assert_allclose(dq[0, 0], gq.numpy(), rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(dk[0, 0], gk.numpy(), rtol=1e-11, atol=1e-13)


def pin_gradient_invariants(o):
    """Rows of dS sum to zero, so sum_j dK_j = 0; both modes vanish at P1 = P2."""
    rng = np.random.default_rng(14)
    q1, k1, q2, k2 = _head(rng, 16, 20, 6, 6)
    dkl = rng.uniform(0.5, 1.5, 16)
    for causal in (False, True):
        for mode in (O.MODE_P2, O.MODE_P1):
            _, dk = o.backward(q1[None, None], k1[None, None], q2[None, None], k2[None, None],
                               0.8, causal, dkl[None, None], mode)
            assert np.abs(dk[0, 0].sum(axis=0)).max() < 1e-12
            dq0, dk0 = o.backward(q1[None, None], k1[None, None], q1[None, None], k1[None, None],
                                  0.8, causal, dkl[None, None], mode)
            assert np.abs(dq0).max() < 1e-14 and np.abs(dk0).max() < 1e-14


def pin_sampled_backward(o):
    rng = np.random.default_rng(15)
    q1, k1, q2, k2 = _head(rng, 21, 26, 4, 3)
    dkl = rng.uniform(0.5, 1.5, 21)
    for causal in (False, True):
        for mode in (O.MODE_P2, O.MODE_P1):
            dq, dk = o.backward_head(q1, k1, q2, k2, 0.8, causal, dkl, mode, row_block=5)
            rows, keys = [0, 7, 20], [1, 13, 25]
            np.testing.assert_allclose(o.backward_dq_rows(q1, k1, q2, k2, 0.8, causal, dkl, mode, rows),
                                       dq[rows], rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(o.backward_dk_keys(q1, k1, q2, k2, 0.8, causal, dkl, mode, keys,
                                                          row_block=4), dk[keys], rtol=1e-12, atol=1e-15)
            if causal:  # rows before key 13 - (26 - 21) = 8 see none of keys 13, 25
                np.testing.assert_allclose(o.backward_dk_keys(q1, k1, q2, k2, 0.8, causal, dkl, mode,
                                                              [13, 25], row_block=4, first_row=8),
                                           dk[[13, 25]], rtol=1e-12, atol=1e-15)


def pin_sampled_forward(o):
    """forward_rows on scattered, unsorted rows equals those rows of the
    full forward (which the closed forms, brute force and library pins fix),
    for causal NQ < NK (bottom-right mask), non-causal and per-side scales."""
    rng = np.random.default_rng(17)
    q1, k1, q2, k2 = _head(rng, 23, 37, 5, 3)
    rows = [22, 0, 9, 3, 17, 9]  # unsorted, one repeated, first and last row
    for causal in (False, True):
        for s2 in (None, 0.45):
            kl, a, b = o.forward_head(q1, k1, q2, k2, 0.8, causal, row_block=4, scale2=s2)
            skl, sa, sb = o.forward_rows(q1, k1, q2, k2, 0.8, causal, rows, scale2=s2)
            for got, want in ((skl, kl), (sa, a), (sb, b)):
                np.testing.assert_allclose(got, want[rows], rtol=1e-13, atol=1e-15)


def pin_underflow_is_finite(o):
    """Unit scale and peaky teacher rows: many probabilities fall below the
    fp32 normal range, yet every oracle output stays finite."""
    rng = np.random.default_rng(16)
    nq, nk, d = 48, 64, 128
    q1, k1 = _rand(rng, nq, d, sd=1.5), _rand(rng, nk, d, sd=1.5)
    q2, k2 = _rand(rng, nq, d), _rand(rng, nk, d)
    kl, a, _ = _fwd_head(o, q1, k1, q2, k2, 1.0, False)
    logp1 = (q1 @ k1.T) - a[:, None]
    assert np.sum(logp1 < -126 * math.log(2)) > 100  # underflow really happens
    assert np.all(np.isfinite(kl)) and np.all(kl > 0)
    for mode in (O.MODE_P2, O.MODE_P1):
        dq, dk = o.backward(q1[None, None], k1[None, None], q2[None, None], k2[None, None],
                            1.0, False, np.ones((1, 1, nq)), mode)
        assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk))


def pin_per_side_scale_uniform_student(o):
    """s2 = 0 makes P2 uniform whatever Q2 is: KL_i = log|A_i| - H(P1_i)."""
    rng = np.random.default_rng(17)
    nq, nk = 10, 14
    for causal in (False, True):
        q1, k1, q2, k2 = _head(rng, nq, nk, 5, 4)
        kl, _, lse2 = o.forward_head(q1, k1, q2, k2, 0.7, causal, scale2=0.0)
        for i in range(nq):
            n_vis = nk if not causal else i + (nk - nq) + 1
            p1 = scipy.special.softmax(0.7 * (q1[i] @ k1[:n_vis].T))
            assert abs(kl[i] - (math.log(n_vis) - scipy.stats.entropy(p1))) < 1e-12
            assert abs(lse2[i] - math.log(n_vis)) < 1e-12


def pin_per_side_scale_matches_prescaled_student(o):
    """(s1, s2) on (Q1, Q2) is s1 on (Q1, (s2/s1) Q2): forward equal; the
    gradient w.r.t. Q2 picks up the factor s2/s1 by the chain rule, w.r.t.
    K2 (and on the P1 side) it is unchanged.  A power-of-two rescale of Q2
    against s2 is exact."""
    rng = np.random.default_rng(18)
    s1, s2 = 0.8, 0.45
    for causal in (False, True):
        q1, k1, q2, k2 = _head(rng, 13, 17, 6, 4, sd=1.2)
        dkl = rng.uniform(0.5, 1.5, 13)
        b = lambda x: x[None, None]
        got = o.forward(b(q1), b(k1), b(q2), b(k2), s1, causal, scale2=s2)
        want = o.forward(b(q1), b(k1), b(q2 * (s2 / s1)), b(k2), s1, causal)
        for g, w in zip(got, want):
            np.testing.assert_allclose(g, w, rtol=1e-12, atol=1e-13)
        exact = o.forward(b(q1), b(k1), b(q2 * 4.0), b(k2), s1, causal, scale2=s2 / 4.0)
        for g, w in zip(got, exact):
            assert np.array_equal(g, w)
        for mode in (O.MODE_P2, O.MODE_P1):
            dq, dk = o.backward(b(q1), b(k1), b(q2), b(k2), s1, causal, b(dkl), mode, scale2=s2)
            dq0, dk0 = o.backward(b(q1), b(k1), b(q2 * (s2 / s1)), b(k2), s1, causal, b(dkl), mode)
            fq = s2 / s1 if mode == O.MODE_P2 else 1.0
            np.testing.assert_allclose(dq, fq * dq0, rtol=1e-11, atol=1e-14)
            np.testing.assert_allclose(dk, dk0, rtol=1e-11, atol=1e-14)


def pin_per_side_scale_finite_differences(o):
    rng = np.random.default_rng(19)
    for causal, nq, nk, d1, d2 in ((False, 5, 6, 3, 4), (True, 5, 7, 4, 2)):
        q1, k1, q2, k2 = _head(rng, nq, nk, d1, d2, sd=1.2)
        dkl = rng.uniform(0.5, 1.5, nq)
        for mode in (O.MODE_P2, O.MODE_P1):
            dq, dk = o.backward(q1[None, None], k1[None, None], q2[None, None], k2[None, None],
                                0.9, causal, dkl[None, None], mode, scale2=0.55)
            gq, gk = _fd_grad(o, q1, k1, q2, k2, 0.9, causal, dkl, mode, s2=0.55)
            for got, want in ((dq[0, 0], gq), (dk[0, 0], gk)):
                err = np.abs(got - want).max() / max(1e-12, np.abs(want).max())
                assert err < 1e-7, (causal, mode, err)


def pin_per_side_scale_online(o):
    rng = np.random.default_rng(20)
    q1, k1, q2, k2 = _head(rng, 29, 41, 6, 4, sd=1.3)
    for causal in (False, True):
        kl, a, b = o.forward_head(q1, k1, q2, k2, 0.9, causal, scale2=0.4)
        for fn in (o.forward_online, o.forward_two_pass):
            kl2, a2, b2 = fn(q1, k1, q2, k2, 0.9, causal, key_tile=8, row_block=6, scale2=0.4)
            np.testing.assert_allclose(kl2, kl, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(a2, a, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(b2, b, rtol=1e-13, atol=1e-13)


def _gqa_inputs(rng, b_, h_, hk1, hk2, nq, nk, d1, d2, sd=1.2):
    return (_rand(rng, b_, h_, nq, d1, sd=sd), _rand(rng, b_, hk1, nk, d1, sd=sd),
            _rand(rng, b_, h_, nq, d2, sd=sd), _rand(rng, b_, hk2, nk, d2, sd=sd))


def pin_grouped_key_heads_are_repeated_heads(o):
    # grouped key heads = every key head repeated over its consecutive group
    # of query heads (np.repeat), run as independent heads; dK of a shared
    # head = the sum of the repeated copies' dK (chain rule of the repeat)
    rng = np.random.default_rng(21)
    for hk1, hk2, causal in ((3, 2, True), (1, 6, False), (2, 1, True)):
        q1, k1, q2, k2 = _gqa_inputs(rng, 2, 6, hk1, hk2, 9, 11, 4, 3)
        r1, r2 = np.repeat(k1, 6 // hk1, axis=1), np.repeat(k2, 6 // hk2, axis=1)
        dkl = rng.uniform(0.5, 1.5, (2, 6, 9))
        got = o.forward(q1, k1, q2, k2, 0.8, causal, scale2=0.6)
        for b in range(2):
            for h in range(6):
                want = o.forward_head(q1[b, h], r1[b, h], q2[b, h], r2[b, h], 0.8, causal, scale2=0.6)
                for g, w in zip(got, want):
                    np.testing.assert_allclose(g[b, h], w, rtol=1e-14, atol=1e-14)
        for mode, hk, rep in ((O.MODE_P2, hk2, r2), (O.MODE_P1, hk1, r1)):
            dq, dk = o.backward(q1, k1, q2, k2, 0.8, causal, dkl, mode, scale2=0.6)
            assert dk.shape == (2, hk) + rep.shape[2:]
            for b in range(2):
                dks = [o.backward_head(q1[b, h], r1[b, h], q2[b, h], r2[b, h], 0.8, causal, dkl[b, h], mode,
                                       scale2=0.6) for h in range(6)]
                for h in range(6):
                    np.testing.assert_allclose(dq[b, h], dks[h][0], rtol=1e-13, atol=1e-14)
                want_dk = np.stack([x[1] for x in dks]).reshape(hk, 6 // hk, *rep.shape[2:]).sum(axis=1)
                np.testing.assert_allclose(dk[b], want_dk, rtol=1e-12, atol=1e-13)


def pin_grouped_key_heads_finite_differences(o):
    # central differences of sum(dKL * KL) w.r.t. a key head shared by three
    # query heads (MQA on the gradient side) and w.r.t. each query head
    rng = np.random.default_rng(22)
    for mode, causal in ((O.MODE_P2, False), (O.MODE_P1, True)):
        hk1, hk2 = (3, 1) if mode == O.MODE_P2 else (1, 3)
        args = list(_gqa_inputs(rng, 1, 3, hk1, hk2, 4, 5, 3, 2))
        dkl = rng.uniform(0.5, 1.5, (1, 3, 4))
        dq, dk = o.backward(*args, 0.9, causal, dkl, mode, scale2=0.7)
        iq, ik = (2, 3) if mode == O.MODE_P2 else (0, 1)
        for idx, got in ((iq, dq), (ik, dk)):
            fd = np.zeros_like(args[idx])
            for e in np.ndindex(*fd.shape):
                old = args[idx][e]
                args[idx][e] = old + 1e-6
                lp = o.loss(*args, 0.9, causal, dkl, scale2=0.7)
                args[idx][e] = old - 1e-6
                lm = o.loss(*args, 0.9, causal, dkl, scale2=0.7)
                args[idx][e] = old
                fd[e] = (lp - lm) / 2e-6
            err = np.abs(got - fd).max() / max(1e-12, np.abs(fd).max())
            assert err < 1e-7, (mode, idx, err)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O)
