"""The pooled row-block evaluation of the oracle's dK (used by the parity
checks at the largest sizes) equals one direct oracle call, for causal
problems with NQ < NK and NQ = NK and for a non-causal one, in both modes
and with a second softmax scale."""

import numpy as np
import pytest

import oracle
from oracle_pool import dk_keys_pooled


@pytest.mark.parametrize("nq,nk,causal", [(70, 70, True), (53, 90, True), (40, 61, False)])
@pytest.mark.parametrize("mode", [oracle.MODE_P2, oracle.MODE_P1])
def test_pooled_dk_equals_direct(nq, nk, causal, mode):
    rng = np.random.default_rng(nq + nk)
    q1, k1 = rng.standard_normal((nq, 6)), rng.standard_normal((nk, 6))
    q2, k2 = rng.standard_normal((nq, 5)), rng.standard_normal((nk, 5))
    dkl = rng.uniform(-1.0, 1.5, nq)
    keys = np.array([0, 3, nk // 2, nk - 9, nk - 1])
    want = oracle.backward_dk_keys(q1, k1, q2, k2, 0.7, causal, dkl, mode, keys, scale2=0.55)
    got = dk_keys_pooled(q1, k1, q2, k2, 0.7, causal, dkl, mode, keys, scale2=0.55, rows_per_task=16,
                         workers=2)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
    # keys late in a causal problem: blocks that see none of them are skipped
    late = np.array([nk - 5, nk - 2])
    want = oracle.backward_dk_keys(q1, k1, q2, k2, 0.7, causal, dkl, mode, late)
    got = dk_keys_pooled(q1, k1, q2, k2, 0.7, causal, dkl, mode, late, rows_per_task=16, workers=2)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
