"""Both-sides backward (streamkl_bwd_both): dQ1, dK1, dQ2, dK2 against the
float64 oracle's two gradient modes on the same inputs.  d1 = d2 = 64 and
d1 = d2 = 32 run the one-recompute kernel (its deterministic mode too, with
both dQ sides on their rows' grids); other head dimensions run the
single-side backward twice; both must match the oracle with the single-side
tolerances, and the deterministic mode must repeat bit for bit."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, to_f64

from common import grad_close, grad_floor, inputs, np_

pytestmark = pytest.mark.gpu

# (B, H, NQ, NK, d1, d2, causal, s1, s2, deterministic)
CASES = [
    (1, 2, 256, 256, 64, 64, False, 0.125, 0.125, False),
    (2, 2, 300, 300, 64, 64, True, 0.125, 0.09, False),
    (1, 3, 130, 390, 64, 64, False, 0.2, 0.125, False),
    (1, 1, 1000, 1000, 64, 64, True, 0.125, 0.125, False),
    (1, 1, 700, 200, 64, 64, False, 0.125, 0.125, False),
    (1, 1, 5, 333, 64, 64, True, 0.125, 0.125, False),
    (1, 2, 257, 257, 64, 64, True, 0.125, 0.125, True),
    (2, 1, 130, 390, 64, 64, False, 0.2, 0.125, True),
    (1, 2, 300, 300, 32, 32, True, 1 / np.sqrt(32), 0.15, True),
    (1, 2, 300, 300, 128, 64, True, 1 / np.sqrt(128), 1 / np.sqrt(64), True),
    (1, 2, 300, 300, 32, 32, True, 1 / np.sqrt(32), 0.15, False),
    (2, 1, 130, 390, 32, 32, False, 0.2, 1 / np.sqrt(32), False),
    (1, 1, 1000, 1000, 32, 32, True, 1 / np.sqrt(32), 1 / np.sqrt(32), False),
    (1, 1, 700, 200, 32, 32, False, 0.15, 0.15, False),
    (1, 2, 300, 300, 128, 64, True, 1 / np.sqrt(128), 1 / np.sqrt(64), False),
    (1, 2, 300, 300, 64, 32, True, 1 / np.sqrt(64), 1 / np.sqrt(32), False),
    (1, 1, 384, 384, 128, 128, False, 1 / np.sqrt(128), 1 / np.sqrt(128), False),
]
IDS = ["x".join(f"{v:.3g}" if isinstance(v, float) else str(v) for v in c) for c in CASES]


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_both_sides_match_the_oracle(c):
    B, H, NQ, NK, d1, d2, causal, s1, s2, det = c
    w = Workload("both", B, H, NQ, NK, d1, d2, causal, s1, "independent", 0.0, 1.2, 95)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform")
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, s1, s2, causal)
    dq1, dk1, dq2, dk2 = skl.streamkl_bwd_both(*dev, s1, s2, causal, kl, l1, l2, dkl.cuda(), det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(t) for t in host]
    d64 = to_f64(dkl)
    r1 = oracle.backward(*f64, s1, causal, d64, oracle.MODE_P1, scale2=s2)
    r2 = oracle.backward(*f64, s1, causal, d64, oracle.MODE_P2, scale2=s2)
    for got, want, g, sg in (((dq1, dk1), r1, 0, s1), ((dq2, dk2), r2, 2, s2)):
        for b in range(B):
            for h in range(H):
                fl = grad_floor(sg, d64[b, h], f64[g][b, h], f64[g + 1][b, h])
                grad_close(np_(got[0])[b, h], want[0][b, h], fl)
                grad_close(np_(got[1])[b, h], want[1][b, h], fl)


@pytest.mark.parametrize("d", [64, 32])
def test_one_pass_agrees_with_the_two_single_side_calls(d):
    w = Workload("both", 1, 4, 1536, 1536, d, d, True, 1 / np.sqrt(d), "independent", 0.0, 1.2, 96)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform").cuda()
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    dq1, dk1, dq2, dk2 = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl)
    sq2, sk2 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2)
    sq1, sk1 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P1)
    torch.cuda.synchronize()
    for got, want in ((dq1, sq1), (dk1, sk1), (dq2, sq2), (dk2, sk2)):
        g, r = np_(got), np_(want)
        assert np.linalg.norm(g - r) <= 1e-5 * np.linalg.norm(r) + 1e-30


def test_both_sides_with_signed_upstream_gradient():
    w = Workload("both", 1, 2, 300, 300, 64, 64, True, 0.125, "independent", 0.0, 1.2, 97)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "signed")
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    got = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl.cuda())
    torch.cuda.synchronize()
    f64 = [to_f64(t) for t in host]
    d64 = to_f64(dkl)
    r1 = oracle.backward(*f64, w.scale, w.causal, d64, oracle.MODE_P1)
    r2 = oracle.backward(*f64, w.scale, w.causal, d64, oracle.MODE_P2)
    for out, want, g in ((got[:2], r1, 0), (got[2:], r2, 2)):
        for h in range(w.H):
            fl = grad_floor(w.scale, d64[0, h], f64[g][0, h], f64[g + 1][0, h])
            grad_close(np_(out[0])[0, h], want[0][0, h], fl)
            grad_close(np_(out[1])[0, h], want[1][0, h], fl)


@pytest.mark.parametrize("d", [64, 32])
def test_deterministic_one_pass_repeats_and_agrees(d):
    """The one-pass deterministic form: bitwise repeatable; each dQ row within
    its grid rounding of the atomic one-pass form (the same kernel, so the
    same per-tile contributions), over upstream gradients spanning the fp32
    range; dK equal bit for bit; and close to the two deterministic
    single-side calls (another kernel: bf16-level agreement)."""
    from test_det_fixed_gpu import compare_modes, row_bound
    w = Workload("both", 1, 4, 1536, 1536, d, d, True, 1 / np.sqrt(d), "independent", 0.0, 1.2, 98)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "wide").cuda()
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    a = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, True)
    b = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, True)
    f = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, False)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
    for x, y in zip(a, b):
        assert torch.equal(x, y), "not bitwise repeatable"
    assert torch.equal(a[1], f[1]) and torch.equal(a[3], f[3])  # dK1, dK2
    tiles = (w.NK + 127) // 128
    for side, mode, kg in ((0, skl.STREAMKL_GRAD_P1, host[1]), (2, skl.STREAMKL_GRAD_P2, host[3])):
        assert np.all(np.isfinite(np_(a[side])))
        bound = row_bound(mode, w.scale, np_(dkl), np_(kl), kg)
        compare_modes(np_(f[side]), np_(a[side]), bound, tiles)
    dklu = generate_dkl(w, "uniform").cuda()
    a = skl.streamkl_bwd_both(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dklu, True)
    s2 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dklu, skl.STREAMKL_GRAD_P2, True)
    s1 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dklu, skl.STREAMKL_GRAD_P1, True)
    torch.cuda.synchronize()
    for got, want in ((a[0], s1[0]), (a[1], s1[1]), (a[2], s2[0]), (a[3], s2[1])):
        g, r = np_(got), np_(want)
        assert np.linalg.norm(g - r) <= 1e-3 * np.linalg.norm(r) + 1e-30
