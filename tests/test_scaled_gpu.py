"""Per-side softmax scales (S1 = s1 Q1 K1^T, S2 = s2 Q2 K2^T) through the
*_scaled C entry points, against the float64 oracle's ``scale2``: forward,
key-split forward and the backward of both gradient modes, fused and
deterministic, with the same tolerances as the single-scale parity tests.
The natural case is a student with its own head dimension and 1/sqrt(d)."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, to_f64

from common import assert_fwd_close, grad_close, grad_floor, inputs, np_

pytestmark = pytest.mark.gpu

# (B, H, NQ, NK, d1, d2, causal, s1, s2)
CASES = [
    (1, 2, 300, 300, 128, 64, True, 1 / np.sqrt(128), 1 / np.sqrt(64)),
    (2, 1, 257, 390, 64, 128, False, 0.2, 0.05),
    (1, 2, 640, 640, 128, 128, True, 1 / np.sqrt(128), 0.25),
    (1, 1, 700, 200, 64, 64, False, 0.1, 0.3),
]
IDS = ["x".join(str(v) if not isinstance(v, float) else f"{v:.3g}" for v in c) for c in CASES]


def workload(c, seed):
    B, H, NQ, NK, d1, d2, causal, s1, _ = c
    return Workload("scaled", B, H, NQ, NK, d1, d2, causal, s1, "independent", 0.0, 1.2, seed)


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_forward_and_split(c):
    w, s2 = workload(c, 91), c[8]
    host, dev = inputs(w)
    f64 = [to_f64(t) for t in host]
    want = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    got = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    assert_fwd_close(*(np_(t) for t in got), *want, "scaled fwd")
    for splits in (1, 3):
        got = skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, splits)
        assert_fwd_close(*(np_(t) for t in got), *want, f"scaled split {splits}")
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)],
                         ids=["P2", "P1"])
@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_backward(c, mode, det):
    gmode, omode = mode
    w, s2 = workload(c, 92), c[8]
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform")
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    dq, dk = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), gmode, det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(t) for t in host]
    rdq, rdk = oracle.backward(*f64, w.scale, w.causal, to_f64(dkl), omode, scale2=s2)
    g = 2 if omode == oracle.MODE_P2 else 0
    sg = s2 if omode == oracle.MODE_P2 else w.scale
    gdq, gdk = np_(dq), np_(dk)
    for b in range(w.B):
        for h in range(w.H):
            fl = grad_floor(sg, to_f64(dkl)[b, h], f64[g][b, h], f64[g + 1][b, h])
            grad_close(gdq[b, h], rdq[b, h], fl)
            grad_close(gdk[b, h], rdk[b, h], fl)


def test_equal_scales_match_the_single_scale_calls():
    w = workload(CASES[2], 93)
    host, dev = inputs(w)
    a = skl.streamkl_fwd(*dev, w.scale, w.causal)
    b = skl.streamkl_fwd_scaled(*dev, w.scale, w.scale, w.causal)
    dkl = torch.ones(w.B, w.H, w.NQ, device="cuda")
    ga = skl.streamkl_bwd(*dev, w.scale, w.causal, *a, dkl, skl.STREAMKL_GRAD_P1, True)
    gb = skl.streamkl_bwd_scaled(*dev, w.scale, w.scale, w.causal, *b, dkl, skl.STREAMKL_GRAD_P1, True)
    torch.cuda.synchronize()
    for x, y in zip(a + ga, b + gb):
        assert torch.equal(x, y)
