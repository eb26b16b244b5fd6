"""Head dims below the kernels' tile widths (any multiple of 16 up to 128:
16 and 32 compute in 32-wide tiles, 48 and 64 in 64-wide, 80 to 128 in
128-wide, the TMA zero-filling the columns past d): forward, key-split
forward, both gradient modes fused and deterministic, and the both-sides
backward, against the float64 oracle at the head dims as given, with the
tolerances of the other parity tests."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, to_f64

from common import assert_fwd_close, grad_close, grad_floor, inputs, np_

pytestmark = pytest.mark.gpu

# (B, H, NQ, NK, d1, d2, causal)
CASES = [
    (1, 2, 130, 129, 16, 16, False),
    (1, 2, 300, 300, 48, 48, True),
    (1, 1, 257, 390, 96, 80, False),
    (1, 2, 100, 333, 112, 48, True),      # causal with NQ < NK
    (2, 1, 384, 384, 16, 128, True),
    (1, 1, 700, 200, 128, 96, False),     # more queries than keys
    (1, 1, 1000, 1000, 80, 16, True),     # several tiles and a ragged tail
]
IDS = ["x".join(map(str, c)) for c in CASES]


def workload(c, seed):
    B, H, NQ, NK, d1, d2, causal = c
    return Workload("padded", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, seed)


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_forward_and_split(c):
    w, s2 = workload(c, 111), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    f64 = [to_f64(t) for t in host]
    want = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    got = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    assert_fwd_close(*(np_(t) for t in got), *want, "padded fwd")
    got = skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, 3)
    assert_fwd_close(*(np_(t) for t in got), *want, "padded split 3")
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


def check_grads(w, s2, host, dq, dk, dkl, omode):
    f64 = [to_f64(t) for t in host]
    rdq, rdk = oracle.backward(*f64, w.scale, w.causal, to_f64(dkl), omode, scale2=s2)
    gdq, gdk = np_(dq), np_(dk)
    assert gdq.shape == rdq.shape and gdk.shape == rdk.shape
    g, sg = (2, s2) if omode == oracle.MODE_P2 else (0, w.scale)
    for b in range(w.B):
        for h in range(w.H):
            fl = grad_floor(sg, to_f64(dkl)[b, h], f64[g][b, h], f64[g + 1][b, h])
            grad_close(gdq[b, h], rdq[b, h], fl)
            grad_close(gdk[b, h], rdk[b, h], fl)


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)],
                         ids=["P2", "P1"])
@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_backward(c, mode, det):
    gmode, omode = mode
    w, s2 = workload(c, 112), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    dkl = generate_dkl(w, "signed")
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    dq, dk = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), gmode, det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    check_grads(w, s2, host, dq, dk, dkl, omode)


@pytest.mark.parametrize("c", [(1, 2, 300, 300, 48, 48, True), (2, 1, 257, 390, 16, 16, False)],
                         ids=["48x48-causal", "16x16"])
def test_both_sides(c):
    w, s2 = workload(c, 113), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform")
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    dq1, dk1, dq2, dk2 = skl.streamkl_bwd_both(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), False)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    check_grads(w, s2, host, dq1, dk1, dkl, oracle.MODE_P1)
    check_grads(w, s2, host, dq2, dk2, dkl, oracle.MODE_P2)
