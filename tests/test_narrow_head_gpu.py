"""Head dimension 32 (operand tiles of one 32-element block with the 64-byte
swizzle) on either side or both, against the float64 oracle: forward,
key-split forward and the backward of both gradient modes, fused and
deterministic, with the tolerances of the other parity tests.  Each side
takes its own 1/sqrt(d) scale, as a narrow student distilled from a wider
teacher would."""

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
    (1, 1, 1, 1, 32, 32, False),
    (1, 2, 17, 17, 32, 32, True),
    (2, 3, 130, 129, 32, 32, False),
    (1, 2, 257, 300, 128, 32, False),
    (1, 2, 100, 333, 32, 128, True),       # causal with NQ < NK
    (1, 1, 1000, 1000, 32, 64, True),      # several tiles and a ragged tail
    (2, 2, 384, 384, 64, 32, False),       # exact multiples of the tile
    (1, 1, 700, 200, 128, 32, False),      # more queries than keys
]
IDS = ["x".join(map(str, c)) for c in CASES]


def workload(c, seed):
    B, H, NQ, NK, d1, d2, causal = c
    return Workload("narrow", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, seed)


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_forward_and_split(c):
    w, s2 = workload(c, 101), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    f64 = [to_f64(t) for t in host]
    want = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    got = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    assert_fwd_close(*(np_(t) for t in got), *want, "narrow fwd")
    for splits in (2, 5):
        got = skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, splits)
        assert_fwd_close(*(np_(t) for t in got), *want, f"narrow split {splits}")
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


def test_forward_single_scale():
    # the one-scale entry point on a 32/32 problem
    w = workload((1, 2, 300, 300, 32, 32, True), 102)
    host, dev = inputs(w)
    f64 = [to_f64(t) for t in host]
    want = oracle.forward(*f64, w.scale, w.causal)
    got = skl.streamkl_fwd(*dev, w.scale, w.causal)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    assert_fwd_close(*(np_(t) for t in got), *want, "narrow fwd, one scale")


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)],
                         ids=["P2", "P1"])
@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_backward(c, mode, det):
    gmode, omode = mode
    w, s2 = workload(c, 103), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    dkl = generate_dkl(w, "signed")
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    dq, dk = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), gmode, det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
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
