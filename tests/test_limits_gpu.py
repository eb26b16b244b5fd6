"""The size limits the library accepts, at their maximum: B*H = 65535 heads
(the largest grid the kernels launch over heads) with tiny rows, through the
forward, key-split forward and both backward modes, fused and
deterministic; and 1024 key splits (the maximum) on problems with far fewer
key tiles, where almost every split is empty and must merge with weight 0.
Checked against the float64 oracle on a sample of heads that includes the
first and the last."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate, generate_dkl, to_f64

from common import assert_fwd_close, grad_close, grad_floor, np_

pytestmark = pytest.mark.gpu


def test_largest_head_count():
    B, H = 3, 21845  # B * H = 65535
    w = Workload("many-heads", B, H, 3, 5, 16, 32, True, 0.25, "independent", 0.0, 1.2, 131)
    sample = [(0, 0), (0, 1), (1, 10922), (2, H - 2), (2, H - 1)]
    host = generate(w, heads=sample)
    dev = [t.cuda() for t in host]
    s2 = 0.17
    dkl = generate_dkl(w, "uniform")
    got = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    split = skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, 2)
    grads = {}
    for mode in (skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1):
        for det in (False, True):
            grads[mode, det] = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, *got, dkl.cuda(), mode, det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    for b, h in sample:
        f64 = [to_f64(t[b, h]) for t in host]
        want = oracle.forward_head(*f64, w.scale, w.causal, scale2=s2)
        for res in (got, split):
            assert_fwd_close(*(np_(t[b, h]) for t in res), *want, f"head ({b}, {h})")
        d64 = to_f64(dkl[b, h])
        for (mode, det), (dq, dk) in grads.items():
            omode = oracle.MODE_P2 if mode == skl.STREAMKL_GRAD_P2 else oracle.MODE_P1
            rdq, rdk = oracle.backward_head(*f64, w.scale, w.causal, d64, omode, scale2=s2)
            g, sg = (2, s2) if omode == oracle.MODE_P2 else (0, w.scale)
            fl = grad_floor(sg, d64, f64[g], f64[g + 1])
            grad_close(np_(dq[b, h]), rdq, fl)
            grad_close(np_(dk[b, h]), rdk, fl)


@pytest.mark.parametrize("shape", [(1, 2, 200, 300, 64, 64, False), (1, 2, 257, 257, 128, 32, True),
                                   (2, 1, 1, 1, 32, 32, False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_maximum_split_count(shape):
    B, H, NQ, NK, d1, d2, causal = shape
    w = Workload("splits", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, 132)
    host = generate(w)
    dev = [t.cuda() for t in host]
    got = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, 1024)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(t) for t in host]
    assert_fwd_close(*(np_(t) for t in got), *oracle.forward(*f64, w.scale, w.causal), "1024 splits")
