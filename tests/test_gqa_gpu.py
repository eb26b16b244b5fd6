"""Grouped key heads (GQA, and MQA with one key head): k1 [B, HK1, NK, d1],
k2 [B, HK2, NK, d2], query head h reading key head h // (H // HK) of its
side; forward, key-split forward and both gradient modes (fused: atomics
into the shared key heads' dK; deterministic: one launch per query head of
a group, bitwise repeatable) against the float64 oracle, which takes the
same grouping as its definition."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, generate_gqa, to_f64

from common import assert_fwd_close, grad_close, grad_floor, np_

pytestmark = pytest.mark.gpu

# (B, H, HK1, HK2, NQ, NK, d1, d2, causal)
CASES = [
    (1, 4, 4, 1, 300, 300, 128, 64, True),     # MQA student
    (2, 6, 2, 3, 257, 390, 64, 64, False),
    (1, 8, 1, 1, 130, 129, 64, 128, False),    # MQA on both sides
    (1, 4, 2, 4, 700, 200, 128, 32, False),    # grouped teacher, more queries than keys
    (1, 6, 3, 2, 1000, 1000, 48, 64, True),    # several tiles, ragged tail, padded head dim
]
IDS = ["x".join(map(str, c)) for c in CASES]


def make(c, seed):
    B, H, HK1, HK2, NQ, NK, d1, d2, causal = c
    w = Workload("gqa", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, seed)
    host = generate_gqa(w, HK1, HK2)
    return w, 1.0 / np.sqrt(d2), host, [x.cuda() for x in host]


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_forward_and_split(c):
    w, s2, host, dev = make(c, 121)
    f64 = [to_f64(x) for x in host]
    want = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    got = skl.streamkl_fwd_gqa(*dev, w.scale, s2, w.causal)
    assert_fwd_close(*(np_(x) for x in got), *want, "gqa fwd")
    got = skl.streamkl_fwd_splitk_gqa(*dev, w.scale, s2, w.causal, 3)
    assert_fwd_close(*(np_(x) for x in got), *want, "gqa split 3")
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)],
                         ids=["P2", "P1"])
@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_backward(c, mode, det):
    gmode, omode = mode
    w, s2, host, dev = make(c, 122)
    dkl = generate_dkl(w, "signed")
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, s2, w.causal)
    dq, dk = skl.streamkl_bwd_gqa(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), gmode, det)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(x) for x in host]
    rdq, rdk = oracle.backward(*f64, w.scale, w.causal, to_f64(dkl), omode, scale2=s2)
    gdq, gdk = np_(dq), np_(dk)
    assert gdq.shape == rdq.shape and gdk.shape == rdk.shape
    g, sg = (2, s2) if omode == oracle.MODE_P2 else (0, w.scale)
    hk = f64[g + 1].shape[1]
    grp = w.H // hk
    d64 = to_f64(dkl)
    for b in range(w.B):
        for h in range(w.H):
            fl = grad_floor(sg, d64[b, h], f64[g][b, h], f64[g + 1][b, h // grp])
            grad_close(gdq[b, h], rdq[b, h], fl)
        for j in range(hk):
            fl = sum(grad_floor(sg, d64[b, h], f64[g][b, h], f64[g + 1][b, j]) for h in range(j * grp, (j + 1) * grp))
            grad_close(gdk[b, j], rdk[b, j], fl)


def test_deterministic_is_bitwise_repeatable():
    w, s2, host, dev = make(CASES[1], 123)
    dkl = generate_dkl(w, "uniform").cuda()
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, s2, w.causal)
    for mode in (skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1):
        a = skl.streamkl_bwd_gqa(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl, mode, True)
        b = skl.streamkl_bwd_gqa(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl, mode, True)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_one_key_head_per_query_head_matches_the_plain_calls():
    c = (1, 4, 4, 4, 300, 300, 64, 64, True)
    w, s2, host, dev = make(c, 124)
    dkl = generate_dkl(w, "uniform").cuda()
    a = skl.streamkl_fwd_gqa(*dev, w.scale, s2, w.causal)
    b = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    ga = skl.streamkl_bwd_gqa(*dev, w.scale, s2, w.causal, *a, dkl, skl.STREAMKL_GRAD_P2, True)
    gb = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, *b, dkl, skl.STREAMKL_GRAD_P2, True)
    torch.cuda.synchronize()
    for x, y in zip(a + ga, b + gb):
        assert torch.equal(x, y)
