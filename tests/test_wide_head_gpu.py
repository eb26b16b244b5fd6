"""Head dimensions above 128 (tile widths 192 and 256, on either side or
both) against the float64 oracle: forward, key-split forward, and the
backward of both gradient modes, which above 128 always runs as the two
atomic-free passes (dK by key tiles, dQ by query tiles) whatever the
deterministic flag says.  Also head dims between tile widths (144, 208, 240)
that run zero-padded, causal NQ < NK, more queries than keys, ragged tails,
grouped key heads, per-side 1/sqrt(d) scales and a signed upstream gradient;
the tolerances are those of the other parity tests."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, generate_gqa, to_f64

from common import assert_fwd_close, grad_close, grad_floor, inputs, np_

pytestmark = pytest.mark.gpu

# (B, H, NQ, NK, d1, d2, causal)
CASES = [
    (1, 1, 1, 1, 256, 256, False),
    (1, 2, 17, 17, 192, 192, True),
    (2, 1, 130, 129, 256, 64, False),
    (1, 2, 257, 300, 128, 256, False),
    (1, 1, 100, 333, 256, 32, True),       # causal with NQ < NK
    (1, 1, 1000, 1000, 256, 256, True),    # several tiles and a ragged tail
    (1, 2, 384, 384, 192, 128, False),     # exact multiples of the tile
    (1, 1, 700, 200, 32, 192, False),      # more queries than keys
    (1, 1, 300, 300, 144, 240, True),      # padded to 192 and 256
    (1, 1, 200, 260, 208, 96, False),      # padded to 256 and 128
]
IDS = ["x".join(map(str, c)) for c in CASES]
MODES = [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)]


def workload(c, seed):
    B, H, NQ, NK, d1, d2, causal = c
    return Workload("wide", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, seed)


@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_forward_and_split(c):
    w, s2 = workload(c, 111), 1.0 / np.sqrt(c[5])
    host, dev = inputs(w)
    f64 = [to_f64(t) for t in host]
    want = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    got = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    assert_fwd_close(*(np_(t) for t in got), *want, "wide fwd")
    for splits in (2, 5):
        got = skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, splits)
        assert_fwd_close(*(np_(t) for t in got), *want, f"wide split {splits}")
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


@pytest.mark.parametrize("det", [False, True], ids=["flag0", "flag1"])
@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
@pytest.mark.parametrize("c", CASES, ids=IDS)
def test_backward(c, mode, det):
    gmode, omode = mode
    w, s2 = workload(c, 113), 1.0 / np.sqrt(c[5])
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


def test_backward_is_bitwise_reproducible():
    w, s2 = workload((1, 2, 500, 500, 256, 192, True), 114), 1.0 / np.sqrt(192)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform").cuda()
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)
    for mode in (skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1):
        a = [t.clone() for t in skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl, mode, False)]
        b = skl.streamkl_bwd_scaled(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl, mode, False)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
def test_grouped_key_heads(mode):
    """Four query heads on two (side 1) and one (side 2) key heads at d = 256 / 192:
    a shared head's dK is the ordered sum of its query heads' contributions."""
    gmode, omode = mode
    w = Workload("wide-gqa", 1, 4, 260, 300, 256, 192, True, 1.0 / 16.0, "independent", 0.0, 1.0, 115)
    host = generate_gqa(w, 2, 1)
    dev = [t.cuda() for t in host]
    s2 = 1.0 / np.sqrt(192)
    dkl = generate_dkl(w, "uniform")
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, s2, w.causal)
    dq, dk = skl.streamkl_bwd_gqa(*dev, w.scale, s2, w.causal, kl, l1, l2, dkl.cuda(), gmode, False)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(x) for x in host]
    rkl, rl1, rl2 = oracle.forward(*f64, w.scale, w.causal, scale2=s2)
    assert_fwd_close(np_(kl), np_(l1), np_(l2), rkl, rl1, rl2, "wide gqa fwd")
    rdq, rdk = oracle.backward(*f64, w.scale, w.causal, to_f64(dkl), omode, scale2=s2)
    g, sg = (2, s2) if omode == oracle.MODE_P2 else (0, w.scale)
    hk = f64[g + 1].shape[1]
    grp = w.H // hk
    d64 = to_f64(dkl)
    gdq, gdk = np_(dq), np_(dk)
    for h in range(w.H):
        grad_close(gdq[0, h], rdq[0, h], grad_floor(sg, d64[0, h], f64[g][0, h], f64[g + 1][0, h // grp]))
    for j in range(hk):
        fl = sum(grad_floor(sg, d64[0, h], f64[g][0, h], f64[g + 1][0, j]) for h in range(j * grp, (j + 1) * grp))
        grad_close(gdk[0, j], rdk[0, j], fl)
