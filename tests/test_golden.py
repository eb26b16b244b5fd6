"""Stored fixtures under tests/golden/ (written by make_golden.py there): the
float64 oracle must reproduce them to rounding, and the CUDA path must match
them within the parity tolerances.  The GPU runs the fixtures with their head
dims zero-padded to 16 (padding changes no dot product; the padded gradient
columns must be zero)."""

import json
import os

import numpy as np
import pytest
import torch

import oracle

from common import assert_fwd_close, grad_close

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = json.load(open(os.path.join(HERE, "golden", "streamkl_small.json")))


def arrays(c):
    return [np.array(c[k], dtype=np.float64) for k in ("q1", "k1", "q2", "k2")]


@pytest.mark.parametrize("name", sorted(CASES))
def test_oracle_reproduces_the_fixture(name):
    c = CASES[name]
    q1, k1, q2, k2 = arrays(c)
    kl, l1, l2 = oracle.forward(q1, k1, q2, k2, c["scale1"], c["causal"], scale2=c["scale2"])
    for got, key in ((kl, "kl"), (l1, "lse1"), (l2, "lse2")):
        np.testing.assert_allclose(got, np.array(c[key]), rtol=1e-13, atol=1e-14)
    if "dq2_p2" in c:
        dkl = np.ones(kl.shape)
        for mode, keys in ((oracle.MODE_P2, ("dq2_p2", "dk2_p2")), (oracle.MODE_P1, ("dq1_p1", "dk1_p1"))):
            dq, dk = oracle.backward(q1, k1, q2, k2, c["scale1"], c["causal"], dkl, mode, scale2=c["scale2"])
            np.testing.assert_allclose(dq, np.array(c[keys[0]]), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(dk, np.array(c[keys[1]]), rtol=1e-12, atol=1e-14)


def pad16(a):
    out = np.zeros(a.shape[:-1] + (16,))
    out[..., :a.shape[-1]] = a
    return torch.from_numpy(out).to(torch.bfloat16).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_cuda_path_matches_the_fixture(name):
    import attention_distillation_kl_gb300 as skl
    c = CASES[name]
    host = arrays(c)
    dev = [pad16(a) for a in host]
    for a, t in zip(host, dev):  # the fixture's values are exact in bf16
        assert np.array_equal(t.float().cpu().numpy()[..., :a.shape[-1]], a)
    kl, l1, l2 = skl.streamkl_fwd_scaled(*dev, c["scale1"], c["scale2"], c["causal"])
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    assert_fwd_close(kl.double().cpu().numpy(), l1.double().cpu().numpy(), l2.double().cpu().numpy(),
                     np.array(c["kl"]), np.array(c["lse1"]), np.array(c["lse2"]), name)
    if "dq2_p2" not in c:
        return
    dkl = torch.ones_like(kl)
    for mode, keys, d in ((skl.STREAMKL_GRAD_P2, ("dq2_p2", "dk2_p2"), host[2].shape[-1]),
                          (skl.STREAMKL_GRAD_P1, ("dq1_p1", "dk1_p1"), host[0].shape[-1])):
        for det in (False, True):
            dq, dk = skl.streamkl_bwd_scaled(*dev, c["scale1"], c["scale2"], c["causal"], kl, l1, l2, dkl, mode, det)
            torch.cuda.synchronize()
            for got, key in ((dq, keys[0]), (dk, keys[1])):
                g = got.double().cpu().numpy()
                assert np.all(g[..., d:] == 0.0), "padded gradient columns must be zero"
                grad_close(g[..., :d], np.array(c[key]), 1e-6)
