"""Failure detection on the GPU without faulting it: a kernel waits on a
barrier that nothing completes, gives up after a short limit, reports
STREAMKL_DEVICE_TIMEOUT through the status word and exits; the context stays
usable and the next call runs normally."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
from attention_distillation_kl_gb300.workloads import WORKLOADS

from common import np_

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK  # clears anything earlier
    skl.streamkl_selftest_wait_timeout(20000)  # 20 ms
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == skl.STREAMKL_DEVICE_TIMEOUT
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK  # read-and-clear
    w = WORKLOADS["pr1"]
    dev = [torch.randn(w.B, w.H, n, d, device="cuda").to(torch.bfloat16)
           for n, d in ((w.NQ, w.d1), (w.NK, w.d1), (w.NQ, w.d2), (w.NK, w.d2))]
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    torch.cuda.synchronize()
    assert np.all(np.isfinite(np_(kl))) and skl.streamkl_get_device_status() == skl.STREAMKL_OK


def test_selftest_argument_checks():
    with pytest.raises(skl.StreamKLError):
        skl.streamkl_selftest_wait_timeout(0)
    with pytest.raises(skl.StreamKLError):
        skl.streamkl_selftest_wait_timeout(2_000_000)


def test_turn_wait_reports_timeout_and_releases_the_launch():
    """The counter wait of the deterministic backward with shared key heads:
    it gives up after the limit, reports a time-out, sets the launch's abort
    word, and a later wait of the same launch gives up at once."""
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
    words = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    skl.streamkl_selftest_turn_timeout(20000, words)  # 20 ms
    torch.cuda.synchronize()
    w = words.cpu().tolist()
    assert w[0] == 0 and w[1] == 1, w          # the count never moved; the launch was aborted
    assert w[2] == 0 and w[3] == 0 and w[4] == 1, w
    assert skl.streamkl_get_device_status() == skl.STREAMKL_DEVICE_TIMEOUT
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK


def test_turn_selftest_argument_checks():
    words = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(skl.StreamKLError):
        skl.streamkl_selftest_turn_timeout(0, words)
    with pytest.raises(skl.StreamKLError):
        skl.streamkl_selftest_turn_timeout(2_000_000, words)
