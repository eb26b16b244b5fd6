"""The allocation-free key-split forward against the caller-workspace one.

streamkl_fwd_splitk_noalloc serves callers that cannot allocate device memory
(for example code under an allocator that owns all of it): its partials live
in a fixed array inside the library.  This checks, through the C ABI, that
two calls in a row give the same results as streamkl_fwd_splitk with a
caller-owned workspace (within the forward tolerances of the parity tests),
that the second call is not disturbed by what the first left in the shared
array, and that a problem whose partials exceed the fixed size is refused.
The file sorts last so a failure here never hides another test.
"""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
from attention_distillation_kl_gb300.workloads import Workload

from common import assert_fwd_close, inputs, np_

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, num_splits): the second is bigger and uses other head dims
    (Workload("na1", 1, 2, 700, 700, 128, 128, True, 1.0 / np.sqrt(128), "independent", 0.0, 1.3, 41), 3),
    (Workload("na2", 2, 3, 1000, 2048, 128, 64, False, 1.0 / np.sqrt(128), "independent", 0.0, 1.3, 42), 8),
]


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    for w, splits in CASES:
        host, dev = inputs(w)
        got = skl.streamkl_fwd_splitk_noalloc(*dev, w.scale, w.causal, splits)
        want = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, splits)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == 0
        assert_fwd_close(*(np_(t) for t in got), *(np_(t) for t in want), f"{w.name} noalloc")


def test_noalloc_larger_call_then_smaller_call():
    """The bigger layout first: partials it leaves past the smaller call's
    extent, or at the smaller call's offsets, must not leak into the latter."""
    for w, splits in reversed(CASES):
        host, dev = inputs(w)
        got = skl.streamkl_fwd_splitk_noalloc(*dev, w.scale, w.causal, splits)
        want = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, splits)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == 0
        assert_fwd_close(*(np_(t) for t in got), *(np_(t) for t in want), f"{w.name} noalloc after larger")


def test_noalloc_repeated_call_is_stable():
    w, splits = CASES[0]
    host, dev = inputs(w)
    a = [t.clone() for t in skl.streamkl_fwd_splitk_noalloc(*dev, w.scale, w.causal, splits)]
    b = skl.streamkl_fwd_splitk_noalloc(*dev, w.scale, w.causal, splits)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_noalloc_refuses_over_the_fixed_size():
    w = Workload("na3", 1, 1, 128, 128, 64, 64, False, 0.125, "independent", 0.0, 1.0, 43)
    host, dev = inputs(w)
    # 5 * 4 * splits * B * H * NQ bytes must fit in the fixed array
    splits = 1024
    big = Workload("na4", 1, 16, 128 * 16, 128, 64, 64, False, 0.125, "independent", 0.0, 1.0, 44)
    assert skl.streamkl_fwd_splitk_workspace_bytes(big.B, big.H, big.NQ, splits) > skl.STREAMKL_STATIC_WORKSPACE_BYTES
    hb, db = inputs(big)
    with pytest.raises(skl.StreamKLError) as e:
        skl.streamkl_fwd_splitk_noalloc(*db, big.scale, big.causal, splits)
    assert e.value.status == skl.STREAMKL_INVALID_ARG
    # the refused call enqueued nothing; a fitting call still works
    got = skl.streamkl_fwd_splitk_noalloc(*dev, w.scale, w.causal, 2)
    want = skl.streamkl_fwd(*dev, w.scale, w.causal)
    assert_fwd_close(*(np_(t) for t in got), *(np_(t) for t in want), "after refusal")
