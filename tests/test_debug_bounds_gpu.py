"""The debug build (libstreamkl_debug.so: the same sources compiled with
STREAMKL_DEBUG, so every global index and staging offset the kernels compute
is checked against the extents they were given, a failed check skipping the
access and setting STREAMKL_DEBUG_BOUNDS in the device status word) on edge
shapes of every kernel: no check may fail, and the results must equal the
normal build's (exactly where the kernels are deterministic)."""

import contextlib
import os

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, generate_gqa

from common import inputs

pytestmark = pytest.mark.gpu

DEBUG_LIB = os.path.join(os.path.dirname(skl.library_path), "libstreamkl_debug.so")


@contextlib.contextmanager
def library(path):
    """Route the binding's calls to the library at `path` for the block."""
    saved = skl._lib, skl.library_path
    skl._lib, skl.library_path = None, path
    try:
        yield skl.lib()
    finally:
        skl._lib, skl.library_path = saved


def run_all(w, s2, dev, dkl):
    out = {}
    out["fwd"] = [t.clone() for t in skl.streamkl_fwd_scaled(*dev, w.scale, s2, w.causal)]
    kl, l1, l2 = out["fwd"]
    out["split3"] = [t.clone() for t in skl.streamkl_fwd_splitk_scaled(*dev, w.scale, s2, w.causal, 3)]
    for mode in (skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1):
        for det in (False, True):
            out[f"bwd{mode}{int(det)}"] = [t.clone() for t in skl.streamkl_bwd_scaled(
                *dev, w.scale, s2, w.causal, kl, l1, l2, dkl, mode, det)]
    torch.cuda.synchronize()
    return out


CASES = [
    (1, 2, 17, 17, 64, 64, True),
    (2, 1, 130, 129, 128, 32, False),
    (1, 1, 100, 333, 128, 128, True),
    (1, 1, 700, 200, 64, 128, False),
    (1, 1, 300, 300, 256, 144, True),
]


@pytest.mark.parametrize("c", CASES, ids=["x".join(map(str, c)) for c in CASES])
def test_debug_build_checks_pass_and_match(c):
    if not os.path.exists(DEBUG_LIB):
        pytest.fail("libstreamkl_debug.so was not built")
    B, H, NQ, NK, d1, d2, causal = c
    w = Workload("dbg", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, 131)
    s2 = 1.0 / np.sqrt(d2)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "signed").cuda()
    ref = run_all(w, s2, dev, dkl)
    with library(DEBUG_LIB):
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
        got = run_all(w, s2, dev, dkl)
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK, "a bounds check failed"
    for key, want in ref.items():
        for x, y in zip(got[key], want):
            if key.endswith("0") and key.startswith("bwd") and max(d1, d2) <= 128:
                # fused backward: dQ is summed with atomics in varying order
                assert torch.allclose(x, y, rtol=1e-4, atol=1e-6), key
            else:
                assert torch.equal(x, y), key


def test_debug_build_grouped_key_heads_and_both_sides():
    if not os.path.exists(DEBUG_LIB):
        pytest.fail("libstreamkl_debug.so was not built")
    w = Workload("dbg-gqa", 1, 4, 200, 260, 64, 64, True, 0.125, "independent", 0.0, 1.0, 132)
    dev = [t.cuda() for t in generate_gqa(w, 2, 1)]
    dkl = generate_dkl(w, "uniform").cuda()
    wb = Workload("dbg-both", 1, 2, 190, 190, 64, 64, False, 0.125, "independent", 0.0, 1.0, 133)
    hb, db = inputs(wb)
    dklb = generate_dkl(wb, "uniform").cuda()
    with library(DEBUG_LIB):
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
        kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal)
        for mode in (skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1):
            for det in (False, True):
                skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, det)
        kb, a1, a2 = skl.streamkl_fwd(*db, wb.scale, wb.causal)
        skl.streamkl_bwd_both(*db, wb.scale, wb.scale, wb.causal, kb, a1, a2, dklb, False)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK, "a bounds check failed"
