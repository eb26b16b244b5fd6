"""Key-split forward (partial statistics per split + merge kernel): equal to
the unsplit forward and to the oracle for any split count, including splits
that receive no key tile."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import WORKLOADS, Workload, to_f64

from common import assert_fwd_close, head64, inputs, np_

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 2, 256, 256, 64, 64, False),
    (1, 2, 1000, 1000, 128, 64, True),
    (2, 1, 300, 777, 128, 128, True),
    (1, 1, 129, 5000, 64, 128, False),
]


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_splits_match_oracle(shape, splits):
    B, H, NQ, NK, d1, d2, causal = shape
    w = Workload("sk", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.3, 31)
    host, dev = inputs(w)
    kl, l1, l2 = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, splits)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    f64 = [to_f64(t) for t in host]
    rkl, rl1, rl2 = oracle.forward(*f64, w.scale, w.causal)
    assert_fwd_close(np_(kl), np_(l1), np_(l2), rkl, rl1, rl2, f"splits={splits}")
    ukl, ul1, ul2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    assert_fwd_close(np_(kl), np_(l1), np_(l2), np_(ukl).astype(np.float64), np_(ul1), np_(ul2), "vs unsplit")


def test_single_split_matches_unsplit():
    """One split runs the same tile loop as the unsplit kernel; only the final
    merge differs (the reduce kernel instead of the in-kernel epilogue)."""
    w = Workload("sk1", 1, 2, 128, 128, 128, 128, False, 0.0884, "independent", 0.0, 1.0, 3)
    host, dev = inputs(w)
    a = skl.streamkl_fwd(*dev, w.scale, False)
    b = skl.streamkl_fwd_splitk(*dev, w.scale, False, 1)
    for x, y in zip(a, b):
        assert torch.allclose(x, y, rtol=1e-6, atol=1e-6)


def test_caller_workspace_is_respected():
    w = Workload("skw", 1, 2, 512, 512, 64, 64, True, 0.125, "independent", 0.0, 1.0, 4)
    host, dev = inputs(w)
    need = skl.streamkl_fwd_splitk_workspace_bytes(1, 2, 512, 4)
    ws = torch.full((need + 64,), 0x7F, dtype=torch.uint8, device="cuda")
    kl, l1, l2 = skl.streamkl_fwd_splitk(*dev, w.scale, True, 4, workspace=ws)
    assert torch.all(ws[need:] == 0x7F)  # nothing written past the stated size
    ukl, _, _ = skl.streamkl_fwd(*dev, w.scale, True)
    assert torch.allclose(kl, ukl, rtol=1e-4, atol=1e-5)
    with pytest.raises(skl.StreamKLError):
        skl.streamkl_fwd_splitk(*dev, w.scale, True, 4, workspace=ws[: need - 16])


def test_suggest_splits():
    assert skl.streamkl_suggest_splits(1, 32, 65536, 65536, 1) == 1  # plenty of CTAs already
    s = skl.streamkl_suggest_splits(1, 4, 131072, 131072, 1)
    assert 1 <= s <= 1024
    assert skl.streamkl_suggest_splits(1, 1, 128, 131072, 0) > 1  # one query tile, long rows


@pytest.mark.parametrize("splits", [8, None], ids=["8", "suggested"])
def test_c5_split(splits):
    w = WORKLOADS["c5"]
    host, dev = inputs(w)
    if splits is None:
        splits = skl.streamkl_suggest_splits(w.B, w.H, w.NQ, w.NK, w.causal)
    kl, l1, l2 = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, splits)
    ukl, ul1, ul2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    torch.cuda.synchronize()
    gkl, gl1, gl2 = np_(kl), np_(l1), np_(l2)
    assert_fwd_close(gkl, gl1, gl2, np_(ukl), np_(ul1), np_(ul2), "c5 split vs unsplit")
    g = np.random.default_rng(5)
    for h in range(w.H):
        rows = np.unique(np.concatenate([[0, 1, 128, w.NQ - 1], g.integers(0, w.NQ, 16)]))
        rkl, rl1, rl2 = oracle.forward_rows(*head64(host, 0, h), w.scale, w.causal, rows)
        assert_fwd_close(gkl[0, h, rows], gl1[0, h, rows], gl2[0, h, rows], rkl, rl1, rl2, f"c5 h{h}")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "non-causal"])
def test_short_queries_long_keys(causal):
    """256 queries against 131072 keys (4 heads, d = 128): the shape the key
    split exists for.  The heuristic's split count (well above 1 here) and a
    fixed 32 against the oracle on rows of every head, and against the plain
    forward on all rows."""
    w = Workload("short-q", 1, 4, 256, 131072, 128, 128, causal, 1.0 / np.sqrt(128), "independent", 0.0, 1.0, 1008)
    host, dev = inputs(w)
    s = skl.streamkl_suggest_splits(w.B, w.H, w.NQ, w.NK, w.causal)
    assert s > 1
    ukl, ul1, ul2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    g = np.random.default_rng(6)
    for splits in (s, 32):
        kl, l1, l2 = skl.streamkl_fwd_splitk(*dev, w.scale, w.causal, splits)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == 0
        gkl, gl1, gl2 = np_(kl), np_(l1), np_(l2)
        assert_fwd_close(gkl, gl1, gl2, np_(ukl), np_(ul1), np_(ul2), f"split {splits} vs unsplit")
        for h in range(w.H):
            rows = np.unique(np.concatenate([[0, 127, 128, w.NQ - 1], g.integers(0, w.NQ, 12)]))
            rkl, rl1, rl2 = oracle.forward_rows(*head64(host, 0, h), w.scale, w.causal, rows)
            assert_fwd_close(gkl[0, h, rows], gl1[0, h, rows], gl2[0, h, rows], rkl, rl1, rl2,
                             f"short queries split {splits} h{h}")
