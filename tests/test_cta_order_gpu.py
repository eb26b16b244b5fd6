"""CTA order: heads whose tiles interleave give the same bits as one head.

The forward and the fused backward hand their CTAs (tile, head) units in
groups of heads whose tiles interleave, longest first, the group sized from
the L2 size and the problem (a pure permutation of the units).  Each row's
forward statistics and each key tile's dK depend only on that head's data,
and the deterministic backward's dQ sums are exact in any order, so a
batched call must reproduce, bit for bit, the same call made head by head
(one head: a single group, head after head).  Seven heads of 16K tokens:
a prime count, so any group size from 2 to 6 (the sizes a GB300's L2 gives
these shapes) leaves a partial last group, and a unit lost or taken twice
at a group boundary would show.  Outputs start as NaN where the library
does not clear them first.
"""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, d, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = [torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda() for _ in range(4)]
    t[2] = (t[0].float() + 0.3 * t[2].float()).to(torch.bfloat16)  # a correlated student
    return t


@pytest.mark.parametrize("causal", [True, False])
def test_grouped_heads_match_head_by_head(causal):
    B, H, N, d = 1, 7, 16384, 128
    q1, k1, q2, k2 = _inputs(B, H, N, d, 7 + int(causal))
    scale = 1.0 / np.sqrt(d)
    nan = lambda *s: torch.full(s, float("nan"), device="cuda")
    kl, l1, l2 = nan(B, H, N), nan(B, H, N), nan(B, H, N)
    skl.streamkl_fwd(q1, k1, q2, k2, scale, causal, kl, l1, l2)
    dkl = torch.rand(B, H, N, device="cuda") - 0.25
    dq, dk = nan(B, H, N, d), nan(B, H, N, d)
    skl.streamkl_bwd(q1, k1, q2, k2, scale, causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2, True, dq, dk)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    for t in (kl, l1, l2, dq, dk):
        assert bool(torch.isfinite(t).all())
    for b in range(B):
        for h in range(H):
            one = [x[b:b + 1, h:h + 1].contiguous() for x in (q1, k1, q2, k2)]
            k_, a_, c_ = skl.streamkl_fwd(*one, scale, causal)
            assert torch.equal(k_[0, 0], kl[b, h]) and torch.equal(a_[0, 0], l1[b, h])
            assert torch.equal(c_[0, 0], l2[b, h])
            q_, kk_ = skl.streamkl_bwd(*one, scale, causal, k_, a_, c_, dkl[b:b + 1, h:h + 1].contiguous(),
                                       skl.STREAMKL_GRAD_P2, True)
            assert torch.equal(q_[0, 0], dq[b, h]), (b, h)
            assert torch.equal(kk_[0, 0], dk[b, h]), (b, h)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0


def _per_head_equal(batched, per_head, B, H):
    for b in range(B):
        for h in range(H):
            got = per_head(b, h)
            for x, y in zip(got, batched):
                assert torch.equal(x[0, 0], y[b, h]), (b, h)


def test_grouped_heads_both_sides_deterministic():
    """The both-sides kernel (d = 64), deterministic."""
    B, H, N, d = 1, 7, 16384, 64
    q1, k1, q2, k2 = _inputs(B, H, N, d, 11)
    scale = 1.0 / np.sqrt(d)
    kl, l1, l2 = skl.streamkl_fwd(q1, k1, q2, k2, scale, True)
    dkl = torch.rand(B, H, N, device="cuda") - 0.25
    out = skl.streamkl_bwd_both(q1, k1, q2, k2, scale, scale, True, kl, l1, l2, dkl, True)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0

    def one(b, h):
        s = (slice(b, b + 1), slice(h, h + 1))
        x = [t[s].contiguous() for t in (q1, k1, q2, k2)]
        return skl.streamkl_bwd_both(*x, scale, scale, True, kl[s].contiguous(), l1[s].contiguous(),
                                     l2[s].contiguous(), dkl[s].contiguous(), True)

    _per_head_equal(out, one, B, H)


def test_grouped_heads_wide_head_dim():
    """Head dim 256 on both sides (block-ring forward, two-pass backward,
    no atomics)."""
    B, H, N, d = 1, 7, 16384, 256
    q1, k1, q2, k2 = _inputs(B, H, N, d, 13)
    scale = 1.0 / np.sqrt(d)
    fwd = skl.streamkl_fwd(q1, k1, q2, k2, scale, True)
    dkl = torch.rand(B, H, N, device="cuda") - 0.25
    bwd = skl.streamkl_bwd(q1, k1, q2, k2, scale, True, *fwd, dkl, skl.STREAMKL_GRAD_P2, False)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0

    def one(b, h):
        s = (slice(b, b + 1), slice(h, h + 1))
        x = [t[s].contiguous() for t in (q1, k1, q2, k2)]
        f = skl.streamkl_fwd(*x, scale, True)
        g = skl.streamkl_bwd(*x, scale, True, *(t[s].contiguous() for t in fwd), dkl[s].contiguous(),
                             skl.STREAMKL_GRAD_P2, False)
        return (*f, *g)

    _per_head_equal((*fwd, *bwd), one, B, H)
