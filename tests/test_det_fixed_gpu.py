"""Deterministic backward: every dQ contribution rounded to a per-row grid
of 2^-e, 2^-22 of a bound on |dQ_i|, so the fp32 sums are exact in any
order.  The per-tile contributions are the same MMA outputs the fused (fp32
atomic) mode adds, so the two modes may differ only by their rounding; the
deterministic result must also be bitwise repeatable, finite and exactly
zero on rows with dKL = 0, over upstream gradients spanning the fp32 range."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
from attention_distillation_kl_gb300.workloads import Workload, generate_dkl, generate_gqa

from common import inputs, np_

pytestmark = pytest.mark.gpu

MODES = [skl.STREAMKL_GRAD_P2, skl.STREAMKL_GRAD_P1]


def row_bound(mode, sg, dkl, kl, kg):
    """The bound the grid is taken from (the kernel's formula, slack
    included): |dQ_id| <= s |dKL_i| max|K_g| C_i with TV_i <= min(1,
    sqrt(KL_i / 2)), C_i = 2 TV_i (mode P2) or 2 KL_i + 2 TV_i (mode P1)."""
    kmax = np.abs(kg.float().cpu().numpy()).reshape(kg.shape[0], kg.shape[1], -1).max(axis=2)
    k = np.maximum(kl, 0.0) + 1e-4
    tv = np.minimum(1.0, np.sqrt(k / 2)) + 1e-4
    c = 2.0 * tv if mode == skl.STREAMKL_GRAD_P2 else 2.0 * (k + tv)
    return sg * np.abs(dkl) * kmax[:, :, None] * c * 1.0078125


def compare_modes(dq_fused, dq_det, bound, n_key_tiles):
    """Per row: |det - fused| <= (key tiles + 1) (2^-24 + 2^-21) bound +
    key tiles 2^-126: the fp32 atomic rounding of partial sums below the
    bound, and the deterministic mode's rounding of each tile's contribution
    to its grid (half a step, a step being at most 2^-21 of the bound, or
    2^-126 for rows whose bound is below 2^-104)."""
    tol = (n_key_tiles + 1) * (2.0 ** -24 + 2.0 ** -21) * bound + n_key_tiles * 2.0 ** -126
    err = np.abs(dq_det - dq_fused).max(axis=-1)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), f"row {worst}: |det - fused| {err[worst]} > {tol[worst]}"


CASES = [
    (1, 2, 300, 300, 128, 128, True),
    (2, 1, 1000, 1000, 64, 64, False),
    (1, 2, 257, 700, 128, 64, True),
    (1, 1, 130, 129, 32, 128, False),
]


@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
@pytest.mark.parametrize("kind", ["uniform", "signed", "wide"])
@pytest.mark.parametrize("c", CASES, ids=lambda c: "x".join(map(str, c)))
def test_fixed_point_matches_fused_sum(c, kind, mode):
    B, H, NQ, NK, d1, d2, causal = c
    w = Workload("fx", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, 211)
    host, dev = inputs(w)
    dkl = generate_dkl(w, kind).cuda()
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    fused = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, mode, False)
    det = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
    det2 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
    dq_f, dk_f, dq_d, dk_d = (np_(t) for t in (*fused, *det))
    assert np.all(np.isfinite(dq_d)) and np.all(np.isfinite(dk_d))
    assert torch.equal(det[0], det2[0]) and torch.equal(det[1], det2[1]), "not bitwise repeatable"
    # dK is written by one CTA per key tile in both modes: the same bits
    assert np.array_equal(dk_d, dk_f)
    zero = np_(dkl) == 0.0
    assert np.all(dq_d[zero] == 0.0)
    kg = host[3] if mode == skl.STREAMKL_GRAD_P2 else host[1]
    bound = row_bound(mode, w.scale, np_(dkl), np_(kl), kg)
    compare_modes(dq_f, dq_d, bound, (NK + 127) // 128)


def test_gqa_fixed_point_repeatable_and_close():
    w = Workload("fxg", 1, 6, 900, 900, 64, 64, True, 0.125, "independent", 0.0, 1.0, 212)
    dev = [t.cuda() for t in generate_gqa(w, 3, 2)]
    dkl = generate_dkl(w, "wide").cuda()
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal)
    for mode in MODES:
        f = skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, False)
        a = skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
        b = skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        kg = dev[3] if mode == skl.STREAMKL_GRAD_P2 else dev[1]
        kg = kg.repeat_interleave(w.H // kg.shape[1], dim=1)  # key head of each query head
        bound = row_bound(mode, w.scale, np_(dkl), np_(kl), kg)
        compare_modes(np_(f[0]), np_(a[0]), bound, (w.NK + 127) // 128)
        # dK of a shared key head: ordered adds against atomics in any order
        dk_f, dk_d = np_(f[1]), np_(a[1])
        assert np.linalg.norm(dk_d - dk_f) <= 1e-5 * np.linalg.norm(dk_f)


def test_mqa_ordered_dk_single_launch():
    """Eight query heads on one key head per side, causal with NQ < NK."""
    w = Workload("fxm", 1, 8, 200, 600, 64, 64, True, 0.125, "independent", 0.0, 1.0, 213)
    dev = [t.cuda() for t in generate_gqa(w, 1, 1)]
    dkl = generate_dkl(w, "signed").cuda()
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal)
    for mode in MODES:
        runs = [skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
                for _ in range(3)]
        f = skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, False)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
        for r in runs[1:]:
            assert torch.equal(r[0], runs[0][0]) and torch.equal(r[1], runs[0][1])
        dk_f, dk_d = np_(f[1]), np_(runs[0][1])
        assert np.all(np.isfinite(dk_d))
        assert np.linalg.norm(dk_d - dk_f) <= 1e-5 * np.linalg.norm(dk_f)


def test_headline_size_deterministic_matches_fused():
    """64K x 32 heads, causal, d = 128 (the benchmark's workload and launch):
    every row of the deterministic dQ within its rounding bound of the fused
    one, dK equal bit for bit, and two deterministic runs identical."""
    from attention_distillation_kl_gb300.workloads import WORKLOADS
    w = WORKLOADS["c4"]
    _, dev = inputs(w)
    dkl = generate_dkl(w, "uniform").cuda()
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    fused = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2, False)
    det = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2, True)
    det2 = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, skl.STREAMKL_GRAD_P2, True)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
    assert torch.equal(det[0], det2[0]) and torch.equal(det[1], det2[1])
    assert torch.equal(det[1], fused[1])
    # the bound of each row, on the device (same formula as row_bound)
    kmax = dev[3].float().abs().amax(dim=(2, 3))  # [B, H]
    k = kl.clamp_min(0.0).double() + 1e-4
    tv = torch.clamp(torch.sqrt(k / 2), max=1.0) + 1e-4
    bound = w.scale * dkl.double().abs() * kmax.double()[:, :, None] * 2.0 * tv * 1.0078125
    tiles = (w.NK + 127) // 128
    tol = (tiles + 1) * (2.0 ** -24 + 2.0 ** -21) * bound + tiles * 2.0 ** -126
    err = (det[0] - fused[0]).abs().amax(dim=-1).double()
    assert bool(torch.all(torch.isfinite(det[0])))
    worst = torch.argmax(err - tol)
    assert bool(torch.all(err <= tol)), f"row {worst.item()}: {err.flatten()[worst].item()} > {tol.flatten()[worst].item()}"


def test_caller_workspace_gives_the_same_bits():
    """streamkl_bwd_gqa_ws with the caller's scratch equals the pooled call bit
    for bit, and rejects a missing or short workspace before enqueuing."""
    w = Workload("fxw", 1, 4, 400, 400, 64, 64, True, 0.125, "independent", 0.0, 1.0, 214)
    dev = [t.cuda() for t in generate_gqa(w, 2, 2)]
    dkl = generate_dkl(w, "signed").cuda()
    kl, l1, l2 = skl.streamkl_fwd_gqa(*dev, w.scale, w.scale, w.causal)
    for mode in MODES:
        need = skl.streamkl_bwd_workspace_bytes(w.B, w.H, 2, 2, w.NK, w.d1, w.d2, mode)
        assert need > 0
        ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")  # contents must not matter
        a = skl.streamkl_bwd_gqa(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, mode, True)
        b = skl.streamkl_bwd_gqa_ws(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, ws, mode, True)
        torch.cuda.synchronize()
        assert skl.streamkl_get_device_status() == skl.STREAMKL_OK
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        with pytest.raises(skl.StreamKLError):
            skl.streamkl_bwd_gqa_ws(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, ws[:need - 16], mode, True)
        with pytest.raises(skl.StreamKLError):
            skl.streamkl_bwd_gqa_ws(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, None, mode, True)
        # the atomic mode needs no scratch
        skl.streamkl_bwd_gqa_ws(*dev, w.scale, w.scale, w.causal, kl, l1, l2, dkl, None, mode, False)
