"""Backward parity: dQ/dK of both gradient modes, fused (atomics) and
deterministic, against the float64 oracle on the same seeded bf16 inputs.
Full tensors at small sizes; at the large workload sizes sampled dQ rows,
dK of keys whose visible rows the oracle can afford, and the zero-sum
property sum_j dK_j = 0 (rows of dS sum to zero) on every head."""

import numpy as np
import pytest
import torch

import attention_distillation_kl_gb300 as skl
import oracle
from attention_distillation_kl_gb300.workloads import WORKLOADS, Workload, generate_dkl, to_f64

from common import GRAD_RTOL, frob_rel, grad_close, grad_floor, head64, inputs, np_

pytestmark = pytest.mark.gpu

MODES = [(skl.STREAMKL_GRAD_P2, oracle.MODE_P2), (skl.STREAMKL_GRAD_P1, oracle.MODE_P1)]


def gpu_grads(w, dev, dkl, mode, deterministic):
    kl, l1, l2 = skl.streamkl_fwd(*dev, w.scale, w.causal)
    dq, dk = skl.streamkl_bwd(*dev, w.scale, w.causal, kl, l1, l2, dkl, mode, deterministic)
    torch.cuda.synchronize()
    assert skl.streamkl_get_device_status() == 0
    return np_(dq), np_(dk)


def check_full(w, mode_pair, deterministic, dkl_kind="ones"):
    gmode, omode = mode_pair
    host, dev = inputs(w)
    dkl = generate_dkl(w, dkl_kind)
    gdq, gdk = gpu_grads(w, dev, dkl.cuda(), gmode, deterministic)
    f64 = [to_f64(t) for t in host]
    rdq, rdk = oracle.backward(*f64, w.scale, w.causal, to_f64(dkl), omode)
    assert gdq.shape == rdq.shape and gdk.shape == rdk.shape
    g = 2 if omode == oracle.MODE_P2 else 0
    for b in range(w.B):
        for h in range(w.H):
            fl = grad_floor(w.scale, to_f64(dkl)[b, h], f64[g][b, h], f64[g + 1][b, h])
            grad_close(gdq[b, h], rdq[b, h], fl)
            grad_close(gdk[b, h], rdk[b, h], fl)


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
@pytest.mark.parametrize("dkl_kind", ["ones", "uniform"])
def test_pr1(mode, det, dkl_kind):
    check_full(WORKLOADS["pr1"], mode, det, dkl_kind)


EDGE = [
    (1, 1, 1, 1, 64, 64, False),
    (1, 2, 17, 17, 64, 64, True),
    (2, 3, 130, 129, 64, 64, False),
    (1, 2, 257, 300, 128, 64, False),
    (1, 2, 100, 333, 64, 128, True),
    (1, 1, 1000, 1000, 128, 128, True),
    (2, 2, 384, 384, 128, 128, False),
    (1, 1, 5, 1000, 128, 128, True),
    (1, 1, 700, 200, 128, 128, False),  # more queries than keys
]


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "x".join(map(str, s)))
def test_edge_shapes(shape, mode, det):
    B, H, NQ, NK, d1, d2, causal = shape
    w = Workload("edge", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, 78)
    check_full(w, mode, det, "uniform")


@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
def test_identical_inputs_give_zero_gradient(mode):
    w = Workload("same", 1, 2, 300, 300, 128, 128, True, 1.0 / np.sqrt(128), "same", 0.0, 1.0, 6)
    host, dev = inputs(w)
    for det in (False, True):
        gdq, gdk = gpu_grads(w, dev, torch.ones(1, 2, 300, device="cuda"), mode[0], det)
        assert np.all(gdq == 0) and np.all(gdk == 0)


def test_deterministic_mode_is_bitwise_reproducible():
    w = WORKLOADS["c2"].with_(B=1, H=4, NQ=1500, NK=1500)
    host, dev = inputs(w)
    dkl = generate_dkl(w, "uniform").cuda()
    a = gpu_grads(w, dev, dkl, skl.STREAMKL_GRAD_P2, True)
    b = gpu_grads(w, dev, dkl, skl.STREAMKL_GRAD_P2, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
def test_c2_all_heads_p2(det):
    check_full(WORKLOADS["c2"], MODES[0], det)


@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
def test_c3u_underflow_both_modes(mode):
    check_full(WORKLOADS["c3u"].with_(H=4), mode, False)


def sampled(n, k, seed):
    g = np.random.default_rng(seed)
    r = set([0, 1, 127, 128, n // 2, n - 129, n - 1])
    r.update(g.integers(0, n, k).tolist())
    return np.array(sorted(x for x in r if 0 <= x < n))


@pytest.mark.parametrize("name,mode", [("c3", MODES[0]), ("c3", MODES[1]), ("c4", MODES[0]), ("c5", MODES[0])],
                         ids=["c3-P2", "c3-P1", "c4-P2", "c5-P2"])
def test_large_workload_sampled(name, mode):
    w = WORKLOADS[name]
    gmode, omode = mode
    host, dev = inputs(w)
    dkl = generate_dkl(w)
    gdq, gdk = gpu_grads(w, dev, dkl.cuda(), gmode, False)
    assert np.all(np.isfinite(gdq)) and np.all(np.isfinite(gdk))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    for i, (b, h) in enumerate(heads):
        # rows of dS sum to zero, so the keys' gradients do too (any size);
        # bf16 rounding of dS leaves a small residue
        colsum = np.abs(gdk[b, h].sum(axis=0))
        assert np.all(colsum <= 5e-2 * np.abs(gdk[b, h]).sum(axis=0) + 1e-30), (name, b, h)
    dk_all = to_f64(dkl)
    for i, (b, h) in enumerate(heads[:: max(1, len(heads) // 4)]):
        f = head64(host, b, h)
        rows = sampled(w.NQ, 8, i)
        rdq = oracle.backward_dq_rows(*f, w.scale, w.causal, dk_all[b, h], omode, rows)
        assert frob_rel(gdq[b, h, rows], rdq) <= GRAD_RTOL, (name, b, h)
    # dK of keys the oracle can afford: the last key tile under a causal mask
    # (few rows see it), any keys of one head otherwise
    b, h = heads[-1]
    f = head64(host, b, h)
    if w.causal:
        keys = np.arange(w.NK - 200, w.NK, 7)
        first = keys.min() - (w.NK - w.NQ)
    else:
        keys = sampled(w.NK, 6, 99)
        first = 0
    rdk = oracle.backward_dk_keys(*f, w.scale, w.causal, dk_all[b, h], omode, keys, first_row=first)
    assert frob_rel(gdk[b, h, keys], rdk) <= GRAD_RTOL, (name, "dk")


@pytest.mark.parametrize("det", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("mode", MODES, ids=["P2", "P1"])
@pytest.mark.parametrize("shape", [(1, 2, 300, 300, 128, 128, True), (2, 1, 200, 333, 64, 128, False)],
                         ids=["300-causal", "200x333"])
def test_signed_upstream_gradient(shape, mode, det):
    """dKL may be negative or zero on some rows (any loss that weights rows)."""
    B, H, NQ, NK, d1, d2, causal = shape
    w = Workload("signed", B, H, NQ, NK, d1, d2, causal, 1.0 / np.sqrt(d1), "independent", 0.0, 1.2, 81)
    check_full(w, mode, det, "signed")


@pytest.mark.parametrize("name,hb", [("c4", (0, 17)), ("c5", (0, 2))], ids=["c4-P2", "c5-P2"])
def test_large_workload_early_key_tiles(name, hb):
    """dK at the headline sizes for keys of the first key tile (summed over
    every query tile of the head: 512 at 64K, 1024 at 128K) and of a middle
    tile, against the oracle over all the rows that see them (row blocks in
    a spawn pool: tests/oracle_pool.py), in the benchmark's launch
    configuration (fused P2 backward over all heads)."""
    from oracle_pool import dk_keys_pooled
    w = WORKLOADS[name]
    host, dev = inputs(w)
    dkl = generate_dkl(w)
    gdq, gdk = gpu_grads(w, dev, dkl.cuda(), skl.STREAMKL_GRAD_P2, False)
    del dev, gdq
    b, h = hb
    mid = (w.NK // 128 // 2) * 128
    keys = np.array([0, 1, 37, 64, 90, 126, 127, mid, mid + 5, mid + 63, mid + 64, mid + 100, mid + 127])
    f = head64(host, b, h)
    rdk = dk_keys_pooled(*f, w.scale, w.causal, to_f64(dkl)[b, h], oracle.MODE_P2, keys)
    assert frob_rel(gdk[b, h, keys[:7]], rdk[:7]) <= GRAD_RTOL, (name, "key tile 0")
    assert frob_rel(gdk[b, h, keys[7:]], rdk[7:]) <= GRAD_RTOL, (name, "middle key tile")
