"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host before touching the device (no GPU needed:
every call here fails validation before any CUDA call)."""

import ctypes
import os
import re

import pytest

import attention_distillation_kl_gb300 as skl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "streamkl.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(skl.library_path):
        import __graft_entry__
        __graft_entry__.build()
    return skl.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(streamkl_\w+)\s*\(", text, re.M)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for want in ("streamkl_fwd", "streamkl_fwd_splitk", "streamkl_bwd",
                 "streamkl_fwd_splitk_workspace_bytes", "streamkl_suggest_splits",
                 "streamkl_status_string", "streamkl_get_device_status"):
        assert want in syms


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
        assert name in skl._SIGS, f"binding lacks {name}"


def test_debug_library_exports_every_declared_symbol():
    # the STREAMKL_DEBUG build of the same sources (bounds checks in the kernels)
    import ctypes
    import os
    path = os.path.join(os.path.dirname(skl.library_path), "libstreamkl_debug.so")
    if not os.path.exists(path):
        pytest.skip("debug library not built")
    D = ctypes.CDLL(path)
    for name in declared_symbols():
        assert hasattr(D, name), name
    D.streamkl_status_string.restype = ctypes.c_char_p
    assert b"bounds" in D.streamkl_status_string(skl.STREAMKL_DEBUG_BOUNDS)


def test_binding_wraps_every_entry_point():
    # each C entry point has a Python function of the same name, exported
    for name in declared_symbols():
        assert callable(getattr(skl, name, None)), f"no Python wrapper for {name}"
        assert name in skl.__all__, f"{name} missing from __all__"


def test_status_strings(L):
    for s in range(5):
        assert skl.status_string(s) and skl.status_string(s) != "unknown status"
    assert skl.status_string(99) == "unknown status"


def test_workspace_bytes(L):
    assert skl.streamkl_fwd_splitk_workspace_bytes(1, 4, 131072, 8) == 5 * 4 * 8 * 4 * 131072
    assert skl.streamkl_fwd_splitk_workspace_bytes(1, 1, 10, 0) == 0
    assert skl.streamkl_fwd_splitk_workspace_bytes(1, 1, 10, 1025) == 0
    assert skl.streamkl_fwd_splitk_workspace_bytes(-1, 1, 10, 2) == 0


def test_suggest_splits_rejects_bad_sizes(L):
    assert skl.streamkl_suggest_splits(0, 4, 128, 128, 0) == 0
    assert skl.streamkl_suggest_splits(1, 4, 256, 128, 1) == 0  # causal NQ > NK


A = 4096  # a 16-byte aligned fake address: never dereferenced, validation fails first


def fwd(L, q=(A, A, A, A), B=1, H=1, NQ=128, NK=128, d1=64, d2=64, scale=0.125, causal=0,
        out=(A, A, A)):
    return L.streamkl_fwd(*q, B, H, NQ, NK, d1, d2, scale, causal, *out, None)


@pytest.mark.parametrize("kw,status", [
    (dict(scale=0.0), skl.STREAMKL_INVALID_ARG),
    (dict(scale=-1.0), skl.STREAMKL_INVALID_ARG),
    (dict(scale=float("nan")), skl.STREAMKL_INVALID_ARG),
    (dict(scale=float("inf")), skl.STREAMKL_INVALID_ARG),
    (dict(causal=2), skl.STREAMKL_INVALID_ARG),
    (dict(d1=8), skl.STREAMKL_UNSUPPORTED),
    (dict(d2=40), skl.STREAMKL_UNSUPPORTED),
    (dict(d1=0), skl.STREAMKL_UNSUPPORTED),
    (dict(d2=136), skl.STREAMKL_UNSUPPORTED),
    (dict(d1=272), skl.STREAMKL_UNSUPPORTED),
    (dict(d2=512), skl.STREAMKL_UNSUPPORTED),
    (dict(NQ=256, NK=128, causal=1), skl.STREAMKL_INVALID_ARG),
    (dict(NK=0), skl.STREAMKL_INVALID_ARG),
    (dict(B=-1), skl.STREAMKL_INVALID_ARG),
    (dict(q=(0, A, A, A)), skl.STREAMKL_INVALID_ARG),
    (dict(q=(A, A + 2, A, A)), skl.STREAMKL_INVALID_ARG),
    (dict(out=(0, A, A)), skl.STREAMKL_INVALID_ARG),
    (dict(out=(A, A, A + 4)), skl.STREAMKL_INVALID_ARG),
    (dict(B=70000), skl.STREAMKL_INVALID_ARG),
])
def test_fwd_validation(L, kw, status):
    assert fwd(L, **kw) == status


def test_empty_problem_is_noop(L):
    # no rows: returns OK without touching any pointer or the device
    assert fwd(L, q=(0, 0, 0, 0), NQ=0, out=(0, 0, 0)) == skl.STREAMKL_OK
    assert fwd(L, q=(0, 0, 0, 0), B=0, out=(0, 0, 0)) == skl.STREAMKL_OK


def test_splitk_validation(L):
    f = L.streamkl_fwd_splitk
    ok_args = (A, A, A, A, 1, 2, 256, 256, 64, 64, 0.125, 0)
    need = skl.streamkl_fwd_splitk_workspace_bytes(1, 2, 256, 4)
    assert f(*ok_args, 0, A, need, A, A, A, None) == skl.STREAMKL_INVALID_ARG      # splits < 1
    assert f(*ok_args, 2000, A, 1 << 40, A, A, A, None) == skl.STREAMKL_INVALID_ARG  # splits > 1024
    assert f(*ok_args, 4, A, need - 1, A, A, A, None) == skl.STREAMKL_INVALID_ARG   # small workspace
    assert f(*ok_args, 4, 0, need, A, A, A, None) == skl.STREAMKL_INVALID_ARG       # null workspace
    assert f(*ok_args, 4, A + 8, need, A, A, A, None) == skl.STREAMKL_INVALID_ARG   # misaligned


def test_bwd_validation(L):
    f = L.streamkl_bwd
    base = (A, A, A, A, 1, 1, 128, 128, 64, 64, 0.125, 0, A, A, A, A)
    assert f(*base, 2, 0, A, A, None) == skl.STREAMKL_INVALID_ARG   # bad mode
    assert f(*base, 0, 3, A, A, None) == skl.STREAMKL_INVALID_ARG   # bad deterministic flag
    assert f(*base, 0, 0, 0, A, None) == skl.STREAMKL_INVALID_ARG   # null dq
    assert f(*base, 0, 0, A, A + 4, None) == skl.STREAMKL_INVALID_ARG  # misaligned dk
    bad_lse = base[:13] + (0,) + base[14:]
    assert f(*bad_lse, 0, 0, A, A, None) == skl.STREAMKL_INVALID_ARG


def test_binding_raises_without_cuda_tensors(L):
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        skl.streamkl_fwd(x, x, x, x, 0.125, False)


def test_noalloc_constant_and_host_refusal(L):
    text = open(HEADER).read()
    m = re.search(r"#define STREAMKL_STATIC_WORKSPACE_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == skl.STREAMKL_STATIC_WORKSPACE_BYTES
    f = L.streamkl_fwd_splitk_noalloc
    # partials of 5*4*1024*16*2048 bytes exceed the fixed array: refused before any device call
    assert f(A, A, A, A, 1, 16, 2048, 128, 64, 64, 0.125, 0, 1024, A, A, A, None) == skl.STREAMKL_INVALID_ARG
    assert f(A, A, A, A, 1, 1, 128, 128, 64, 64, 0.125, 0, 0, A, A, A, None) == skl.STREAMKL_INVALID_ARG
    assert f(0, 0, 0, 0, 1, 1, 0, 128, 64, 64, 0.125, 0, 2, 0, 0, 0, None) == skl.STREAMKL_OK  # no rows


@pytest.mark.parametrize("s1,s2", [(0.125, 0.0), (0.125, -1.0), (0.125, float("nan")), (0.125, 2e4),
                                   (0.0, 0.125), (float("inf"), 0.125)])
def test_scaled_calls_validate_both_scales(L, s1, s2):
    out = (A, A, A)
    assert L.streamkl_fwd_scaled(A, A, A, A, 1, 1, 128, 128, 64, 64, s1, s2, 0, *out, None) == \
        skl.STREAMKL_INVALID_ARG
    need = skl.streamkl_fwd_splitk_workspace_bytes(1, 1, 128, 2)
    assert L.streamkl_fwd_splitk_scaled(A, A, A, A, 1, 1, 128, 128, 64, 64, s1, s2, 0, 2, A, need,
                                        *out, None) == skl.STREAMKL_INVALID_ARG
    assert L.streamkl_bwd_scaled(A, A, A, A, 1, 1, 128, 128, 64, 64, s1, s2, 0, A, A, A, A, 0, 0, A, A,
                                 None) == skl.STREAMKL_INVALID_ARG


def test_scaled_calls_empty_problem_is_noop(L):
    assert L.streamkl_fwd_scaled(0, 0, 0, 0, 1, 1, 0, 128, 64, 64, 0.1, 0.2, 0, 0, 0, 0, None) == skl.STREAMKL_OK


def test_bwd_both_validation(L):
    f = L.streamkl_bwd_both
    base = (A, A, A, A, 1, 1, 128, 128, 64, 64)
    tail = (A, A, A, A)
    assert f(*base, 0.125, 0.0, 0, *tail, 0, A, A, A, A, None) == skl.STREAMKL_INVALID_ARG     # scale2
    assert f(*base, 0.125, 0.125, 0, *tail, 2, A, A, A, A, None) == skl.STREAMKL_INVALID_ARG   # deterministic flag
    assert f(*base, 0.125, 0.125, 0, *tail, 0, A, A, 0, A, None) == skl.STREAMKL_INVALID_ARG   # null dq2
    assert f(*base, 0.125, 0.125, 0, *tail, 0, A, A, A, A + 4, None) == skl.STREAMKL_INVALID_ARG  # misaligned dk2
    assert f(A, A, A, A, 1, 1, 128, 128, 72, 64, 0.1, 0.1, 0, *tail, 0, A, A, A, A, None) == skl.STREAMKL_UNSUPPORTED


@pytest.mark.parametrize("H,HK1,HK2,ok", [
    (8, 8, 8, True), (8, 2, 8, True), (8, 1, 4, True),
    (8, 3, 8, False),    # 3 does not divide 8
    (8, 8, 16, False),   # more key heads than query heads
    (8, 0, 8, False),
    (8, 8, -1, False),
])
def test_gqa_head_counts(L, H, HK1, HK2, ok):
    # a bad head layout is INVALID_ARG before anything else is looked at; a
    # good one is accepted (shown on an empty problem, which needs no GPU)
    fwd_args = (A, A, A, A, 1, H, HK1, HK2, 128, 128, 64, 64, 0.125, 0.125, 0)
    if ok:
        # empty problem (NQ = 0) with the same head layout is a no-op
        assert L.streamkl_fwd_gqa(0, 0, 0, 0, 1, H, HK1, HK2, 0, 128, 64, 64, 0.125, 0.125, 0, 0, 0, 0,
                                  None) == skl.STREAMKL_OK
    else:
        assert L.streamkl_fwd_gqa(*fwd_args, A, A, A, None) == skl.STREAMKL_INVALID_ARG
        assert L.streamkl_fwd_splitk_gqa(*fwd_args, 2, A, 1 << 20, A, A, A, None) == skl.STREAMKL_INVALID_ARG
        assert L.streamkl_bwd_gqa(*fwd_args, A, A, A, A, 0, 0, A, A, None) == skl.STREAMKL_INVALID_ARG


def test_gqa_empty_backward_zeroes_key_heads_only(L):
    # NQ = 0: nothing to compute, and with no dk buffer (size 0) nothing to zero
    assert L.streamkl_bwd_gqa(0, 0, 0, 0, 0, 8, 2, 2, 0, 128, 64, 64, 0.125, 0.125, 0, 0, 0, 0, 0, 0, 0, 0, 0,
                              None) == skl.STREAMKL_OK


def test_backward_workspace_bytes():
    # the deterministic backward's scratch: 4 bytes per gradient-side key head,
    # 8 more, and 4 per key head and key tile when query heads share key heads
    assert skl.streamkl_bwd_workspace_bytes(1, 32, 32, 32, 65536, 128, 128) == 144
    assert skl.streamkl_bwd_workspace_bytes(1, 32, 8, 8, 16384, 128, 128) == (8 + 2 + 8 * 128) * 4 + 8
    assert skl.streamkl_bwd_workspace_bytes(2, 4, 4, 1, 300, 64, 64, skl.STREAMKL_GRAD_P1) == 48
    assert skl.streamkl_bwd_workspace_bytes(2, 4, 4, 1, 300, 64, 64, skl.STREAMKL_GRAD_P2) == \
        (2 + 2 + 2 * 3) * 4 + 8
    # none: the atomic mode, heads above 128 (two passes without atomics), bad arguments
    assert skl.streamkl_bwd_workspace_bytes(1, 32, 32, 32, 4096, 128, 128, deterministic=False) == 0
    assert skl.streamkl_bwd_workspace_bytes(1, 8, 8, 8, 4096, 256, 256) == 0
    assert skl.streamkl_bwd_workspace_bytes(1, 6, 4, 4, 4096, 64, 64) == 0   # 4 does not divide 6
    assert skl.streamkl_bwd_workspace_bytes(1, 4, 4, 4, 4096, 72, 64) == 0   # not a multiple of 16
    assert skl.streamkl_bwd_workspace_bytes(1, 4, 4, 4, 4096, 64, 64, mode=2) == 0
