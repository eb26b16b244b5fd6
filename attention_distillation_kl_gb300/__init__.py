"""Python binding for libstreamkl (fused attention KL divergence, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libstreamkl.so``.  PyTorch supplies device memory and streams.
There is no CPU fallback: if the library is missing or the device is not a
GB300 (sm_103a), calls raise.

Functions mirror the C ABI in ``include/streamkl.h`` and keep its names.
"""

import ctypes
import os

import torch

__all__ = [
    "StreamKLError", "lib", "library_path",
    "streamkl_fwd", "streamkl_fwd_splitk", "streamkl_fwd_splitk_workspace_bytes",
    "streamkl_suggest_splits", "streamkl_fwd_splitk_noalloc", "streamkl_bwd", "streamkl_status_string",
    "streamkl_fwd_scaled", "streamkl_fwd_splitk_scaled", "streamkl_bwd_scaled",
    "streamkl_fwd_gqa", "streamkl_fwd_splitk_gqa", "streamkl_bwd_gqa", "streamkl_bwd_both",
    "streamkl_bwd_workspace_bytes", "streamkl_bwd_gqa_ws",
    "status_string", "STREAMKL_STATIC_WORKSPACE_BYTES",
    "streamkl_get_device_status", "streamkl_probe_ex2", "streamkl_selftest_wait_timeout",
    "streamkl_selftest_turn_timeout",
    "STREAMKL_OK", "STREAMKL_INVALID_ARG", "STREAMKL_UNSUPPORTED", "STREAMKL_CUDA_ERROR",
    "STREAMKL_DEVICE_TIMEOUT", "STREAMKL_DEBUG_BOUNDS", "STREAMKL_GRAD_P2", "STREAMKL_GRAD_P1",
]

STREAMKL_OK = 0
STREAMKL_INVALID_ARG = 1
STREAMKL_UNSUPPORTED = 2
STREAMKL_CUDA_ERROR = 3
STREAMKL_DEVICE_TIMEOUT = 4
STREAMKL_DEBUG_BOUNDS = 5
STREAMKL_GRAD_P2 = 0
STREAMKL_GRAD_P1 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libstreamkl.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "streamkl_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "streamkl_fwd_splitk": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ,
                                 _P, _P, _P, _P]),
    "streamkl_fwd_splitk_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "streamkl_fwd_splitk_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                                         _P, _P, _P, _P]),
    "streamkl_suggest_splits": (_I, [_I, _I, _I, _I, _I]),
    "streamkl_bwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _I, _I,
                          _P, _P, _P]),
    "streamkl_fwd_scaled": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P]),
    "streamkl_fwd_splitk_scaled": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _I, _I, _P, _SZ,
                                        _P, _P, _P, _P]),
    "streamkl_bwd_scaled": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P, _I,
                                 _I, _P, _P, _P]),
    "streamkl_fwd_gqa": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P]),
    "streamkl_fwd_splitk_gqa": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I, _I, _P, _SZ,
                                     _P, _P, _P, _P]),
    "streamkl_bwd_gqa": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P, _I,
                              _I, _P, _P, _P]),
    "streamkl_bwd_both": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P, _I,
                               _P, _P, _P, _P, _P]),
    "streamkl_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "streamkl_bwd_gqa_ws": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _I, _P, _P, _P, _P, _I,
                                 _I, _P, _P, _P, _SZ, _P]),
    "streamkl_status_string": (ctypes.c_char_p, [_I]),
    "streamkl_get_device_status": (_I, []),
    "streamkl_probe_ex2": (_I, [_P, _I, _I, _P]),
    "streamkl_selftest_wait_timeout": (_I, [_I, _P]),
    "streamkl_selftest_turn_timeout": (_I, [_I, _P, _P]),
}


class StreamKLError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


def lib():
    """The loaded ``libstreamkl.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status):
    return lib().streamkl_status_string(int(status)).decode()


streamkl_status_string = status_string


def _check(status, where):
    if status != STREAMKL_OK:
        raise StreamKLError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dims(q1, k1, q2, k2):
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA bf16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, NQ, d1 = q1.shape
    NK = k1.shape[2]
    d2 = q2.shape[3]
    if tuple(k1.shape) != (B, H, NK, d1) or tuple(q2.shape) != (B, H, NQ, d2) or \
            tuple(k2.shape) != (B, H, NK, d2):
        raise ValueError("inconsistent shapes: want q1 [B,H,NQ,d1], k1 [B,H,NK,d1], "
                         "q2 [B,H,NQ,d2], k2 [B,H,NK,d2]")
    return B, H, NQ, NK, d1, d2


def _dims_gqa(q1, k1, q2, k2):
    """Like _dims, with k1 and k2 allowed their own head counts (grouped key
    heads; the library checks that each divides the query head count)."""
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA bf16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, NQ, d1 = q1.shape
    HK1, NK = k1.shape[1], k1.shape[2]
    HK2, d2 = k2.shape[1], q2.shape[3]
    if tuple(k1.shape) != (B, HK1, NK, d1) or tuple(q2.shape) != (B, H, NQ, d2) or \
            tuple(k2.shape) != (B, HK2, NK, d2):
        raise ValueError("inconsistent shapes: want q1 [B,H,NQ,d1], k1 [B,HK1,NK,d1], "
                         "q2 [B,H,NQ,d2], k2 [B,HK2,NK,d2]")
    return B, H, HK1, HK2, NQ, NK, d1, d2


def _out(t, shape, device, name):
    if t is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() \
            or t.device != device:
        raise ValueError(f"{name} must be a contiguous fp32 tensor of shape {tuple(shape)} on {device}")
    return t


def streamkl_fwd(q1, k1, q2, k2, scale, causal, kl=None, lse1=None, lse2=None, stream=None):
    """Per-row KL(P1 || P2), LSE1, LSE2 (fp32 [B, H, NQ]); see include/streamkl.h."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                              B, H, NQ, NK, d1, d2, float(scale), int(bool(causal)),
                              kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd")
    return kl, lse1, lse2


def streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits):
    return int(lib().streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits))


def streamkl_suggest_splits(B, H, NQ, NK, causal):
    return int(lib().streamkl_suggest_splits(B, H, NQ, NK, int(bool(causal))))


def streamkl_fwd_splitk(q1, k1, q2, k2, scale, causal, num_splits, workspace=None,
                        kl=None, lse1=None, lse2=None, stream=None):
    """Key-split forward plus merge; ``workspace`` is a caller-owned byte buffer."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    need = streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_splitk(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                     B, H, NQ, NK, d1, d2, float(scale), int(bool(causal)),
                                     int(num_splits), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_splitk")
    return kl, lse1, lse2


# Size in bytes of the library's fixed key-split workspace (see the header).
STREAMKL_STATIC_WORKSPACE_BYTES = 32 << 20


def streamkl_fwd_splitk_noalloc(q1, k1, q2, k2, scale, causal, num_splits, kl=None, lse1=None,
                                lse2=None, stream=None):
    """Key-split forward that allocates no device memory inside the library.

    For callers that cannot provide scratch memory (for example code running
    under an allocator that owns all device memory): the per-split partials
    live in a fixed array of STREAMKL_STATIC_WORKSPACE_BYTES inside the
    library.  Calls overlapping on the GPU race on that array; the first call
    on a device should precede any stream capture there.  Pass preallocated
    ``kl``/``lse1``/``lse2`` to keep this wrapper allocation-free as well.
    """
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_splitk_noalloc(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                             B, H, NQ, NK, d1, d2, float(scale), int(bool(causal)),
                                             int(num_splits), kl.data_ptr(), lse1.data_ptr(),
                                             lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_splitk_noalloc")
    return kl, lse1, lse2


def streamkl_bwd(q1, k1, q2, k2, scale, causal, kl, lse1, lse2, dkl, mode=STREAMKL_GRAD_P2,
                 deterministic=False, dq=None, dk=None, stream=None):
    """(dQ, dK) fp32 for the side ``mode`` selects; see include/streamkl.h."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    dg = d2 if mode == STREAMKL_GRAD_P2 else d1
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        _out(t, (B, H, NQ), q1.device, name)
    dq = _out(dq, (B, H, NQ, dg), q1.device, "dq")
    dk = _out(dk, (B, H, NK, dg), q1.device, "dk")
    _check(lib().streamkl_bwd(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                              B, H, NQ, NK, d1, d2, float(scale), int(bool(causal)),
                              kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), dkl.data_ptr(),
                              int(mode), int(bool(deterministic)), dq.data_ptr(), dk.data_ptr(),
                              _stream(stream)),
           "streamkl_bwd")
    return dq, dk


def streamkl_fwd_scaled(q1, k1, q2, k2, scale1, scale2, causal, kl=None, lse1=None, lse2=None, stream=None):
    """streamkl_fwd with S1 = scale1 Q1 K1^T and S2 = scale2 Q2 K2^T."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_scaled(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                     B, H, NQ, NK, d1, d2, float(scale1), float(scale2), int(bool(causal)),
                                     kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_scaled")
    return kl, lse1, lse2


def streamkl_fwd_splitk_scaled(q1, k1, q2, k2, scale1, scale2, causal, num_splits, workspace=None,
                               kl=None, lse1=None, lse2=None, stream=None):
    """streamkl_fwd_splitk with a softmax scale per side."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    need = streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_splitk_scaled(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                            B, H, NQ, NK, d1, d2, float(scale1), float(scale2),
                                            int(bool(causal)), int(num_splits), workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_splitk_scaled")
    return kl, lse1, lse2


def streamkl_bwd_scaled(q1, k1, q2, k2, scale1, scale2, causal, kl, lse1, lse2, dkl, mode=STREAMKL_GRAD_P2,
                        deterministic=False, dq=None, dk=None, stream=None):
    """streamkl_bwd with a softmax scale per side (kl/lse from streamkl_fwd_scaled)."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    dg = d2 if mode == STREAMKL_GRAD_P2 else d1
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        _out(t, (B, H, NQ), q1.device, name)
    dq = _out(dq, (B, H, NQ, dg), q1.device, "dq")
    dk = _out(dk, (B, H, NK, dg), q1.device, "dk")
    _check(lib().streamkl_bwd_scaled(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                     B, H, NQ, NK, d1, d2, float(scale1), float(scale2), int(bool(causal)),
                                     kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), dkl.data_ptr(),
                                     int(mode), int(bool(deterministic)), dq.data_ptr(), dk.data_ptr(),
                                     _stream(stream)),
           "streamkl_bwd_scaled")
    return dq, dk


def streamkl_fwd_gqa(q1, k1, q2, k2, scale1, scale2, causal, kl=None, lse1=None, lse2=None, stream=None):
    """streamkl_fwd_scaled with grouped key heads: k1 [B, HK1, NK, d1] and
    k2 [B, HK2, NK, d2], query head h reading key head h // (H // HK)."""
    B, H, HK1, HK2, NQ, NK, d1, d2 = _dims_gqa(q1, k1, q2, k2)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_gqa(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                  B, H, HK1, HK2, NQ, NK, d1, d2, float(scale1), float(scale2), int(bool(causal)),
                                  kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_gqa")
    return kl, lse1, lse2


def streamkl_fwd_splitk_gqa(q1, k1, q2, k2, scale1, scale2, causal, num_splits, workspace=None,
                            kl=None, lse1=None, lse2=None, stream=None):
    """streamkl_fwd_splitk_scaled with grouped key heads."""
    B, H, HK1, HK2, NQ, NK, d1, d2 = _dims_gqa(q1, k1, q2, k2)
    need = streamkl_fwd_splitk_workspace_bytes(B, H, NQ, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    kl = _out(kl, (B, H, NQ), q1.device, "kl")
    lse1 = _out(lse1, (B, H, NQ), q1.device, "lse1")
    lse2 = _out(lse2, (B, H, NQ), q1.device, "lse2")
    _check(lib().streamkl_fwd_splitk_gqa(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                         B, H, HK1, HK2, NQ, NK, d1, d2, float(scale1), float(scale2),
                                         int(bool(causal)), int(num_splits), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), _stream(stream)),
           "streamkl_fwd_splitk_gqa")
    return kl, lse1, lse2


def streamkl_bwd_gqa(q1, k1, q2, k2, scale1, scale2, causal, kl, lse1, lse2, dkl, mode=STREAMKL_GRAD_P2,
                     deterministic=False, dq=None, dk=None, stream=None):
    """streamkl_bwd_scaled with grouped key heads: dq [B, H, NQ, dg] per query
    head, dk [B, HK_g, NK, dg] per key head of the gradient side (summed over
    the query heads that read it)."""
    B, H, HK1, HK2, NQ, NK, d1, d2 = _dims_gqa(q1, k1, q2, k2)
    dg, hkg = (d2, HK2) if mode == STREAMKL_GRAD_P2 else (d1, HK1)
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        _out(t, (B, H, NQ), q1.device, name)
    dq = _out(dq, (B, H, NQ, dg), q1.device, "dq")
    dk = _out(dk, (B, hkg, NK, dg), q1.device, "dk")
    _check(lib().streamkl_bwd_gqa(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                  B, H, HK1, HK2, NQ, NK, d1, d2, float(scale1), float(scale2), int(bool(causal)),
                                  kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), dkl.data_ptr(),
                                  int(mode), int(bool(deterministic)), dq.data_ptr(), dk.data_ptr(),
                                  _stream(stream)),
           "streamkl_bwd_gqa")
    return dq, dk


def streamkl_bwd_workspace_bytes(B, H, HK1, HK2, NK, d1, d2, mode=STREAMKL_GRAD_P2, deterministic=True):
    """Scratch bytes streamkl_bwd_gqa_ws needs (see the header)."""
    return int(lib().streamkl_bwd_workspace_bytes(B, H, HK1, HK2, NK, d1, d2, int(mode), int(bool(deterministic))))


def streamkl_bwd_gqa_ws(q1, k1, q2, k2, scale1, scale2, causal, kl, lse1, lse2, dkl, workspace,
                        mode=STREAMKL_GRAD_P2, deterministic=True, dq=None, dk=None, stream=None):
    """streamkl_bwd_gqa with the deterministic mode's scratch in `workspace`
    (a CUDA tensor of at least streamkl_bwd_workspace_bytes bytes, or None
    when that is 0)."""
    B, H, HK1, HK2, NQ, NK, d1, d2 = _dims_gqa(q1, k1, q2, k2)
    dg, hkg = (d2, HK2) if mode == STREAMKL_GRAD_P2 else (d1, HK1)
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        _out(t, (B, H, NQ), q1.device, name)
    dq = _out(dq, (B, H, NQ, dg), q1.device, "dq")
    dk = _out(dk, (B, hkg, NK, dg), q1.device, "dk")
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().streamkl_bwd_gqa_ws(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                     B, H, HK1, HK2, NQ, NK, d1, d2, float(scale1), float(scale2),
                                     int(bool(causal)), kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(),
                                     dkl.data_ptr(), int(mode), int(bool(deterministic)), dq.data_ptr(),
                                     dk.data_ptr(), ws_ptr, ws_bytes, _stream(stream)),
           "streamkl_bwd_gqa_ws")
    return dq, dk


def streamkl_bwd_both(q1, k1, q2, k2, scale1, scale2, causal, kl, lse1, lse2, dkl, deterministic=False,
                      dq1=None, dk1=None, dq2=None, dk2=None, stream=None):
    """(dQ1, dK1, dQ2, dK2) fp32: the gradients of sum(dkl * KL) on both sides."""
    B, H, NQ, NK, d1, d2 = _dims(q1, k1, q2, k2)
    for name, t in (("kl", kl), ("lse1", lse1), ("lse2", lse2), ("dkl", dkl)):
        _out(t, (B, H, NQ), q1.device, name)
    dq1 = _out(dq1, (B, H, NQ, d1), q1.device, "dq1")
    dk1 = _out(dk1, (B, H, NK, d1), q1.device, "dk1")
    dq2 = _out(dq2, (B, H, NQ, d2), q1.device, "dq2")
    dk2 = _out(dk2, (B, H, NK, d2), q1.device, "dk2")
    _check(lib().streamkl_bwd_both(q1.data_ptr(), k1.data_ptr(), q2.data_ptr(), k2.data_ptr(),
                                   B, H, NQ, NK, d1, d2, float(scale1), float(scale2), int(bool(causal)),
                                   kl.data_ptr(), lse1.data_ptr(), lse2.data_ptr(), dkl.data_ptr(),
                                   int(bool(deterministic)), dq1.data_ptr(), dk1.data_ptr(), dq2.data_ptr(),
                                   dk2.data_ptr(), _stream(stream)),
           "streamkl_bwd_both")
    return dq1, dk1, dq2, dk2


def streamkl_get_device_status():
    return int(lib().streamkl_get_device_status())


def streamkl_probe_ex2(out, blocks, iters, stream=None):
    _check(lib().streamkl_probe_ex2(out.data_ptr(), int(blocks), int(iters), _stream(stream)),
           "streamkl_probe_ex2")


def streamkl_selftest_wait_timeout(limit_us, stream=None):
    """Runs a kernel whose barrier wait must time out (see the header)."""
    _check(lib().streamkl_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "streamkl_selftest_wait_timeout")


def streamkl_selftest_turn_timeout(limit_us, words, stream=None):
    """Runs a kernel whose turn wait must time out (see the header); `words`
    is a CUDA int32 tensor of at least 5 elements."""
    _check(lib().streamkl_selftest_turn_timeout(int(limit_us), words.data_ptr(), _stream(stream)),
           "streamkl_selftest_turn_timeout")
