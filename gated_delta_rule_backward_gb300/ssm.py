"""ctypes binding of the selective scan's C ABI (include/ssm.h) in libgdn.so.

Argument marshalling only: every step of the scan and its reverse walk runs in the
library's kernels.  Tensors are torch tensors on the device (their data pointers are
passed through); the functions check shapes and dtypes and raise on a non-zero status.
"""
from __future__ import annotations

import ctypes

import torch

from . import gdn

_lib = gdn._lib

# Every symbol include/ssm.h declares.
EXPORTS = ["ssm_checkpoint_interval", "ssm_num_checkpoints", "ssm_packed_out_elems", "ssm_packed_grad_elems",
           "ssm_backward_workspace_bytes", "ssm_supported", "ssm_chunked", "ssm_form", "ssm_forward_launches",
           "ssm_backward_launches", "ssm_forward", "ssm_backward"]


class SsmParams(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("P", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("G", ctypes.c_int64),
        ("a_per_state", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("reserved1", ctypes.c_int32),
    ]


_PP = ctypes.POINTER(SsmParams)
_V = ctypes.c_void_p
_lib.ssm_checkpoint_interval.argtypes = [_PP]
_lib.ssm_checkpoint_interval.restype = ctypes.c_int64
_lib.ssm_num_checkpoints.argtypes = [_PP]
_lib.ssm_num_checkpoints.restype = ctypes.c_int64
_lib.ssm_packed_out_elems.argtypes = [_PP]
_lib.ssm_packed_out_elems.restype = ctypes.c_size_t
_lib.ssm_packed_grad_elems.argtypes = [_PP]
_lib.ssm_packed_grad_elems.restype = ctypes.c_size_t
_lib.ssm_backward_workspace_bytes.argtypes = [_PP]
_lib.ssm_backward_workspace_bytes.restype = ctypes.c_size_t
_lib.ssm_supported.argtypes = [_PP]
_lib.ssm_supported.restype = ctypes.c_int
_lib.ssm_chunked.argtypes = [_PP]
_lib.ssm_chunked.restype = ctypes.c_int
_lib.ssm_form.argtypes = [_PP]
_lib.ssm_form.restype = ctypes.c_int
_lib.ssm_forward_launches.argtypes = [_PP]
_lib.ssm_forward_launches.restype = ctypes.c_int
_lib.ssm_backward_launches.argtypes = [_PP]
_lib.ssm_backward_launches.restype = ctypes.c_int
_lib.ssm_forward.argtypes = [_PP] + [_V] * 9
_lib.ssm_forward.restype = ctypes.c_int
_lib.ssm_backward.argtypes = [_PP] + [_V] * 9 + [ctypes.c_size_t, _V]
_lib.ssm_backward.restype = ctypes.c_int


def make_params(N, T, H, P, S, G=1, mamba1=False, K=0):
    return SsmParams(int(N), int(T), int(H), int(P), int(S), int(G), 1 if mamba1 else 0, int(K), 0, 0)


def params_for(x, A, B, K=0):
    """Sizes from x [N,T,H,P], A ([H] or [H,S]) and B [N,T,G,S]."""
    N, T, H, P = x.shape
    G, S = B.shape[2], B.shape[3]
    return make_params(N, T, H, P, S, G, mamba1=(A.dim() == 2), K=K)


def checkpoint_interval(p) -> int:
    return int(_lib.ssm_checkpoint_interval(ctypes.byref(p)))


def num_checkpoints(p) -> int:
    return int(_lib.ssm_num_checkpoints(ctypes.byref(p)))


def packed_out_elems(p) -> int:
    return int(_lib.ssm_packed_out_elems(ctypes.byref(p)))


def packed_grad_elems(p) -> int:
    return int(_lib.ssm_packed_grad_elems(ctypes.byref(p)))


def backward_workspace_bytes(p) -> int:
    return int(_lib.ssm_backward_workspace_bytes(ctypes.byref(p)))


def supported(p) -> int:
    return int(_lib.ssm_supported(ctypes.byref(p)))


def chunked(p) -> bool:
    """True when these sizes run the chunked form."""
    return bool(_lib.ssm_chunked(ctypes.byref(p)))


FORMS = {0: "token-serial", 1: "chunked", 2: "segmented"}


def form(p) -> str:
    """The form these sizes run: "token-serial", "chunked" or "segmented" (a decay per state)."""
    f = int(_lib.ssm_form(ctypes.byref(p)))
    if f < 0:
        raise gdn.GdnError(int(_lib.ssm_supported(ctypes.byref(p))), "ssm_form")
    return FORMS[f]


def launches(p):
    """(kernels a forward call launches, kernels a backward call launches)."""
    return int(_lib.ssm_forward_launches(ctypes.byref(p))), int(_lib.ssm_backward_launches(ctypes.byref(p)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.dtype != torch.float32 and t.dtype != torch.uint8:
        raise TypeError("fp32 tensors expected")
    if t.numel() and not t.is_contiguous():
        raise ValueError("dense (contiguous) tensors expected")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc, what):
    if rc != 0:
        raise gdn.GdnError(rc, what)


def ssm_forward(p, s0, x, dt, A, B, C, out_packed, ckpt, stream=None):
    rc = _lib.ssm_forward(ctypes.byref(p), _ptr(s0), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                          _ptr(out_packed), _ptr(ckpt), _stream(stream))
    _check(rc, "ssm_forward")
    return rc


def ssm_backward(p, x, dt, A, B, C, ckpt, grad_in, grad_out, ws, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = _lib.ssm_backward(ctypes.byref(p), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(ckpt),
                           _ptr(grad_in), _ptr(grad_out), _ptr(ws), nbytes, _stream(stream))
    _check(rc, "ssm_backward")
    return rc


def split_out(p, out_packed):
    """Views (y [N,T,H,P], s_T [N,H,P,S]) of the packed forward output."""
    n_x = p.N * p.T * p.H * p.P
    return (out_packed[:n_x].view(p.N, p.T, p.H, p.P), out_packed[n_x:].view(p.N, p.H, p.P, p.S))


def split_grads(p, grad_out):
    """Views (d_s, d_x, d_dt, d_B, d_C) of the packed backward output."""
    n_s, n_x, n_dt, n_bc = p.N * p.H * p.P * p.S, p.N * p.T * p.H * p.P, p.N * p.T * p.H, p.N * p.T * p.G * p.S
    o = 0
    out = []
    for n, shape in ((n_s, (p.N, p.H, p.P, p.S)), (n_x, (p.N, p.T, p.H, p.P)), (n_dt, (p.N, p.T, p.H)),
                     (n_bc, (p.N, p.T, p.G, p.S)), (n_bc, (p.N, p.T, p.G, p.S))):
        out.append(grad_out[o:o + n].view(*shape))
        o += n
    return tuple(out)


def pack_grad_in(p, dy, ds_T):
    """The packed cotangent [dy | ds_T] (a new device tensor)."""
    return torch.cat([dy.reshape(-1), ds_T.reshape(-1)]).contiguous()
