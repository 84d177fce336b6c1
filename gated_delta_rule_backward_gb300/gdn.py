"""ctypes binding of libgdn (include/gdn.h): argument marshalling only.

Every step of the gated delta rule runs in the CUDA kernels behind the C ABI; this
module builds the parameter struct from tensors, allocates outputs with PyTorch (device
memory and streams are all PyTorch is used for) and raises on a non-OK status.  There is
no fallback: importing this module fails loudly when libgdn.so has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libgdn.so not found at {LIB_PATH}; build it first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

GDN_OK = 0
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIAS",
          4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_CUDA", 6: "GDN_ERR_TIMEOUT"}
GATE_SCALAR, GATE_KDA = 0, 1
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2

# Every symbol include/gdn.h declares.
EXPORTS = ["gdn_checkpoint_interval", "gdn_num_checkpoints", "gdn_ckpt_elems", "gdn_forward",
           "gdn_packed_grad_elems", "gdn_packed_grad_offsets", "gdn_backward_workspace_bytes",
           "gdn_backward", "gdn_status_str", "gdn_last_error", "gdn_forward_launches",
           "gdn_backward_launches", "gdn_set_timing_events", "gdn_backward_noalloc",
           "gdn_forward_workspace_bytes", "gdn_device_status", "gdn_selftest_wait_timeout",
           "gdn_timing_stages"]


class GdnParams(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int64), ("T", ctypes.c_int64), ("H_k", ctypes.c_int64),
        ("H_v", ctypes.c_int64), ("S_k", ctypes.c_int64), ("S_v", ctypes.c_int64),
        ("gate", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("C", ctypes.c_int64),
        ("scale", ctypes.c_float), ("seq_rep", ctypes.c_int32),
        ("q_s", ctypes.c_int64 * 3), ("k_s", ctypes.c_int64 * 3),
        ("v_s", ctypes.c_int64 * 3), ("gy_s", ctypes.c_int64 * 3),
    ]


_P = ctypes.POINTER(GdnParams)
_vp = ctypes.c_void_p
_lib.gdn_checkpoint_interval.argtypes = [_P]
_lib.gdn_checkpoint_interval.restype = ctypes.c_int64
_lib.gdn_num_checkpoints.argtypes = [_P]
_lib.gdn_num_checkpoints.restype = ctypes.c_int64
_lib.gdn_ckpt_elems.argtypes = [_P]
_lib.gdn_ckpt_elems.restype = ctypes.c_size_t
_lib.gdn_packed_grad_elems.argtypes = [_P]
_lib.gdn_packed_grad_elems.restype = ctypes.c_size_t
_lib.gdn_packed_grad_offsets.argtypes = [_P, ctypes.POINTER(ctypes.c_size_t)]
_lib.gdn_packed_grad_offsets.restype = None
_lib.gdn_backward_workspace_bytes.argtypes = [_P]
_lib.gdn_backward_workspace_bytes.restype = ctypes.c_size_t
_lib.gdn_forward.argtypes = [_P] + [_vp] * 10 + [ctypes.c_size_t, _vp]
_lib.gdn_forward.restype = ctypes.c_int
_lib.gdn_backward.argtypes = [_P] + [_vp] * 10 + [ctypes.c_size_t, _vp]
_lib.gdn_backward.restype = ctypes.c_int
_lib.gdn_status_str.argtypes = [ctypes.c_int]
_lib.gdn_status_str.restype = ctypes.c_char_p
_lib.gdn_last_error.argtypes = []
_lib.gdn_last_error.restype = ctypes.c_char_p
_lib.gdn_forward_launches.argtypes = [_P]
_lib.gdn_forward_launches.restype = ctypes.c_int
_lib.gdn_backward_launches.argtypes = [_P]
_lib.gdn_backward_launches.restype = ctypes.c_int
_lib.gdn_backward_noalloc.argtypes = [_P] + [_vp] * 10
_lib.gdn_backward_noalloc.restype = ctypes.c_int
_lib.gdn_set_timing_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
_lib.gdn_set_timing_events.restype = None
_lib.gdn_forward_workspace_bytes.argtypes = [_P]
_lib.gdn_forward_workspace_bytes.restype = ctypes.c_size_t
_lib.gdn_timing_stages.argtypes = [_P, ctypes.c_int]
_lib.gdn_timing_stages.restype = ctypes.c_int
_lib.gdn_device_status.argtypes = [_vp]
_lib.gdn_device_status.restype = ctypes.c_int
_lib.gdn_selftest_wait_timeout.argtypes = [_vp]
_lib.gdn_selftest_wait_timeout.restype = ctypes.c_int


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = _lib.gdn_last_error().decode()
        super().__init__(f"{what}: {STATUS.get(status, status)}: {detail}")


def library():
    return _lib


def make_params(N, T, H_k, H_v, S, kda, C=None, scale=None, q_s=None, k_s=None, v_s=None,
                gy_s=None, in_dtype=DTYPE_F32, S_v=None, seq_rep=1) -> GdnParams:
    """Parameter struct; S is the key head size S_k, S_v the value head size (default S);
    N counts the value sequences and q, k hold N / seq_rep; strides default to the
    contiguous [N,T,H,S] layouts."""
    SV = S if S_v is None else int(S_v)
    p = GdnParams()
    p.n_seq, p.T, p.H_k, p.H_v, p.S_k, p.S_v = N, T, H_k, H_v, S, SV
    p.gate = GATE_KDA if kda else GATE_SCALAR
    p.in_dtype, p.seq_rep = int(in_dtype), int(seq_rep)
    p.C = 0 if C is None else int(C)
    p.scale = (1.0 / math.sqrt(S)) if scale is None else float(scale)
    p.q_s[:] = q_s or (T * H_k * S, H_k * S, S)  # per q/k sequence
    p.k_s[:] = k_s or (T * H_k * S, H_k * S, S)
    p.v_s[:] = v_s or (T * H_v * SV, H_v * SV, SV)
    p.gy_s[:] = gy_s or (T * H_v * SV, H_v * SV, SV)
    return p


def strides3(t):
    """Element strides of a [N,T,H,S] tensor view (its last dim must be contiguous)."""
    if t.numel() == 0:  # empty views carry no meaningful strides
        N, T, H, S = t.shape
        return (T * H * S, H * S, S)
    if t.stride(-1) != 1:
        raise ValueError("the head dimension must be contiguous")
    return tuple(int(s) for s in t.stride()[:3])


def input_dtype(t) -> int:
    """gdn_dtype_t of an input tensor: fp32, bf16 or fp16."""
    import torch
    code = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}.get(t.dtype)
    if code is None:
        raise TypeError(f"inputs must be float32, bfloat16 or float16, not {t.dtype}")
    return code


def params_for(q, k, v, g, gy=None, C=None, scale=None) -> GdnParams:
    """Parameters for these input tensors: sizes, strides and their storage type (q, k, v,
    g and gy must all have that type).  q, k may hold fewer sequences than v (a divisor of
    its count): the sequence broadcast."""
    Nq, T, H_k, S = q.shape
    N, H_v = v.shape[0], v.shape[2]
    if Nq == 0 or N % Nq:
        raise ValueError("v's sequences must be a multiple of q's")
    kda = g.dim() == 4
    dt = input_dtype(q)
    for t in (k, v, g) + ((gy,) if gy is not None else ()):
        if input_dtype(t) != dt:
            raise TypeError("q, k, v, g (and gy) must share one storage type")
    return make_params(N, T, H_k, H_v, S, kda, C=C, scale=scale, q_s=strides3(q),
                       k_s=strides3(k), v_s=strides3(v),
                       gy_s=strides3(gy) if gy is not None else None, in_dtype=dt,
                       S_v=v.shape[3], seq_rep=N // Nq)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def num_checkpoints(p: GdnParams) -> int:
    return int(_lib.gdn_num_checkpoints(ctypes.byref(p)))


def checkpoint_interval(p: GdnParams) -> int:
    return int(_lib.gdn_checkpoint_interval(ctypes.byref(p)))


def packed_grad_elems(p: GdnParams) -> int:
    return int(_lib.gdn_packed_grad_elems(ctypes.byref(p)))


def packed_grad_offsets(p: GdnParams):
    off = (ctypes.c_size_t * 6)()
    _lib.gdn_packed_grad_offsets(ctypes.byref(p), off)
    return [int(x) for x in off]


def backward_workspace_bytes(p: GdnParams) -> int:
    return int(_lib.gdn_backward_workspace_bytes(ctypes.byref(p)))


def launches(p: GdnParams):
    """(forward kernels, backward kernels) one call of each enqueues."""
    return (int(_lib.gdn_forward_launches(ctypes.byref(p))),
            int(_lib.gdn_backward_launches(ctypes.byref(p))))


def timing_stages(p: GdnParams):
    """(forward stages, backward stages) that set_timing_events brackets."""
    return (int(_lib.gdn_timing_stages(ctypes.byref(p), 0)),
            int(_lib.gdn_timing_stages(ctypes.byref(p), 1)))


_EVENTS = None


def set_timing_events(events):
    """A list of recorded torch.cuda.Event(enable_timing=True) objects, or None.  Each
    gdn_forward / gdn_backward call then records events[0] before its first stage and
    events[i] after its i-th stage (see timing_stages)."""
    global _EVENTS
    if events is None:
        _EVENTS = None
        _lib.gdn_set_timing_events(None, 0)
        return
    _EVENTS = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _lib.gdn_set_timing_events(_EVENTS, len(events))


def forward_workspace_bytes(p: GdnParams) -> int:
    return int(_lib.gdn_forward_workspace_bytes(ctypes.byref(p)))


def gdn_forward(p: GdnParams, q, k, v, g, beta, state0, y, state_T, ckpt, workspace=None,
                stream=None):
    """Raw C-ABI call on caller-provided tensors (all on the current CUDA device)."""
    st = _lib.gdn_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                          _ptr(state0), _ptr(y), _ptr(state_T), _ptr(ckpt), _ptr(workspace),
                          ctypes.c_size_t(0 if workspace is None else workspace.numel()),
                          _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_forward")


def gdn_backward(p: GdnParams, q, k, v, g, beta, ckpt, gy, dstate_T, packed, workspace,
                 stream=None):
    st = _lib.gdn_backward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(ckpt), _ptr(gy), _ptr(dstate_T), _ptr(packed),
                           _ptr(workspace),
                           ctypes.c_size_t(0 if workspace is None else workspace.numel()),
                           _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_backward")


def gdn_backward_noalloc(p: GdnParams, q, k, v, g, beta, ckpt, gy, dstate_T, packed,
                         stream=None):
    """gdn_backward with the library's fixed device scratch instead of a workspace."""
    st = _lib.gdn_backward_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(ckpt), _ptr(gy), _ptr(dstate_T),
                                   _ptr(packed), _stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_backward_noalloc")


def device_status(stream=None) -> int:
    """Synchronise `stream` and return (and clear) the device status: GDN_OK, or
    6 (GDN_ERR_TIMEOUT) when a tensor-core kernel's bounded wait gave up."""
    return int(_lib.gdn_device_status(_stream_handle(stream)))


def selftest_wait_timeout(stream=None):
    """Enqueue the kernel whose bounded wait gives up (test of the timeout path)."""
    st = _lib.gdn_selftest_wait_timeout(_stream_handle(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_selftest_wait_timeout")


def forward(q, k, v, g, beta, state0, C=None, scale=None, stream=None):
    """Allocate y, state_T, ckpt and run gdn_forward.  Returns (y, state_T, ckpt, params)."""
    import torch
    p = params_for(q, k, v, g, C=C, scale=scale)
    _, T, H_k, S = q.shape
    N, H_v, SV = v.shape[0], v.shape[2], v.shape[3]
    dev = q.device
    y = torch.empty((N, T, H_v, SV), dtype=torch.float32, device=dev)
    state_T = torch.empty((N, H_v, SV, S), dtype=torch.float32, device=dev)
    ckpt = torch.empty((N, H_v, num_checkpoints(p), SV, S), dtype=torch.float32, device=dev)
    nws = forward_workspace_bytes(p)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
    gdn_forward(p, q, k, v, g, beta, state0, y, state_T, ckpt, ws, stream)
    return y, state_T, ckpt, p


def split_packed(p: GdnParams, packed):
    """Views of the six regions of a packed gradient buffer."""
    N, T, H_k, H_v, S, SV = p.n_seq, p.T, p.H_k, p.H_v, p.S_k, p.S_v
    Nq = N // max(1, p.seq_rep)
    off = packed_grad_offsets(p) + [packed_grad_elems(p)]
    shapes = [(Nq, T, H_k, S), (Nq, T, H_k, S), (N, T, H_v, SV),
              (N, T, H_v, S) if p.gate == GATE_KDA else (N, T, H_v), (N, T, H_v),
              (N, H_v, SV, S)]
    names = ["dq", "dk", "dv", "dg", "dbeta", "dstate0"]
    return {nm: packed[off[i]:off[i + 1]].view(shapes[i]) for i, nm in enumerate(names)}


def backward(p: GdnParams, q, k, v, g, beta, ckpt, gy, dstate_T=None, stream=None,
             workspace=None):
    """Allocate the packed buffer (and workspace unless given) and run gdn_backward.

    Returns (packed, views) where views maps dq, dk, dv, dg, dbeta, dstate0 to regions."""
    import torch
    dev = q.device
    if tuple(int(s) for s in p.gy_s) != strides3(gy):
        p.gy_s[:] = strides3(gy)
    packed = torch.empty(packed_grad_elems(p), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(backward_workspace_bytes(p), 1), dtype=torch.uint8,
                                device=dev)
    gdn_backward(p, q, k, v, g, beta, ckpt, gy, dstate_T, packed, workspace, stream)
    return packed, split_packed(p, packed)
