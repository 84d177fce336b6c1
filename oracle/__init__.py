"""Float64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and
``--impl reference``) may import this package.  The product path (``libgdn`` and its
Python binding) never calls it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, float64, OpenMP over
(sequence, value head)); this module compiles it with gcc and marshals numpy arrays.
What it computes, and which passage each step follows, is stated in the C file's
header.  Every function here is argument handling only.

Parity status: every output (y, state_T, checkpoints, dq, dk, dv, dg, dbeta, dstate0)
is pinned by the tests in ``tests/test_oracle_pins.py`` (finite differences, closed
forms, invariants, exact symbolic gradients, planted-defect kill list).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_DEFAULT = os.path.join(_HERE, "libgdn_oracle.so")


class Dims(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("H_k", ctypes.c_int64),
        ("H_v", ctypes.c_int64),
        ("S_k", ctypes.c_int64),
        ("S_v", ctypes.c_int64),
        ("kda", ctypes.c_int64),
        ("C", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("rep", ctypes.c_int64),
    ]


def build(out_path: str = _LIB_DEFAULT, mutation: int = 0, openmp: bool = True) -> str:
    """Compile the oracle into a shared library (gcc, -O2, no fast-math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math"]
    if openmp:
        cmd.append("-fopenmp")
    if mutation:
        cmd.append(f"-DGDN_ORACLE_MUTATION={int(mutation)}")
    cmd += [_SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


_DP = ctypes.POINTER(ctypes.c_double)


def _bind(lib):
    lib.gdn_oracle_forward.argtypes = [ctypes.POINTER(Dims)] + [_DP] * 9
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_backward.argtypes = (
        [ctypes.POINTER(Dims), ctypes.c_int] + [_DP] * 14
    )
    lib.gdn_oracle_backward.restype = ctypes.c_int
    lib.gdn_oracle_num_checkpoints.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.gdn_oracle_num_checkpoints.restype = ctypes.c_int64
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    lib.gdn_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.gdn_oracle_set_threads.restype = None
    lib.gdn_oracle_mutation.restype = ctypes.c_int
    return lib


_LIBS: dict = {}


def load(path: str | None = None, mutation: int = 0):
    """Load (building first if needed) the oracle library; mutants build into a temp dir."""
    key = (path, mutation)
    if key in _LIBS:
        return _LIBS[key]
    if mutation:
        out = os.path.join(tempfile.mkdtemp(prefix="gdn_oracle_mut"), f"libm{mutation}.so")
        build(out, mutation=mutation)
        lib = ctypes.CDLL(out)
    else:
        p = path or _LIB_DEFAULT
        if not os.path.exists(p) or os.path.getmtime(p) < os.path.getmtime(_SRC):
            build(p)
        lib = ctypes.CDLL(p)
    _LIBS[key] = _bind(lib)
    return _LIBS[key]


def default_C(T: int) -> int:
    """Default checkpoint interval ceil(sqrt(T)) (PR #16: C ~ sqrt(T), window 8192 -> 91)."""
    return max(1, math.isqrt(max(T, 0) - 1) + 1) if T > 1 else 1


def num_checkpoints(T: int, C: int) -> int:
    return 0 if T <= 0 else (T + C - 1) // C


def max_threads(lib=None) -> int:
    return int((lib or load()).gdn_oracle_max_threads())


def set_threads(n: int, lib=None) -> None:
    """Threads of the oracle's loop over (sequence, value head) units from now on."""
    (lib or load()).gdn_oracle_set_threads(int(n))


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def _dims(q, v, g, C, scale):
    """Sizes from the arrays: v holds the N value sequences, q the N / rep q/k sequences."""
    N, T, H_v, S_v = v.shape
    H_k, S_k = q.shape[2], q.shape[3]
    if q.shape[0] == 0 or N % q.shape[0]:
        raise ValueError("v's sequences must be a multiple of q's")
    kda = 1 if g.ndim == 4 else 0
    return Dims(N, T, H_k, H_v, S_k, S_v, kda, int(C), float(scale), N // q.shape[0])


def forward(q, k, v, g, beta, state0, scale, C=None, lib=None):
    """Oracle forward.  Arrays are promoted to float64 (contiguous semantic layouts); q, k
    may hold fewer sequences than v (a divisor of its count: the sequence broadcast).

    Returns (y [N,T,H_v,S_v], state_T [N,H_v,S_v,S_k], ckpt [N,H_v,n_ck,S_v,S_k]).
    """
    lib = lib or load()
    q, k, v, g, beta, state0 = map(_f64, (q, k, v, g, beta, state0))
    N, T, H_v, S_v = v.shape
    H_k, S_k = q.shape[2], q.shape[3]
    C = default_C(T) if C is None else int(C)
    d = _dims(q, v, g, C, scale)
    n_ck = num_checkpoints(T, C)
    y = np.zeros((N, T, H_v, S_v))
    sT = np.zeros((N, H_v, S_v, S_k))
    ck = np.zeros((N, H_v, n_ck, S_v, S_k))
    rc = lib.gdn_oracle_forward(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(state0), _ptr(y), _ptr(sT), _ptr(ck))
    if rc != 0:
        raise ValueError(f"gdn_oracle_forward rejected its arguments (code {rc})")
    return y, sT, ck


def backward(q, k, v, g, beta, state0, gy, dstate_T, scale, C=None, mode="checkpointed",
             ckpt=None, lib=None):
    """Oracle backward.  mode = "store_all" or "checkpointed".

    Returns a dict with dq, dk [N,T,H_k,S_k], dv [N,T,H_v,S_v], dg (like g),
    dbeta [N,T,H_v] and dstate0 [N,H_v,S_v,S_k].  dstate_T may be None (zero).
    """
    lib = lib or load()
    q, k, v, g, beta, state0, gy = map(_f64, (q, k, v, g, beta, state0, gy))
    dsT = None if dstate_T is None else _f64(dstate_T)
    N, T, H_v, S_v = v.shape
    Nq, H_k, S_k = q.shape[0], q.shape[2], q.shape[3]
    C = default_C(T) if C is None else int(C)
    d = _dims(q, v, g, C, scale)
    m = {"store_all": 0, "checkpointed": 1}[mode]
    if m == 1 and ckpt is None:
        _, _, ckpt = forward(q, k, v, g, beta, state0, scale, C=C, lib=lib)
    ck = None if m == 0 else _f64(ckpt)
    out = {
        "dq": np.zeros((Nq, T, H_k, S_k)),
        "dk": np.zeros((Nq, T, H_k, S_k)),
        "dv": np.zeros((N, T, H_v, S_v)),
        "dg": np.zeros(g.shape),
        "dbeta": np.zeros((N, T, H_v)),
        "dstate0": np.zeros((N, H_v, S_v, S_k)),
    }
    rc = lib.gdn_oracle_backward(
        ctypes.byref(d), m, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(state0) if m == 0 else None, _ptr(ck), _ptr(gy), _ptr(dsT),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
        _ptr(out["dbeta"]), _ptr(out["dstate0"]))
    if rc != 0:
        raise ValueError(f"gdn_oracle_backward rejected its arguments (code {rc})")
    return out
