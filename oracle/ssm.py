"""Float64 CPU oracle of the selective scan (Mamba-1 / Mamba-2) and its reverse walk --
TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU legs) may import
this module.  The product path never calls it and shares no code with it.

The arithmetic lives in ``ssm_oracle.c`` (plain C, float64, OpenMP over (sequence, head)
in the forward and over (sequence, group) in the walk); this module compiles it with gcc
and marshals numpy arrays.  What it computes, and the reading of each step, is stated in
the C file's header (llama.cpp PR #26, the SSM_SCAN_BACK section).

Parity status: every output (y, the final states, the checkpoints, d_s, d_x, d_dt, d_B,
d_C) is pinned by ``tests/test_ssm_oracle_pins.py`` (finite differences under an objective
that weights the state region, closed forms, invariants, store-all against checkpointed
bit for bit, and a six-defect kill list).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_DEFAULT = os.path.join(_HERE, "libssm_oracle.so")


class Dims(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("P", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("G", ctypes.c_int64),
        ("a_per_state", ctypes.c_int64),
        ("K", ctypes.c_int64),
    ]


def build(out_path: str = _LIB_DEFAULT, mutation: int = 0, openmp: bool = True) -> str:
    """Compile the oracle into a shared library (gcc, -O2, no fast-math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math"]
    if openmp:
        cmd.append("-fopenmp")
    if mutation:
        cmd.append(f"-DSSM_ORACLE_MUTATION={int(mutation)}")
    cmd += [_SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


_DP = ctypes.POINTER(ctypes.c_double)
_LIBS: dict = {}


def _bind(lib):
    lib.ssm_oracle_forward.argtypes = [ctypes.POINTER(Dims)] + [_DP] * 9
    lib.ssm_oracle_forward.restype = ctypes.c_int
    lib.ssm_oracle_backward.argtypes = [ctypes.POINTER(Dims), ctypes.c_int] + [_DP] * 14
    lib.ssm_oracle_backward.restype = ctypes.c_int
    lib.ssm_oracle_num_checkpoints.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.ssm_oracle_num_checkpoints.restype = ctypes.c_int64
    lib.ssm_oracle_max_threads.restype = ctypes.c_int
    lib.ssm_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.ssm_oracle_set_threads.restype = None
    lib.ssm_oracle_mutation.restype = ctypes.c_int
    return lib


def load(path: str | None = None, mutation: int = 0):
    """Load (building first if needed) the oracle library; mutants build into a temp dir."""
    key = (path, mutation)
    if key in _LIBS:
        return _LIBS[key]
    if mutation:
        out = os.path.join(tempfile.mkdtemp(prefix="ssm_oracle_mut"), f"libm{mutation}.so")
        build(out, mutation=mutation)
        lib = ctypes.CDLL(out)
    else:
        p = path or _LIB_DEFAULT
        if not os.path.exists(p) or os.path.getmtime(p) < os.path.getmtime(_SRC):
            build(p)
        lib = ctypes.CDLL(p)
    _LIBS[key] = _bind(lib)
    return _LIBS[key]


def num_checkpoints(T: int, K: int) -> int:
    return 1 if T <= 0 else (T + K - 1) // K


def set_threads(n: int, lib=None) -> None:
    (lib or load()).ssm_oracle_set_threads(int(n))


def max_threads(lib=None) -> int:
    return int((lib or load()).ssm_oracle_max_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def _dims(x, A, B, K):
    N, T, H, P = x.shape
    G, S = B.shape[2], B.shape[3]
    per_state = 1 if A.ndim == 2 else 0
    return Dims(N, T, H, P, S, G, per_state, int(K))


def forward(s0, x, dt, A, B, C, K=1, lib=None):
    """Returns (y [N,T,H,P], s_T [N,H,P,S], checkpoints [N,H,n_ck,P,S])."""
    lib = lib or load()
    s0, x, dt, A, B, C = map(_f64, (s0, x, dt, A, B, C))
    d = _dims(x, A, B, K)
    N, T, H, P = x.shape
    S = B.shape[3]
    y = np.zeros((N, T, H, P))
    sT = np.zeros((N, H, P, S))
    ck = np.zeros((N, H, num_checkpoints(T, K), P, S))
    rc = lib.ssm_oracle_forward(ctypes.byref(d), _ptr(s0), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(y), _ptr(sT), _ptr(ck))
    if rc != 0:
        raise ValueError(f"ssm_oracle_forward rejected its arguments (code {rc})")
    return y, sT, ck


def backward(s0, x, dt, A, B, C, dy, ds_T, K=1, mode="checkpointed", ckpt=None, lib=None):
    """The reverse walk.  mode = "store_all" (every state recomputed from s0) or
    "checkpointed" (each segment of K tokens recomputed from its checkpoint).

    Returns a dict with ds0 [N,H,P,S], dx [N,T,H,P], ddt [N,T,H], dB, dC [N,T,G,S].
    """
    lib = lib or load()
    s0, x, dt, A, B, C, dy, ds_T = map(_f64, (s0, x, dt, A, B, C, dy, ds_T))
    d = _dims(x, A, B, K)
    N, T, H, P = x.shape
    G, S = B.shape[2], B.shape[3]
    m = {"store_all": 1, "checkpointed": 0}[mode]
    if m == 0 and ckpt is None:
        _, _, ckpt = forward(s0, x, dt, A, B, C, K=K, lib=lib)
    ck = None if m == 1 else _f64(ckpt)
    out = {
        "ds0": np.zeros((N, H, P, S)),
        "dx": np.zeros((N, T, H, P)),
        "ddt": np.zeros((N, T, H)),
        "dB": np.zeros((N, T, G, S)),
        "dC": np.zeros((N, T, G, S)),
    }
    rc = lib.ssm_oracle_backward(ctypes.byref(d), m, _ptr(s0), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(ck), _ptr(dy), _ptr(ds_T), _ptr(out["ds0"]), _ptr(out["dx"]),
                                 _ptr(out["ddt"]), _ptr(out["dB"]), _ptr(out["dC"]))
    if rc != 0:
        raise ValueError(f"ssm_oracle_backward rejected its arguments (code {rc})")
    return out
