"""Seeded synthetic inputs for the gated delta rule (shared by tests and bench).

This module holds none of the recurrence's arithmetic: it only draws random numbers
and applies the caller-side input transforms the workloads prescribe (L2-normalised
q/k, g = -softplus(.), beta = sigmoid(.)).  Both the CUDA path's tests and the oracle's
tests take their inputs from here.

Recipe (numpy PCG64 ``default_rng(seed)``, drawn in float64, cast to float32):
  q, k   ~ N(0, 1), L2-normalised over the head dimension per (token, head)
  v      ~ N(0, 1)
  g      = -softplus(N(0, g_std^2))   [N,T,H_v] (scalar gate) or [N,T,H_v,S_k] (KDA)
  beta   = sigmoid(N(0, 1))           [N,T,H_v]
  state0 ~ N(0, 0.1^2)                [N,H_v,S_v,S_k]
  gy     ~ N(0, 1)                    [N,T,H_v,S_v]
  dstate_T = 0, or ~ N(0, 0.1^2)
  scale  = 1/sqrt(S_k)
With ``packed=True`` q, k and v are row views of one qkv buffer [N, T, (2H_k+H_v)*d]
(q at column 0, k at H_k*d, v at 2*H_k*d), as a fused projection would lay them out.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Problem:
    N: int
    T: int
    H_k: int
    H_v: int
    d: int
    kda: bool
    C: int | None
    scale: float
    q: np.ndarray       # [N,T,H_k,d] float32 (possibly a strided view of qkv)
    k: np.ndarray
    v: np.ndarray       # [N,T,H_v,d]
    g: np.ndarray       # [N,T,H_v] or [N,T,H_v,d]
    beta: np.ndarray    # [N,T,H_v]
    state0: np.ndarray  # [N,H_v,d,d]
    gy: np.ndarray      # [N,T,H_v,d]
    dstate_T: np.ndarray | None
    qkv: np.ndarray | None  # the packed buffer when packed=True
    d_v: int | None = None  # value head size (S_v); d is the key head size (S_k)


def _normal(rng, shape, std=1.0):
    return rng.standard_normal(shape, dtype=np.float64) * std


def _l2norm(x):
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / n


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def make_problem(N, T, H_k, H_v, d, kda=False, seed=0, g_std=1.0, C=None,
                 packed=False, dstate_T=False, d_v=None, seq_rep=1):
    """Draw one seeded problem.  Draw order is fixed: q, k, v, g, beta, state0, gy, dstate_T.
    d is the key head size S_k; d_v the value head size S_v (default d).  With seq_rep > 1
    q and k hold N / seq_rep sequences, value sequence n reading q/k sequence n / seq_rep
    (not with packed=True)."""
    if H_v % H_k:
        raise ValueError("H_v must be a multiple of H_k")
    if N % seq_rep or (packed and seq_rep != 1):
        raise ValueError("seq_rep must divide N (and the packed layout has one q/k per sequence)")
    dv = d if d_v is None else d_v
    Nq = N // seq_rep
    rng = np.random.default_rng(seed)
    f32 = np.float32
    q = _l2norm(_normal(rng, (Nq, T, H_k, d))).astype(f32)
    k = _l2norm(_normal(rng, (Nq, T, H_k, d))).astype(f32)
    v = _normal(rng, (N, T, H_v, dv)).astype(f32)
    gshape = (N, T, H_v, d) if kda else (N, T, H_v)
    g = (-_softplus(_normal(rng, gshape, g_std))).astype(f32)
    beta = _sigmoid(_normal(rng, (N, T, H_v))).astype(f32)
    state0 = _normal(rng, (N, H_v, dv, d), 0.1).astype(f32)
    gy = _normal(rng, (N, T, H_v, dv)).astype(f32)
    dsT = _normal(rng, (N, H_v, dv, d), 0.1).astype(f32) if dstate_T else None
    qkv = None
    if packed:
        width = 2 * H_k * d + H_v * dv
        qkv = np.empty((N, T, width), dtype=f32)
        qkv[:, :, : H_k * d] = q.reshape(N, T, H_k * d)
        qkv[:, :, H_k * d: 2 * H_k * d] = k.reshape(N, T, H_k * d)
        qkv[:, :, 2 * H_k * d:] = v.reshape(N, T, H_v * dv)
        q = qkv[:, :, : H_k * d].reshape(N, T, H_k, d)
        k = qkv[:, :, H_k * d: 2 * H_k * d].reshape(N, T, H_k, d)
        v = qkv[:, :, 2 * H_k * d:].reshape(N, T, H_v, dv)
    return Problem(N, T, H_k, H_v, d, kda, C, 1.0 / float(np.sqrt(d)), q, k, v, g, beta,
                   state0, gy, dsT, qkv, dv)


# The named workloads (shapes and distributions of the gated delta rule configurations).
WORKLOADS = {
    # 1 seq, one head, d=32, T=16, scalar gate, C=4
    "tiny_d32_T16": dict(N=1, T=16, H_k=1, H_v=1, d=32, kda=False, C=4, seed=1000),
    # 2 seqs, 4 heads, d=64, T=61 (partial last segment), KDA gate, C=8, dstate_T != 0
    "kda_d64_T61": dict(N=2, T=61, H_k=4, H_v=4, d=64, kda=True, C=8, seed=1001,
                        dstate_T=True),
    # 4 seqs, H_k=16 broadcast to H_v=48, d=128, T=2048, packed qkv views, default C
    "bcast_d128_T2048": dict(N=4, T=2048, H_k=16, H_v=48, d=128, kda=False, C=None,
                             seed=1002, packed=True),
    # 1 seq, H_k=16/H_v=48, d=128, T=16384, KDA with strong decay mix, C=128
    "kda_d128_T16384": dict(N=1, T=16384, H_k=16, H_v=48, d=128, kda=True, C=128,
                            seed=1003, packed=True, g_std=2.0),
    # the throughput shape: 1 seq, H_k=16/H_v=48, d=128, T=4096, scalar gate, default C
    "bench_d128_T4096": dict(N=1, T=4096, H_k=16, H_v=48, d=128, kda=False, C=None,
                             seed=1004, packed=True),
    # the throughput shape cut to T=1024 with the same C=64 (two chunks per segment): the
    # size a many-pass profiler capture of one kernel launch stays small at
    "profile_d128_T1024": dict(N=1, T=1024, H_k=16, H_v=48, d=128, kda=False, C=64,
                               seed=1005, packed=True),
    # the per-key-column gate at the same heads and C as the 16384-token workload, cut to
    # 1024 tokens for many-pass profiler captures of the token-recurrence kernels
    "profile_kda_d128_T1024": dict(N=1, T=1024, H_k=16, H_v=48, d=128, kda=True, C=128,
                                   seed=1006, packed=True, g_std=2.0),
    # sweep shapes at head sizes 64 and 32 (4 sequences, 16 key heads over 48 value heads,
    # 4096 tokens, scalar gate): the FP32-pipe chunked path, for stage times and captures
    "d64_T4096_N4": dict(N=4, T=4096, H_k=16, H_v=48, d=64, kda=False, C=None, seed=1007, packed=True),
    "d32_T4096_N4": dict(N=4, T=4096, H_k=16, H_v=48, d=32, kda=False, C=None, seed=1008, packed=True),
    # the head-size-64 shape at one sequence and 1024 tokens, for many-pass captures
    "profile_d64_T1024": dict(N=1, T=1024, H_k=16, H_v=48, d=64, kda=False, C=64, seed=1009, packed=True),
}


def workload(name, **overrides):
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return make_problem(**kw)


def sweep_points():
    """The throughput sweep: d x T x batch*H_v (H_v = 48 = 3 H_k, N = 1/4/8) x gate."""
    pts = []
    idx = 0
    for d in (32, 64, 128):
        for T in (512, 4096, 16384):
            for N in (1, 4, 8):
                for kda in (False, True):
                    pts.append(dict(N=N, T=T, H_k=16, H_v=48, d=d, kda=kda, C=None,
                                    seed=2000 + idx, packed=True))
                    idx += 1
    return pts
