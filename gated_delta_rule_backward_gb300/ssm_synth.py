"""Seeded synthetic inputs for the selective scan (shared by its tests and bench).

This module holds none of the scan's arithmetic: it only draws random numbers in the
shapes and ranges of Mamba-1 / Mamba-2 layers.  Both the CUDA path's tests and the
oracle's tests take their inputs from here.

Recipe (numpy PCG64 ``default_rng(seed)``, drawn in float64, cast to float32):
  x      ~ N(0, 1)                                  [N,T,H,P]
  dt     = exp(U(log 1e-3, log 1e-1))               [N,T,H]   (Mamba's dt range, after
                                                               the caller's softplus)
  A      Mamba-2: -U(1, 16) per head                [H]
         Mamba-1: -(j + 1) for state j (S4D-real)   [H,S]
  B, C   ~ N(0, 1)                                  [N,T,G,S]
  s0     ~ N(0, 0.1^2)                              [N,H,P,S]
  dy     ~ N(0, 1)                                  [N,T,H,P]
  ds_T   ~ N(0, 0.1^2)                              [N,H,P,S] (the state region of the
                                                               packed cotangent is not zero)
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class SsmProblem:
    N: int
    T: int
    H: int
    P: int
    S: int
    G: int
    mamba1: bool        # A per state ([H,S]); else one per head ([H])
    K: int              # checkpoint interval
    s0: np.ndarray
    x: np.ndarray
    dt: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    dy: np.ndarray
    ds_T: np.ndarray


def make_ssm_problem(N, T, H, P, S, G=1, mamba1=False, K=None, seed=0):
    if H % G:
        raise ValueError("H must be a multiple of G")
    rng = np.random.default_rng(seed)
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    x = rng.standard_normal((N, T, H, P))
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), (N, T, H)))
    if mamba1:
        A = -np.tile(np.arange(1, S + 1, dtype=np.float64), (H, 1))
    else:
        A = -rng.uniform(1.0, 16.0, (H,))
    B = rng.standard_normal((N, T, G, S))
    C = rng.standard_normal((N, T, G, S))
    s0 = rng.standard_normal((N, H, P, S)) * 0.1
    dy = rng.standard_normal((N, T, H, P))
    ds_T = rng.standard_normal((N, H, P, S)) * 0.1
    if K is None:
        K = max(1, int(np.ceil(np.sqrt(max(T, 1)))))
    return SsmProblem(N, T, H, P, S, G, bool(mamba1), int(K), f32(s0), f32(x), f32(dt), f32(A), f32(B), f32(C),
                      f32(dy), f32(ds_T))


# Workloads: Mamba-2 2.7B-like (d_inner 5120 = 80 heads of 64, 128 states, one group) and
# Mamba-1 130M-like (d_inner 1536 channels of one, 16 states); small cases for parity.
SSM_WORKLOADS = {
    "mamba2_h80_T4096": dict(N=1, T=4096, H=80, P=64, S=128, G=1, mamba1=False, K=64, seed=11),
    "mamba1_d1536_T4096": dict(N=1, T=4096, H=1536, P=1, S=16, G=1, mamba1=True, K=64, seed=12),
    "mamba2_small": dict(N=2, T=100, H=8, P=64, S=128, G=2, mamba1=False, K=16, seed=13),
    "mamba1_small": dict(N=2, T=100, H=96, P=1, S=16, G=1, mamba1=True, K=16, seed=14),
    # the two layers cut to 512 tokens, for kernel captures of a few hundred MB
    "profile_mamba2_h80_T512": dict(N=1, T=512, H=80, P=64, S=128, G=1, mamba1=False, K=16, seed=11),
    "profile_mamba1_d1536_T512": dict(N=1, T=512, H=1536, P=1, S=16, G=1, mamba1=True, K=16, seed=12),
    # the Mamba-2 layer in chunked form at 2048 tokens (about 0.5 GB on the device)
    "profile_mamba2_h80_T2048": dict(N=1, T=2048, H=80, P=64, S=128, G=1, mamba1=False, K=64, seed=11),
}


def ssm_workload(name, **overrides):
    kw = dict(SSM_WORKLOADS[name])
    kw.update(overrides)
    return make_ssm_problem(**kw)
