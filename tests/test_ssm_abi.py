"""The selective scan's C ABI (include/ssm.h) on the CPU: exports, sizes and argument
validation.  Every call below fails its checks before any device work is enqueued."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_backward_gb300 import gdn, ssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIAS, WORKSPACE = 0, 1, 2, 3, 4
BASE = 0x7F0000000000  # fake, 256-byte aligned device addresses (never dereferenced)


def test_header_symbols_exported():
    hdr = open(os.path.join(ROOT, "include", "ssm.h")).read()
    declared = set(re.findall(r"^\w[\w\s\*]*?\b(ssm_\w+)\(", hdr, flags=re.M))
    assert declared == set(ssm.EXPORTS)
    for name in declared:
        assert hasattr(gdn.library(), name), name


def test_sizes():
    p = ssm.make_params(2, 10, 4, 8, 16, G=2, K=3)
    assert ssm.checkpoint_interval(p) == 3 and ssm.num_checkpoints(p) == 4
    assert ssm.packed_out_elems(p) == 2 * 10 * 4 * 8 + 2 * 4 * 8 * 16
    assert ssm.packed_grad_elems(p) == 2 * 4 * 8 * 16 + 2 * 10 * 4 * 8 + 2 * 10 * 4 + 2 * 2 * 10 * 2 * 16
    p = ssm.make_params(1, 100, 4, 8, 16)   # K = 0: ceil(sqrt(T))
    assert ssm.checkpoint_interval(p) == 10 and ssm.num_checkpoints(p) == 10
    p = ssm.make_params(1, 0, 4, 8, 16)
    assert ssm.num_checkpoints(p) == 1
    assert ssm.backward_workspace_bytes(ssm.make_params(1, 4096, 80, 64, 128, K=64)) > 0


def test_chunked_dispatch():
    """Which form runs, its default checkpoint interval and its launch counts."""
    p = ssm.make_params(1, 100, 8, 64, 128)            # K = 0: ceil(sqrt(100)) = 10, rounded up to 64
    assert ssm.chunked(p) and ssm.checkpoint_interval(p) == 64 and ssm.num_checkpoints(p) == 2
    assert ssm.launches(p) == (3, 4)
    p = ssm.make_params(1, 5000, 8, 64, 128)           # ceil(sqrt(5000)) = 71 -> 128
    assert ssm.chunked(p) and ssm.checkpoint_interval(p) == 128
    for p in (ssm.make_params(1, 100, 8, 64, 128, K=16),          # K off the chunk grid
              ssm.make_params(1, 100, 8, 64, 64, K=64),           # other state counts
              ssm.make_params(1, 100, 8, 32, 128, K=64),          # other head sizes
              ssm.make_params(1, 100, 8, 64, 128, mamba1=True, K=64),
              ssm.make_params(1, 0, 8, 64, 128, K=64)):           # no tokens
        assert not ssm.chunked(p)
    assert ssm.launches(ssm.make_params(1, 100, 8, 64, 128, K=16)) == (1, 2)
    assert ssm.launches(ssm.make_params(1, 0, 8, 64, 128, K=64)) == (1, 0)
    assert ssm.launches(ssm.make_params(0, 10, 8, 64, 128, K=64)) == (0, 0)
    assert ssm.launches(ssm.make_params(1, 10, 8, 64, 24)) == (0, 0)
    # the segmented form: a decay per state, one channel a head, 16 states, whole blocks of 16
    # channels in a group, and ceil(T / K) 16 <= T
    assert ssm.form(ssm.make_params(1, 4096, 1536, 1, 16, mamba1=True, K=64)) == "segmented"
    assert ssm.launches(ssm.make_params(1, 4096, 1536, 1, 16, mamba1=True, K=64)) == (3, 4)
    for p in (ssm.make_params(1, 100, 96, 1, 16, mamba1=True, K=6),     # 17 segments x 16 > 100
              ssm.make_params(1, 100, 40, 1, 16, mamba1=True, K=20),    # 40 channels: not blocks of 16
              ssm.make_params(1, 100, 96, 2, 16, mamba1=True, K=20),    # two channels a head
              ssm.make_params(1, 100, 96, 1, 32, mamba1=True, K=20)):   # 32 states
        assert ssm.form(p) == "token-serial"
    assert ssm.form(ssm.make_params(1, 100, 8, 64, 128, K=64)) == "chunked"
    # its workspace: four per-sub-block slabs (entry states, U, G, carries: 32-token sub-blocks
    # of every segment, 16 states a channel) and the dB/dC partials of the 16-channel blocks
    N, T, H, G, K = 2, 4096, 1536, 2, 100
    nsb = -(-T // K) * -(-K // 32)
    per = 4 * N * nsb * H * 16
    parts = 4 * N * T * G * (H // G // 16) * 2 * 16
    up = lambda b: (b + 255) // 256 * 256
    assert ssm.backward_workspace_bytes(ssm.make_params(N, T, H, 1, 16, G, mamba1=True, K=K)) == 4 * up(per) + up(parts)
    # the chunked workspace: the per-chunk state slabs (one, or two with inner chunks to
    # replay), the chunk decays and the dB/dC block partials
    st = 4 * 64 * 8 * 64 * 128
    w1 = ssm.backward_workspace_bytes(ssm.make_params(1, 4096, 8, 64, 128, K=64))
    w2 = ssm.backward_workspace_bytes(ssm.make_params(1, 4096, 8, 64, 128, K=128))
    assert w1 > st and w2 - w1 == st


@pytest.mark.parametrize("args,code", [
    (dict(S=24), UNSUPPORTED), (dict(S=512), UNSUPPORTED), (dict(H=6, G=4), INVALID),
    (dict(P=3), UNSUPPORTED), (dict(K=-1), INVALID), (dict(T=-1), INVALID), (dict(S=0), INVALID),
])
def test_supported_rejects(args, code):
    kw = dict(N=1, T=8, H=4, P=8, S=16, G=1, K=0)
    kw.update(args)
    p = ssm.make_params(kw["N"], kw["T"], kw["H"], kw["P"], kw["S"], kw["G"], K=kw["K"])
    assert ssm.supported(p) == code


def _fwd(p, **ptrs):
    mb = 1 << 20
    d = dict(s0=BASE, x=BASE + mb, dt=BASE + 2 * mb, A=BASE + 3 * mb, B=BASE + 4 * mb, C=BASE + 5 * mb,
             out=BASE + 6 * mb, ck=BASE + 7 * mb)
    d.update(ptrs)
    return gdn.library().ssm_forward(ctypes.byref(p), d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["out"],
                                     d["ck"], None)


def _bwd(p, ws_bytes=None, **ptrs):
    mb = 1 << 26
    d = dict(x=BASE, dt=BASE + mb, A=BASE + 2 * mb, B=BASE + 3 * mb, C=BASE + 4 * mb, ck=BASE + 5 * mb,
             gin=BASE + 6 * mb, gout=BASE + 7 * mb, ws=BASE + 8 * mb)
    d.update(ptrs)
    if ws_bytes is None:
        ws_bytes = ssm.backward_workspace_bytes(p)
    return gdn.library().ssm_backward(ctypes.byref(p), d["x"], d["dt"], d["A"], d["B"], d["C"], d["ck"], d["gin"],
                                      d["gout"], d["ws"], ws_bytes, None)


def test_forward_validation():
    p = ssm.make_params(1, 8, 4, 8, 16)
    assert _fwd(p, x=None) == INVALID
    assert _fwd(p, A=BASE + 4) == INVALID                       # misaligned
    assert _fwd(p, out=BASE + 16) == ALIAS                      # the output over s0
    assert _fwd(ssm.make_params(1, 8, 4, 8, 24)) == UNSUPPORTED


def test_backward_validation():
    p = ssm.make_params(1, 8, 4, 8, 16)
    assert _bwd(p, gin=None) == INVALID
    assert _bwd(p, ws_bytes=ssm.backward_workspace_bytes(p) - 256) == WORKSPACE
    assert _bwd(p, gout=BASE + 16) == ALIAS                     # the output over x
    assert _bwd(p, ws=BASE + (1 << 26) + 64) == ALIAS           # the workspace over dt
    assert _bwd(p, C=BASE + (4 << 26) + 8) == INVALID           # misaligned
