"""libgdn's C ABI on the host (no GPU needed): it loads, exports every symbol that
include/gdn.h declares, sizes its buffers as documented, and rejects bad arguments
with the documented status codes before touching the device."""
import ctypes
import json
import os
import re

import pytest

from gated_delta_rule_backward_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIAS, WORKSPACE = 0, 1, 2, 3, 4


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 12
    lib = gdn.library()
    for nm in names:
        assert hasattr(lib, nm), nm
    assert sorted(gdn.EXPORTS) == names


def test_status_strings():
    lib = gdn.library()
    for code, name in gdn.STATUS.items():
        assert lib.gdn_status_str(code).decode() == name


def test_packed_layout_and_sizes():
    for kda in (False, True):
        p = gdn.make_params(3, 61, 4, 12, 64, kda, C=8)
        off = gdn.packed_grad_offsets(p)
        N, T, Hk, Hv, S = 3, 61, 4, 12, 64
        sizes = [N * T * Hk * S, N * T * Hk * S, N * T * Hv * S,
                 N * T * Hv * (S if kda else 1), N * T * Hv, N * Hv * S * S]
        exp = [0]
        for s in sizes[:-1]:
            exp.append(exp[-1] + s)
        assert off == exp
        assert gdn.packed_grad_elems(p) == sum(sizes)
        assert gdn.num_checkpoints(p) == 8                        # ceil(61 / 8)
        assert gdn.library().gdn_ckpt_elems(ctypes.byref(p)) == N * Hv * 8 * S * S
        assert gdn.backward_workspace_bytes(p) > 0
        # scalar gate: chunked kernels (prep + state chain; prep + dM chain + gradients),
        # KDA gate: token recurrence (forward; backward + reduction)
        assert gdn.launches(p) == ((1, 2) if kda else (2, 3))
        assert gdn.timing_stages(p) == gdn.launches(p)
        assert (gdn.forward_workspace_bytes(p) == 0) == kda


def test_default_checkpoint_interval_matches_pages():
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "checkpoint_interval.json")))
    for case in gold["cases"]:
        p = gdn.make_params(1, case["T"], 1, 1, 32, False, C=None)
        assert gdn.checkpoint_interval(p) == case["C"]
    p = gdn.make_params(1, 2048, 16, 48, 128, False)
    assert gdn.checkpoint_interval(p) == 46 and gdn.num_checkpoints(p) == 45


def test_empty_batch_launches_nothing():
    p = gdn.make_params(0, 16, 1, 1, 32, False)
    assert gdn.launches(p) == (0, 0)
    p = gdn.make_params(2, 0, 1, 1, 32, False)
    assert gdn.launches(p) == (1, 1)
    assert gdn.num_checkpoints(p) == 0


def test_chunked_launch_count_with_several_chunks_per_segment():
    # C = 64 > 32-token chunks.  Head size 128 pipelines over chunk ranges: the forward
    # launches a prep and a state chain for each of 4 ranges; the backward launches, for
    # each of 2, a prep, a dM chain, one gradient launch per place of a chunk in its segment
    # (the first parks the second's entry states) and a sum over value heads.  With timing
    # events the backward runs 3 stages one after another.
    p = gdn.make_params(1, 4096, 16, 48, 128, False)
    assert gdn.checkpoint_interval(p) == 64
    assert gdn.launches(p) == (8, 10)
    assert gdn.timing_stages(p) == (1, 3)
    p = gdn.make_params(1, 100, 1, 2, 128, False, C=64)   # 2 segments -> 2 ranges
    assert gdn.launches(p) == (4, 10)
    p = gdn.make_params(1, 100, 1, 2, 128, False, C=32)   # one chunk per segment
    assert gdn.launches(p) == (8, 8)
    p = gdn.make_params(1, 100, 1, 2, 128, False, C=96)   # 3 places; the last segment has 1 chunk
    assert gdn.launches(p) == (4, 6 + 4)
    p = gdn.make_params(1, 4096, 16, 48, 64, False)
    assert gdn.launches(p) == (2, 4)


def test_forward_workspace_checks():
    p = gdn.make_params(1, 64, 1, 3, 64, False)
    need = gdn.forward_workspace_bytes(p)
    assert need > 0
    assert call_forward(p, ws_bytes=need - 256) == WORKSPACE


# ---- argument validation: every case below fails before any device work ----

BASE = 0x7f0000000000  # fake, 256-byte aligned device addresses


def fake(i):
    return ctypes.c_void_p(BASE + i * (1 << 32))


def call_forward(p, ptrs=None, ws_bytes=None):
    ptrs = ptrs or [fake(i) for i in range(9)]
    if ws_bytes is None:
        ws_bytes = gdn.forward_workspace_bytes(p)
    return gdn.library().gdn_forward(ctypes.byref(p), *ptrs, fake(10), ctypes.c_size_t(ws_bytes),
                                     None)


def call_backward(p, ws_bytes, ptrs=None):
    ptrs = ptrs or [fake(i) for i in range(10)]
    return gdn.library().gdn_backward(ctypes.byref(p), *ptrs[:10], ctypes.c_size_t(ws_bytes), None)


def test_unsupported_head_sizes():
    """Key head sizes 16, 32, 64, 128, 256; value head sizes multiples of 16 up to 256, in
    any combination (S_k != S_v included)."""
    for sk in (8, 48, 512):
        assert call_forward(gdn.make_params(1, 8, 1, 1, sk, False)) == UNSUPPORTED
        assert b"S_k" in gdn.library().gdn_last_error()
    for sv in (8, 24, 272):
        assert call_forward(gdn.make_params(1, 8, 1, 1, 64, False, S_v=sv)) == UNSUPPORTED
        assert b"S_v" in gdn.library().gdn_last_error()


def test_head_shapes_beyond_the_chunked_form_run_the_token_recurrence():
    """Square heads of 32, 64, 128 run the chunked kernels (the per-key-column gate at 128
    only); head sizes 16 and 256 and S_k != S_v run the token recurrence (forward; backward +
    reduction), with its work-proportional backward workspace."""
    for sk, sv, kda in ((64, 32, False), (32, 128, True), (16, 16, False), (16, 64, True),
                        (256, 256, False), (256, 64, True), (128, 256, False)):
        p = gdn.make_params(2, 61, 2, 4, sk, kda, C=8, S_v=sv)
        assert gdn.launches(p) == (1, 2), (sk, sv, kda)
        assert gdn.forward_workspace_bytes(p) == 0
        assert gdn.backward_workspace_bytes(p) > 0
        off = gdn.packed_grad_offsets(p)
        N, T, Hk, Hv = 2, 61, 2, 4
        assert off[2] - off[1] == N * T * Hk * sk                 # dk
        assert off[3] - off[2] == N * T * Hv * sv                 # dv
        assert gdn.packed_grad_elems(p) - off[5] == N * Hv * sv * sk  # dstate
    for sk in (32, 64):  # the FP32-pipe chunked kernels (head size 128: the pipelined ones)
        assert gdn.launches(gdn.make_params(2, 61, 2, 4, sk, False, C=8)) == (2, 3)


def test_invalid_arguments():
    assert call_forward(gdn.make_params(1, 8, 2, 3, 32, False)) == INVALID  # H_v % H_k
    p = gdn.make_params(1, 8, 1, 1, 32, False)
    p.q_s[1] = -32
    assert call_forward(p) == INVALID                                       # negative stride
    p = gdn.make_params(1, 8, 1, 1, 32, False)
    p.gate = 7
    assert call_forward(p) == INVALID
    p = gdn.make_params(1, 8, 1, 1, 32, False)
    p.in_dtype = 3                                                          # unknown input dtype
    assert call_forward(p) == INVALID
    p = gdn.make_params(3, 8, 1, 1, 32, False)
    p.seq_rep = 2                                                           # 3 % 2 != 0
    assert call_forward(p) == INVALID
    p = gdn.make_params(2, 8, 1, 1, 32, False)
    p.seq_rep = -1
    assert call_forward(p) == INVALID
    p = gdn.make_params(-1, 8, 1, 1, 32, False)
    assert call_forward(p) == INVALID
    assert gdn.library().gdn_forward(None, *[fake(i) for i in range(10)], ctypes.c_size_t(0),
                                     None) == INVALID
    p = gdn.make_params(1, 8, 1, 1, 32, False)
    ptrs = [fake(i) for i in range(9)]
    ptrs[0] = ctypes.c_void_p(BASE + 2)                                     # q not 4-byte aligned
    assert call_forward(p, ptrs) == INVALID
    ptrs = [fake(i) for i in range(9)]
    ptrs[7] = ctypes.c_void_p(BASE + 7 * (1 << 32) + 4)                     # state_T not 16-aligned
    assert call_forward(p, ptrs) == INVALID
    ptrs = [fake(i) for i in range(9)]
    ptrs[0] = None                                                          # q missing
    assert call_forward(p, ptrs) == INVALID


def test_alias_is_rejected():
    p = gdn.make_params(1, 8, 1, 1, 32, False)
    ptrs = [fake(i) for i in range(9)]
    ptrs[7] = ptrs[5]                                                       # state_T == state0
    assert call_forward(p, ptrs) == ALIAS
    ptrs = [fake(i) for i in range(9)]
    ptrs[6] = ctypes.c_void_p(BASE + 2 * (1 << 32) + 64)                    # y inside v
    assert call_forward(p, ptrs) == ALIAS
    ws = gdn.backward_workspace_bytes(p)
    ptrs = [fake(i) for i in range(10)]
    ptrs[8] = ptrs[6]                                                       # packed over gy
    assert call_backward(p, ws, ptrs) == ALIAS


def test_workspace_too_small():
    p = gdn.make_params(1, 64, 1, 3, 64, True)
    ws = gdn.backward_workspace_bytes(p)
    assert call_backward(p, ws - 256) == WORKSPACE
    ptrs = [fake(i) for i in range(10)]
    ptrs[9] = ctypes.c_void_p(BASE + 9 * (1 << 32) + 16)                    # not 256-aligned
    assert call_backward(p, ws, ptrs) == WORKSPACE


def test_16bit_inputs_add_their_widened_copies_to_the_workspace():
    """bf16 / fp16 inputs are widened into dense fp32 copies at the start of the workspace:
    q, k, v, g, beta (and gy in the backward), each 256-byte aligned; then the fp32 path's
    own workspace.  The widening adds one kernel per input."""
    al = lambda b: (b + 255) // 256 * 256
    for kda, S in ((False, 64), (True, 64), (False, 128), (True, 128)):
        N, T, Hk, Hv = 2, 61, 2, 6
        p32 = gdn.make_params(N, T, Hk, Hv, S, kda, C=8)
        for dt in (gdn.DTYPE_BF16, gdn.DTYPE_F16):
            p16 = gdn.make_params(N, T, Hk, Hv, S, kda, C=8, in_dtype=dt)
            gw = S if kda else 1
            wide_f = 2 * al(N * T * Hk * S * 4) + al(N * T * Hv * S * 4) + al(N * T * Hv * gw * 4) + al(N * T * Hv * 4)
            wide_b = wide_f + al(N * T * Hv * S * 4)
            assert gdn.forward_workspace_bytes(p16) == wide_f + gdn.forward_workspace_bytes(p32)
            assert gdn.backward_workspace_bytes(p16) == wide_b + gdn.backward_workspace_bytes(p32)
            f32, b32 = gdn.launches(p32)
            assert gdn.launches(p16) == (f32 + 5, b32 + 6)
