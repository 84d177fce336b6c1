"""gdn_backward_noalloc: the backward for callers that cannot allocate device memory when
they run it (a host framework that has handed out its whole budget, a plugin host with no
device allocator for its extensions).  It uses the library's fixed 64 MiB device scratch
instead of a caller workspace.

Checked through the C ABI against gdn_backward on the same inputs, on two calls in a row.
Before each of them the scratch is filled by a call on an unrelated problem, so that a
scratch element read before being written would show; and the rejection of a problem
whose scratch would exceed 64 MiB.  This file is collected
last so that a failure here cannot hide any other test.
"""
import ctypes

import numpy as np
import pytest

import gpu_helpers as H
from gated_delta_rule_backward_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _noalloc_other_problem(gdn, kda, seed):
    """Runs the no-allocation backward on an unrelated problem (other seed, length, C and
    gate), so that the shared scratch holds values that have nothing to do with the next
    call's."""
    prob = synth.make_problem(1, 203 + seed % 50, 2, 6, 128, kda=not kda, seed=seed, C=23,
                              packed=True, dstate_T=True)
    dev = H.upload(prob)
    _, _, ck, p = gdn.forward(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                              dev["state0"], C=prob.C, scale=prob.scale)
    p.gy_s[:] = gdn.strides3(dev["gy"])
    assert gdn.backward_workspace_bytes(p) <= 64 << 20
    out = torch.empty(gdn.packed_grad_elems(p), device="cuda")
    gdn.gdn_backward_noalloc(p, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ck,
                             dev["gy"], dev["dstate_T"], out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_noalloc_matches_workspace_backward_twice(kda):
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(2, 300, 2, 6, 128, kda=kda, seed=77, C=17, packed=True,
                              dstate_T=True)
    dev = H.upload(prob)
    y, sT, ck, p = gdn.forward(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                               dev["state0"], C=prob.C, scale=prob.scale)
    p.gy_s[:] = gdn.strides3(dev["gy"])
    assert gdn.backward_workspace_bytes(p) <= 64 << 20
    ref, _ = gdn.backward(p, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ck,
                          dev["gy"], dev["dstate_T"])
    tol = H.tolerance(prob.T)
    for call in range(2):
        # the scratch first holds an unrelated problem's values: a scratch element read
        # before this call writes it would change the result
        _noalloc_other_problem(gdn, kda, seed=900 + 10 * call + int(kda))
        out = torch.full_like(ref, float("nan"))
        gdn.gdn_backward_noalloc(p, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ck,
                                 dev["gy"], dev["dstate_T"], out)
        torch.cuda.synchronize()
        H.compare("packed (noalloc vs workspace)", out.cpu().numpy(), ref.cpu().numpy(), tol)
        assert torch.equal(out, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    from gated_delta_rule_backward_gb300 import gdn
    p = gdn.make_params(1, 4096, 16, 48, 128, False)
    assert gdn.backward_workspace_bytes(p) > 64 << 20
    e = torch.empty(16, device="cuda")
    ptr = ctypes.c_void_p(e.data_ptr())
    # q, k, v, g, beta, ckpt, gy, dstate_T (none), packed, stream (default)
    st = gdn.library().gdn_backward_noalloc(ctypes.byref(p), *[ptr] * 7, None, ptr, None)
    assert st == 4  # GDN_ERR_WORKSPACE
    assert b"64" in gdn.library().gdn_last_error() or b"67108864" in gdn.library().gdn_last_error()
