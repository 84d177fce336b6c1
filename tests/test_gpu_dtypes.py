"""16-bit input storage (bf16, fp16) against the float64 oracle.

q, k, v, g, beta and gy are stored in the 16-bit type; states and every output are fp32
(meTile "Training kernels and gradients": 16-bit inputs beside fp32 state and gradients).
The oracle runs on exactly the stored values (each 16-bit value is an fp32 value, promoted
to float64), so the tolerance is the fp32 path's: 2e-4 (1 + |ref|) at these lengths.  The
library widens the inputs exactly and runs its fp32 path on the copies, so the results
are also the fp32 path's own on the widened tensors, bit for bit.
"""
import numpy as np
import pytest

import gpu_helpers as H
from gated_delta_rule_backward_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("kda,d", [(False, 64), (True, 64), (False, 128), (True, 128)],
                         ids=["scalar-64", "kda-64", "scalar-128", "kda-128"])
def test_16bit_inputs(dtype, kda, d):
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(2, 150, 2, 6, d, kda=kda, seed=70, C=40, packed=True, dstate_T=True)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    N, T, Hk, Hv = prob.N, prob.T, prob.H_k, prob.H_v
    to16 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(tdt).cuda()
    qkv = to16(prob.qkv)
    q = qkv[:, :, : Hk * d].view(N, T, Hk, d)
    k = qkv[:, :, Hk * d: 2 * Hk * d].view(N, T, Hk, d)
    v = qkv[:, :, 2 * Hk * d:].view(N, T, Hv, d)
    g, beta, gy = to16(prob.g), to16(prob.beta), to16(prob.gy)
    s0 = torch.from_numpy(prob.state0).cuda()
    dsT = torch.from_numpy(prob.dstate_T).cuda()
    y, sT, ck, p = gdn.forward(q, k, v, g, beta, s0, C=prob.C, scale=prob.scale)
    assert p.in_dtype == (gdn.DTYPE_BF16 if dtype == "bf16" else gdn.DTYPE_F16)
    packed, views = gdn.backward(p, q, k, v, g, beta, ck, gy, dsT)
    torch.cuda.synchronize()
    H.assert_device_ok()
    wide = {nm: t.float().cpu().numpy() for nm, t in (("q", q), ("k", k), ("v", v), ("g", g),
                                                      ("beta", beta), ("gy", gy))}
    wide.update(state0=prob.state0, dstate_T=prob.dstate_T)
    ref = H.run_oracle(wide, prob.scale, prob.C)
    got = {"y": y, "state_T": sT, "ckpt": ck}
    got.update(views)
    H.compare_all({kk: t.cpu().numpy() for kk, t in got.items()}, ref, H.tolerance(T))
    # the same bits as the fp32 path on the widened inputs
    f = lambda t: t.float()
    y2, sT2, ck2, p2 = gdn.forward(f(q), f(k), f(v), f(g), f(beta), s0, C=prob.C, scale=prob.scale)
    packed2, _ = gdn.backward(p2, f(q), f(k), f(v), f(g), f(beta), ck2, f(gy), dsT)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(sT, sT2) and torch.equal(ck, ck2)
    assert torch.equal(packed, packed2)
