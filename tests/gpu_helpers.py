"""Shared plumbing of the GPU parity tests: upload a synthetic problem, run libgdn through
its C ABI, run the float64 oracle on the whole problem or on sampled key-head groups, and
compare element by element."""
from __future__ import annotations

import numpy as np

import oracle


def tolerance(T: int) -> float:
    """max |err| <= tol (1 + |ref|): 2e-4 up to T = 2048 tokens, 1e-3 beyond."""
    return 2e-4 if T <= 2048 else 1e-3


def upload(prob, device="cuda"):
    import torch
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
    d = {}
    if prob.qkv is not None:
        N, T, H_k, H_v, S = prob.N, prob.T, prob.H_k, prob.H_v, prob.d
        SV = prob.d_v or S
        qkv = t(prob.qkv)
        d["qkv"] = qkv
        d["q"] = qkv[:, :, : H_k * S].view(N, T, H_k, S)
        d["k"] = qkv[:, :, H_k * S: 2 * H_k * S].view(N, T, H_k, S)
        d["v"] = qkv[:, :, 2 * H_k * S:].view(N, T, H_v, SV)
    else:
        d["q"], d["k"], d["v"] = t(prob.q), t(prob.k), t(prob.v)
    for name in ("g", "beta", "state0", "gy", "dstate_T"):
        d[name] = t(getattr(prob, name))
    return d


def assert_device_ok():
    """No bounded wait of a tensor-core kernel gave up since the last check."""
    from gated_delta_rule_backward_gb300 import gdn
    st = gdn.device_status()
    assert st == 0, f"device status {st}: {gdn.library().gdn_last_error().decode()}"


def run_gpu(prob, C=None, dev=None, dstate_T="from_problem"):
    """Forward + backward through the C ABI.  Returns numpy outputs."""
    import torch
    from gated_delta_rule_backward_gb300 import gdn
    dev = dev or upload(prob)
    dsT = dev["dstate_T"] if dstate_T == "from_problem" else dstate_T
    y, sT, ck, p = gdn.forward(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                               dev["state0"], C=C if C is not None else prob.C,
                               scale=prob.scale)
    packed, views = gdn.backward(p, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ck,
                                 dev["gy"], dsT)
    torch.cuda.synchronize()
    assert_device_ok()
    out = {"y": y, "state_T": sT, "ckpt": ck}
    out.update(views)
    return {k: v.cpu().numpy() for k, v in out.items()}, packed


def group_problem(prob, n, hk):
    """The sub-problem of sequence n and the value heads served by key head hk."""
    heads = list(range(hk, prob.H_v, prob.H_k))  # ascending h_v
    sl = slice(n, n + 1)
    sub = dict(q=prob.q[sl][:, :, hk:hk + 1], k=prob.k[sl][:, :, hk:hk + 1],
               v=prob.v[sl][:, :, heads], g=prob.g[sl][:, :, heads],
               beta=prob.beta[sl][:, :, heads], state0=prob.state0[sl][:, heads],
               gy=prob.gy[sl][:, :, heads],
               dstate_T=None if prob.dstate_T is None else prob.dstate_T[sl][:, heads])
    return sub, heads


def run_oracle(x, scale, C, dstate_T="from_problem"):
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)
    dsT = x["dstate_T"] if dstate_T == "from_problem" else dstate_T
    y, sT, ck = oracle.forward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                               f(x["state0"]), scale, C=C)
    gr = oracle.backward(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]),
                         f(x["state0"]), f(x["gy"]), f(dsT), scale, C=C, ckpt=ck)
    out = {"y": y, "state_T": sT, "ckpt": ck}
    out.update(gr)
    return out


def problem_dict(prob):
    return dict(q=prob.q, k=prob.k, v=prob.v, g=prob.g, beta=prob.beta, state0=prob.state0,
                gy=prob.gy, dstate_T=prob.dstate_T)


def compare(name, got, ref, tol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    if got.size == 0:
        return 0.0
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    worst = float(err.max())
    assert worst <= tol, f"{name}: max rel err {worst:.3e} > {tol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return worst


KEYS = ("y", "state_T", "ckpt", "dq", "dk", "dv", "dg", "dbeta", "dstate0")


def compare_all(gpu, ref, tol, select=None):
    """select(name, array) -> the GPU slice matching the oracle's array."""
    worst = {}
    for k in KEYS:
        g = gpu[k] if select is None else select(k, gpu[k])
        worst[k] = compare(k, g, ref[k], tol)
    return worst


def compare_group(gpu, prob, n, hk, C):
    sub, heads = group_problem(prob, n, hk)
    ref = run_oracle(sub, prob.scale, C)

    def select(k, a):
        if k in ("y", "dv", "dg", "dbeta"):
            return a[n:n + 1][:, :, heads]
        if k in ("state_T", "ckpt", "dstate0"):
            return a[n:n + 1][:, heads]
        return a[n:n + 1][:, :, hk:hk + 1]  # dq, dk

    return compare_all(gpu, ref, tolerance(prob.T), select)
