"""Pins that tie the float64 oracle to facts outside itself.

Each pin takes an oracle library handle (the real one, or a copy built with a planted
defect) and returns (ok, detail).  ``tests/test_oracle_pins.py`` asserts that every pin
holds for the real oracle and that every planted defect fails at least one of them.

What each pin rests on:
  fd           central finite differences of the oracle's own forward, for every input
               element, under a random-weight objective over y AND state_T (so the
               final-state seed and the incoming gradient are both exercised: llama.cpp
               PR #26, SSM_SCAN_BACK section, "the state region is NOT zero").
  symbolic     exact gradients from sympy's differentiation of the recurrence written
               out symbolically (an independent derivation of the backward).
  beta0        beta = 0: the state only decays, M_t = (prod a) (.) M_0.
  reset        a = 0 (g = -inf): u = 0, M_t[j][i] = beta v_j k_i, y = scale beta (k.q) v.
  exact_write  a = 1, beta = 1, |k| = 1: the delta rule writes v exactly, M_t k_t = v_t.
  homogeneity  y and state_T are jointly linear in (state0, v).
  euler        sum<gy,y> = sum<dq,q>;  sum<gy,y> + <dsT,sT> = <dv,v> + <ds0,s0>.
  kda_equal    a KDA gate with equal columns equals the scalar gate (dg sums over i).
  broadcast    H_v = r H_k broadcast equals explicit replication with h_k = h_v mod H_k
               (PR #16: "iv1 % neq1"), dq/dk summed over the replicas.
  ckpt_exact   checkpointed backward equals store-all bit for bit (PR #26).
"""
from __future__ import annotations

import numpy as np

import oracle
from gated_delta_rule_backward_gb300 import synth


def _as64(p):
    f = lambda x: None if x is None else np.array(x, dtype=np.float64)
    return dict(q=f(p.q), k=f(p.k), v=f(p.v), g=f(p.g), beta=f(p.beta),
                state0=f(p.state0), gy=f(p.gy), dstate_T=f(p.dstate_T), scale=p.scale)


def _fwd(lib, x, C=None):
    return oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                          x["scale"], C=C, lib=lib)


def _bwd(lib, x, C=None, mode="checkpointed"):
    return oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                           x["gy"], x["dstate_T"], x["scale"], C=C, mode=mode, lib=lib)


def tiny(kda, seed, T=5, H_k=1, H_v=2, S_k=3, S_v=4):
    """A tiny problem with S_k != S_v (a transposed operand cannot go unnoticed)."""
    rng = np.random.default_rng(seed)
    p = synth.make_problem(1, T, H_k, H_v, S_k, kda=kda, seed=seed, dstate_T=True)
    x = _as64(p)
    # widen v / state / gy / dsT to S_v rows (synth draws square heads)
    x["v"] = rng.standard_normal((1, T, H_v, S_v))
    x["state0"] = 0.3 * rng.standard_normal((1, H_v, S_v, S_k))
    x["gy"] = rng.standard_normal((1, T, H_v, S_v))
    x["dstate_T"] = rng.standard_normal((1, H_v, S_v, S_k))
    return x


def pin_fd(lib, kda, seed=7, h=1e-6, tol=1e-6):
    x = tiny(kda, seed)
    W_y, W_s = x["gy"], x["dstate_T"]

    def objective(xx):
        y, sT, _ = _fwd(lib, xx, C=2)
        return float(np.sum(W_y * y) + np.sum(W_s * sT))

    grads = _bwd(lib, x, C=2)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "state0": "dstate0"}
    worst = 0.0
    for name, gname in names.items():
        base = x[name]
        an = grads[gname]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            xp = dict(x); xm = dict(x)
            xp[name] = base.copy(); xm[name] = base.copy()
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (objective(xp) - objective(xm)) / (2 * h)
        err = float(np.max(np.abs(fd - an) / (1.0 + np.abs(an))))
        worst = max(worst, err)
        if not err <= tol:
            return False, f"fd mismatch on {name}: {err:.3e}"
    return True, f"worst {worst:.2e}"


def pin_symbolic(lib, kda, seed=11, tol=1e-11):
    """Exact gradients by sympy, T=3, H_k=1, H_v=2, S_k=2, S_v=2."""
    import sympy as sp

    x = tiny(kda, seed, T=3, H_k=1, H_v=2, S_k=2, S_v=2)
    N, T, H_k, S_k = x["q"].shape
    H_v, S_v = x["v"].shape[2], x["v"].shape[3]
    syms = {}

    def sym_array(name, arr):
        out = np.empty(arr.shape, dtype=object)
        for idx in np.ndindex(arr.shape):
            s = sp.Symbol(name + "_" + "_".join(map(str, idx)))
            syms[s] = arr[idx]
            out[idx] = s
        return out

    S = {n: sym_array(n, x[n]) for n in ("q", "k", "v", "g", "beta", "state0")}
    L = 0
    for hv in range(H_v):
        hk = hv % H_k
        M = [[S["state0"][0, hv, j, i] for i in range(S_k)] for j in range(S_v)]
        for t in range(T):
            if kda:
                a = [sp.exp(S["g"][0, t, hv, i]) for i in range(S_k)]
            else:
                a = [sp.exp(S["g"][0, t, hv])] * S_k
            kk = [S["k"][0, t, hk, i] for i in range(S_k)]
            qq = [S["q"][0, t, hk, i] for i in range(S_k)]
            b = S["beta"][0, t, hv]
            dec = [[a[i] * M[j][i] for i in range(S_k)] for j in range(S_v)]
            err = [S["v"][0, t, hv, j] - sum(dec[j][i] * kk[i] for i in range(S_k))
                   for j in range(S_v)]
            M = [[dec[j][i] + b * kk[i] * err[j] for i in range(S_k)] for j in range(S_v)]
            for j in range(S_v):
                y = x["scale"] * sum(M[j][i] * qq[i] for i in range(S_k))
                L += x["gy"][0, t, hv, j] * y
        for j in range(S_v):
            for i in range(S_k):
                L += x["dstate_T"][0, hv, j, i] * M[j][i]
    grads = _bwd(lib, x, C=2)
    names = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "state0": "dstate0"}
    subs = {s: sp.Float(val, 40) for s, val in syms.items()}
    worst = 0.0
    for name, gname in names.items():
        for idx in np.ndindex(S[name].shape):
            exact = float(sp.diff(L, S[name][idx]).evalf(30, subs=subs))
            got = grads[gname][idx]
            err = abs(exact - got) / (1.0 + abs(exact))
            worst = max(worst, err)
            if not err <= tol:
                return False, f"symbolic mismatch {name}{idx}: {got} vs {exact}"
    return True, f"worst {worst:.2e}"


def pin_beta0(lib, kda, seed=3):
    p = synth.make_problem(1, 9, 2, 4, 8, kda=kda, seed=seed)
    x = _as64(p)
    x["beta"] = np.zeros_like(x["beta"])
    y, sT, _ = _fwd(lib, x, C=3)
    a = np.exp(x["g"])
    M = x["state0"].copy()  # [N,H_v,S_v,S_k]
    worst = 0.0
    for t in range(x["q"].shape[1]):
        at = a[:, t]  # [N,H_v] or [N,H_v,S_k]
        M = M * (at[:, :, None, None] if not kda else at[:, :, None, :])
        hk = np.arange(x["v"].shape[2]) % x["q"].shape[2]
        yt = x["scale"] * np.einsum("nhji,nhi->nhj", M, x["q"][:, t, hk])
        worst = max(worst, float(np.max(np.abs(yt - y[:, t]))))
    worst = max(worst, float(np.max(np.abs(M - sT))))
    return worst < 1e-12, f"max dev {worst:.2e}"


def pin_reset(lib, kda, seed=4):
    p = synth.make_problem(1, 6, 2, 4, 8, kda=kda, seed=seed)
    x = _as64(p)
    x["g"] = np.full_like(x["g"], -np.inf)
    y, sT, _ = _fwd(lib, x, C=4)
    T = x["q"].shape[1]
    hk = np.arange(x["v"].shape[2]) % x["q"].shape[2]
    worst = 0.0
    for t in range(T):
        kt, qt = x["k"][:, t, hk], x["q"][:, t, hk]         # [N,H_v,S_k]
        bt, vt = x["beta"][:, t], x["v"][:, t]              # [N,H_v], [N,H_v,S_v]
        kq = np.sum(kt * qt, axis=-1)
        yt = x["scale"] * (bt * kq)[..., None] * vt
        worst = max(worst, float(np.max(np.abs(yt - y[:, t]))))
    Mt = x["beta"][:, T - 1][..., None, None] * x["v"][:, T - 1][..., :, None] \
        * x["k"][:, T - 1, hk][..., None, :]
    worst = max(worst, float(np.max(np.abs(Mt - sT))))
    return worst < 1e-12, f"max dev {worst:.2e}"


def pin_exact_write(lib, kda, seed=5):
    p = synth.make_problem(1, 7, 1, 2, 8, kda=kda, seed=seed)
    x = _as64(p)
    x["g"] = np.zeros_like(x["g"])
    x["beta"] = np.ones_like(x["beta"])
    x["k"] = x["k"] / np.linalg.norm(x["k"], axis=-1, keepdims=True)  # |k| = 1 in float64
    T = x["q"].shape[1]
    worst = 0.0
    for t in range(1, T + 1):
        xt = {kk: (vv[:, :t] if kk in ("q", "k", "v", "g", "beta", "gy") else vv)
              for kk, vv in x.items()}
        _, sT, _ = _fwd(lib, xt, C=3)
        kt = x["k"][:, t - 1, np.arange(2) % 1]
        Mk = np.einsum("nhji,nhi->nhj", sT, kt)
        worst = max(worst, float(np.max(np.abs(Mk - x["v"][:, t - 1]))))
    return worst < 1e-12, f"max dev {worst:.2e}"


def pin_homogeneity(lib, kda, seed=6, lam=-2.5):
    x = _as64(synth.make_problem(2, 8, 2, 4, 8, kda=kda, seed=seed))
    y1, s1, _ = _fwd(lib, x, C=3)
    x2 = dict(x); x2["v"] = lam * x["v"]; x2["state0"] = lam * x["state0"]
    y2, s2, _ = _fwd(lib, x2, C=3)
    dev = max(float(np.max(np.abs(y2 - lam * y1))), float(np.max(np.abs(s2 - lam * s1))))
    return dev < 1e-12, f"max dev {dev:.2e}"


def pin_euler(lib, kda, seed=8):
    x = _as64(synth.make_problem(2, 11, 2, 4, 8, kda=kda, seed=seed, dstate_T=True))
    y, sT, _ = _fwd(lib, x, C=3)
    gr = _bwd(lib, x, C=3)
    L_y = float(np.sum(x["gy"] * y))
    L_s = float(np.sum(x["dstate_T"] * sT))
    e1 = abs(L_y - float(np.sum(gr["dq"] * x["q"])))
    e2 = abs(L_y + L_s - float(np.sum(gr["dv"] * x["v"]) + np.sum(gr["dstate0"] * x["state0"])))
    ok = e1 < 1e-10 * (1 + abs(L_y)) and e2 < 1e-10 * (1 + abs(L_y + L_s))
    return ok, f"e1 {e1:.2e} e2 {e2:.2e}"


def pin_kda_equal(lib, seed=9):
    xs = _as64(synth.make_problem(1, 10, 2, 4, 8, kda=False, seed=seed, dstate_T=True))
    xk = dict(xs)
    xk["g"] = np.repeat(xs["g"][..., None], 8, axis=-1)
    ys, ss, _ = _fwd(lib, xs, C=4)
    yk, sk, _ = _fwd(lib, xk, C=4)
    gs = _bwd(lib, xs, C=4)
    gk = _bwd(lib, xk, C=4)
    dev = max(float(np.max(np.abs(ys - yk))), float(np.max(np.abs(ss - sk))))
    for n in ("dq", "dk", "dv", "dbeta", "dstate0"):
        dev = max(dev, float(np.max(np.abs(gs[n] - gk[n]))))
    dev = max(dev, float(np.max(np.abs(gs["dg"] - gk["dg"].sum(-1)))))
    return dev < 1e-11, f"max dev {dev:.2e}"


def pin_broadcast(lib, kda, seed=10):
    H_k, H_v = 2, 6
    x = _as64(synth.make_problem(1, 7, H_k, H_v, 8, kda=kda, seed=seed, dstate_T=True))
    rep = dict(x)
    hk = np.arange(H_v) % H_k
    rep["q"] = x["q"][:, :, hk].copy()
    rep["k"] = x["k"][:, :, hk].copy()
    yb, sb, _ = _fwd(lib, x, C=3)
    yr, sr, _ = _fwd(lib, rep, C=3)
    gb = _bwd(lib, x, C=3)
    gr = _bwd(lib, rep, C=3)
    dev = max(float(np.max(np.abs(yb - yr))), float(np.max(np.abs(sb - sr))))
    for h in range(H_k):
        heads = [hv for hv in range(H_v) if hv % H_k == h]  # ascending h_v
        for n in ("dq", "dk"):
            acc = np.zeros_like(gr[n][:, :, 0])
            for hv in heads:
                acc = acc + gr[n][:, :, hv]
            dev = max(dev, float(np.max(np.abs(acc - gb[n][:, :, h]))))
    for n in ("dv", "dg", "dbeta", "dstate0"):
        dev = max(dev, float(np.max(np.abs(gb[n] - gr[n]))))
    return dev < 1e-12, f"max dev {dev:.2e}"


def pin_seq_broadcast(lib, kda, seed=13):
    """Sequence broadcast (PR #16 "iv3/rq3"): value sequence n reads q/k sequence n / rep.
    It must equal the same problem with q, k repeated per value sequence (np.repeat: rows
    0, 0, 1, 1, ...), with dq/dk summed over each group of rep sequences."""
    rep_, N = 2, 4
    x = _as64(synth.make_problem(N, 7, 1, 2, 8, kda=kda, seed=seed, dstate_T=True, seq_rep=rep_))
    r = dict(x)
    r["q"] = np.repeat(x["q"], rep_, axis=0)
    r["k"] = np.repeat(x["k"], rep_, axis=0)
    yb, sb, _ = _fwd(lib, x, C=3)
    yr, sr, _ = _fwd(lib, r, C=3)
    gb = _bwd(lib, x, C=3)
    gr = _bwd(lib, r, C=3)
    dev = max(float(np.max(np.abs(yb - yr))), float(np.max(np.abs(sb - sr))))
    for n in ("dq", "dk"):
        acc = gr[n][0::rep_] + gr[n][1::rep_]  # ascending value sequence within each group
        dev = max(dev, float(np.max(np.abs(acc - gb[n]))))
    for n in ("dv", "dg", "dbeta", "dstate0"):
        dev = max(dev, float(np.max(np.abs(gb[n] - gr[n]))))
    return dev < 1e-12, f"max dev {dev:.2e}"


def pin_ckpt_exact(lib, kda, seed=12, T=13):
    x = _as64(synth.make_problem(2, T, 1, 2, 8, kda=kda, seed=seed, dstate_T=True))
    ref = _bwd(lib, x, mode="store_all", C=1)
    for C in (1, 3, oracle.default_C(T), T, T + 5):
        got = _bwd(lib, x, C=C)
        for n in ref:
            if not np.array_equal(ref[n], got[n]):
                return False, f"C={C}: {n} differs from store-all"
    return True, "bit-identical"


def battery(lib, quick=False):
    """All pins, both gates.  Returns {name: (ok, detail)}."""
    res = {}
    for kda in (False, True):
        tag = "kda" if kda else "scalar"
        res[f"fd_{tag}"] = pin_fd(lib, kda)
        res[f"beta0_{tag}"] = pin_beta0(lib, kda)
        res[f"reset_{tag}"] = pin_reset(lib, kda)
        res[f"exact_write_{tag}"] = pin_exact_write(lib, kda)
        res[f"homogeneity_{tag}"] = pin_homogeneity(lib, kda)
        res[f"euler_{tag}"] = pin_euler(lib, kda)
        res[f"broadcast_{tag}"] = pin_broadcast(lib, kda)
        res[f"seq_broadcast_{tag}"] = pin_seq_broadcast(lib, kda)
        res[f"ckpt_exact_{tag}"] = pin_ckpt_exact(lib, kda)
    res["kda_equal"] = pin_kda_equal(lib)
    return res
