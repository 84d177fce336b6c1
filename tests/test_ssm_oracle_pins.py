"""The float64 selective-scan oracle against facts outside itself (CPU only).

Pins (llama.cpp PR #26, the SSM_SCAN_BACK section, and the mathematics of a linear scan):
  fd            central differences of an objective that weights y AND the final states
                (the packed cotangent's state region is not zero), every input element,
                both branches, two groups, store-all and checkpointed walks
  ckpt_exact    checkpointed walks (several K) equal the store-all walk bit for bit, and
                the forward's checkpoints are the store-all states
  prefix_sum    A = 0 (no decay): s_t = s0 + cumulative sum of B x dt, in numpy
  dt_zero       dt = 0: the state never moves, and every gradient has a closed form
  scalar        P = S = 1: the scalar linear recurrence written with explicit products
  group_fold    G groups against one group per head with B, C replicated: y equal, and dB,
                dC of a group the sums over its heads
  mamba2_is_mamba1  one decay per head equals the per-state form with equal entries
Every planted defect (a copy built with -DSSM_ORACLE_MUTATION=m) must break one of them.
"""
import numpy as np
import pytest

from oracle import ssm
from gated_delta_rule_backward_gb300.ssm_synth import make_ssm_problem


def _prob(N=2, T=5, H=4, P=2, S=3, G=2, mamba1=False, seed=3, K=2):
    p = make_ssm_problem(N, T, H, P, S, G=G, mamba1=mamba1, K=K, seed=seed)
    d = {k: getattr(p, k).astype(np.float64) for k in ("s0", "x", "dt", "A", "B", "C", "dy", "ds_T")}
    # larger steps than the recipe's so that every path of d(dt) is well above FD noise
    d["dt"] = d["dt"] * 5.0
    return d, p.K


def _objective(lib, d, K):
    y, sT, _ = ssm.forward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], K=K, lib=lib)
    return float(np.sum(d["dy"] * y) + np.sum(d["ds_T"] * sT))


def pin_fd(lib, mamba1, mode):
    d, K = _prob(mamba1=mamba1)
    g = ssm.backward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["dy"], d["ds_T"], K=K, mode=mode, lib=lib)
    worst = 0.0
    for name, gname in (("s0", "ds0"), ("x", "dx"), ("dt", "ddt"), ("B", "dB"), ("C", "dC")):
        base = d[name]
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            h = 1e-6 * max(1.0, abs(base[i]))
            orig = base[i]
            base[i] = orig + h
            fp = _objective(lib, d, K)
            base[i] = orig - h
            fm = _objective(lib, d, K)
            base[i] = orig
            fd = (fp - fm) / (2 * h)
            an = g[gname][i]
            err = abs(fd - an) / (1.0 + abs(an))
            worst = max(worst, err)
            if err > 1e-7:
                return False, f"{gname}{i}: fd {fd:.12g} analytic {an:.12g}"
    return True, f"worst {worst:.2e}"


def pin_ckpt_exact(lib, mamba1):
    d, _ = _prob(N=1, T=7, mamba1=mamba1)
    args = (d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"])
    ref = ssm.backward(*args, d["dy"], d["ds_T"], K=1, mode="store_all", lib=lib)
    y1, s1, ck1 = ssm.forward(*args, K=1, lib=lib)
    for K in (1, 2, 3, 7, 9):
        got = ssm.backward(*args, d["dy"], d["ds_T"], K=K, mode="checkpointed", lib=lib)
        for k in ref:
            if not np.array_equal(ref[k], got[k]):
                return False, f"K={K}: {k} differs from store-all"
        y, s, ck = ssm.forward(*args, K=K, lib=lib)
        if not (np.array_equal(y, y1) and np.array_equal(s, s1)):
            return False, f"K={K}: forward differs"
        for c in range(ck.shape[2]):
            if not np.array_equal(ck[:, :, c], ck1[:, :, c * K]):
                return False, f"K={K}: checkpoint {c} is not the state entering token {c * K}"
    return True, ""


def _route(H, G):
    return np.arange(H) // (H // G)


def pin_prefix_sum(lib, mamba1):
    d, K = _prob(mamba1=mamba1)
    d["A"] = np.zeros_like(d["A"])
    y, sT, _ = ssm.forward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], K=K, lib=lib)
    Bh = d["B"][:, :, _route(4, 2)]                                   # [N,T,H,S]
    Ch = d["C"][:, :, _route(4, 2)]
    write = Bh[:, :, :, None, :] * (d["x"] * d["dt"][..., None])[..., None]  # [N,T,H,P,S]
    st = d["s0"][:, None] + np.cumsum(write, axis=1)                  # [N,T,H,P,S]
    y_ref = np.einsum("nthps,nths->nthp", st, Ch)
    ok = np.allclose(y, y_ref, rtol=1e-12, atol=1e-12) and np.allclose(sT, st[:, -1], rtol=1e-12, atol=1e-12)
    return ok, f"max |y - ref| {np.max(np.abs(y - y_ref)):.2e}"


def pin_dt_zero(lib, mamba1):
    d, K = _prob(mamba1=mamba1)
    d["dt"] = np.zeros_like(d["dt"])
    y, sT, _ = ssm.forward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], K=K, lib=lib)
    g = ssm.backward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["dy"], d["ds_T"], K=K, lib=lib)
    r = _route(4, 2)
    Bh, Ch = d["B"][:, :, r], d["C"][:, :, r]
    y_ref = np.einsum("nhps,nths->nthp", d["s0"], Ch)
    # the state gradient after token t: ds_T plus every later (and this) token's dy C^T
    outer = d["dy"][..., None] * Ch[:, :, :, None, :]                 # [N,T,H,P,S]
    ds_t = d["ds_T"][:, None] + np.flip(np.cumsum(np.flip(outer, 1), 1), 1)
    Ah = d["A"][:, :] if mamba1 else d["A"][:, None]                  # [H,S] or [H,1]
    ddt_ref = (np.einsum("nthps,nths,nthp->nth", ds_t, Bh, d["x"])
               + np.einsum("nthps,hs,nhps->nth", ds_t, np.broadcast_to(Ah, (4, 3)), d["s0"]))
    dC_h = np.einsum("nthp,nhps->nths", d["dy"], d["s0"])
    dC_ref = dC_h.reshape(2, 5, 2, 2, 3).sum(axis=3)                 # heads folded into groups
    checks = [
        ("y", np.allclose(y, y_ref, rtol=1e-12, atol=1e-12)),
        ("sT", np.array_equal(sT, d["s0"])),
        ("dx", np.array_equal(g["dx"], np.zeros_like(g["dx"]))),
        ("dB", np.array_equal(g["dB"], np.zeros_like(g["dB"]))),
        ("ds0", np.allclose(g["ds0"], ds_t[:, 0], rtol=1e-12, atol=1e-12)),
        ("ddt", np.allclose(g["ddt"], ddt_ref, rtol=1e-11, atol=1e-11)),
        ("dC", np.allclose(g["dC"], dC_ref, rtol=1e-12, atol=1e-12)),
    ]
    bad = [n for n, ok in checks if not ok]
    return not bad, f"failed: {bad}"


def pin_scalar(lib):
    d, K = _prob(N=1, T=6, H=1, P=1, S=1, G=1, mamba1=True)
    y, sT, _ = ssm.forward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], K=K, lib=lib)
    a = np.exp(d["dt"][0, :, 0] * d["A"][0, 0])
    b = d["B"][0, :, 0, 0] * d["x"][0, :, 0, 0] * d["dt"][0, :, 0]
    c = d["C"][0, :, 0, 0]
    s0 = d["s0"][0, 0, 0, 0]
    ref = []
    for t in range(6):
        st = np.prod(a[: t + 1]) * s0 + sum(np.prod(a[tau + 1: t + 1]) * b[tau] for tau in range(t + 1))
        ref.append(st * c[t])
    ok = np.allclose(y[0, :, 0, 0], ref, rtol=1e-13, atol=1e-14)
    return ok, f"{y[0, :, 0, 0]} vs {ref}"


def pin_group_fold(lib, mamba1):
    d, K = _prob(N=1, T=6, H=4, P=2, S=3, G=2, mamba1=mamba1)
    r = _route(4, 2)
    args_g = (d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"])
    args_h = (d["s0"], d["x"], d["dt"], d["A"], d["B"][:, :, r], d["C"][:, :, r])
    yg, sg, _ = ssm.forward(*args_g, K=K, lib=lib)
    yh, sh, _ = ssm.forward(*args_h, K=K, lib=lib)
    gg = ssm.backward(*args_g, d["dy"], d["ds_T"], K=K, lib=lib)
    gh = ssm.backward(*args_h, d["dy"], d["ds_T"], K=K, lib=lib)
    fold = lambda a: a.reshape(a.shape[0], a.shape[1], 2, 2, a.shape[3]).sum(axis=3)
    checks = [
        ("y", np.array_equal(yg, yh)), ("sT", np.array_equal(sg, sh)),
        ("dx", np.array_equal(gg["dx"], gh["dx"])), ("ddt", np.array_equal(gg["ddt"], gh["ddt"])),
        ("ds0", np.array_equal(gg["ds0"], gh["ds0"])),
        ("dB", np.allclose(gg["dB"], fold(gh["dB"]), rtol=1e-13, atol=1e-14)),
        ("dC", np.allclose(gg["dC"], fold(gh["dC"]), rtol=1e-13, atol=1e-14)),
    ]
    bad = [n for n, ok in checks if not ok]
    return not bad, f"failed: {bad}"


def pin_mamba2_is_mamba1(lib):
    d, K = _prob(mamba1=False)
    A1 = np.repeat(d["A"][:, None], 3, axis=1)
    a2 = (d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"])
    a1 = (d["s0"], d["x"], d["dt"], A1, d["B"], d["C"])
    y2, s2, _ = ssm.forward(*a2, K=K, lib=lib)
    y1, s1, _ = ssm.forward(*a1, K=K, lib=lib)
    g2 = ssm.backward(*a2, d["dy"], d["ds_T"], K=K, lib=lib)
    g1 = ssm.backward(*a1, d["dy"], d["ds_T"], K=K, lib=lib)
    ok = np.array_equal(y1, y2) and np.array_equal(s1, s2) and all(np.array_equal(g1[k], g2[k]) for k in g1)
    return ok, ""


@pytest.fixture(scope="module")
def lib():
    return ssm.load()


@pytest.mark.parametrize("mode", ["store_all", "checkpointed"])
@pytest.mark.parametrize("mamba1", [False, True], ids=["mamba2", "mamba1"])
def test_fd_every_input(lib, mamba1, mode):
    ok, detail = pin_fd(lib, mamba1, mode)
    assert ok, detail


@pytest.mark.parametrize("mamba1", [False, True], ids=["mamba2", "mamba1"])
@pytest.mark.parametrize("pin", ["ckpt_exact", "prefix_sum", "dt_zero", "group_fold"])
def test_invariant(lib, pin, mamba1):
    ok, detail = globals()["pin_" + pin](lib, mamba1)
    assert ok, detail


def test_scalar_recurrence(lib):
    ok, detail = pin_scalar(lib)
    assert ok, detail


def test_mamba2_is_mamba1_with_equal_states(lib):
    ok, detail = pin_mamba2_is_mamba1(lib)
    assert ok, detail


def test_empty_sequence(lib):
    d, _ = _prob(T=0)
    y, sT, ck = ssm.forward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], K=2, lib=lib)
    g = ssm.backward(d["s0"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["dy"], d["ds_T"], K=2, lib=lib)
    assert y.size == 0 and np.array_equal(sT, d["s0"]) and np.array_equal(ck[:, :, 0], d["s0"])
    assert np.array_equal(g["ds0"], d["ds_T"])


def _all_pins_hold(lib):
    checks = [pin_fd(lib, False, "checkpointed"), pin_fd(lib, True, "store_all"), pin_ckpt_exact(lib, False),
              pin_prefix_sum(lib, True), pin_dt_zero(lib, False), pin_scalar(lib), pin_group_fold(lib, False),
              pin_mamba2_is_mamba1(lib)]
    return all(ok for ok, _ in checks)


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5, 6])
def test_planted_defect_is_caught(mutation):
    mlib = ssm.load(mutation=mutation)
    assert mlib.ssm_oracle_mutation() == mutation
    assert not _all_pins_hold(mlib), f"planted defect {mutation} passed every pin"
