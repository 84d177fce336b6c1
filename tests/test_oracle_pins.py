"""The float64 oracle against facts outside itself (CPU only).

Every pin in ``oracle_pins`` must hold for the oracle, and every planted defect (a copy
of the oracle built with -DGDN_ORACLE_MUTATION=m) must break at least one pin.
"""
import numpy as np
import pytest

import oracle
import oracle_pins as P
from gated_delta_rule_backward_gb300 import synth


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_fd_every_input(lib, kda):
    ok, detail = P.pin_fd(lib, kda)
    assert ok, detail


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_symbolic_exact_gradients(lib, kda):
    pytest.importorskip("sympy")
    ok, detail = P.pin_symbolic(lib, kda)
    assert ok, detail


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("pin", ["beta0", "reset", "exact_write", "homogeneity", "euler",
                                 "broadcast", "seq_broadcast", "ckpt_exact"])
def test_invariant(lib, pin, kda):
    ok, detail = getattr(P, "pin_" + pin)(lib, kda)
    assert ok, detail


def test_kda_equal_columns_is_scalar_gate(lib):
    ok, detail = P.pin_kda_equal(lib)
    assert ok, detail


def test_forward_t1_matrix_form(lib):
    """T = 1 against the matrix statement of the step (meTile, Recurrent delta attention):
    decayed = a (.) S, error = v - decayed^T k, S' = decayed + beta outer(k, error),
    y = scale S'^T q -- written here with S [K,V] (the transposed layout of M)."""
    for kda in (False, True):
        x = P._as64(synth.make_problem(1, 1, 1, 1, 16, kda=kda, seed=21))
        y, sT, ck = P._fwd(lib, x, C=1)
        S0 = x["state0"][0, 0].T                       # [K, V]
        a = np.exp(x["g"][0, 0, 0]) * np.ones(16) if not kda else np.exp(x["g"][0, 0, 0])
        k, q, v, b = x["k"][0, 0, 0], x["q"][0, 0, 0], x["v"][0, 0, 0], x["beta"][0, 0, 0]
        dec = a[:, None] * S0
        err = v - dec.T @ k
        S1 = dec + b * np.outer(k, err)
        assert np.allclose(sT[0, 0], S1.T, rtol=0, atol=1e-13)
        assert np.allclose(y[0, 0, 0], x["scale"] * S1.T @ q, rtol=0, atol=1e-13)
        assert np.array_equal(ck[0, 0, 0], x["state0"][0, 0])


def test_checkpoints_are_states_entering_each_segment(lib):
    x = P._as64(synth.make_problem(1, 10, 1, 1, 8, seed=22))
    _, _, ck = P._fwd(lib, x, C=4)                     # n_ck = 3: tokens 0, 4, 8
    assert ck.shape[2] == 3
    for c, t in enumerate((0, 4, 8)):
        xt = {kk: (vv[:, :t] if kk in ("q", "k", "v", "g", "beta", "gy") else vv)
              for kk, vv in x.items()}
        _, sT, _ = P._fwd(lib, xt, C=4)
        assert np.array_equal(sT, ck[:, :, c])


def test_empty_sequence(lib):
    x = P._as64(synth.make_problem(1, 3, 1, 2, 8, seed=23, dstate_T=True))
    x0 = {kk: (vv[:, :0] if kk in ("q", "k", "v", "g", "beta", "gy") else vv)
          for kk, vv in x.items()}
    y, sT, ck = P._fwd(lib, x0, C=2)
    assert y.shape[1] == 0 and ck.shape[2] == 0
    assert np.array_equal(sT, x["state0"])
    g = P._bwd(lib, x0, C=2)
    assert np.array_equal(g["dstate0"], x["dstate_T"])


def test_default_checkpoint_interval():
    import json, os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "checkpoint_interval.json")))
    for case in gold["cases"]:
        assert oracle.default_C(case["T"]) == case["C"]
    assert oracle.default_C(2048) == 46
    assert oracle.default_C(4096) == 64
    assert oracle.default_C(61) == 8
    assert oracle.default_C(1) == 1


@pytest.mark.parametrize("mutation,expect", [
    (1, "dstate_T seed dropped"),
    (2, "undecayed M_{t-1} in dk"),
    (3, "dM read after the du update in dk"),
    (4, "scale dropped from dq"),
    (5, "h_v / r head mapping"),
    (6, "gy ignored"),
    (7, "interleaved q/k sequence mapping"),
])
def test_planted_defect_is_caught(mutation, expect):
    mlib = oracle.load(mutation=mutation)
    assert mlib.gdn_oracle_mutation() == mutation
    res = P.battery(mlib)
    failed = [k for k, (ok, _) in res.items() if not ok]
    assert failed, f"defect '{expect}' passed every pin"


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_state_chaining_across_calls(lib, kda):
    """meTile "Recurrent delta attention": the final state is an output with its own
    cotangent and the initial state an input with its own gradient, so a sequence cut in
    two calls chains through them.  The forward of tokens [T1, T) from the state_T of
    tokens [0, T1), and the backward of [0, T1) seeded with the dstate0 of [T1, T), equal
    the single call on [0, T) bit for bit (every state is recomputed exactly)."""
    p = synth.make_problem(2, 37, 1, 2, 8, kda=kda, seed=61, dstate_T=True)
    f = lambda x: np.asarray(x, dtype=np.float64)
    T1 = 15
    y, sT, _ = oracle.forward(p.q, p.k, p.v, p.g, p.beta, p.state0, p.scale, C=4, lib=lib)
    gr = oracle.backward(p.q, p.k, p.v, p.g, p.beta, p.state0, p.gy, p.dstate_T, p.scale, C=4,
                         lib=lib)
    a, b = slice(0, T1), slice(T1, None)
    part = lambda x, s: np.ascontiguousarray(f(x)[:, s])
    y1, s1, _ = oracle.forward(part(p.q, a), part(p.k, a), part(p.v, a), part(p.g, a),
                               part(p.beta, a), p.state0, p.scale, C=4, lib=lib)
    y2, s2, _ = oracle.forward(part(p.q, b), part(p.k, b), part(p.v, b), part(p.g, b),
                               part(p.beta, b), s1, p.scale, C=4, lib=lib)
    g2 = oracle.backward(part(p.q, b), part(p.k, b), part(p.v, b), part(p.g, b), part(p.beta, b),
                         s1, part(p.gy, b), p.dstate_T, p.scale, C=4, lib=lib)
    g1 = oracle.backward(part(p.q, a), part(p.k, a), part(p.v, a), part(p.g, a), part(p.beta, a),
                         p.state0, part(p.gy, a), g2["dstate0"], p.scale, C=4, lib=lib)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(s2, sT)
    for k in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.array_equal(np.concatenate([g1[k], g2[k]], axis=1), gr[k]), k
    assert np.array_equal(g1["dstate0"], gr["dstate0"])
