"""The selective scan's CUDA path (include/ssm.h) against the float64 oracle, element by
element, through the C ABI.

Tolerance: every output's largest absolute difference over its largest magnitude, at most
2e-5 up to 512 tokens and 1e-4 at 4096 (fp32 states: the rounding of a step is ~6e-8 of
the state, and a decayed sum over T steps collects ~sqrt(T) of them; the oracle is
float64).  The token-serial walk's results at different checkpoint intervals, and every
path's results over repeated calls, must agree bit for bit (the walk recomputes the
forward's own states; every sum runs in a fixed order).

All three forms run here: one decay per head with P = 64, S = 128 and K a multiple of 64
takes the chunked form (64-token chunks); a decay per state with P = 1, S = 16, H / G a
multiple of 16 and ceil(T / K) 16 <= T the segmented form; every other size the token-serial
walk.  Each case asserts which one it exercises.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_backward_gb300 import ssm
from gated_delta_rule_backward_gb300.ssm_synth import make_ssm_problem, ssm_workload

pytestmark = pytest.mark.gpu

NAMES = ("y", "sT", "ckpt", "ds0", "dx", "ddt", "dB", "dC")


def _tol(T):
    return 2e-5 if T <= 512 else 1e-4


def run_gpu(prob, K=None, heads=None):
    """Forward and backward on cuda:0; returns numpy arrays of every output."""
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    s0, x, dt, A, B, C, dy, dsT = map(t, (prob.s0, prob.x, prob.dt, prob.A, prob.B, prob.C, prob.dy, prob.ds_T))
    p = ssm.params_for(x, A, B, K=prob.K if K is None else K)
    out = torch.empty(ssm.packed_out_elems(p), device=dev)
    ck = torch.empty((p.N, p.H, ssm.num_checkpoints(p), p.P, p.S), device=dev)
    ssm.ssm_forward(p, s0, x, dt, A, B, C, out, ck)
    gin = ssm.pack_grad_in(p, dy, dsT)
    gout = torch.empty(ssm.packed_grad_elems(p), device=dev)
    ws = torch.empty(max(ssm.backward_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    ssm.ssm_backward(p, x, dt, A, B, C, ck, gin, gout, ws)
    torch.cuda.synchronize()
    y, sT = ssm.split_out(p, out)
    ds0, dx, ddt, dB, dC = ssm.split_grads(p, gout)
    r = dict(y=y, sT=sT, ckpt=ck, ds0=ds0, dx=dx, ddt=ddt, dB=dB, dC=dC)
    return {k: v.cpu().numpy() for k, v in r.items()}


def run_oracle(prob, K=None, lib=None):
    from oracle import ssm as oss
    K = prob.K if K is None else K
    y, sT, ck = oss.forward(prob.s0, prob.x, prob.dt, prob.A, prob.B, prob.C, K=K, lib=lib)
    g = oss.backward(prob.s0, prob.x, prob.dt, prob.A, prob.B, prob.C, prob.dy, prob.ds_T, K=K, ckpt=ck, lib=lib)
    return dict(y=y, sT=sT, ckpt=ck, **g)


def compare(gpu, ref, tol, names=NAMES):
    worst = {}
    for k in names:
        a, b = gpu[k].astype(np.float64), ref[k]
        assert a.shape == b.shape, (k, a.shape, b.shape)
        if b.size == 0:
            continue
        scale = max(np.max(np.abs(b)), 1e-30)
        err = np.max(np.abs(a - b)) / scale
        worst[k] = err
        assert np.all(np.isfinite(a)), k
        assert err <= tol, f"{k}: {err:.3e} > {tol:.1e}"
    return worst


CASES = [
    dict(N=2, T=100, H=8, P=64, S=128, G=2, mamba1=False, K=16),     # token-serial at Mamba-2 sizes
    dict(N=2, T=100, H=8, P=64, S=128, G=2, mamba1=False, K=64),     # chunked: a ragged 2nd chunk
    dict(N=1, T=300, H=4, P=64, S=128, G=1, mamba1=False, K=128),    # chunked: 2 chunks a segment
    dict(N=1, T=200, H=6, P=64, S=128, G=3, mamba1=False, K=192),    # chunked: 3 a segment, 1 used
    dict(N=3, T=64, H=2, P=64, S=128, G=1, mamba1=False, K=64),      # chunked: one full chunk
    dict(N=1, T=1, H=2, P=64, S=128, G=2, mamba1=False, K=64),       # chunked: one token
    dict(N=2, T=100, H=96, P=1, S=16, G=1, mamba1=True, K=16),
    dict(N=1, T=37, H=4, P=32, S=64, G=4, mamba1=False, K=5),     # ragged last segment
    dict(N=3, T=1, H=2, P=16, S=32, G=1, mamba1=True, K=1),
    dict(N=1, T=50, H=2, P=8, S=256, G=2, mamba1=False, K=7),
    dict(N=1, T=64, H=64, P=2, S=16, G=2, mamba1=True, K=64),     # several heads per block
    dict(N=2, T=29, H=6, P=48, S=32, G=3, mamba1=False, K=4),
    dict(N=2, T=300, H=32, P=1, S=16, G=2, mamba1=True, K=37),       # segmented: ragged segments
    dict(N=1, T=200, H=16, P=1, S=16, G=1, mamba1=True, K=100),      # segmented: 4 sub-blocks a segment
    dict(N=3, T=64, H=48, P=1, S=16, G=3, mamba1=True, K=16),        # segmented: n_ck 16 = T
]


def expected_form(c):
    n_ck = -(-c["T"] // c["K"])
    if not c["mamba1"] and c["P"] == 64 and c["S"] == 128 and c["K"] % 64 == 0:
        return "chunked"
    if c["mamba1"] and c["P"] == 1 and c["S"] == 16 and (c["H"] // c["G"]) % 16 == 0 and n_ck * 16 <= c["T"]:
        return "segmented"
    return "token-serial"


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"N{c['N']}T{c['T']}H{c['H']}P{c['P']}S{c['S']}G{c['G']}"
                                               f"{'m1' if c['mamba1'] else 'm2'}K{c['K']}")
def test_parity(case):
    prob = make_ssm_problem(seed=7, **case)
    p = ssm.make_params(prob.N, prob.T, prob.H, prob.P, prob.S, prob.G, prob.mamba1, prob.K)
    assert ssm.form(p) == expected_form(case)
    assert ssm.chunked(p) == (ssm.form(p) == "chunked")
    gpu = run_gpu(prob)
    ref = run_oracle(prob)
    compare(gpu, ref, _tol(prob.T))


def test_empty_sequence():
    prob = make_ssm_problem(N=2, T=0, H=8, P=8, S=16, G=2, K=3, seed=2)
    gpu = run_gpu(prob)
    assert gpu["y"].size == 0
    assert np.array_equal(gpu["sT"], prob.s0) and np.array_equal(gpu["ckpt"][:, :, 0], prob.s0)
    assert np.array_equal(gpu["ds0"], prob.ds_T)


@pytest.mark.parametrize("mamba1", [False, True], ids=["mamba2", "mamba1"])
def test_checkpoint_interval_invariance_bitwise(mamba1):
    """The token-serial walk's results do not depend on K (two channels a head keep a decay per
    state on the walk at every K)."""
    prob = make_ssm_problem(N=1, T=77, H=8 if not mamba1 else 32, P=16 if not mamba1 else 2,
                            S=64 if not mamba1 else 16, G=2, mamba1=mamba1, K=8, seed=9)
    base = run_gpu(prob, K=1)
    for K in (3, 8, 77, 100):
        assert ssm.form(ssm.make_params(1, 77, prob.H, prob.P, prob.S, 2, mamba1, K)) == "token-serial"
        got = run_gpu(prob, K=K)
        for k in NAMES:
            if k == "ckpt":
                continue
            assert np.array_equal(got[k], base[k]), f"K={K}: {k}"
        ck = got["ckpt"]
        for c in range(ck.shape[2]):
            assert np.array_equal(ck[:, :, c], base["ckpt"][:, :, c * K]), f"K={K}: checkpoint {c}"


@pytest.mark.parametrize("wl,K,form", [("mamba2_small", 16, "token-serial"), ("mamba2_small", 64, "chunked"),
                                       ("mamba1_small", 20, "segmented")], ids=["serial", "chunked", "segmented"])
def test_run_to_run_bitwise(wl, K, form):
    prob = ssm_workload(wl, K=K)
    assert ssm.form(ssm.make_params(prob.N, prob.T, prob.H, prob.P, prob.S, prob.G, prob.mamba1, prob.K)) == form
    a, b = run_gpu(prob), run_gpu(prob)
    for k in NAMES:
        assert np.array_equal(a[k], b[k]), k


def test_chunked_strong_decay():
    """dt up to 3 (a chunk's decay exp(64 dt A) far below fp32's range): the masks and the
    carried state underflow to zero, as the token-serial products do."""
    prob = make_ssm_problem(N=1, T=130, H=4, P=64, S=128, G=1, K=64, seed=5)
    prob.dt = np.ascontiguousarray(prob.dt * 30, dtype=np.float32)
    assert ssm.chunked(ssm.make_params(1, 130, 4, 64, 128, 1, False, 64))
    compare(run_gpu(prob), run_oracle(prob), _tol(prob.T))


def test_chunked_head_blocks_groups_sequences():
    """Head blocks over two groups and two sequences (N = 2, G = 2, 32 heads, 1024 tokens: two
    heads a block), against the oracle on every output."""
    prob = make_ssm_problem(N=2, T=1024, H=32, P=64, S=128, G=2, K=64, seed=21)
    assert ssm.chunked(ssm.make_params(2, 1024, 32, 64, 128, 2, False, 64))
    compare(run_gpu(prob), run_oracle(prob), _tol(prob.T))


def test_mamba2_all_heads_chunked():
    """Every head of the Mamba-2 workload at 1024 tokens in chunked form: the gradient kernel
    takes two heads a block here, so dB and dC fold 40 block partials of 2 heads each."""
    prob = ssm_workload("mamba2_h80_T4096", T=1024, K=64)
    assert ssm.chunked(ssm.params_for(torch.from_numpy(prob.x), torch.from_numpy(prob.A),
                                      torch.from_numpy(prob.B), K=64))
    compare(run_gpu(prob), run_oracle(prob), _tol(prob.T))


def test_mamba1_full_size():
    """The Mamba-1 workload (1536 channels of 16 states, 4096 tokens, segmented form) against
    the oracle."""
    prob = ssm_workload("mamba1_d1536_T4096")
    assert ssm.form(ssm.make_params(1, 4096, 1536, 1, 16, 1, True, 64)) == "segmented"
    compare(run_gpu(prob), run_oracle(prob), _tol(prob.T))


def test_mamba2_all_heads_short():
    """Every head of the Mamba-2 workload (80 heads of 64 channels, 128 states, one group),
    cut to 256 tokens, so that dB and dC fold all 80 heads."""
    prob = ssm_workload("mamba2_h80_T4096", T=256, K=16)
    compare(run_gpu(prob), run_oracle(prob), _tol(prob.T))


def test_mamba2_full_size_sampled():
    """The Mamba-2 workload at 4096 tokens.  Heads 0, 27, 53, 79 against the oracle run on
    those heads alone (their y, s_T, checkpoints, d_s, d_x, d_dt depend on no other head);
    dB and dC through identities that hold per token at any size:
        sum_j dC[t][j] C[t][j] = sum_{h,p} dy[t][h][p] y[t][h][p]
        sum_j dB[t][j] B[t][j] = sum_{h,p} x[t][h][p] dx[t][h][p]."""
    prob = ssm_workload("mamba2_h80_T4096")
    gpu = run_gpu(prob)
    heads = [0, 27, 53, 79]
    sub = make_ssm_problem(1, 1, 4, 64, 128, G=1, K=prob.K, seed=0)
    for f in ("x", "dt", "dy"):
        setattr(sub, f, np.ascontiguousarray(getattr(prob, f)[:, :, heads]))
    for f in ("s0", "ds_T"):
        setattr(sub, f, np.ascontiguousarray(getattr(prob, f)[:, heads]))
    sub.A = np.ascontiguousarray(prob.A[heads])
    sub.B, sub.C, sub.T = prob.B, prob.C, prob.T
    ref = run_oracle(sub)
    sel = dict(y=gpu["y"][:, :, heads], sT=gpu["sT"][:, heads], ckpt=gpu["ckpt"][:, heads],
               ds0=gpu["ds0"][:, heads], dx=gpu["dx"][:, :, heads], ddt=gpu["ddt"][:, :, heads])
    compare(sel, ref, _tol(prob.T), names=tuple(sel))
    f64 = lambda a: a.astype(np.float64)
    lhs_c = np.einsum("ntgj,ntgj->nt", f64(gpu["dC"]), f64(prob.C))
    rhs_c = np.einsum("nthp,nthp->nt", f64(prob.dy), f64(gpu["y"]))
    lhs_b = np.einsum("ntgj,ntgj->nt", f64(gpu["dB"]), f64(prob.B))
    rhs_b = np.einsum("nthp,nthp->nt", f64(prob.x), f64(gpu["dx"]))
    for lhs, rhs, what in ((lhs_c, rhs_c, "dC"), (lhs_b, rhs_b, "dB")):
        err = np.max(np.abs(lhs - rhs)) / np.max(np.abs(rhs))
        assert err <= 1e-4, f"{what} identity: {err:.2e}"
