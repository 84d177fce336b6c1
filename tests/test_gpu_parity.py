"""libgdn (CUDA, sm_103a) against the float64 oracle, element by element.

Tolerance (fp32 kernels vs float64 oracle): max |err| <= 2e-4 (1 + |ref|) for T <= 2048
and <= 1e-3 (1 + |ref|) beyond, on every output: y, state_T, the checkpoints and every
region of the packed gradient.  The problems here are small and mid-size and are checked
in full: they span several tiles, several sub-segments and a ragged last segment, and
cover the degenerate cases (one token, empty sequences, an empty batch).  The full-size
workloads and the throughput sweep are in test_gpu_fullsize.py.
"""
import numpy as np
import pytest

import gpu_helpers as H
from gated_delta_rule_backward_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def full_check(prob, C=None):
    gpu, _ = H.run_gpu(prob, C=C)
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, C if C is not None else prob.C)
    return H.compare_all(gpu, ref, H.tolerance(prob.T))


def test_tiny_d32_T16_scalar():
    prob = synth.workload("tiny_d32_T16")
    full_check(prob)


def test_tiny_d32_T16_scalar_with_final_state_cotangent():
    prob = synth.workload("tiny_d32_T16", dstate_T=True)
    full_check(prob)


def test_kda_d64_T61_partial_last_segment():
    prob = synth.workload("kda_d64_T61")
    full_check(prob)


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_mid_size_full(kda, d):
    # 2 seqs, H_k=2 -> H_v=6 broadcast, packed qkv views, T=300 with C=17 (ragged tail)
    prob = synth.make_problem(2, 300, 2, 6, d, kda=kda, seed=31 + d, C=17, packed=True,
                              dstate_T=True)
    full_check(prob)


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_run_to_run_bit_identical(kda):
    prob = synth.make_problem(2, 300, 2, 6, 128, kda=kda, seed=41, C=17, packed=True,
                              dstate_T=True)
    dev = H.upload(prob)
    a, pa = H.run_gpu(prob, dev=dev)
    b, pb = H.run_gpu(prob, dev=dev)
    assert torch.equal(pa, pb)
    for k in ("y", "state_T", "ckpt"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_checkpoint_interval_invariance(kda):
    """States are recomputed bit-exactly, so gradients do not depend on C.  The token
    recurrence (KDA gate) is exact for every C; the chunked form (scalar gate) for every C
    that keeps its 32-token chunk boundaries (multiples of 32, or C >= T)."""
    prob = synth.make_problem(2, 300, 2, 6, 64, kda=kda, seed=42, packed=True, dstate_T=True)
    dev = H.upload(prob)
    base, pbase = H.run_gpu(prob, C=17 if kda else 32, dev=dev)
    for C in ((1, 5, 64, 300, 1000) if kda else (64, 96, 128, 300, 1000)):
        got, pk = H.run_gpu(prob, C=C, dev=dev)
        assert torch.equal(pk, pbase), C
        assert np.array_equal(got["y"], base["y"]) and np.array_equal(got["state_T"], base["state_T"])


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_checkpoint_interval_invariance_head128(kda):
    """Head size 128 (both gates run the chunked form): the forward is the same state chain
    for every chunk-aligned C, so y and state_T are bit-identical.  The backward takes a
    segment's later entry states from its own gradient step (not from the forward's chain),
    so its gradients agree across C to rounding: within 5e-5 (1 + |ref|), some 40 times
    inside the parity tolerance."""
    prob = synth.make_problem(1, 300, 2, 6, 128, kda=kda, seed=50, packed=True, dstate_T=True)
    dev = H.upload(prob)
    base, pbase = H.run_gpu(prob, C=32, dev=dev)
    ref = pbase.double().cpu().numpy()
    for C in (64, 96, 160, 1000):
        got, pk = H.run_gpu(prob, C=C, dev=dev)
        err = np.abs(pk.double().cpu().numpy() - ref) / (1.0 + np.abs(ref))
        assert err.max() <= 5e-5, (C, float(err.max()))
        assert np.array_equal(got["y"], base["y"]) and np.array_equal(got["state_T"], base["state_T"])


def test_staged_backward_equals_overlapped():
    """A backward call with timing events runs its stages one after another as one chunk
    range; without them it overlaps the gradient work of one range with the chains of the
    next.  Every chunk is computed by the same kernels either way: bit-identical."""
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(1, 700, 2, 6, 128, kda=False, seed=51, C=64, packed=True,
                              dstate_T=True)
    dev = H.upload(prob)
    free, pfree = H.run_gpu(prob, dev=dev)
    p = gdn.params_for(dev["q"], dev["k"], dev["v"], dev["g"], gy=dev["gy"], C=prob.C,
                       scale=prob.scale)
    n_f, n_b = gdn.timing_stages(p)
    assert (n_f, n_b) == (1, 3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_b + 1)]
    for e in ev:
        e.record()
    gdn.set_timing_events(ev)
    try:
        staged, pstaged = H.run_gpu(prob, dev=dev)
    finally:
        gdn.set_timing_events(None)
    assert torch.equal(pfree, pstaged)
    for k in ("y", "state_T", "ckpt"):
        assert np.array_equal(free[k], staged[k]), k


def test_strided_views_equal_contiguous_copies():
    prob = synth.make_problem(2, 100, 2, 6, 64, kda=False, seed=43, C=9, packed=True,
                              dstate_T=True)
    dev = H.upload(prob)
    a, pa = H.run_gpu(prob, dev=dev)
    dev2 = dict(dev)
    for k in ("q", "k", "v"):
        dev2[k] = dev[k].contiguous()
    gy_wide = torch.zeros((2, 100, 6, 80), device="cuda")
    gy_wide[..., :64] = dev["gy"]
    dev2["gy"] = gy_wide[..., :64]                 # a strided gy view as well
    b, pb = H.run_gpu(prob, dev=dev2)
    assert torch.equal(pa, pb)
    assert np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_broadcast_equals_explicit_replication(kda):
    prob = synth.make_problem(1, 120, 2, 6, 64, kda=kda, seed=44, C=11, dstate_T=True)
    dev = H.upload(prob)
    a, _ = H.run_gpu(prob, dev=dev)
    hk = torch.arange(6, device="cuda") % 2
    rep = dict(dev)
    rep["q"] = dev["q"][:, :, hk].contiguous()
    rep["k"] = dev["k"][:, :, hk].contiguous()
    b, _ = H.run_gpu(prob, dev=rep)
    for k in ("y", "state_T", "ckpt", "dv", "dg", "dbeta", "dstate0"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("dq", "dk"):
        for h in range(2):
            acc = np.zeros_like(b[k][:, :, 0])
            for hv in range(h, 6, 2):                  # ascending value heads, fp32 adds
                acc = (acc + b[k][:, :, hv]).astype(np.float32)
            assert np.array_equal(acc, a[k][:, :, h]), (k, h)


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_single_token(kda):
    prob = synth.make_problem(1, 1, 1, 2, 32, kda=kda, seed=45, dstate_T=True)
    full_check(prob)


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_chunk_boundaries_and_long_segments(kda):
    """Chunked form at head size 128: C = 100 (4 chunks per segment, ragged last chunk in
    every segment), T = 333 (ragged last segment), broadcast r = 3."""
    prob = synth.make_problem(1, 333, 2, 6, 128, kda=kda, seed=48, C=100, packed=True,
                              dstate_T=True)
    full_check(prob)


def test_kda_head128_extreme_decay():
    """Per-key-column gate at head size 128 with state resets: every 17th token has
    g = -100 in every column (a = exp(-100), below fp32's normal range), column 5 has
    g = -60 throughout, on top of g = -softplus(N(0, 2^2)).  The chunked form carries the
    decay between tokens as running products of a, so nothing overflows: parity as usual."""
    prob = synth.make_problem(1, 200, 2, 6, 128, kda=True, seed=52, g_std=2.0, C=64,
                              packed=True, dstate_T=True)
    prob.g[:, ::17] = -100.0
    prob.g[..., 5] = -60.0
    full_check(prob)


def test_strong_decay_scalar_gate():
    """g = -softplus(N(0, 2^2)): gamma underflows inside chunks; the chunked form only
    ever evaluates exp(G_t - G_tau) <= 1."""
    prob = synth.make_problem(2, 256, 2, 4, 64, kda=False, seed=49, g_std=2.0, C=64,
                              dstate_T=True)
    full_check(prob)


def test_empty_sequence():
    prob = synth.make_problem(2, 0, 1, 2, 32, kda=False, seed=46, dstate_T=True)
    gpu, _ = H.run_gpu(prob)
    assert np.array_equal(gpu["state_T"], prob.state0)
    assert np.array_equal(gpu["dstate0"], prob.dstate_T)
    assert gpu["y"].size == 0 and gpu["ckpt"].size == 0


def test_empty_batch_is_a_no_op():
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(1, 4, 1, 1, 32, seed=47)
    dev = H.upload(prob)
    p = gdn.make_params(0, 4, 1, 1, 32, False)
    e = torch.empty(0, device="cuda")
    gdn.gdn_forward(p, e, e, e, e, e, e, e, e, e, None)
    gdn.gdn_backward(p, e, e, e, e, e, e, e, None, e, None)
    torch.cuda.synchronize()


def test_device_status_reports_bounded_wait_timeouts():
    """A kernel whose bounded wait gives up returns early and leaves GDN_ERR_TIMEOUT in the
    device status word; reading it clears it; normal head-size-128 runs report GDN_OK."""
    from gated_delta_rule_backward_gb300 import gdn
    assert gdn.device_status() == gdn.GDN_OK
    gdn.selftest_wait_timeout()
    assert gdn.device_status() == 6
    assert b"bounded wait" in gdn.library().gdn_last_error()
    assert gdn.device_status() == gdn.GDN_OK
    prob = synth.make_problem(1, 100, 1, 2, 128, kda=False, seed=51, C=64)
    H.run_gpu(prob)
    assert gdn.device_status() == gdn.GDN_OK


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_head128_outputs_only_4_byte_aligned(kda):
    """The packed buffer's dstate region starts after dg and dbeta, so it is 16-byte aligned
    only when N T H_v (scalar gate: 2 N T H_v) is a multiple of 4; here N T H_v = 999 leaves it
    12 bytes off (KDA) or 8 (scalar).  y is a view starting one float into its buffer (the
    API asks only 4-byte alignment of y).  Both paths store those with 4-byte writes: parity
    as usual and the same bits as an aligned y."""
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(1, 333, 1, 3, 128, kda=kda, seed=53, C=64, packed=True,
                              dstate_T=True)
    dev = H.upload(prob)
    gpu, _ = H.run_gpu(prob, dev=dev)
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, prob.C)
    H.compare_all(gpu, ref, H.tolerance(prob.T))
    p = gdn.params_for(dev["q"], dev["k"], dev["v"], dev["g"], gy=dev["gy"], C=prob.C,
                       scale=prob.scale)
    ybuf = torch.empty(1 + 333 * 3 * 128, device="cuda")
    y = ybuf[1:].view(1, 333, 3, 128)
    sT = torch.empty((1, 3, 128, 128), device="cuda")
    ck = torch.empty((1, 3, gdn.num_checkpoints(p), 128, 128), device="cuda")
    nws = gdn.forward_workspace_bytes(p)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda") if nws else None
    gdn.gdn_forward(p, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["state0"], y,
                    sT, ck, ws)
    torch.cuda.synchronize()
    H.assert_device_ok()
    assert np.array_equal(y.cpu().numpy(), gpu["y"])
    assert np.array_equal(sT.cpu().numpy(), gpu["state_T"])


@pytest.mark.parametrize("kda,d", [(False, 64), (True, 64), (False, 128), (True, 128)],
                         ids=["scalar-64", "kda-64", "scalar-128", "kda-128"])
def test_state_chaining_across_calls(kda, d):
    """A sequence cut in two calls, chained through the states: the second forward starts
    from the first's state_T, and the first backward is seeded with the second's dstate0
    (meTile "Recurrent delta attention": state edges between calls take part in the
    reverse pass).  The pieces, put together, match the oracle's single call."""
    from gated_delta_rule_backward_gb300 import gdn
    prob = synth.make_problem(1, 300, 2, 6, d, kda=kda, seed=62, C=64, dstate_T=True)
    T1 = 128
    cut = lambda x, s: torch.from_numpy(np.ascontiguousarray(x[:, s])).cuda()
    a, b = slice(0, T1), slice(T1, None)
    ins = lambda s: [cut(getattr(prob, nm), s) for nm in ("q", "k", "v", "g", "beta")]
    s0 = torch.from_numpy(prob.state0).cuda()
    dsT = torch.from_numpy(prob.dstate_T).cuda()
    qa, ka, va, ga, ba = ins(a)
    qb, kb, vb, gb, bb = ins(b)
    y1, s1, ck1, p1 = gdn.forward(qa, ka, va, ga, ba, s0, C=prob.C, scale=prob.scale)
    y2, s2, ck2, p2 = gdn.forward(qb, kb, vb, gb, bb, s1, C=prob.C, scale=prob.scale)
    _, g2 = gdn.backward(p2, qb, kb, vb, gb, bb, ck2, cut(prob.gy, b), dsT)
    _, g1 = gdn.backward(p1, qa, ka, va, ga, ba, ck1, cut(prob.gy, a), g2["dstate0"].contiguous())
    torch.cuda.synchronize()
    H.assert_device_ok()
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, prob.C)
    tol = H.tolerance(prob.T)
    cat = lambda u, w: np.concatenate([u.cpu().numpy(), w.cpu().numpy()], axis=1)
    H.compare("y", cat(y1, y2), ref["y"], tol)
    H.compare("state_T", s2.cpu().numpy(), ref["state_T"], tol)
    for k in ("dq", "dk", "dv", "dg", "dbeta"):
        H.compare(k, cat(g1[k], g2[k]), ref[k], tol)
    H.compare("dstate0", g1["dstate0"].cpu().numpy(), ref["dstate0"], tol)
