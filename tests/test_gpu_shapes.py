"""Head shapes beyond the square 32/64/128 of the chunked form, against the float64 oracle:
S_k != S_v (meTile "Recurrent delta attention": separate key and value dimensions, state
[B, H, K, V]), and the head sizes 16 and 256 ("metal: GATED_DELTA_NET_BACK", PR #16: the
other configurations of its test set are head size 16).  They run the token recurrence.

Every problem is checked in full, element by element: 2 sequences, q/k broadcast over
r = 2 value heads, packed qkv views, T = 70 with C = 9 (a ragged last segment), nonzero
dstate_T.  Tolerance 2e-4 (1 + |ref|).
"""
import pytest

import gpu_helpers as H
from gated_delta_rule_backward_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

SHAPES = [(64, 32), (32, 128), (16, 16), (16, 64), (64, 16), (256, 256), (256, 64), (128, 256),
          (128, 48)]


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("sk,sv", SHAPES, ids=[f"Sk{a}-Sv{b}" for a, b in SHAPES])
def test_head_shape(sk, sv, kda):
    prob = synth.make_problem(2, 70, 2, 4, sk, kda=kda, seed=80 + sk + sv, C=9, packed=True,
                              dstate_T=True, d_v=sv)
    gpu, _ = H.run_gpu(prob)
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, prob.C)
    H.compare_all(gpu, ref, H.tolerance(prob.T))


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
def test_head_size_16_checkpoint_interval_invariance(kda):
    """The token recurrence recomputes the forward's states bit for bit, so head size 16's
    zero-padded columns change nothing across C: the gradients are the same bits."""
    import numpy as np
    prob = synth.make_problem(1, 90, 1, 2, 16, kda=kda, seed=90, packed=True, dstate_T=True)
    dev = H.upload(prob)
    base, pbase = H.run_gpu(prob, C=7, dev=dev)
    for C in (1, 30, 90, 200):
        got, pk = H.run_gpu(prob, C=C, dev=dev)
        assert torch.equal(pk, pbase), C
        assert np.array_equal(got["y"], base["y"])


BCAST = [(128, 128, 2, 64), (128, 128, 2, 9), (64, 64, 2, 9), (32, 32, 3, 40), (64, 32, 2, 9),
         (16, 16, 2, 9)]


@pytest.mark.parametrize("kda", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("sk,sv,rep,C", BCAST, ids=[f"Sk{a}-Sv{b}-rep{r}-C{c}" for a, b, r, c in BCAST])
def test_sequence_broadcast(sk, sv, rep, C, kda):
    """The sequence broadcast ("metal: GATED_DELTA_NET_BACK", PR #16: head mapping iv3/rq3):
    q, k hold N / rep sequences and value sequence n reads q/k sequence n / rep; dq, dk sum
    over the rep value sequences of each.  Every path: the tensor-core chunked form (both
    gates, one and two chunks per segment), the FP32-pipe chunked form and the token
    recurrence."""
    N = 2 * rep
    prob = synth.make_problem(N, 150 if C == 64 else 70, 2, 4, sk, kda=kda, seed=95 + sk + rep, C=C,
                              dstate_T=True, d_v=sv, seq_rep=rep)
    gpu, _ = H.run_gpu(prob)
    assert gpu["dq"].shape[0] == N // rep
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, prob.C)
    H.compare_all(gpu, ref, H.tolerance(prob.T))
