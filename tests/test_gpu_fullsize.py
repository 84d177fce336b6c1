"""libgdn against the float64 oracle at full size: the workloads' own shapes, seeds and
launch configurations, element by element.

* The throughput sweep's parity subset: every point with T <= 4096 tokens, plus the
  16384-token points at one sequence (42 points, the sweep's own seeds from
  ``synth.sweep_points()``, default C = ceil(sqrt(T))).  Each point is checked on one
  complete (sequence, key-head group) unit -- the r = 3 value heads of one key head, an
  independent problem the oracle solves on its own -- and the unit rotates over the
  sequences and key heads from point to point, so that every head index and every
  sequence slot is reached across the set.
* The 4096-token throughput workload, the 2048-token broadcast workload and the
  16384-token strong-decay KDA workload, checked on every one of their units (the oracle
  runs the whole problem).
* Run-to-run bit identity on the throughput workload, in the launch configuration the
  benchmark times (the backward overlaps the gradient step of one chunk range with the
  chains of the next on library streams).

Tolerance: max |err| <= 2e-4 (1 + |ref|) for T <= 2048, 1e-3 (1 + |ref|) beyond.
"""
import numpy as np
import pytest

import gpu_helpers as H
from gated_delta_rule_backward_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _parity_points():
    pts = []
    for i, pt in enumerate(synth.sweep_points()):
        if pt["T"] <= 4096 or pt["N"] == 1:
            pts.append((i, pt))
    return pts


_POINTS = _parity_points()


def _point_id(ip):
    i, pt = ip
    return f"{i}-d{pt['d']}-T{pt['T']}-N{pt['N']}-{'kda' if pt['kda'] else 'scalar'}"


def test_parity_subset_size():
    # 3 head sizes x 2 lengths (512, 4096) x 3 batch sizes x 2 gates, plus 3 x 2 at 16384
    assert len(_POINTS) == 42


@pytest.mark.parametrize("ip", _POINTS, ids=_point_id)
def test_sweep_point(ip):
    i, pt = ip
    prob = synth.make_problem(**pt)
    gpu, _ = H.run_gpu(prob)
    n = i % prob.N
    hk = (7 * i + 3) % prob.H_k
    H.compare_group(gpu, prob, n, hk, prob.C)


@pytest.mark.parametrize("name", ["bcast_d128_T2048", "bench_d128_T4096", "kda_d128_T16384"])
def test_workload_every_unit(name):
    prob = synth.workload(name)
    gpu, _ = H.run_gpu(prob)
    ref = H.run_oracle(H.problem_dict(prob), prob.scale, prob.C)
    H.compare_all(gpu, ref, H.tolerance(prob.T))


def test_bench_workload_run_to_run_bit_identical():
    prob = synth.workload("bench_d128_T4096")
    dev = H.upload(prob)
    a, pa = H.run_gpu(prob, dev=dev)
    b, pb = H.run_gpu(prob, dev=dev)
    assert torch.equal(pa, pb)
    for k in ("y", "state_T", "ckpt"):
        assert np.array_equal(a[k], b[k]), k
