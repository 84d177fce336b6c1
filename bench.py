"""Throughput of the gated delta rule forward + backward (libgdn, sm_103a).

One step = gdn_forward + gdn_backward over one batch: 1 sequence, H_k = 16 key heads
broadcast to H_v = 48 value heads, head size 128, T = 4096 tokens, scalar gate, default
checkpoint interval C = ceil(sqrt(T)) = 64, q/k/v as row views of a packed qkv buffer.
Metric: head-tokens/s = N * H_v * T / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  --impl reference times the float64 CPU oracle (the only other
implementation of this path) on the host cores, on a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN fwd+bwd head-tokens/s at d=128,H_v=48,T=4096; % of FP32/HBM roofline"
UNIT = "head-tokens/s"
WORKLOAD = "bench_d128_T4096"

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
# Algorithmic flops per head-token of the path (FMA = 2): forward 7 d^2; backward = one
# recompute 5 d^2 + reverse step 15 d^2.
FWD_FLOPS = lambda d: 7 * d * d
BWD_FLOPS = lambda d: 20 * d * d
BC = 32  # chunk length of the chunked kernels


def chunk_kernel_flops(N, T, H_v, d, C, which):
    """Flops (FMA = 2) each chunked kernel executes per launch: the dense products of the
    WY form per (sequence, value head, 32-token chunk)."""
    cps = -(-C // BC)
    n_ck = -(-T // C)
    last = T - (n_ck - 1) * C
    n_chunks = (n_ck - 1) * cps + -(-last // BC)
    ch = N * H_v * n_chunks
    recomputed = N * H_v * (n_chunks - n_ck)
    b2d, bd2 = BC * BC * d, BC * d * d
    fma = {
        "prep_fwd": ch * 4 * b2d,
        "state_fwd": ch * (3 * bd2 + b2d),
        "prep_bwd": ch * (4 if cps > 1 else 2) * b2d,
        "recompute": recomputed * 2 * bd2,
        "dstate": ch * (3 * bd2 + 2 * b2d),
        "grad": ch * (4 * bd2 + 6 * b2d + 2 * BC ** 3),
        # head size 128: the gradient step also builds the entry state of each chunk's
        # successor in its segment, M' = gamma M + (r Delta)^T K (B d^2)
        "grad_tc": ch * (4 * bd2 + 6 * b2d + 2 * BC ** 3) + recomputed * bd2,
        "dqdk_sum": 0,
        "fwd_pipe": ch * 4 * b2d + ch * (3 * bd2 + b2d),
        # head size 128: prep ([QK^T; KK^T], E = s dY^T QD) and the dM chain
        "bwd_pipe": ch * 3 * b2d + ch * (3 * bd2 + 2 * b2d),
    }[which]
    return 2.0 * fma


# The head-size-128 chunked kernels run their products on the tensor cores as three-pass
# split products (bf16 hi/lo, part of the gradient step in tf32); their flop peak is
# tensor_peak_tflops().
TENSOR_KINDS = {"state_fwd", "dstate", "grad_tc"}


def kernel_plan(chunked, d, n_bwd, cps):
    """(stage name, flop kind) per timed stage of one forward and one backward, in order."""
    if not chunked:
        return [("gdn_fwd_kernel", None)], [("gdn_bwd_kernel", None), ("gdn_reduce_kernel", None)]
    if d == 128:  # forward: chunk-range preps pipelined with the state chain; backward, as
        # timed stage by stage (its calls with timing events run the stages in sequence)
        fwd = [("gdn_chunk_prep_kernel + gdn_tc_state_kernel (pipelined)", "fwd_pipe")]
        bwd = [("gdn_chunk_prep_kernel + gdn_tc_dstate_kernel", "bwd_pipe"),
               ("gdn_tc_grad_kernel", "grad_tc"), ("gdn_tc_dqdk_sum_kernel", "dqdk_sum")]
        return fwd, bwd
    fwd = [("gdn_chunk_prep_kernel", "prep_fwd"), ("gdn_chunk_state_kernel", "state_fwd")]
    bwd = [("gdn_chunk_prep_kernel", "prep_bwd")]
    if cps > 1:
        bwd.append(("gdn_chunk_state_kernel(recompute)", "recompute"))
    bwd += [("gdn_chunk_dstate_kernel", "dstate"), ("gdn_chunk_grad_kernel", "grad")]
    assert len(bwd) == n_bwd, (len(bwd), n_bwd)
    return fwd, bwd


# stages that pipeline several kernels: reported, but not a roofline "kernel"
PIPELINED_KINDS = {"fwd_pipe", "bwd_pipe"}


def chunk_kernel_bytes(N, T, H_k, H_v, d, C, which):
    """Algorithmic DRAM bytes per launch (fp32): what the kernel has to read and write, with
    no re-reads and its operands stored once, unsplit (None where not counted).  The gradient
    step per (chunk, value head): the chunk-entry state M and dM_end (2 d^2); the dDelta,
    dX, V and dY rows (4 BC d); the chunk factors T, Z, KK^T, QK^T, Dm and gamma, r, beta
    (5 BC^2 + 3 BC); the key head's q and k rows (2 BC d); written: this value head's dq
    and dk parts and dv (3 BC d), dg and dbeta (2 BC).  The parked successor states are the
    design's own traffic, not counted."""
    if which != "grad_tc":
        return None
    cps = -(-C // BC)
    n_ck = -(-T // C)
    last = T - (n_ck - 1) * C
    n_chunks = (n_ck - 1) * cps + -(-last // BC)
    per = 4 * (2 * d * d + 4 * BC * d + 5 * BC * BC + 3 * BC + 2 * BC * d + 3 * BC * d + 2 * BC)
    return N * H_v * n_chunks * per


def fp32_peak(dev=None):
    """FP32 CUDA-core peak of the device: its SM count (device properties) x 128 FP32 lanes
    x 2 flop (FMA) x the maximum SM clock (MEASURED_PEAKS.json, else 2070 MHz).  Returns
    (TFLOP/s, SMs, MHz, how it was derived)."""
    import torch
    sms = int(torch.cuda.get_device_properties(dev).multi_processor_count)
    try:
        mhz, src = float(json.load(open(PEAKS_FILE))["sm_max_mhz"]), "sm_max_mhz of MEASURED_PEAKS.json"
    except (OSError, KeyError, ValueError):
        mhz, src = 2070.0, "maximum SM clock 2070 MHz"
    peak = sms * 128 * 2 * mhz * 1e6 / 1e12
    return peak, sms, mhz, (f"derived: {sms} SMs (device properties) x 128 FP32 lanes x 2 flop x "
                            f"{mhz:.0f} MHz ({src})")


def compulsory_bytes(d, r, T, kda):
    """Compulsory DRAM bytes per head-token of a whole step (fp32; every input read once per
    pass that needs it and every output written once; q, k shared by the r value heads of a
    key head; checkpoints excluded): q, k read by both passes and dq, dk written (6 d / r);
    v read twice, y, dv written, dY read (5 d); g, beta read twice, dg, dbeta written (6);
    state0, state_T, dstate_T, dstate0 (16 d^2 / T); the per-key-column gate reads and writes
    d values where the scalar gate has one (12 d - 12 more)."""
    b = 4 * (6 * d / r + 5 * d + 6) + 16 * d * d / T
    return b + (12 * d - 12 if kda else 0)


# Arithmetic of the path, by head size and gate (stated in every bench line).
ARITH_TC = ("fp32 inputs, outputs, state and accumulators; the state-sized products on the "
            "tcgen05 tensor cores as three-pass split products (bf16 hi/lo, kind::f16, and tf32 "
            "hi/lo for one product of the gradient step), the chunk-sized ones as three-pass "
            "tf32 warp-level MMAs")
ARITH_FP32 = "fp32 throughout (FP32 pipe), with three-pass tf32 warp-level MMAs for chunk-sized products"


def hbm_peak_gbs():
    """Measured copy bandwidth (GB/s) of the GB300s, and where it came from."""
    try:
        return float(json.load(open(PEAKS_FILE))["hbm_gbs"]), "measured copy bandwidth (MEASURED_PEAKS.json)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


# Share of the gradient step's tensor-core multiply-adds done in kind::tf32 (the first part of
# D2, 128 x 64 x 128 of the 3,538,944 per (chunk, value head)); the rest is bf16 (kind::f16).
GRAD_TF32_SHARE = 128 * 64 * 128 / 3538944


def tensor_peak_tflops(tf32_share=GRAD_TF32_SHARE):
    """fp32-equivalent peak of three-pass split products, tf32_share of them in tf32 and the
    rest in bf16: measured bf16 / 3 for the bf16 passes, x nominal tf32/bf16 (1.1 / 2.25) for
    the tf32 ones, combined by time per flop; and where it came from."""
    try:
        bf16 = float(json.load(open(PEAKS_FILE))["bf16_tflops"])
        src = "measured bf16 burst"
    except (OSError, KeyError, ValueError):
        bf16, src = 1900.0, "fallback bf16 1.9 PFLOP/s"
    p_bf16 = bf16 / 3.0
    p_tf32 = bf16 * (1.1 / 2.25) / 3.0
    peak = 1.0 / (tf32_share / p_tf32 + (1.0 - tf32_share) / p_bf16)
    return peak, (src + " / 3 passes, %.0f %% of the flops at the nominal tf32/bf16 rate (1.1/2.25)"
                  % (100 * tf32_share))


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="throughput of every sweep point (d x T x N x gate), one JSON line each")
    ap.add_argument("--op", choices=["gdn", "ssm"], default="gdn",
                    help="gdn: the gated delta rule (default); ssm: the selective scan (SSM_SCAN_BACK)")
    return ap.parse_args()


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- traffic
# The sources each family of kernels is built from, launch code included: the chunked
# (tensor-core and FP32) path and the token recurrence.
CHUNKED_SOURCES = ("gdn_api.cu", "gdn_chunk.cu", "gdn_gemm.cuh", "gdn_internal.h", "gdn_tc.cuh",
                   "gdn_tc_chain.cu", "gdn_tc_grad.cu", "gdn_kda_prep.cuh")
TOKEN_SOURCES = ("gdn_api.cu", "gdn_internal.h", "gdn_device.cuh", "gdn_fwd.cu", "gdn_bwd.cu")


def _kernel_sha(kernel):
    """Hash of the sources `kernel` is built from: a recorded ncu figure stays valid while
    they do not change."""
    token = kernel.split("(")[0] in ("gdn_fwd_kernel", "gdn_bwd_kernel", "gdn_reduce_kernel")
    return _sources_sha(not token)


def _sources_sha(chunked):
    """Hash of the chunked path's or the token recurrence's sources."""
    h = hashlib.sha256()
    for f in CHUNKED_SOURCES if chunked else TOKEN_SOURCES:
        h.update(open(os.path.join(ROOT, "gated_delta_rule_backward_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def _recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel.split('(')[0]}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha") != _kernel_sha(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _recorded_step_traffic(workload, chunked):
    """DRAM bytes of one whole step (every launch of a forward and a backward call) from the
    committed ncu summary of the workload, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"step_dram_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha") != _sources_sha(chunked):
        return None
    try:
        return float(vals["dram_bytes_per_step"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- oracle
def _unit_sample(prob, units):
    """The sub-problem of `units` (sequence n, value head h) of prob, one unit per value head:
    each unit's key-head q, k rows sit beside its own v, g, beta, state0, dY (H_k = H_v)."""
    import numpy as np
    st = lambda xs: np.ascontiguousarray(np.stack(xs, axis=1)[None], dtype=np.float64)
    hk = lambda h: h % prob.H_k
    q = st([prob.q[n, :, hk(h)] for n, h in units])
    k = st([prob.k[n, :, hk(h)] for n, h in units])
    v = st([prob.v[n, :, h] for n, h in units])
    g = st([prob.g[n, :, h] for n, h in units])
    b = st([prob.beta[n, :, h] for n, h in units])
    gy = st([prob.gy[n, :, h] for n, h in units])
    s0 = np.ascontiguousarray(np.stack([prob.state0[n, h] for n, h in units])[None], dtype=np.float64)
    return q, k, v, g, b, s0, gy


def _oracle_sample(prob, units, lib=None):
    """The oracle's forward + checkpointed backward on `units` (sequence, value head) of
    prob.  Returns (head_tokens, seconds)."""
    import oracle
    q, k, v, g, b, s0, gy = _unit_sample(prob, units)
    t0 = time.perf_counter()
    _, _, ck = oracle.forward(q, k, v, g, b, s0, prob.scale, C=prob.C, lib=lib)
    oracle.backward(q, k, v, g, b, s0, gy, None, prob.scale, C=prob.C, ckpt=ck, lib=lib)
    dt = time.perf_counter() - t0
    return len(units) * prob.T, dt


def _first_units(prob, count):
    """The first `count` (sequence, value head) units in (sequence, head) order."""
    units = [(n, h) for n in range(prob.N) for h in range(prob.H_v)]
    return units[:max(1, min(count, len(units)))]


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# The oracle's timed sample: the throughput workload, the 2048-token broadcast workload and
# the 16384-token strong-decay KDA workload, each on all host cores and on one.
CPU_WORKLOADS = ("bench_d128_T4096", "bcast_d128_T2048", "kda_d128_T16384")


def cpu_baseline(target):
    """The oracle (float64 C, OpenMP over (sequence, value head)) on the host cores.  On each
    workload of CPU_WORKLOADS: all cores (one value head per thread, as many value heads as
    threads) and one core (one value head), every unit over all of the workload's tokens,
    forward + checkpointed backward.  `value` is the all-core figure on `target`."""
    import oracle
    from gated_delta_rule_backward_gb300 import synth
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    runs = []
    head = None
    for wl in (target,) + tuple(w for w in CPU_WORKLOADS if w != target):
        prob = synth.workload(wl)
        for nt in (threads, 1):
            oracle.set_threads(nt, lib)
            units = _first_units(prob, nt)
            ht, dt = _oracle_sample(prob, units, lib)
            run = {"workload": wl, "threads": nt, "value_heads": len(units), "tokens": prob.T,
                   "seconds": round(dt, 3), "head_tokens_per_s": ht / dt}
            runs.append(run)
            if wl == target and nt == threads:
                head = run
        del prob
    oracle.set_threads(threads, lib)
    return {"value": head["head_tokens_per_s"], "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{head['value_heads']} of the value heads of {target} (sequence 0, heads "
                      f"0..{head['value_heads'] - 1}) over all {head['tokens']} tokens, forward + "
                      f"checkpointed backward, float64, one value head per thread: "
                      f"{head['seconds']:.2f} s wall on {threads} threads",
            "nproc": os.cpu_count(), "omp_threads": threads, "cpu_model": _cpu_model(),
            "runs": runs}


def run_reference(args):
    rank, world, _ = _dist_env()
    if rank != 0:
        return
    from gated_delta_rule_backward_gb300 import synth
    import oracle
    prob = synth.workload(args.workload)
    lib = oracle.load()
    cores = oracle.max_threads(lib)
    units = _first_units(prob, cores)
    for _ in range(args.warmup):
        _oracle_sample(prob, units[:1], lib)
    tot_ht, tot_s = 0, 0.0
    for _ in range(args.steps):
        ht, dt = _oracle_sample(prob, units, lib)
        tot_ht += ht
        tot_s += dt
    value = tot_ht / tot_s
    sample = (f"per step {len(units)} of {prob.N * prob.H_v} value heads (sequence 0) over "
              f"all {prob.T} tokens, forward + checkpointed backward, float64 C oracle, one "
              f"value head per thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "N": prob.N, "T": prob.T, "H_k": prob.H_k,
                   "H_v": prob.H_v, "d": prob.d, "gate": "kda" if prob.kda else "scalar",
                   "C": prob.C or math.isqrt(prob.T - 1) + 1, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, len(units)),
                         "kind": "oracle", "sample": sample, "nproc": os.cpu_count(),
                         "cpu_model": _cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- ours
def max_over_ranks(x, dist, device):
    """The slowest rank's value (whole-job time is the max over ranks)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    import torch
    from gated_delta_rule_backward_gb300 import gdn, synth

    rank, world, local = _dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    prob = synth.workload(args.workload)
    N, T, H_k, H_v, d = prob.N, prob.T, prob.H_k, prob.H_v, prob.d
    qkv = torch.from_numpy(prob.qkv).to(dev)
    q = qkv[:, :, : H_k * d].view(N, T, H_k, d)
    k = qkv[:, :, H_k * d: 2 * H_k * d].view(N, T, H_k, d)
    v = qkv[:, :, 2 * H_k * d:].view(N, T, H_v, d)
    g = torch.from_numpy(prob.g).to(dev)
    beta = torch.from_numpy(prob.beta).to(dev)
    state0 = torch.from_numpy(prob.state0).to(dev)
    gy = torch.from_numpy(prob.gy).to(dev)
    p = gdn.params_for(q, k, v, g, gy=gy, C=prob.C, scale=prob.scale)
    C = gdn.checkpoint_interval(p)
    y = torch.empty((N, T, H_v, d), device=dev)
    sT = torch.empty((N, H_v, d, d), device=dev)
    ck = torch.empty((N, H_v, gdn.num_checkpoints(p), d, d), device=dev)
    packed = torch.empty(gdn.packed_grad_elems(p), device=dev)
    ws = torch.empty(max(gdn.backward_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    fws_n = gdn.forward_workspace_bytes(p)
    fws = torch.empty(fws_n, dtype=torch.uint8, device=dev) if fws_n else None
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)  # 256 MiB > 129 MB of L2
    stream = torch.cuda.current_stream(dev)
    n_launch_fwd, n_launch_bwd = gdn.launches(p)
    n_fwd, n_bwd = gdn.timing_stages(p)
    # the chunked (WY) kernels: the scalar gate at every head size, the KDA gate at 128
    chunked = (not prob.kda) or d == 128
    fplan, bplan = kernel_plan(chunked, d, n_bwd, -(-C // BC))
    fwd_names, bwd_names = [nm for nm, _ in fplan], [nm for nm, _ in bplan]
    kinds = [k for _, k in fplan + bplan] if chunked else None

    def step():
        gdn.gdn_forward(p, q, k, v, g, beta, state0, y, sT, ck, fws, stream)
        gdn.gdn_backward(p, q, k, v, g, beta, ck, gy, None, packed, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # Timed steps: events on the stream around each call only (no per-stage events), so the
    # calls run exactly as a user's do.
    mk = lambda: torch.cuda.Event(enable_timing=True)
    sev = [(mk(), mk(), mk()) for _ in range(args.steps)]
    for trio in sev:
        for e in trio:
            e.record(stream)  # materialise the event handles
    # Per-stage times, from separate steps with the library's stage events (a backward call
    # with stage events runs its kernels one after another, so each stage is one kernel).
    n_stage_steps = max(3, min(args.steps, 5))
    ev = [([mk() for _ in range(n_fwd + 1)], [mk() for _ in range(n_bwd + 1)])
          for _ in range(n_stage_steps)]
    for fe, be in ev:
        for e in fe + be:
            e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps (not inside the events)
        e0, e1, e2 = sev[i]
        e0.record(stream)
        gdn.gdn_forward(p, q, k, v, g, beta, state0, y, sT, ck, fws, stream)
        e1.record(stream)
        gdn.gdn_backward(p, q, k, v, g, beta, ck, gy, None, packed, ws, stream)
        e2.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    fwd_ms = [e0.elapsed_time(e1) for e0, e1, _ in sev]
    bwd_ms = [e1.elapsed_time(e2) for _, e1, e2 in sev]
    steps_ms = [e0.elapsed_time(e2) for e0, _, e2 in sev]
    for i in range(n_stage_steps):
        flush.zero_()
        fe, be = ev[i]
        gdn.set_timing_events(fe)
        gdn.gdn_forward(p, q, k, v, g, beta, state0, y, sT, ck, fws, stream)
        gdn.set_timing_events(be)
        gdn.gdn_backward(p, q, k, v, g, beta, ck, gy, None, packed, ws, stream)
    gdn.set_timing_events(None)
    torch.cuda.synchronize()
    check_device(stream, "the timed steps")
    kern_ms = [0.0] * (n_fwd + n_bwd)
    for fe, be in ev:
        for j in range(n_fwd):
            kern_ms[j] += fe[j].elapsed_time(fe[j + 1]) / n_stage_steps
        for j in range(n_bwd):
            kern_ms[n_fwd + j] += be[j].elapsed_time(be[j + 1]) / n_stage_steps
    step_ms = sum(steps_ms) / args.steps
    if dist:
        step_ms = max_over_ranks(step_ms, dist, dev)
    head_tokens = N * H_v * T
    value = world * head_tokens / (step_ms * 1e-3)

    # end to end through the public API: pinned host inputs in, results back out
    e2e = None
    if not args.no_e2e:
        # End to end through the same calls, as a training loop runs them: every step's
        # inputs go host -> device from pinned memory and its y, state_T and packed gradients
        # come back device -> host, on two copy streams with double buffers, so that step i's
        # compute overlaps the upload of step i + 1 and the download of step i - 1.
        host = {nm: torch.from_numpy(getattr(prob, nm)).pin_memory()
                for nm in ("g", "beta", "state0", "gy")}
        host["qkv"] = torch.from_numpy(prob.qkv).pin_memory()
        bufs = []
        for _ in range(2):
            d_in = {nm: torch.empty(t.shape, device=dev) for nm, t in host.items()}
            qv = d_in["qkv"]
            bufs.append({
                "in": d_in,
                "q": qv[:, :, : H_k * d].view(N, T, H_k, d),
                "k": qv[:, :, H_k * d: 2 * H_k * d].view(N, T, H_k, d),
                "v": qv[:, :, 2 * H_k * d:].view(N, T, H_v, d),
                "y": torch.empty(y.shape, device=dev), "sT": torch.empty(sT.shape, device=dev),
                "packed": torch.empty(packed.shape, device=dev),
                "out_h": {"y": torch.empty(y.shape).pin_memory(), "sT": torch.empty(sT.shape).pin_memory(),
                          "packed": torch.empty(packed.shape).pin_memory()},
            })
        h2d = sum(t.numel() * 4 for t in host.values())
        d2h = sum(t.numel() * 4 for t in bufs[0]["out_h"].values())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()

        def run_steps(k):
            comp, outd = [None] * k, [None] * k
            for i in range(k):
                b = bufs[i % 2]
                e_in = ev()
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp[i - 2])  # step i - 2 has read this input buffer
                    for nm, t in host.items():
                        b["in"][nm].copy_(t, non_blocking=True)
                    e_in.record(s_in)
                stream.wait_event(e_in)
                if i >= 2:
                    stream.wait_event(outd[i - 2])    # step i - 2's results are on the host
                gdn.gdn_forward(p, b["q"], b["k"], b["v"], b["in"]["g"], b["in"]["beta"], b["in"]["state0"],
                                b["y"], b["sT"], ck, fws, stream)
                gdn.gdn_backward(p, b["q"], b["k"], b["v"], b["in"]["g"], b["in"]["beta"], ck, b["in"]["gy"],
                                 None, b["packed"], ws, stream)
                comp[i] = ev()
                comp[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp[i])
                    for nm in ("y", "sT", "packed"):
                        b["out_h"][nm].copy_(b[nm], non_blocking=True)
                    outd[i] = ev()
                    outd[i].record(s_out)
            stream.wait_event(outd[k - 1])

        run_steps(2)
        torch.cuda.synchronize()
        k_e2e = max(3, args.steps)  # the first upload and the last download are not overlapped
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_event(a)
        run_steps(k_e2e)
        b_.record(stream)
        torch.cuda.synchronize()
        check_device(stream, "the end-to-end steps")
        e2e_ms = a.elapsed_time(b_) / k_e2e
        e2e = {"value": world * head_tokens / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "overlap": "double-buffered: step i's compute beside step i + 1's upload and step i - 1's download"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    bwd_avg = sum(bwd_ms) / len(bwd_ms)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    names = fwd_names + bwd_names
    single = [j for j in range(len(kern_ms)) if not (chunked and kinds[j] in PIPELINED_KINDS)]
    top = max(single, key=lambda j: kern_ms[j])
    # The roofline of the method: its algorithmic flops, 27 d^2
    # per head-token (forward 7, one recompute 5, backward 15), against the FP32 pipe of this
    # device; the compulsory bytes at the measured HBM bandwidth are the other floor, far lower.
    peak32, sms, mhz, peak32_src = fp32_peak(dev)
    hbm, hbm_src = hbm_peak_gbs()
    path_flops = (FWD_FLOPS(d) + BWD_FLOPS(d)) * head_tokens
    path_tflops = path_flops / (step_ms * 1e-3) / 1e12
    comp = compulsory_bytes(d, H_v // H_k, T, prob.kda) * head_tokens
    fp32_floor_ms = path_flops / (peak32 * 1e12) * 1e3
    hbm_floor_ms = comp / (hbm * 1e9) * 1e3
    step_traffic = _recorded_step_traffic(args.workload, chunked)
    # the dominant kernel (largest staged stage time): what it executes and moves
    top_ms = kern_ms[top]
    top_traffic = _recorded_traffic(names[top], args.workload)
    dom = {"kernel": names[top], "ms": top_ms, "share_of_staged_stages": top_ms / sum(kern_ms),
           "dram_bytes_per_launch": top_traffic,
           "dram_over_step_compulsory": (top_traffic / comp) if top_traffic else None,
           "dram_gbs": (top_traffic / (top_ms * 1e-3) / 1e9) if top_traffic else None,
           "hbm_peak_gbs": hbm}
    if chunked:
        ex = chunk_kernel_flops(N, T, H_v, d, C, kinds[top])
        dom["executed_flops_per_launch"] = ex
        if kinds[top] in TENSOR_KINDS:
            tpk, tsrc = tensor_peak_tflops()
            dom["tensor"] = {"achieved": ex / (top_ms * 1e-3) / 1e12, "peak": tpk, "unit": "TFLOP/s",
                             "frac": ex / (top_ms * 1e-3) / 1e12 / tpk, "peak_source": tsrc}
    kernels = [{"kernel": nm, "ms": kern_ms[j],
                "tflops": (chunk_kernel_flops(N, T, H_v, d, C, kinds[j]) / (kern_ms[j] * 1e-3) / 1e12)
                if chunked and kinds[j] != "dqdk_sum" else None} for j, nm in enumerate(names)]
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "N": N, "T": T, "H_k": H_k, "H_v": H_v, "d": d,
                   "gate": "kda" if prob.kda else "scalar", "C": C, "qkv": "packed row views",
                   "arithmetic": ARITH_TC if (chunked and d == 128) else ARITH_FP32,
                   "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "per_rank": "each rank runs the whole workload on its own GPU"},
        "roofline": {"bound": "alu", "kernel": "whole step: gdn_forward + gdn_backward",
                     "achieved": path_tflops, "peak": peak32, "unit": "TFLOP/s",
                     "frac": path_tflops / peak32, "traffic": step_traffic,
                     "flops_per_launch": path_flops, "launch_ms": step_ms,
                     "flops_per_head_token": FWD_FLOPS(d) + BWD_FLOPS(d),
                     "frac_without_recompute": 22 * d * d * head_tokens / (step_ms * 1e-3) / 1e12 / peak32,
                     "compulsory_bytes_per_launch": comp,
                     "traffic_over_compulsory": (step_traffic / comp) if step_traffic else None,
                     "fp32_floor_ms": fp32_floor_ms, "hbm_floor_ms": hbm_floor_ms,
                     "sm_count": sms, "peak_source": peak32_src, "hbm_peak_gbs": hbm,
                     "hbm_peak_source": hbm_src, "fwd_ms": fwd_avg, "bwd_ms": bwd_avg,
                     "dominant_kernel": dom},
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (n_launch_fwd + n_launch_bwd) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_sweep(args):
    """Throughput of every sweep point: d in {32, 64, 128} x T in {512, 4096, 16384} x
    N in {1, 4, 8} (H_v = 48 over H_k = 16) x {scalar, KDA}, C = ceil(sqrt(T)).  Inputs follow
    the recipe's distributions but are drawn on the device (seeded torch generators): the
    points reach 6.3 M head-tokens, too large to draw in float64 on the host.  Each point:
    one warm-up step, then timed steps (about 0.5 s of them, at most --steps) with the L2
    flushed between them; one JSON line each."""
    import torch
    from gated_delta_rule_backward_gb300 import gdn, synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    for pt in synth.sweep_points():
        N, T, H_k, H_v, d, kda = pt["N"], pt["T"], pt["H_k"], pt["H_v"], pt["d"], pt["kda"]
        gen = torch.Generator(device=dev)
        gen.manual_seed(pt["seed"])
        rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev)
        qkv = rnd(N, T, (2 * H_k + H_v) * d)
        q = qkv[:, :, : H_k * d].view(N, T, H_k, d)
        k = qkv[:, :, H_k * d: 2 * H_k * d].view(N, T, H_k, d)
        v = qkv[:, :, 2 * H_k * d:].view(N, T, H_v, d)
        q /= q.norm(dim=-1, keepdim=True)
        k /= k.norm(dim=-1, keepdim=True)
        g = -torch.nn.functional.softplus(rnd(N, T, H_v, d) if kda else rnd(N, T, H_v))
        beta = torch.sigmoid(rnd(N, T, H_v))
        state0 = 0.1 * rnd(N, H_v, d, d)
        gy = rnd(N, T, H_v, d)
        p = gdn.params_for(q, k, v, g, gy=gy, C=None, scale=1.0 / math.sqrt(d))
        y = torch.empty((N, T, H_v, d), device=dev)
        sT = torch.empty((N, H_v, d, d), device=dev)
        ck = torch.empty((N, H_v, gdn.num_checkpoints(p), d, d), device=dev)
        packed = torch.empty(gdn.packed_grad_elems(p), device=dev)
        ws = torch.empty(max(gdn.backward_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
        fws_n = gdn.forward_workspace_bytes(p)
        fws = torch.empty(fws_n, dtype=torch.uint8, device=dev) if fws_n else None

        def step():
            gdn.gdn_forward(p, q, k, v, g, beta, state0, y, sT, ck, fws, stream)
            gdn.gdn_backward(p, q, k, v, g, beta, ck, gy, None, packed, ws, stream)

        step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        torch.cuda.synchronize()
        est = time.perf_counter() - t0
        steps = max(1, min(args.steps, int(0.5 / max(est, 1e-6))))
        mk = lambda: torch.cuda.Event(enable_timing=True)
        evs = [(mk(), mk()) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        check_device(stream, f"the sweep point d={d} T={T} N={N}")
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        head_tokens = N * H_v * T
        tflops = (FWD_FLOPS(d) + BWD_FLOPS(d)) * head_tokens / (ms * 1e-3) / 1e12
        peak32 = fp32_peak(dev)[0]
        print(json.dumps({"point": {"d": d, "T": T, "N": N, "H_k": H_k, "H_v": H_v,
                                    "gate": "kda" if kda else "scalar", "C": gdn.checkpoint_interval(p)},
                          "metric": METRIC, "value": head_tokens / (ms * 1e-3), "unit": UNIT,
                          "ms_per_step": ms, "steps": steps, "dtype": "f32", "data": "synthetic",
                          "roofline": {"bound": "alu", "achieved": tflops, "peak": peak32, "unit": "TFLOP/s",
                                       "frac": tflops / peak32}}), flush=True)
        del qkv, q, k, v, g, beta, state0, gy, y, sT, ck, packed, ws, fws
        torch.cuda.empty_cache()


def check_device(stream, what):
    """A run in which a kernel's bounded wait gave up has invalid outputs: no number."""
    from gated_delta_rule_backward_gb300 import gdn
    st = gdn.device_status(stream)
    if st:
        raise RuntimeError(f"device status {st} after {what}: {gdn.library().gdn_last_error().decode()}")


# --------------------------------------------------------------------------- selective scan
SSM_METRIC = "SSM scan fwd+bwd channel-tokens/s; % of FP32 roofline"
SSM_UNIT = "channel-tokens/s"
SSM_WORKLOAD = "mamba2_h80_T4096"
# Algorithmic flops per state element and token (FMA = 2): forward 5 (s = a s + B (x dt): a
# multiply and an FMA; y: an FMA); backward 13 (ds += dy C: 2; the dC and dB terms and their
# sums over rows: 2 + 2; dx: 2; d(dt): B x, A a, an FMA with s_{t-1} and an FMA into the sum:
# 4; ds = a ds: 1).  The walk's recompute of the states and the exps are not counted.
SSM_FWD_FLOPS, SSM_BWD_FLOPS = 5, 13


def ssm_compulsory_bytes(prob):
    """Bytes a fwd+bwd step must move at least: x, dt, B, C read twice (forward, backward),
    y written, dy, ds_T read, every gradient written, s0 read, s_T written, the checkpoints
    written and read back."""
    N, T, H, P, S, G = prob.N, prob.T, prob.H, prob.P, prob.S, prob.G
    n_ck = max(1, -(-T // prob.K))
    per_tok = 4 * (2 * H * P + 2 * H + 4 * G * S)          # x, dt, B, C twice
    per_tok += 4 * (H * P + H * P + H * P + H + 2 * G * S)  # y; dy; dx, ddt, dB, dC
    state = 4 * H * P * S
    return N * (T * per_tok + state * (4 + 2 * n_ck))


def ssm_cpu_baseline(prob, workload):
    """The selective-scan oracle on the host cores: a sample of the workload's heads over all
    of its tokens (forward + checkpointed walk), all cores (the forward runs a head per
    thread; the walk a group per thread) and one core."""
    import numpy as np
    from oracle import ssm as oss
    lib = oss.load()
    threads = oss.max_threads(lib)
    heads = list(range(min(prob.H, 4 if prob.P > 1 else prob.H)))  # Mamba-2: 4 heads; Mamba-1: every channel
    sub = {f: np.ascontiguousarray(getattr(prob, f)[:, :, heads]) for f in ("x", "dt", "dy")}
    sub.update({f: np.ascontiguousarray(getattr(prob, f)[:, heads]) for f in ("s0", "ds_T")})
    A = np.ascontiguousarray(prob.A[heads])
    # the sample keeps one group, with every group's B and C rows (heads of one group)
    B, C = np.ascontiguousarray(prob.B[:, :, :1]), np.ascontiguousarray(prob.C[:, :, :1])
    runs = []
    for nt in (threads, 1):
        oss.set_threads(nt, lib)
        t0 = time.perf_counter()
        y, sT, ck = oss.forward(sub["s0"], sub["x"], sub["dt"], A, B, C, K=prob.K, lib=lib)
        oss.backward(sub["s0"], sub["x"], sub["dt"], A, B, C, sub["dy"], sub["ds_T"], K=prob.K, ckpt=ck, lib=lib)
        dt = time.perf_counter() - t0
        runs.append({"threads": nt, "seconds": round(dt, 3),
                     "channel_tokens_per_s": prob.N * prob.T * len(heads) * prob.P / dt})
    oss.set_threads(threads, lib)
    return {"value": runs[0]["channel_tokens_per_s"], "unit": SSM_UNIT, "cores": threads, "kind": "oracle",
            "sample": f"heads 0..{len(heads) - 1} of {workload} ({len(heads) * prob.P} of its {prob.H * prob.P} "
                      f"channels) over all {prob.T} tokens, forward + checkpointed walk, float64: "
                      f"{runs[0]['seconds']:.2f} s wall on {threads} threads, {runs[1]['seconds']:.2f} s on 1",
            "nproc": os.cpu_count(), "omp_threads": threads, "cpu_model": _cpu_model(), "runs": runs}


def run_ssm(args):
    """The selective scan: ssm_forward + ssm_backward per step on one synthetic batch."""
    import numpy as np
    import torch
    from gated_delta_rule_backward_gb300 import ssm
    from gated_delta_rule_backward_gb300.ssm_synth import ssm_workload

    rank, world, local = _dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = args.workload if args.workload != WORKLOAD else SSM_WORKLOAD
    prob = ssm_workload(wl)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    s0, x, dt, A, B, C, dy, dsT = map(t, (prob.s0, prob.x, prob.dt, prob.A, prob.B, prob.C, prob.dy, prob.ds_T))
    p = ssm.params_for(x, A, B, K=prob.K)
    out = torch.empty(ssm.packed_out_elems(p), device=dev)
    ck = torch.empty((p.N, p.H, ssm.num_checkpoints(p), p.P, p.S), device=dev)
    gin = ssm.pack_grad_in(p, dy, dsT)
    gout = torch.empty(ssm.packed_grad_elems(p), device=dev)
    ws = torch.empty(max(ssm.backward_workspace_bytes(p), 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(xx=x, dtt=dt, BB=B, CC=C, s00=s0, gi=gin, o=out, go=gout):
        ssm.ssm_forward(p, s00, xx, dtt, A, BB, CC, o, ck, stream)
        ssm.ssm_backward(p, xx, dtt, A, BB, CC, ck, gi, go, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    sev = [(mk(), mk(), mk()) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()
        e0, e1, e2 = sev[i]
        e0.record(stream)
        ssm.ssm_forward(p, s0, x, dt, A, B, C, out, ck, stream)
        e1.record(stream)
        ssm.ssm_backward(p, x, dt, A, B, C, ck, gin, gout, ws, stream)
        e2.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    check_device(stream, "the timed steps")
    fwd_ms = sum(a.elapsed_time(b) for a, b, _ in sev) / args.steps
    bwd_ms = sum(b.elapsed_time(c) for _, b, c in sev) / args.steps
    step_ms = sum(a.elapsed_time(c) for a, _, c in sev) / args.steps
    if dist:
        step_ms = max_over_ranks(step_ms, dist, dev)
    ch_tok = prob.N * prob.T * prob.H * prob.P
    value = world * ch_tok / (step_ms * 1e-3)

    e2e = None
    if not args.no_e2e:
        # through the same calls with every step's inputs uploaded from pinned host memory and
        # its outputs (the packed forward output and the packed gradients) downloaded
        names_in = ("s0", "x", "dt", "B", "C")
        host = {nm: torch.from_numpy(np.ascontiguousarray(getattr(prob, nm))).pin_memory() for nm in names_in}
        host["gin"] = gin.cpu().pin_memory()
        d_in = {nm: torch.empty(h.shape, device=dev) for nm, h in host.items()}
        out_h, gout_h = torch.empty(out.shape).pin_memory(), torch.empty(gout.shape).pin_memory()
        h2d = sum(h.numel() * 4 for h in host.values())
        d2h = (out.numel() + gout.numel()) * 4
        a, b = mk(), mk()
        k_e2e = max(3, args.steps)
        a.record(stream)
        for _ in range(k_e2e):
            for nm, h in host.items():
                d_in[nm].copy_(h, non_blocking=True)
            step(d_in["x"], d_in["dt"], d_in["B"], d_in["C"], d_in["s0"], d_in["gin"])
            out_h.copy_(out, non_blocking=True)
            gout_h.copy_(gout, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / k_e2e
        e2e = {"value": world * ch_tok / (e2e_ms * 1e-3), "unit": SSM_UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": "none (copies in stream order)"}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peak32, sms, mhz, peak32_src = fp32_peak(dev)
    hbm, hbm_src = hbm_peak_gbs()
    flops = (SSM_FWD_FLOPS + SSM_BWD_FLOPS) * ch_tok * prob.S
    tflops = flops / (step_ms * 1e-3) / 1e12
    comp = ssm_compulsory_bytes(prob)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = ssm_cpu_baseline(prob, wl)
    line = {
        "metric": SSM_METRIC, "value": value, "unit": SSM_UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl, "N": prob.N, "T": prob.T, "H": prob.H, "P": prob.P, "S": prob.S,
                   "G": prob.G, "decay": "per state (Mamba-1)" if prob.mamba1 else "per head (Mamba-2)",
                   "K": prob.K, "form": {"chunked": "chunked (64-token chunks)", "segmented": "segmented (a decay per state, by "
                            "checkpoint segments)", "token-serial": "token-serial"}[ssm.form(p)],
                   "arithmetic": "fp32 FP32-pipe, expf",
                   "l2": "flushed between timed steps (256 MiB write outside the events)"},
        "roofline": {"bound": "alu", "kernel": "whole step: ssm_forward + ssm_backward",
                     "achieved": tflops, "peak": peak32, "unit": "TFLOP/s", "frac": tflops / peak32,
                     "traffic": None, "flops_per_launch": flops, "launch_ms": step_ms,
                     "flops_per_state_token": SSM_FWD_FLOPS + SSM_BWD_FLOPS,
                     "compulsory_bytes_per_launch": comp, "hbm_floor_ms": comp / (hbm * 1e9) * 1e3,
                     "fp32_floor_ms": flops / (peak32 * 1e12) * 1e3, "sm_count": sms, "peak_source": peak32_src,
                     "hbm_peak_gbs": hbm, "hbm_peak_source": hbm_src, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                     "workspace_bytes": ws.numel()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(ssm.launches(p)) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    args = _args()
    if args.op == "ssm":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the selective scan's reference arm is "
                              "the oracle timed by this line's cpu_baseline"}), flush=True)
            return
        run_ssm(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
