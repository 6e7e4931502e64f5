#!/usr/bin/env python3
"""Benchmark of the kernelized linear attention library on GB300.

Metric: tokens/s/GPU of the causal FAVOR+ forward (r = 256, d = 64), with the
dominant kernel's fraction of the tensor-core / HBM roofline.  Workload: the
long causal FAVOR+ case, B=1, H=16, N=65536, d_k=d_v=64, r=256, bf16 q/k/v,
fp32 state, eps 1e-6, synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one forward call (every phase: plan, segment states, scan,
outputs) over the whole batch with inputs resident in HBM.  The inputs (402
MB) exceed the 126 MB L2, so no flush is needed between steps.  Under
torchrun (N > 1) every rank runs an independent replica on its own GPU (the
path has no exchange step); value = all ranks' tokens / max-over-ranks time.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

WORKLOAD = "favor_causal_b1h16n65536"
METRIC = "tokens/s/GPU causal FAVOR+ r=256 d=64; % tensor-core / HBM roofline"
DECODE_METRIC = "tokens/s/GPU causal FAVOR+ decode step (one new token per sequence), r=256 d=64; % HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PHASE_NAMES = ["plan", "state", "scan", "output"]
# source file of each phase's kernel on the tensor-core (tc) and CUDA-core (simt) paths
KERNEL_SOURCES = {"tc": {"output": "tc.cu", "state": "tc.cu", "scan": "plan.cu", "plan": "plan.cu"},
                  "simt": {"output": "simt.cu", "state": "simt.cu", "scan": "plan.cu", "plan": "plan.cu",
                           "decode": "decode.cu"}}
# second measured line: the bidirectional state pass (phi(k)^T [v|1] over every token)
BIDIR_WORKLOAD = "favor_bidir_b4h8n16384"
# the other bf16 workloads of the benchmark plan, each timed as a whole forward
CONFIG_WORKLOADS = ("elu_causal_b8h8n4096", "favor_bidir_b4h8n16384", "favor_causal_varlen64_h8")
# the decode-step and backward lines of the default run
DECODE_WORKLOAD = "favor_decode_b256h16"
BACKWARD_WORKLOAD = "favor_causal_b4h8n4096_bwd"
# fp32 FMA peak of the CUDA-core kernels: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the bidirectional state-pass line")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# Algorithmic work (per token-head), from the method's definition
# ----------------------------------------------------------------------------
def algorithmic(w: synthetic.Workload) -> dict:
    """FLOPs, bytes and exponentials one token of one head needs.

    FAVOR+ projection of q and k: 2 * 2 * d_k * r; state update phi(k)[v|1]^T:
    2 * r * (d_v + 1); readout phi(q)^T [S|z]: 2 * r * (d_v + 1).  HBM: q, k,
    v read once, out written once.  Exponentials: r for q and r for k.
    """
    esz = 2 if w.dtype == "bf16" else 4
    proj = 2 * 2 * w.dk * w.r if w.map == "favor" else 0
    flops = proj + 2 * 2 * w.r * (w.dv + 1)
    byts = (2 * w.dk + 2 * w.dv) * esz
    exps = 2 * w.r if w.map == "favor" else (2 * w.dk if w.map == "elu1" else 0)
    return {"flops": flops, "bytes": byts, "exps": exps}


def roofline_of(w: synthetic.Workload, phase_ms: dict, peaks: dict) -> dict:
    """Roofline of the dominant phase's kernel: algorithmic FLOPs or bytes of one
    launch (the per-token-head figures of algorithmic() times the token-heads the
    launch processes) over its measured duration, against the measured peak of
    the roofline that bounds it (the larger of FLOPs / tensor peak and bytes /
    HBM peak).  The causal output kernel performs the whole method for every
    token-head (it reads q, k, v, writes out, computes both projections, the state
    terms and the readout); the bidirectional output kernel reads q and writes out
    (the q projection and the readout); the state kernel reads k and v of every
    token (the k projection and the state update)."""
    token_heads = w.T * w.H
    esz = 2 if w.dtype == "bf16" else 4
    proj1 = 2 * w.dk * w.r if w.map == "favor" else 0     # one projection (q or k)
    term = 2 * w.r * (w.dv + 1)                            # the state update or the readout
    if w.causal:
        out_flops, out_bytes = algorithmic(w)["flops"], algorithmic(w)["bytes"]
    else:
        out_flops, out_bytes = proj1 + term, (w.dk + w.dv) * esz
    dom = max(phase_ms, key=phase_ms.get)
    dom_ms = phase_ms[dom]
    if dom == "state":
        flops = (proj1 + term) * token_heads
        byts = (w.dk + w.dv) * esz * token_heads
    else:
        flops = out_flops * token_heads
        byts = out_bytes * token_heads
    tflop = peaks["bf16_tflops"] if w.dtype == "bf16" else FP32_ALU_TFLOPS
    t_flop = flops / (tflop * 1e12)
    t_byte = byts / (peaks["hbm_gbs"] * 1e9)
    if dom in ("output", "state") and t_flop >= t_byte:
        achieved = flops / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor" if w.dtype == "bf16" else "alu", "achieved": achieved, "peak": tflop,
                "unit": "TFLOP/s"}
    else:
        achieved = byts / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["phase"] = dom
    roof["kernel"] = {"output": "tc_causal_out_kernel" if w.causal else "tc_bidir_out_kernel",
                      "state": "tc_state_kernel", "scan": "scan_kernel", "plan": "plan_kernel"}[dom]
    roof["alg_flops_per_launch"] = flops
    roof["alg_bytes_per_launch"] = byts
    roof["peak_source"] = peaks["source"] + (" (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "")
    if "output" in phase_ms and phase_ms["output"] > 0:
        roof["tensor_frac_of_output"] = out_flops * token_heads / (phase_ms["output"] * 1e-3) / 1e12 / tflop
        roof["hbm_frac_of_output"] = out_bytes * token_heads / (phase_ms["output"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    roof["phase_ms"] = phase_ms
    roof["kernel_timing"] = ("CUDA events between la_forward_phase calls on the launching stream, over as many "
                             "forwards as the timed steps, right after them")
    return roof


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def code_only(text: str) -> str:
    """C++/CUDA source with its comments removed and whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(path: str, phase: str) -> str:
    """Fingerprint of a kernel's source as compiled: its .cu file and every header of the
    library, comments and whitespace removed (an edit of comments alone leaves a capture
    valid; any change of code, in the file or a header, invalidates it)."""
    csrc = os.path.join(ROOT, "kernelized_linear_attention_gb300", "csrc")
    names = [KERNEL_SOURCES[path][phase]] + sorted(f for f in os.listdir(csrc) if f.endswith((".cuh", ".h")))
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(csrc, n)) as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(path: str, phase: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current source of that kernel on this path (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[workload][path][phase]
        if e.get("source_sha256_16") == kernel_source_hash(path, phase):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------
# Clock sampling (nvidia-smi, during the timed region)
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        smax = float(rows[0][2])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if _isnum(r[3])) if any(
                    _isnum(r[3]) for r in rows) else None}


def _isnum(s):
    try:
        float(s)
        return True
    except Exception:
        return False


# ----------------------------------------------------------------------------
# Distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for one process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(tokens_per_step_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_step_per_rank * steps * world / (max_ms / 1e3)


# ----------------------------------------------------------------------------
# CPU baseline: the oracle, timed on a bounded sample of the workload
# ----------------------------------------------------------------------------
def _oracle_rows(job):
    """Worker (spawned process, one BLAS thread): the oracle on one head's rows;
    returns the seconds it took."""
    import oracle
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(limits=1)
    except Exception:
        pass
    causal, kind, q, k, v, om, eps, norm, state_in = job
    f = oracle.causal if causal else oracle.bidir
    t0 = time.perf_counter()
    f(q, k, v, kind, omega=om, eps=eps, norm=norm, state_in=state_in)
    return time.perf_counter() - t0


def oracle_pool():
    """Process pool for the CPU baseline: spawned (never forked after CUDA is
    initialised), one worker per host core, each with one BLAS thread."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    n = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))
    return ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")), n


def cpu_baseline(w: synthetic.Workload, seconds: float, inputs=None, pool=None) -> dict:
    """Time the oracle, as it stands, on rows [0, n) of every head of the first
    sequence: one head per worker of `pool` (one process per host core, one
    BLAS thread each), n sized from a single-core calibration run so that the
    sample takes about `seconds` of CPU time.  tokens/s = token-heads/s / H,
    with the wall time of the parallel sample."""
    import oracle
    if inputs is None:
        inputs = synthetic.make_qkv(w)
    om = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        om = oracle.orthogonal_random_features(blocks, lengths, r=w.r).astype(np.float32)
    if w.decode:
        return cpu_baseline_decode(w, seconds, inputs, om)
    a, b = int(inputs.cu_seqlens[0]), int(inputs.cu_seqlens[1])
    st = carried_state(w, 1) if w.carry else None

    def job(h, n):
        sl = slice(a, a + n)
        state_in = None
        if st is not None:
            state_in = (st[:, h:h + 1, :, :-1].astype(np.float64), st[:, h:h + 1, :, -1].astype(np.float64))
        return (w.causal, w.map, np.ascontiguousarray(inputs.q[sl, h:h + 1]), np.ascontiguousarray(inputs.k[sl, h:h + 1]),
                np.ascontiguousarray(inputs.v[sl, h:h + 1]), om, w.eps, w.norm, state_in)

    n0 = min(1024, b - a)
    t_cal = _oracle_rows(job(0, n0))
    if pool is None:
        pool, workers = oracle_pool()
    else:
        pool, workers = pool
    used = min(workers, w.H)
    # each worker gets ceil(H / used) heads; size n so that one worker's share takes ~seconds / used
    per_worker = -(-w.H // used)
    n = int(min(b - a, max(n0, n0 * (seconds / max(1, used)) / max(1e-9, t_cal * per_worker))))
    t1 = time.perf_counter()
    list(pool.map(_oracle_rows, [job(h, n) for h in range(w.H)]))
    el = time.perf_counter() - t1
    th = n * w.H
    return {"value": th / w.H / el, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 oracle ({'causal recurrence' if w.causal else 'bidirectional'}) on rows 0..{n - 1} "
                      f"of all {w.H} heads of sequence 0 ({th} token-heads) in {el:.1f} s wall, one head per "
                      f"process on {used} host cores, 1 BLAS thread each; tokens/s = token-heads/s / H"}


def carried_state(w: synthetic.Workload, nseq: int) -> np.ndarray:
    """The carried state a carry or decode workload starts from (seeded)."""
    return synthetic.random_state(nseq, w.H, w.r, w.dv, seed=w.seed + 1000,
                                  z_mean=synthetic.mean_feature(w.map, w.r), n_prior=w.n_prior)


def cpu_baseline_decode(w: synthetic.Workload, seconds: float, inputs, om) -> dict:
    """The oracle's decode step on a sample of (sequence, head) pairs, one at a
    time; tokens/s = (sequence, head) steps per second / H."""
    import oracle
    st = carried_state(w, w.nseq)
    S = st[..., :-1].astype(np.float64); z = st[..., -1].astype(np.float64)
    n, t0 = 0, time.perf_counter()
    while True:
        b, h = n % w.nseq, (n // w.nseq) % w.H
        oracle.decode_step(inputs.q[b:b + 1, h:h + 1], inputs.k[b:b + 1, h:h + 1], inputs.v[b:b + 1, h:h + 1],
                           w.map, S[b:b + 1, h:h + 1], z[b:b + 1, h:h + 1], omega=om, eps=w.eps, norm=w.norm)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= w.nseq * w.H:
            break
    return {"value": n / w.H / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 oracle decode step on {n} (sequence, head) pairs of the {w.name} workload in "
                      f"{el:.1f} s, 1 BLAS thread; tokens/s = pair-steps/s / H"}


def cpu_baseline_backward(w: synthetic.Workload, seconds: float) -> dict:
    """The oracle's backward (quadratic form) on the first n tokens of one
    head of sequence 0, n grown until the sample takes about `seconds`;
    tokens/s = token-heads/s / H."""
    import oracle
    try:
        from threadpoolctl import threadpool_limits
        limiter = threadpool_limits(limits=1)  # noqa: F841  (held for the duration of the sample)
    except Exception:
        limiter = None  # noqa: F841
    inputs = synthetic.make_qkv(w)
    om = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        om = oracle.orthogonal_random_features(blocks, lengths, r=w.r).astype(np.float32)
    rng = np.random.Generator(np.random.PCG64(w.seed + 1))
    dout = rng.standard_normal(inputs.v.shape).astype(np.float32)
    n, el = 256, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.backward(inputs.q[:n, :1], inputs.k[:n, :1], inputs.v[:n, :1], dout[:n, :1], w.map, w.causal,
                        omega=om, eps=w.eps, norm=w.norm)
        el = time.perf_counter() - t0
        if el >= seconds / 3 or n >= w.lengths[0]:
            break
        n = min(w.lengths[0], n * 2)
    return {"value": n / w.H / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 oracle backward (quadratic form) on tokens 0..{n - 1} of head 0 of sequence 0 of "
                      f"{w.name} in {el:.2f} s, 1 BLAS thread; tokens/s = token-heads/s / H"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_ours(args):
    world, rank, local = dist_env()
    # the oracle's worker processes are spawned before CUDA is touched (rank 0, one GPU)
    pool = oracle_pool() if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    import torch
    import kernelized_linear_attention_gb300 as la

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    la.load_library()

    w = synthetic.workloads()[args.workload]
    if w.decode:
        return run_decode(args, la, w, dev, world, rank, local)
    if w.backward:
        return run_backward(args, la, w, dev, world, rank)
    inputs = synthetic.make_qkv(w)
    T, H, dk, dv, r = w.T, w.H, w.dk, w.dv, w.r
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {}
    for n in ("q", "k", "v"):
        a = torch.from_numpy(np.ascontiguousarray(inputs.storage(n)))
        if w.dtype == "bf16":
            a = a.view(torch.bfloat16)
        host[n] = a.pin_memory()
    dq, dk_, dvv = (host[n].to(dev) for n in ("q", "k", "v"))
    omega = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(r, dk)
        omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), r)
    cu = None if w.equal_lengths else torch.from_numpy(inputs.cu_seqlens).to(dev)
    nseq = w.nseq
    out = torch.empty((T, H, dv), dtype=tdt, device=dev)
    ws_bytes = la.la_workspace_bytes(w.causal, w.map, tdt, cu is not None, nseq, T, H, dk, dv, r)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    call_args = (ptr(dq), ptr(dk_), ptr(dvv), ptr(omega), w.map, tdt, ptr(cu), nseq, T, H, dk, dv, r, w.eps,
                 ptr(out), ptr(ws), ws_bytes, stream.cuda_stream)

    state_in = state_out = None
    if w.carry:
        state_in = torch.from_numpy(carried_state(w, nseq)).to(dev)
        state_out = torch.empty_like(state_in)
    state_kw = dict(norm=w.norm, state_in=ptr(state_in), state_out=ptr(state_out))

    plain = w.norm == "attention" and not w.carry

    def step():
        """One forward through the boundary entry point a user calls: la_forward_causal /
        la_forward_bidir (la_forward for the norm and carried-state variants)."""
        if plain:
            la.forward_ptrs(w.causal, *call_args)
        else:
            la.forward_general_ptrs(w.causal, *call_args, **state_kw)
        return launches_per_call

    launches_per_call = sum(la.la_forward_phase(w.causal, ph, *call_args, **state_kw) for ph in range(4))
    warmup = max(args.warmup, 3)      # timing rules: at least 3 untimed warm-up steps
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if la.la_workspace_error(ws) != 0:
        raise RuntimeError(f"device error {la.la_workspace_error(ws)} during warm-up")

    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    launches = 0
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        launches += step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_total = t_start.elapsed_time(t_end)
    ms_total_max = max_over_ranks(ms_total, world, dev)
    if la.la_workspace_error(ws) != 0:
        raise RuntimeError("device error during the timed steps")
    # the same forwards phase by phase (la_forward_phase runs exactly the kernels of the call
    # above, in order), CUDA events between the phases on the launching stream: the duration
    # of each kernel for the roofline
    phase_ms, _ = _phase_timed(la, stream, K, (w.causal,) + call_args, **state_kw)

    tokens = T  # tokens per step per GPU (all heads)
    value = aggregate_value(tokens, K, world, ms_total_max)
    peaks = measured_peaks()
    roof = roofline_of(w, phase_ms, peaks)
    path = "tc" if la.la_selected_path(w.causal, w.map, tdt, dk, dv, r) == 1 and not (w.norm == "sum" and w.carry) \
        else "simt"
    roof["traffic"] = recorded_traffic(path, roof["phase"], w.name)

    # end to end through the C ABI with host buffers: every step copies its q, k, v from pinned host
    # memory, runs the forward and copies out back.  Pipelined over two device buffer sets on three
    # streams: step i+1's host-to-device copy overlaps step i's forward and its device-to-host copy
    # (events order every reuse of a buffer set).
    Ke = args.e2e_steps if args.e2e_steps is not None else max(3, min(K, 20))
    sets = [(dq, dk_, dvv, out), tuple(torch.empty_like(t) for t in (dq, dk_, dvv, out))]
    out_host = [torch.empty((T, H, dv), dtype=tdt).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def forward_on(bset):
        a = (ptr(bset[0]), ptr(bset[1]), ptr(bset[2]), ptr(omega), w.map, tdt, ptr(cu), nseq, T, H, dk, dv, r,
             w.eps, ptr(bset[3]), ptr(ws), ws_bytes, stream.cuda_stream)
        if plain:
            la.forward_ptrs(w.causal, *a)
        else:
            la.forward_general_ptrs(w.causal, *a, **state_kw)

    def pipelined(nsteps, e_begin=None, e_end=None):
        done, copied = [None, None], [None, None]
        if e_begin is not None:
            e_begin.record(s_in)
        for i in range(nsteps):
            b = i % 2
            qb, kb, vb, ob = sets[b]
            with torch.cuda.stream(s_in):
                if done[b] is not None:
                    s_in.wait_event(done[b])          # the forward that read this set has finished
                qb.copy_(host["q"], non_blocking=True); kb.copy_(host["k"], non_blocking=True)
                vb.copy_(host["v"], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            if copied[b] is not None:
                stream.wait_event(copied[b])          # this set's previous output has been copied out
            forward_on(sets[b])
            done[b] = torch.cuda.Event()
            done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[b])
                out_host[b].copy_(ob, non_blocking=True)
                copied[b] = torch.cuda.Event()
                copied[b].record(s_out)
        if e_end is not None:
            for c in copied:
                if c is not None:
                    s_out.wait_event(c)
            e_end.record(s_out)

    pipelined(2)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    pipelined(Ke, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / Ke
    h2d = sum(host[n].numel() * host[n].element_size() for n in ("q", "k", "v"))
    d2h = out_host[0].numel() * out_host[0].element_size()
    e2e = {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "pipelining": "two buffer sets; step i+1's H2D overlaps step i's forward and D2H"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": warmup, "ms_per_step": ms_total_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1) q,k scaled by d^-1/4, v)",
        "config": {"workload": w.name, "B": w.nseq, "H": H, "N": w.lengths[0], "d_k": dk, "d_v": dv, "r": r,
                   "map": w.map, "causal": w.causal, "eps": w.eps, "norm": w.norm, "carried_state": w.carry,
                   "parallelism": f"replicas x{world}",
                   "l2": "no flush: q, k, v (402 MB) exceed the 126 MB L2",
                   "path": "tcgen05" if path == "tc" else "cuda-core"},
        "roofline": roof, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if not args.no_secondary and w.name == WORKLOAD:
        line["bidir_state_pass"] = bidir_state_pass(la, dev, stream, peaks, K)
        line["variants"] = forward_variants(la, dev, stream, peaks, K, w, (dq, dk_, dvv), omega)
        line["decode_step"] = decode_line(la, dev, stream, peaks, max(3, min(K, 20)), DECODE_WORKLOAD)
        line["backward"] = backward_line(la, dev, stream, max(3, min(K, 10)), BACKWARD_WORKLOAD)
        line["fp32_n1024"] = small_config_line(la, dev, stream, max(5, min(K, 20)))
        line["configs"] = {name: config_line(la, dev, stream, peaks, K, name) for name in CONFIG_WORKLOADS}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, inputs, pool)
        if "variants" in line:
            # the oracle beside each further row, on a bounded sample of its workload
            secs = max(2.0, args.cpu_seconds / 4)
            for key, wname in (("none", "favor_causal_b1h16n65536_none"), ("carry", "favor_causal_b1h16n65536_carry"),
                               ("sum", "elu_causal_b8h8n4096_sum")):
                line["variants"][key]["cpu_baseline"] = cpu_baseline(synthetic.workloads()[wname], secs, pool=pool)
            for name in CONFIG_WORKLOADS:
                line["configs"][name]["cpu_baseline"] = cpu_baseline(synthetic.workloads()[name], secs, pool=pool)
            line["fp32_n1024"]["cpu_baseline"] = cpu_baseline_single(synthetic.workloads()["fp32_n1024"])
            line["decode_step"]["cpu_baseline"] = cpu_baseline(synthetic.workloads()[DECODE_WORKLOAD], secs)
            line["backward"]["cpu_baseline"] = cpu_baseline_backward(synthetic.workloads()[BACKWARD_WORKLOAD], secs)
    if pool is not None:
        pool[0].shutdown()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _phase_timed(la, stream, steps, call_args, **kw):
    """Mean per-phase ms of `steps` forward calls (after 3 warm-up calls)."""
    import torch
    for _ in range(3):
        for ph in range(4):
            la.la_forward_phase(call_args[0], ph, *call_args[1:], **kw)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    n = 0
    for i in range(steps):
        for ph in range(4):
            evs[i][ph].record(stream)
            n += la.la_forward_phase(call_args[0], ph, *call_args[1:], **kw)
        evs[i][4].record(stream)
    torch.cuda.synchronize()
    phase_ms = {PHASE_NAMES[p]: statistics.mean(evs[i][p].elapsed_time(evs[i][p + 1]) for i in range(steps))
                for p in range(4)}
    return phase_ms, n // steps


def forward_variants(la, dev, stream, peaks, steps, w, dev_qkv, omega) -> dict:
    """The headline workload's forward with unnormalised output and with a
    carried state in and out (same q, k, v on the device), and the ELU+1
    workload with sum normalisation (its own inputs, CUDA-core path): mean
    per-phase ms over `steps` calls each."""
    import torch
    out = {}
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def args_for(wl, qkv, om):
        o = torch.empty((wl.T, wl.H, wl.dv), dtype=tdt, device=dev)
        nb = la.la_workspace_bytes(wl.causal, wl.map, tdt, False, wl.nseq, wl.T, wl.H, wl.dk, wl.dv, wl.r)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        a = (wl.causal, ptr(qkv[0]), ptr(qkv[1]), ptr(qkv[2]), ptr(om), wl.map, tdt, None, wl.nseq, wl.T, wl.H,
             wl.dk, wl.dv, wl.r, wl.eps, ptr(o), ptr(ws), nb, stream.cuda_stream)
        return a, (o, ws)

    def summary(wl, phase_ms, launches, note):
        ms = sum(phase_ms.values())
        return {"workload": wl.name, "norm": wl.norm, "carried_state": wl.carry, "ms": ms,
                "tokens_per_s": wl.T / (ms * 1e-3), "phase_ms": phase_ms, "launches": launches, "note": note}

    wl = w.with_(name=w.name + "_none", norm="none")
    a, keep = args_for(wl, dev_qkv, omega)
    pm, n = _phase_timed(la, stream, steps, a, norm="none")
    out["none"] = summary(wl, pm, n, "unnormalised output, tensor-core kernels")

    wl = synthetic.workloads()["favor_causal_b1h16n65536_carry"]
    st_in = torch.from_numpy(carried_state(wl, wl.nseq)).to(dev)
    st_out = torch.empty_like(st_in)
    a, keep = args_for(wl, dev_qkv, omega)
    pm, n = _phase_timed(la, stream, steps, a, state_in=ptr(st_in), state_out=ptr(st_out))
    out["carry"] = summary(wl, pm, n, "state_in and state_out; same q, k, v as the headline line; "
                                      "the state pass also sums the last segment")

    wl = synthetic.workloads()["elu_causal_b8h8n4096_sum"]
    inputs = synthetic.make_qkv(wl)
    qkv = [torch.from_numpy(np.ascontiguousarray(inputs.storage(n))).view(torch.bfloat16).to(dev)
           for n in ("q", "k", "v")]
    a, keep = args_for(wl, qkv, None)
    pm, n = _phase_timed(la, stream, steps, a, norm="sum")
    alg = algorithmic(wl)
    s = summary(wl, pm, n, "sum normalisation on tensor cores: feature sums, values / sigma_k, unnormalised "
                           "kernels, output / sigma_q")
    s["hbm_frac_of_output"] = alg["bytes"] * wl.T * wl.H / (pm["output"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    out["sum"] = s
    return out


def run_backward(args, la, w, dev, world, rank):
    """Main line for a backward workload: one step = one la_backward call."""
    import torch
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    res = backward_line(la, dev, stream, args.steps, w.name, warmup=max(args.warmup, 3), world=world)
    clocks = sampler.stop()
    line = {
        "metric": "tokens/s/GPU backward (dq, dk, dv) of causal FAVOR+ r=256 d=64; % fp32 ALU roofline",
        "value": res["tokens_per_s"] * world, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded q, k, v, dout)",
        "config": {"workload": w.name, "B": w.nseq, "H": w.H, "N": w.lengths[0], "d_k": w.dk, "d_v": w.dv,
                   "r": w.r, "map": w.map, "causal": w.causal, "norm": w.norm, "eps": w.eps,
                   "parallelism": f"replicas x{world}", "l2": "no flush: inputs and fp32 workspace rows exceed L2",
                   "path": res["path"]},
        "roofline": res["roofline"], "gpu_launches": res["launches_per_call"] * args.steps, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_backward(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_decode(args, la, w, dev, world, rank, local):
    """Main line for a decode workload: one step = one decode step of every sequence."""
    import torch
    stream = torch.cuda.current_stream(dev)
    res = decode_line(la, dev, stream, measured_peaks(), args.steps, w.name, warmup=max(args.warmup, 3),
                      world=world, e2e_steps=args.e2e_steps)
    line = {
        "metric": DECODE_METRIC,
        "value": res["tokens_per_s"] * world, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded q, k, v and carried state)",
        "config": {"workload": w.name, "B": w.nseq, "H": w.H, "d_k": w.dk, "d_v": w.dv, "r": w.r, "map": w.map,
                   "norm": w.norm, "eps": w.eps, "parallelism": f"replicas x{world}",
                   "l2": "no flush: the carried state (272 MB) exceeds the 126 MB L2", "path": "cuda-core"},
        "roofline": res["roofline"], "e2e": res["e2e"], "gpu_launches": res["launches"], "clocks": res["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, synthetic.make_qkv(w))
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_line(la, dev, stream, peaks, steps, name, warmup=3, world=1, e2e_steps=None) -> dict:
    """Decode steps of a decode workload, timed with CUDA events on the
    launching stream.  Algorithmic bytes per (sequence, head): the fp32 state
    read and written once (2 * 4 * r * (d_v + 1)) plus q, k, v read and out
    written.  The state updates in place from step to step."""
    import torch
    w = synthetic.workloads()[name]
    inputs = synthetic.make_qkv(w)
    B, H, dk, dv, r = w.nseq, w.H, w.dk, w.dv, w.r
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {}
    for n in ("q", "k", "v"):
        t = torch.from_numpy(np.ascontiguousarray(inputs.storage(n)).reshape(B, H, -1))
        host[n] = (t.view(torch.bfloat16) if w.dtype == "bf16" else t).pin_memory()
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    omega = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(r, dk)
        omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), r)
    state = torch.from_numpy(carried_state(w, B)).to(dev)
    out = torch.empty((B, H, dv), dtype=tdt, device=dev)
    for _ in range(warmup):
        la.la_decode_step(q, k, v, state, w.map, omega=omega, norm=w.norm, eps=w.eps, out=out)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        e0.record(stream)
        la.la_decode_step(q, k, v, state, w.map, omega=omega, norm=w.norm, eps=w.eps, out=out)
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs), world, dev)
    esz = 2 if w.dtype == "bf16" else 4
    byts = B * H * (2 * 4 * r * (dv + 1) + esz * (2 * dk + 2 * dv))
    gbs = byts / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "traffic": recorded_traffic("simt", "decode", w.name),
            "kernel": "decode_kernel", "alg_bytes_per_launch": byts,
            "peak_source": peaks["source"] + (" (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "")}
    # end to end: H2D of the new tokens' q, k, v, the step, D2H of out (the state stays resident)
    out_host = torch.empty((B, H, dv), dtype=tdt).pin_memory()
    Ke = e2e_steps if e2e_steps is not None else max(3, min(steps, 20))
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True); a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(Ke):
        q.copy_(host["q"], non_blocking=True); k.copy_(host["k"], non_blocking=True)
        v.copy_(host["v"], non_blocking=True)
        la.la_decode_step(q, k, v, state, w.map, omega=omega, norm=w.norm, eps=w.eps, out=out)
        out_host.copy_(out, non_blocking=True)
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), world, dev) / Ke
    h2d = sum(host[n].numel() * host[n].element_size() for n in ("q", "k", "v"))
    e2e = {"value": B * world / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": out_host.numel() * out_host.element_size(), "ms_per_step": e2e_ms}
    return {"workload": w.name, "ms": ms, "tokens_per_s": B / (ms * 1e-3), "launches": steps,
            "roofline": roof, "e2e": e2e, "clocks": clocks}


def config_line(la, dev, stream, peaks, steps, name) -> dict:
    """One whole forward of a workload through la_forward_causal / la_forward_bidir
    (cu_seqlens for packed workloads), timed with CUDA events on the launching
    stream after 3 warm-up calls; then the same forwards phase by phase for the
    roofline of the dominant kernel.  Inputs stay resident in HBM."""
    import torch
    w = synthetic.workloads()[name]
    inputs = synthetic.make_qkv(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    qkv = []
    for n in ("q", "k", "v"):
        a = torch.from_numpy(np.ascontiguousarray(inputs.storage(n)))
        qkv.append((a.view(torch.bfloat16) if w.dtype == "bf16" else a).to(dev))
    omega = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), w.r)
    cu = None if w.equal_lengths else torch.from_numpy(inputs.cu_seqlens).to(dev)
    out = torch.empty((w.T, w.H, w.dv), dtype=tdt, device=dev)
    nb = la.la_workspace_bytes(w.causal, w.map, tdt, cu is not None, w.nseq, w.T, w.H, w.dk, w.dv, w.r)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    args = (ptr(qkv[0]), ptr(qkv[1]), ptr(qkv[2]), ptr(omega), w.map, tdt, ptr(cu), w.nseq, w.T, w.H, w.dk, w.dv,
            w.r, w.eps, ptr(out), ptr(ws), nb, stream.cuda_stream)
    for _ in range(3):
        la.forward_ptrs(w.causal, *args)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        la.forward_ptrs(w.causal, *args)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if la.la_workspace_error(ws) != 0:
        raise RuntimeError(f"device error in the {name} forward")
    ms = e0.elapsed_time(e1) / steps
    phase_ms, launches = _phase_timed(la, stream, steps, (w.causal,) + args)
    roof = roofline_of(w, phase_ms, peaks)
    roof["traffic"] = recorded_traffic("tc", roof["phase"], name)
    alg = algorithmic(w)
    return {"workload": name, "call": "la_forward_causal" if w.causal else "la_forward_bidir",
            "B": w.nseq, "H": w.H, "N": w.lengths[0] if w.equal_lengths else "varlen",
            "T": w.T, "map": w.map, "causal": w.causal, "r": w.r, "ms": ms, "tokens_per_s": w.T / (ms * 1e-3),
            "launches_per_call": launches, "roofline": roof,
            "whole_forward": {"alg_bytes": alg["bytes"] * w.T * w.H, "alg_flops": alg["flops"] * w.T * w.H,
                              "hbm_frac": alg["bytes"] * w.T * w.H / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                              "tensor_frac": alg["flops"] * w.T * w.H / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
            "l2": "no flush: inputs exceed L2" if 3 * w.T * w.H * w.dk * 2 > (126 << 20)
                  else "inputs below L2 (100 MB): consecutive forwards may hit L2",
            "clocks": clocks}


def cpu_baseline_single(w: synthetic.Workload) -> dict:
    """The oracle on the whole (small) workload on one core, one BLAS thread."""
    import oracle
    inputs = synthetic.make_qkv(w)
    om = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        om = oracle.orthogonal_random_features(blocks, lengths, r=w.r).astype(np.float32)
    el = _oracle_rows((w.causal, w.map, inputs.q, inputs.k, inputs.v, om, w.eps, w.norm, None))
    return {"value": w.T / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 oracle ({'causal recurrence' if w.causal else 'bidirectional'}) on the whole "
                      f"{w.name} problem ({w.T} tokens x {w.H} head, {w.map}) in {el:.3f} s on one core, 1 BLAS thread"}


def small_config_line(la, dev, stream, steps) -> dict:
    """Latency of the fp32 single-head N=1024 case (a parity configuration,
    reported as time only): whole forwards on the fp32 CUDA-core kernels, for
    both maps and both forms, CUDA events on the launching stream."""
    import torch
    w = synthetic.workloads()["fp32_n1024"]
    inputs = synthetic.make_qkv(w)
    q, k, v = (torch.from_numpy(np.ascontiguousarray(inputs.storage(n))).to(dev) for n in ("q", "k", "v"))
    blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
    omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), w.r)
    res = {"workload": w.name, "path": "cuda-core fp32", "unit": "ms per forward"}
    for kind in ("favor", "elu1"):
        for causal in (True, False):
            om = omega if kind == "favor" else None
            out, ws = la.attention(q, k, v, kind, om, causal=causal, return_workspace=True, stream=stream)
            for _ in range(3):
                la.attention(q, k, v, kind, om, causal=causal, out=out, workspace=ws, stream=stream)
            e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(steps):
                la.attention(q, k, v, kind, om, causal=causal, out=out, workspace=ws, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            res[f"{kind}_{'causal' if causal else 'bidir'}_ms"] = e0.elapsed_time(e1) / steps
    return res


def backward_flops(w: synthetic.Workload) -> int:
    """Algorithmic FLOPs of the backward per token-head: the features of q and
    k (FAVOR+: 2 * 2 d r) and their chain rule (2 * 2 d r), the output
    recomputed (readout and state, 2 * 2 r (d_v + 1)), dphi(q) = S g, the
    reverse sum R, dphi(k) = R [v|1] (3 * 2 r (d_v + 1)) and dv = R^T phi(k)
    (2 r d_v)."""
    dvx = w.dv + 1
    proj = 8 * w.dk * w.r if w.map == "favor" else 0
    return proj + 10 * w.r * dvx + 2 * w.r * w.dv - 2 * w.r


def backward_line(la, dev, stream, steps, name, warmup=3, world=1) -> dict:
    """la_backward on a backward workload, timed with CUDA events on the
    launching stream; inputs (q, k, v, dout: 134 MB) and the 268 MB of fp32
    workspace rows exceed L2."""
    import torch
    w = synthetic.workloads()[name]
    inputs = synthetic.make_qkv(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(tdt).to(dev)  # noqa: E731
    q, k, v = (to(inputs.storage(n)) for n in ("q", "k", "v"))
    rng = np.random.Generator(np.random.PCG64(w.seed + 1))
    dout_np = synthetic.quantise(rng.standard_normal(inputs.v.shape).astype(np.float32), w.dtype)
    dout = to(dout_np if w.dtype == "f32" else synthetic.bf16_bits(dout_np).view(np.int16))
    omega = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), w.r)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = la.la_backward_workspace_bytes(w.causal, w.map, tdt, False, w.nseq, w.T, w.H, w.dk, w.dv, w.r)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    call = lambda: la.la_backward(q, k, v, dout, w.map, omega=omega, causal=w.causal, norm=w.norm,  # noqa: E731
                                  nseq=w.nseq, eps=w.eps, dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if la.la_workspace_error(ws) != 0:
        raise RuntimeError("device error in the backward warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    flops = backward_flops(w) * w.T * w.H
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": w.name, "ms": ms, "tokens_per_s": w.T / (ms * 1e-3),
            "launches_per_call": 7 if w.map == "favor" else 6,
            "path": "cuda-core fp32",
            "roofline": {"bound": "alu", "achieved": tf, "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                         "frac": tf / FP32_ALU_TFLOPS, "alg_flops_per_call": flops,
                         "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 FLOP x 2.07 GHz"}}


def bidir_state_pass(la, dev, stream, peaks, steps: int) -> dict:
    """The state phase of the bidirectional FAVOR+ forward (the per-segment
    sum of phi(k_j) [v_j | 1]^T over every token) on its own workload, timed
    with CUDA events on the launching stream after warm-up.  Algorithmic
    bytes: k and v read once (2 * d * 2 B per token-head; the state written is
    negligible).  q, k, v (100 MB) are below L2, so L2 is flushed between
    launches by writing a 256 MB buffer (outside the timed intervals)."""
    import torch
    w = synthetic.workloads()[BIDIR_WORKLOAD]
    inputs = synthetic.make_qkv(w)
    dev_t = {n: torch.from_numpy(np.ascontiguousarray(inputs.storage(n))).view(torch.bfloat16).to(dev)
             for n in ("q", "k", "v")}
    blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
    omega = la.la_orthogonal_features(torch.from_numpy(blocks).to(dev), torch.from_numpy(lengths).to(dev), w.r)
    out = torch.empty((w.T, w.H, w.dv), dtype=torch.bfloat16, device=dev)
    nb = la.la_workspace_bytes(False, w.map, torch.bfloat16, False, w.nseq, w.T, w.H, w.dk, w.dv, w.r)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    args = (dev_t["q"].data_ptr(), dev_t["k"].data_ptr(), dev_t["v"].data_ptr(), omega.data_ptr(), w.map,
            torch.bfloat16, None, w.nseq, w.T, w.H, w.dk, w.dv, w.r, w.eps, out.data_ptr(), ws.data_ptr(), nb,
            stream.cuda_stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    la.la_forward_phase(False, 0, *args)
    for _ in range(3):
        la.la_forward_phase(False, 1, *args)
    times = []
    for _ in range(max(3, steps)):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        la.la_forward_phase(False, 1, *args)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if la.la_workspace_error(ws) != 0:
        raise RuntimeError("device error in the bidirectional state pass")
    ms = statistics.mean(times)
    byts = w.T * w.H * 2 * w.dk * 2
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": w.name, "kernel": "state (tc_state_kernel)", "ms": ms, "bound": "hbm",
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "alg_bytes": byts, "l2": "flushed (256 MB write) before each timed launch",
            "traffic": recorded_traffic("tc", "state", w.name)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = synthetic.workloads()[args.workload]
    inputs = synthetic.make_qkv(w)
    import oracle
    om = None
    if w.map == "favor":
        blocks, lengths = synthetic.omega_gaussians(w.r, w.dk)
        om = oracle.orthogonal_random_features(blocks, lengths, r=w.r).astype(np.float32)
    metric = DECODE_METRIC if w.decode else METRIC
    if w.decode:
        st = carried_state(w, w.nseq)
        n_sample = min(w.nseq, 16)
        S = st[:n_sample, :1, :, :-1].astype(np.float64); z = st[:n_sample, :1, :, -1].astype(np.float64)

        def one():
            oracle.decode_step(inputs.q[:n_sample, :1], inputs.k[:n_sample, :1], inputs.v[:n_sample, :1], w.map,
                               S, z, omega=om, eps=w.eps, norm=w.norm)
        sample = (f"each step: fp64 oracle decode step of head 0 of the first {n_sample} sequences of the "
                  f"{w.name} workload (1 of {w.H} heads); tokens/s = (sequence, head) steps/s / H")
    else:
        # each step: the oracle on the first n_sample tokens of every head, one head per
        # process on the host's cores (spawned pool, one BLAS thread per process)
        n_sample = 2048
        sl = slice(0, n_sample)
        st = carried_state(w, 1) if w.carry else None
        jobs = []
        for h in range(w.H):
            state_in = None
            if st is not None:
                state_in = (st[:, h:h + 1, :, :-1].astype(np.float64), st[:, h:h + 1, :, -1].astype(np.float64))
            jobs.append((w.causal, w.map, np.ascontiguousarray(inputs.q[sl, h:h + 1]),
                         np.ascontiguousarray(inputs.k[sl, h:h + 1]), np.ascontiguousarray(inputs.v[sl, h:h + 1]),
                         om, w.eps, w.norm, state_in))
        pool, workers = oracle_pool()
        cores = min(workers, w.H)

        def one():
            list(pool.map(_oracle_rows, jobs))
        sample = (f"each step: fp64 oracle on the first {n_sample} tokens of all {w.H} heads of the "
                  f"{w.name} workload, one head per process on {cores} host cores; tokens/s = token-heads/s / H")
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    heads_per_step = 1 if w.decode else w.H
    value = n_sample * heads_per_step * args.steps / w.H / el
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1 if w.decode else cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
