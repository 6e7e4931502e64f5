"""GPU parity of the backward pass: dq, dk, dv from la_backward (through the
C ABI) against the fp64 oracle's gradients on the same seeded inputs.

The backward runs in fp32 on CUDA cores for both dtypes, so the fp32 rule
(relative error <= 1e-4 with an RMS floor) applies to fp32 inputs and the
output-RMS rule (2e-2 RMS + the 2^-8 rounding of the stored bf16 gradient)
to bf16 inputs.
"""
import numpy as np
import pytest

import oracle
import synthetic
from parity_util import assert_close, from_torch, omega_for, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

QK_SCALE = {"elu1": 1.0, "favor": 64 ** -0.25, "dpfp1": 0.5, "identity": 0.5}


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kernelized_linear_attention_gb300 as m
    m.load_library()
    return m


def _dout(inp, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    d = rng.standard_normal(inp.v.shape).astype(np.float32)
    return synthetic.quantise(d, inp.dtype)


def _to_dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a if dtype == "f32" else synthetic.bf16_bits(a).view(np.int16)))
    return (t if dtype == "f32" else t.view(torch.bfloat16)).cuda()


def _run(la, inp, kind, causal, norm, om, cu=True, seed=5):
    q, k, v = to_torch(inp)
    dout = _dout(inp, seed)
    om_t = torch.from_numpy(om).cuda() if om is not None else None
    cu_t = torch.from_numpy(inp.cu_seqlens).cuda() if cu else None
    nseq = len(inp.cu_seqlens) - 1
    dq, dk, dv = la.la_backward(q, k, v, _to_dev(dout, inp.dtype), kind, omega=om_t, causal=causal, norm=norm,
                                cu_seqlens=cu_t, nseq=nseq)
    torch.cuda.synchronize()
    ref = oracle.backward(inp.q, inp.k, inp.v, dout, kind, causal, omega=om, cu_seqlens=inp.cu_seqlens, norm=norm)
    return [from_torch(t) for t in (dq, dk, dv)], ref


RAGGED = [0, 1, 15, 16, 17, 40, 0, 129]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor", "dpfp1"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
def test_backward_ragged_packed(la, dtype, kind, causal, norm):
    inp = synthetic.random_inputs(RAGGED, H=2, dk=64, dv=64, dtype=dtype, seed=51, qk_scale=QK_SCALE[kind])
    om = omega_for(256, 64) if kind == "favor" else None
    got, ref = _run(la, inp, kind, causal, norm, om)
    for g, r_, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(g, r_, dtype, f"{kind} causal={causal} norm={norm} {name}")


@pytest.mark.parametrize("causal", [True, False])
def test_backward_identity_map_fp32(la, causal):
    # positive inputs keep the identity-map denominators away from the eps clamp
    inp = synthetic.random_inputs([37, 200], H=2, dk=32, dv=48, dtype="f32", seed=52, qk_scale=0.3)
    inp.q = np.abs(inp.q) + 0.05
    inp.k = np.abs(inp.k) + 0.05
    got, ref = _run(la, inp, "identity", causal, "attention", None)
    for g, r_, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(g, r_, "f32", f"identity {name}")


# r = 30 (even, not a multiple of 4) and r = 33 (odd) take the backward's plain loops
@pytest.mark.parametrize("shape", [(16, 48, 96), (32, 16, 64), (16, 48, 30), (32, 16, 33)])
def test_backward_other_head_sizes_fp32(la, shape):
    dk, dv, r = shape
    inp = synthetic.random_inputs([90, 3, 250], H=2, dk=dk, dv=dv, dtype="f32", seed=53, qk_scale=dk ** -0.25)
    om = omega_for(r, dk)
    for causal in (True, False):
        got, ref = _run(la, inp, "favor", causal, "attention", om)
        for g, r_, name in zip(got, ref, ("dq", "dk", "dv")):
            assert_close(g, r_, "f32", f"favor {shape} causal={causal} {name}")


def test_backward_long_sequence_spans_many_segments(la):
    """An equal-length batch long enough to be split into several segments per
    sequence: the forward and reverse scans join the segments."""
    inp = synthetic.random_inputs([1500] * 2, H=2, dk=64, dv=64, dtype="f32", seed=54)
    om = omega_for(256, 64)
    for causal in (True, False):
        got, ref = _run(la, inp, "favor", causal, "attention", om, cu=False)
        for g, r_, name in zip(got, ref, ("dq", "dk", "dv")):
            assert_close(g, r_, "f32", f"long causal={causal} {name}")


def test_backward_empty_batch_and_deterministic(la):
    z = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = la.la_backward(z, z, z, z, "elu1", nseq=1)
    assert dq.shape == (0, 2, 64)
    inp = synthetic.random_inputs([300, 77], H=2, dk=64, dv=64, dtype="bf16", seed=55)
    q, k, v = to_torch(inp)
    dout = _to_dev(_dout(inp, 6), "bf16")
    om = torch.from_numpy(omega_for(256, 64)).cuda()
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    a = la.la_backward(q, k, v, dout, "favor", omega=om, cu_seqlens=cu)
    b = la.la_backward(q, k, v, dout, "favor", omega=om, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_full_size_backward_workload_sampled_heads(la):
    """The benchmark's backward workload in its launch configuration; the oracle
    checks two whole (sequence, head) pairs."""
    w = synthetic.workloads()["favor_causal_b4h8n4096_bwd"]
    inp = synthetic.make_qkv(w)
    om = omega_for(w.r, w.dk)
    q, k, v = to_torch(inp)
    dout = _dout(inp, w.seed + 1)
    dq, dk, dv = la.la_backward(q, k, v, _to_dev(dout, w.dtype), "favor", omega=torch.from_numpy(om).cuda(),
                                causal=True, nseq=w.nseq)
    torch.cuda.synchronize()
    got = [from_torch(t) for t in (dq, dk, dv)]
    n = w.lengths[0]
    for s, h in ((0, 0), (w.nseq - 1, w.H - 1)):
        sl = slice(s * n, (s + 1) * n)
        ref = oracle.backward(inp.q[sl, h:h + 1], inp.k[sl, h:h + 1], inp.v[sl, h:h + 1], dout[sl, h:h + 1],
                              "favor", True, omega=om)
        for g, r_, name in zip(got, ref, ("dq", "dk", "dv")):
            assert_close(g[sl, h:h + 1], r_, "bf16", f"full-size seq {s} head {h} {name}")
