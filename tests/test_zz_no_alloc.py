"""The no-allocation causal entry point against the workspace entry point and
the oracle.

la_forward_causal_noalloc serves callers that may not allocate device memory
on their hot path (a serving loop with a fixed memory budget, a plug-in inside
a framework that owns all device memory): its scratch is a fixed array inside
the library instead of a caller-provided workspace.  This file is collected
last so that a run stopping at its first failure has run everything else.
It must pass alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synthetic
from parity_util import assert_close, from_torch, omega_for, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LA_ERR_WORKSPACE = 3


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kernelized_linear_attention_gb300 as m
    m.load_library()
    return m


def _call_noalloc(lib, q, k, v, omega, kind, dtype_id, cu, nseq, T, H, dk, dv, r, out):
    fn = lib.la_forward_causal_noalloc
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return fn(ptr(q), ptr(k), ptr(v), ptr(omega), {"identity": 0, "elu1": 1, "favor": 2}[kind], dtype_id,
              ptr(cu), nseq, T, H, dk, dv, r, ctypes.c_float(1e-6), ptr(out),
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(la):
    lib = la.load_library()
    cases = [([300, 1, 700, 129], "favor", "bf16", 21), ([1000, 64, 5], "elu1", "f32", 22)]
    for lengths, kind, dtype, seed in cases:
        inp = synthetic.random_inputs(lengths, H=3, dk=64, dv=64, dtype=dtype, seed=seed,
                                      qk_scale=64 ** -0.25 if kind == "favor" else 1.0)
        q, k, v = to_torch(inp)
        cu = torch.from_numpy(inp.cu_seqlens).cuda()
        om = torch.from_numpy(omega_for(256, 64)).cuda() if kind == "favor" else None
        r = 256 if kind == "favor" else 64
        ref = la.la_forward_causal(q, k, v, kind, omega=om, cu_seqlens=cu)
        out = torch.full_like(ref, float("nan"))
        st = _call_noalloc(lib, q, k, v, om, kind, 1 if dtype == "bf16" else 0, cu, len(lengths), q.shape[0], 3,
                           64, 64, r, out)
        assert st == 0, la.la_status_string(st)
        torch.cuda.synchronize()
        assert la.la_noalloc_error() == 0
        assert_close(from_torch(out), from_torch(ref), dtype, f"no-alloc {kind} {dtype}")
        exact = oracle.forward(inp.q, inp.k, inp.v, kind, True, omega=omega_for(256, 64) if kind == "favor" else None,
                               cu_seqlens=inp.cu_seqlens)
        assert_close(from_torch(out), exact, dtype, f"no-alloc {kind} {dtype} against the oracle")


def test_noalloc_rejects_problems_beyond_its_scratch(la):
    lib = la.load_library()
    # 16 sequences x 16 heads of r = 256 states need more than the fixed scratch; the
    # buffers are sized for the call, so that it would stay in bounds even if it ran
    nseq, H = 16, 16
    T = nseq * 128
    need = la.la_workspace_bytes(True, "favor", torch.bfloat16, False, nseq, T, H, 64, 64, 256)
    assert need > (32 << 20)
    q = torch.zeros((T, H, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 7.0)
    om = torch.zeros((256, 64), dtype=torch.float32, device="cuda")
    st = _call_noalloc(lib, q, q, q, om, "favor", 1, None, nseq, T, H, 64, 64, 256, out)
    assert st == LA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_noalloc_reports_bad_cu_seqlens_through_its_error_accessor(la):
    """cu_seqlens that decrease: the planner records LA_DEVERR_CU_SEQLENS in the
    fixed scratch's error word and every kernel skips its work (nothing faults);
    la_noalloc_error reads it, and the next valid call clears it."""
    lib = la.load_library()
    inp = synthetic.random_inputs([100, 50, 80], H=2, dk=64, dv=64, dtype="bf16", seed=27, qk_scale=1.0)
    q, k, v = to_torch(inp)
    bad = torch.tensor([0, 120, 60, 230], dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    assert _call_noalloc(lib, q, k, v, None, "elu1", 1, bad, 3, q.shape[0], 2, 64, 64, 64, out) == 0
    torch.cuda.synchronize()
    assert la.la_noalloc_error() == 1
    good = torch.from_numpy(inp.cu_seqlens).cuda()
    assert _call_noalloc(lib, q, k, v, None, "elu1", 1, good, 3, q.shape[0], 2, 64, 64, 64, out) == 0
    torch.cuda.synchronize()
    assert la.la_noalloc_error() == 0
