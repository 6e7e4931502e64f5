"""The bounded in-kernel waits, made to run out on purpose.

Every wait of the tensor-core kernels gives up after a limit and records
LA_DEVERR_WAIT_TIMEOUT in the workspace's error word instead of trapping.  The
test hook la_test_force_wait_timeout makes the causal output kernel's projection
epilogue wait on a barrier that nothing arrives at (1 ms limit); the other roles
then give up on their own bounded waits, drain what they started and return.
The host reads the status, and the next call on the same context is exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from parity_util import assert_close, from_torch, omega_for, to_torch

pytestmark = pytest.mark.gpu

LA_DEVERR_WAIT_TIMEOUT = 2


@pytest.fixture(scope="module")
def la():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kernelized_linear_attention_gb300 as m
    m.load_library()   # raises if the library was not built: no fallback
    return m


def _causal_favor(la, inp, om):
    q, k, v = to_torch(inp)
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    nseq = len(inp.cu_seqlens) - 1
    T, H, dk = q.shape
    nb = la.la_workspace_bytes(True, "favor", q.dtype, True, nseq, T, H, dk, v.shape[2], om.shape[0])
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    out = la.la_forward_causal(q, k, v, "favor", omega=om, cu_seqlens=cu, nseq=nseq, workspace=ws)
    torch.cuda.synchronize()
    return out, la.la_workspace_error(ws)


def test_forced_wait_timeout_is_reported_and_the_next_call_is_exact(la):
    inp = synthetic.random_inputs([700, 129], H=2, dk=64, dv=64, dtype="bf16", seed=31,
                                  qk_scale=64 ** -0.25)
    omega = omega_for(256, 64)
    om = torch.from_numpy(omega).cuda()
    assert la.la_selected_path(True, "favor", torch.bfloat16, 64, 64, 256) == 1   # the tensor-core kernels
    la.la_test_force_wait_timeout(True)
    try:
        _, code = _causal_favor(la, inp, om)
    finally:
        la.la_test_force_wait_timeout(False)
    assert code == LA_DEVERR_WAIT_TIMEOUT
    # the context is usable and the kernels are whole again
    out, code = _causal_favor(la, inp, om)
    assert code == 0
    ref = oracle.forward(inp.q, inp.k, inp.v, "favor", True, omega=omega, cu_seqlens=inp.cu_seqlens)
    assert_close(from_torch(out), ref, "bf16", "causal FAVOR+ after a forced timeout")
