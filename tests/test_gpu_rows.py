"""GPU parity of the normalisation variants, the carried state and the decode
step: the CUDA library (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Tolerances are those of parity_util: fp32 relative error
<= 1e-4 (RMS floor); bf16 |error| beyond the rounding of the exact value to
bf16 <= 2e-2 RMS (row by row where rows span orders of magnitude).  States are
fp32 on both paths: the CUDA-core path's are held to the fp32 rule, the
tensor-core path's (sums of f16 features) to 2e-2 of the RMS of S and of z."""
import numpy as np
import pytest

import oracle
import synthetic
from parity_util import (abs_err_over_rms, assert_close, assert_rowwise_close, assert_state_close, from_torch,
                         omega_for, rel_err_rms_floor, to_torch)

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


def _omega(kind, r=256, d=64):
    if kind != "favor":
        return None, None
    om = omega_for(r, d)
    return om, torch.from_numpy(om).cuda()


def _pair(st):
    """[.., r, dv + 1] state -> (S, z) float64."""
    st = np.asarray(st, np.float64)
    return st[..., :-1], st[..., -1]


def _state_array(finals, nseq, H):
    S = np.stack([np.stack([finals[(s, h)][0] for h in range(H)]) for s in range(nseq)])
    z = np.stack([np.stack([finals[(s, h)][1] for h in range(H)]) for s in range(nseq)])
    return np.concatenate([S, z[..., None]], axis=-1)


def _assert_state(got, ref, tensor_path, what):
    """fp32 sums on the CUDA-core path: relative error <= 1e-4 (RMS floor).
    Tensor-core path (fp32 sums of f16 features): S and z each within 2e-2 of
    the RMS of their own oracle values, per sequence and head."""
    if tensor_path:
        assert_state_close(got, ref, what)
    else:
        e = rel_err_rms_floor(got, ref)
        assert e <= 1e-4, f"{what}: state relative error {e:.3e}"


def _tensor_path(la, causal, kind, dtype, norm, r, d=64, carried=False):
    """Whether the call runs the tensor-core kernels (sum normalisation with a
    carried state stays on CUDA cores)."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return not (norm == "sum" and carried) and la.la_selected_path(causal, kind, tdt, d, d, r) == 1


# ----------------------------------------------------------------------------
# Normalisation variants
# ----------------------------------------------------------------------------
RAGGED = [0, 1, 15, 16, 17, 127, 128, 129, 300, 0, 700]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor", "dpfp1"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("norm", ["none", "sum"])
def test_norm_variants_ragged_packed(la, dtype, kind, causal, norm):
    inp = synthetic.random_inputs(RAGGED, H=2, dk=64, dv=64, dtype=dtype, seed=21, qk_scale=QK_SCALE[kind])
    om, om_t = _omega(kind)
    q, k, v = to_torch(inp)
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    out = la.la_forward(q, k, v, kind, omega=om_t, causal=causal, norm=norm, cu_seqlens=cu)
    torch.cuda.synchronize()
    ref = oracle.forward(inp.q, inp.k, inp.v, kind, causal, omega=om, cu_seqlens=inp.cu_seqlens, norm=norm)
    tensor = _tensor_path(la, causal, kind, dtype, norm, 256 if kind == "favor" else (128 if kind == "dpfp1" else 64))
    if tensor:
        # unnormalised and sum-normalised rows grow with position: each row against its own RMS
        assert_rowwise_close(from_torch(out), ref, f"{kind} causal={causal} norm={norm}")
    else:
        assert_close(from_torch(out), ref, dtype, f"{kind} causal={causal} norm={norm}")


def test_norm_attention_through_the_general_call_equals_the_plain_call(la):
    inp = synthetic.random_inputs([300, 129], H=2, dk=64, dv=64, dtype="bf16", seed=4)
    om, om_t = _omega("favor")
    q, k, v = to_torch(inp)
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    for causal in (True, False):
        a = la.la_forward(q, k, v, "favor", omega=om_t, causal=causal, norm="attention", cu_seqlens=cu,
                          state_in=torch.zeros((2, 2, 256, 65), device="cuda"))
        b = la.attention(q, k, v, "favor", om_t, causal=causal, cu_seqlens=cu)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


# ----------------------------------------------------------------------------
# Carried state
# ----------------------------------------------------------------------------
def _prefix_state(kind, om, nseq, H, seed, dtype):
    """state_in = the oracle's final state over a random earlier segment per sequence."""
    pre = synthetic.random_inputs([57] * nseq, H=H, dk=64, dv=64, dtype=dtype, seed=seed, qk_scale=QK_SCALE[kind])
    _, _, _, fin = oracle.causal(pre.q, pre.k, pre.v, kind, omega=om, cu_seqlens=pre.cu_seqlens,
                                 return_parts=True)
    return _state_array(fin, nseq, H).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("packing", ["cu_seqlens", "equal_lengths"])
def test_state_in_and_out_match_oracle(la, dtype, kind, causal, packing):
    lengths = [300, 1, 129, 0, 1000] if packing == "cu_seqlens" else [333] * 3
    H = 2
    inp = synthetic.random_inputs(lengths, H=H, dk=64, dv=64, dtype=dtype, seed=23, qk_scale=QK_SCALE[kind])
    om, om_t = _omega(kind)
    st_in = _prefix_state(kind, om, len(lengths), H, 24, dtype)
    q, k, v = to_torch(inp)
    cu = torch.from_numpy(inp.cu_seqlens).cuda() if packing == "cu_seqlens" else None
    out, st_out = la.la_forward(q, k, v, kind, omega=om_t, causal=causal, cu_seqlens=cu, nseq=len(lengths),
                                state_in=torch.from_numpy(st_in).cuda(), return_state=True)
    torch.cuda.synchronize()
    f = oracle.causal if causal else oracle.bidir
    ref, _, den, fin = f(inp.q, inp.k, inp.v, kind, omega=om, cu_seqlens=inp.cu_seqlens, state_in=_pair(st_in),
                         return_parts=True)
    tensor = _tensor_path(la, causal, kind, dtype, "attention", 256 if kind == "favor" else 64)
    got = from_torch(out)
    assert_close(got, ref, dtype, f"{kind} causal={causal} {packing} out")
    _assert_state(st_out.cpu().numpy(), _state_array(fin, len(lengths), H), tensor,
                  f"{kind} causal={causal} {packing} state_out")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor"])
def test_split_causal_run_with_carried_state_equals_whole(la, dtype, kind):
    """A long causal sequence run as two calls, the second starting from the
    first call's final state, gives the outputs of one run over the whole."""
    whole = [700, 129, 1, 40, 0]
    split = [300, 0, 1, 17, 0]
    H = 2
    inp = synthetic.random_inputs(whole, H=H, dk=64, dv=64, dtype=dtype, seed=25, qk_scale=QK_SCALE[kind])
    om, om_t = _omega(kind)
    cu = inp.cu_seqlens
    idx1 = np.concatenate([np.arange(cu[s], cu[s] + split[s]) for s in range(len(whole))]).astype(int)
    idx2 = np.concatenate([np.arange(cu[s] + split[s], cu[s + 1]) for s in range(len(whole))]).astype(int)
    cu1 = np.concatenate([[0], np.cumsum(split)]).astype(np.int32)
    cu2 = np.concatenate([[0], np.cumsum(np.subtract(whole, split))]).astype(np.int32)
    q, k, v = to_torch(inp)
    i1, i2 = torch.from_numpy(idx1).cuda(), torch.from_numpy(idx2).cuda()
    part = lambda t, i: t.index_select(0, i).contiguous()  # noqa: E731
    _, st1 = la.la_forward(part(q, i1), part(k, i1), part(v, i1), kind, omega=om_t, causal=True,
                           cu_seqlens=torch.from_numpy(cu1).cuda(), return_state=True)
    out2, st2 = la.la_forward(part(q, i2), part(k, i2), part(v, i2), kind, omega=om_t, causal=True,
                              cu_seqlens=torch.from_numpy(cu2).cuda(), state_in=st1, return_state=True)
    torch.cuda.synchronize()
    ref, _, den, fin = oracle.causal(inp.q, inp.k, inp.v, kind, omega=om, cu_seqlens=cu, return_parts=True)
    tensor = _tensor_path(la, True, kind, dtype, "attention", 256 if kind == "favor" else 64)
    got = from_torch(out2)
    assert_close(got, ref[idx2], dtype, f"{kind} second segment")
    _assert_state(st2.cpu().numpy(), _state_array(fin, len(whole), H), tensor, "final state")
    # in place: state_in and state_out the same array
    st = st1.clone()
    out3 = la.la_forward(part(q, i2), part(k, i2), part(v, i2), kind, omega=om_t, causal=True,
                         cu_seqlens=torch.from_numpy(cu2).cuda(), state_in=st, state_out=st)
    torch.cuda.synchronize()
    assert torch.equal(out3, out2) and torch.equal(st, st2)


def test_state_out_of_empty_sequences_is_state_in(la):
    H = 2
    st_in = synthetic.random_state(3, H, 64, 64, seed=3, z_mean=1.0, n_prior=100)
    z = torch.empty((0, H, 64), dtype=torch.bfloat16, device="cuda")
    for causal in (True, False):
        for cu in (None, torch.zeros(4, dtype=torch.int32, device="cuda")):
            _, st_out = la.la_forward(z, z, z, "elu1", causal=causal, cu_seqlens=cu, nseq=3,
                                      state_in=torch.from_numpy(st_in).cuda(), return_state=True)
            torch.cuda.synchronize()
            assert np.array_equal(st_out.cpu().numpy(), st_in)
    _, st0 = la.la_forward(z, z, z, "elu1", causal=True, nseq=3, return_state=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st0) == 0


# ----------------------------------------------------------------------------
# Decode step
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor", "dpfp1", "identity"])
@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
def test_decode_step_matches_oracle(la, dtype, kind, norm):
    if kind == "identity" and norm != "none":
        pytest.skip("identity features can make the denominator vanish; sum normalisation rejects them")
    B, H, d = 5, 3, 64
    om, om_t = _omega(kind)
    r = oracle.feature_dim("dpfp1" if kind == "dpfp1" else kind, d, om)
    inp = synthetic.random_inputs([1] * B, H=H, dk=d, dv=d, dtype=dtype, seed=31, qk_scale=QK_SCALE[kind])
    st = synthetic.random_state(B, H, r, d, seed=32, z_mean=synthetic.mean_feature(kind, r), n_prior=500)
    q, k, v = to_torch(inp)
    st_t = torch.from_numpy(st).cuda()
    out = la.la_decode_step(q, k, v, st_t, kind, omega=om_t, norm=norm)
    torch.cuda.synchronize()
    S, z = _pair(st)
    ref, S2, z2 = oracle.decode_step(inp.q, inp.k, inp.v, kind, S, z, omega=om, norm=norm)
    assert_close(from_torch(out), ref, dtype, f"decode {kind} {norm}")
    _assert_state(st_t.cpu().numpy(), np.concatenate([S2, z2[..., None]], axis=-1), False, "decode state")


@pytest.mark.parametrize("shape", [(16, 48, 96), (32, 8, 32), (128, 256, 512)])
def test_decode_step_other_head_sizes_fp32(la, shape):
    dk, dv, r = shape
    B, H = 3, 2
    om = omega_for(r, dk)
    inp = synthetic.random_inputs([1] * B, H=H, dk=dk, dv=dv, dtype="f32", seed=33, qk_scale=dk ** -0.25)
    st = synthetic.random_state(B, H, r, dv, seed=34, z_mean=r ** -0.5, n_prior=50)
    q, k, v = to_torch(inp)
    st_t = torch.from_numpy(st).cuda()
    out = la.la_decode_step(q, k, v, st_t, "favor", omega=torch.from_numpy(om).cuda())
    torch.cuda.synchronize()
    S, z = _pair(st)
    ref, S2, z2 = oracle.decode_step(inp.q, inp.k, inp.v, "favor", S, z, omega=om)
    assert_close(from_torch(out), ref, "f32", f"decode {shape}")
    _assert_state(st_t.cpu().numpy(), np.concatenate([S2, z2[..., None]], axis=-1), False, "decode state")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["elu1", "favor"])
def test_prefill_then_decode_equals_causal_attention(la, dtype, kind):
    """A causal forward over the prompts that returns its final state, then
    one decode step per new token, gives the causal outputs of the whole
    sequences at the new tokens."""
    prompts = [37, 300, 1, 0]
    n_new, H, d = 4, 2, 64
    B = len(prompts)
    om, om_t = _omega(kind)
    whole = [p + n_new for p in prompts]
    inp = synthetic.random_inputs(whole, H=H, dk=d, dv=d, dtype=dtype, seed=35, qk_scale=QK_SCALE[kind])
    cu = inp.cu_seqlens
    q, k, v = to_torch(inp)
    pidx = torch.from_numpy(np.concatenate([np.arange(cu[s], cu[s] + prompts[s]) for s in range(B)])
                            .astype(np.int64)).cuda()
    pcu = torch.from_numpy(np.concatenate([[0], np.cumsum(prompts)]).astype(np.int32)).cuda()
    sel = lambda t, i: t.index_select(0, i).contiguous()  # noqa: E731
    _, st = la.la_forward(sel(q, pidx), sel(k, pidx), sel(v, pidx), kind, omega=om_t, causal=True,
                          cu_seqlens=pcu, return_state=True)
    ref = oracle.causal(inp.q, inp.k, inp.v, kind, omega=om, cu_seqlens=cu)
    for t in range(n_new):
        rows = torch.from_numpy(np.array([cu[s] + prompts[s] + t for s in range(B)], np.int64)).cuda()
        out = la.la_decode_step(sel(q, rows), sel(k, rows), sel(v, rows), st, kind, omega=om_t)
        torch.cuda.synchronize()
        assert_close(from_torch(out), ref[rows.cpu().numpy()], dtype, f"{kind} decode token {t}")


# ----------------------------------------------------------------------------
# Full-size workloads of these rows, sampled, in the benchmark's launch configuration
# ----------------------------------------------------------------------------
def test_full_size_decode_workload_sampled(la):
    w = synthetic.workloads()["favor_decode_b256h16"]
    inp = synthetic.make_qkv(w)
    om, om_t = _omega("favor")
    B, H = w.nseq, w.H
    st = synthetic.random_state(B, H, w.r, w.dv, seed=w.seed + 1000, z_mean=synthetic.mean_feature("favor", w.r),
                                n_prior=w.n_prior)
    q, k, v = to_torch(inp)
    st_t = torch.from_numpy(st).cuda()
    out = from_torch(la.la_decode_step(q, k, v, st_t, "favor", omega=om_t))
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    bs = sorted(set([0, B - 1] + list(rng.integers(0, B, 6))))
    S, z = _pair(st[bs])
    ref, S2, z2 = oracle.decode_step(inp.q[bs], inp.k[bs], inp.v[bs], "favor", S, z, omega=om)
    assert_close(out[bs], ref, "bf16", "full-size decode")
    _assert_state(st_t.cpu().numpy()[bs], np.concatenate([S2, z2[..., None]], axis=-1), False, "full-size state")


def test_full_size_carry_workload_sampled(la):
    w = synthetic.workloads()["favor_causal_b1h16n65536_carry"]
    inp = synthetic.make_qkv(w)
    om, om_t = _omega("favor")
    st = synthetic.random_state(1, w.H, w.r, w.dv, seed=w.seed + 1000, z_mean=synthetic.mean_feature("favor", w.r),
                                n_prior=w.n_prior)
    q, k, v = to_torch(inp)
    out, st_out = la.la_forward(q, k, v, "favor", omega=om_t, causal=True, nseq=1,
                                state_in=torch.from_numpy(st).cuda(), return_state=True)
    torch.cuda.synchronize()
    out = from_torch(out)
    st_out = st_out.cpu().numpy()
    T = w.T
    for h in (0, w.H - 1):
        rows = [0, 1, 127, 128, 4095, T // 2, T - 1]
        S0, z0 = _pair(st[0, h])
        ref = oracle.causal_rows(inp.q, inp.k, inp.v, "favor", om, 0, T, h, rows, state0=(S0, z0))
        assert_close(out[rows, h], ref, "bf16", f"carry rows head {h}")
        pk = oracle.feature_map(np.asarray(inp.k[:, h], np.float64), "favor", om)
        vv = np.asarray(inp.v[:, h], np.float64)
        S_end = S0 + pk.T @ vv
        z_end = z0 + pk.sum(axis=0)
        _assert_state(st_out[0, h], np.concatenate([S_end, z_end[:, None]], axis=-1), True, f"final state head {h}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_unaligned_state_and_odd_r(la, dtype):
    """A state that is only 4-byte aligned, or r not a multiple of 4, cannot be
    moved by 16-byte bulk copies: the step then runs the register-staged
    kernel, which must give the same results."""
    B, H, dk, dv = 3, 2, 16, 20
    for r, offset in ((32, 1), (30, 0), (30, 3)):
        om = omega_for(r, dk)
        inp = synthetic.random_inputs([1] * B, H=H, dk=dk, dv=dv, dtype=dtype, seed=36, qk_scale=dk ** -0.25)
        st = synthetic.random_state(B, H, r, dv, seed=37, z_mean=r ** -0.5, n_prior=80)
        store = torch.zeros(st.size + 4, dtype=torch.float32, device="cuda")
        st_t = store[offset:offset + st.size].view(st.shape)
        st_t.copy_(torch.from_numpy(st))
        q, k, v = to_torch(inp)
        out = la.la_decode_step(q, k, v, st_t, "favor", omega=torch.from_numpy(om).cuda())
        torch.cuda.synchronize()
        S, z = _pair(st)
        ref, S2, z2 = oracle.decode_step(inp.q, inp.k, inp.v, "favor", S, z, omega=om)
        assert_close(from_torch(out), ref, dtype, f"decode r={r} offset={offset}")
        _assert_state(st_t.cpu().numpy(), np.concatenate([S2, z2[..., None]], axis=-1), False,
                      f"decode state r={r} offset={offset}")
        assert torch.count_nonzero(store[:offset]) == 0 and torch.count_nonzero(store[offset + st.size:]) == 0
