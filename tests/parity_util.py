"""Helpers shared by the GPU parity tests.

Tolerances (written out here and asserted in the tests):
* fp32 path: max over elements of |gpu - oracle| / max(|oracle|, RMS(oracle))
  <= 1e-4 (relative error, with the output RMS as the floor below which an
  element's size does not shrink the allowance);
* bf16 inputs, fp32 accumulation, bf16 output: for every element,
  |gpu - oracle| - |bf16(oracle) - oracle| <= 2e-2 * RMS(oracle).  The only
  allowance beyond 2e-2 RMS is the rounding of that element's exact value to
  the stored bf16 output (an oracle-side quantity): early causal rows average
  few values and sit far above the RMS, where that rounding alone can exceed
  2e-2 RMS.
* results whose rows span orders of magnitude (the unnormalised fast-weight
  output, the sum-normalised output, whose rows grow with the number of keys
  they sum): the same rule row by row, each row against the RMS of its own
  oracle values;
* states (fp32 sums [S|z] of one sequence and head): S and z each against
  2e-2 of the RMS of their own oracle values.
"""
import numpy as np

import oracle
import synthetic

FP32_REL_TOL = 1e-4
BF16_RMS_TOL = 2e-2


def rel_err_rms_floor(got, ref):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    denom = np.maximum(np.abs(ref), rms)
    denom = np.where(denom == 0, 1.0, denom)
    return float(np.max(np.abs(got - ref) / denom)) if ref.size else 0.0


def bf16_round(x):
    """Values rounded to bf16 (round to nearest even), as float64."""
    return synthetic.bf16_to_f32(synthetic.bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def store_excess(got, ref):
    """|got - ref| beyond the bf16 rounding of the exact value: |got - ref| - |bf16(ref) - ref|."""
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) - np.abs(bf16_round(ref) - ref)


def abs_err_over_rms(got, ref, rms=None):
    """max over elements of (|got - ref| - |bf16(ref) - ref|) / RMS(ref)."""
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    if rms is None:
        rms = np.sqrt(np.mean(ref * ref))
    return float(max(0.0, np.max(store_excess(got, ref))) / (rms if rms > 0 else 1.0))


def rows_over_bar(got, ref, rms=None, tol=BF16_RMS_TOL):
    """Number of rows (last axis = channels) with an element beyond the bar."""
    ref = np.asarray(ref, np.float64)
    if rms is None:
        rms = np.sqrt(np.mean(ref * ref))
    return int(np.sum(np.max(store_excess(got, ref), axis=-1) > tol * rms))


def rowwise_err_over_rms(got, ref):
    """max over rows (last axis = channels) of the bf16 rule against the row's own RMS."""
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    ex = store_excess(got, ref)
    ratio = np.where(rms > 0, ex / np.where(rms > 0, rms, 1.0), np.where(ex > 0, np.inf, 0.0))
    return float(max(0.0, np.max(ratio)))


def assert_close(got, ref, dtype, what=""):
    if dtype == "f32":
        e = rel_err_rms_floor(got, ref)
        assert e <= FP32_REL_TOL, f"{what}: fp32 relative error {e:.3e} > {FP32_REL_TOL}"
    else:
        e = abs_err_over_rms(got, ref)
        assert e <= BF16_RMS_TOL, f"{what}: bf16 abs error / RMS {e:.3e} > {BF16_RMS_TOL}"
    return e


def assert_rowwise_close(got, ref, what=""):
    e = rowwise_err_over_rms(got, ref)
    assert e <= BF16_RMS_TOL, f"{what}: bf16 abs error / row RMS {e:.3e} > {BF16_RMS_TOL}"
    return e


def assert_state_close(got, ref, what=""):
    """[.., r, dv + 1] states: per leading index (sequence, head), S and z each
    within 2e-2 of the RMS of their own oracle values (fp32, nothing stored in bf16)."""
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    g2 = got.reshape(-1, *got.shape[-2:]); r2 = ref.reshape(-1, *ref.shape[-2:])
    worst = 0.0
    for gs, rs in zip(g2, r2):
        for part in (np.s_[:, :-1], np.s_[:, -1]):
            rp = rs[part]
            rms = np.sqrt(np.mean(rp * rp))
            err = np.max(np.abs(gs[part] - rp)) if rp.size else 0.0
            worst = max(worst, err / rms if rms > 0 else (np.inf if err > 0 else 0.0))
    assert worst <= BF16_RMS_TOL, f"{what}: state abs error / RMS {worst:.3e} > {BF16_RMS_TOL}"
    return worst


def omega_for(r, d, seed=synthetic.OMEGA_SEED):
    """fp32 orthogonal random features (chi lengths) drawn from the oracle."""
    blocks, lengths = synthetic.omega_gaussians(r, d, seed)
    return oracle.orthogonal_random_features(blocks, lengths, r=r).astype(np.float32)


def to_torch(inputs, device="cuda"):
    """Inputs -> (q, k, v) torch tensors on device, in storage dtype."""
    import torch
    out = []
    for name in ("q", "k", "v"):
        a = inputs.storage(name)
        t = torch.from_numpy(np.ascontiguousarray(a))
        if inputs.dtype == "bf16":
            t = t.view(torch.bfloat16)
        out.append(t.to(device))
    return out


def from_torch(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()
