"""Helpers shared by the GPU parity tests.

Tolerances (written out here and asserted in the tests):
* fp32 path: max over elements of |gpu - oracle| / max(|oracle|, RMS(oracle))
  <= 1e-4 (relative error, with the output RMS as the floor below which an
  element's size does not shrink the allowance);
* bf16 inputs, fp32 accumulation, bf16 output: |gpu - oracle| <= 2e-2 * RMS(oracle)
  + 2^-8 * |oracle| for every element.  The second term is the rounding of the
  stored bf16 output itself (at most half an ulp, 2^-8 of the value): early
  causal rows average few values and sit far above the RMS, so the storage
  rounding alone can exceed 2e-2 * RMS there.

Bounds from the arithmetic, for results the output-RMS rule does not fit.
bf16 keeps 8 significant bits, so one rounding has relative error at most
u = 2^-8.  The tensor-core path rounds phi(q) and phi(k) to bf16 once each and
rounds every in-chunk score, or the carried state it reads, once more; sums
are fp32.  With non-negative features every weight w_ij = phi(q_i) . phi(k_j)
it effectively uses is within 3u of the exact one.  Hence, with
M_ic = sum_j w_ij |v_jc| (plus phi(q_i) . |S_in[:, c]| for a carried state):
* unnormalised output (norm "none"), whose rows span orders of magnitude
  (FAVOR+ weights are heavy-tailed), so one global RMS means little:
  |error| <= 3u M_ic;
* normalised output: |error| <= 3u (M_ic / den_i + |out_ic|), the worst case
  for rows with a long history (a carried state, or far into a sequence),
  where outputs are small averages and bf16 noise is a larger part of them;
* a state (a sum, no normalisation): one rounding of phi(k), so
  |error| <= u M with M the state computed with |v| (z: M = z).
The tests allow 3.25u instead of 3u (0.25u for the fp32 exponentials, sums and
the 1 / (1 - 3u) of the division) and 1.25u instead of u, plus u |ref| for the
rounding of a stored bf16 output.
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


BF16_STORE_REL = 2.0 ** -8


def abs_err_over_rms(got, ref, rms=None):
    """max over elements of (|got - ref| - 2^-8 |ref|) / RMS(ref): the error
    beyond the bf16 rounding of the stored output, in units of the RMS."""
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    if rms is None:
        rms = np.sqrt(np.mean(ref * ref))
    excess = np.abs(got - ref) - BF16_STORE_REL * np.abs(ref)
    return float(max(0.0, np.max(excess)) / (rms if rms > 0 else 1.0))


def assert_close(got, ref, dtype, what=""):
    if dtype == "f32":
        e = rel_err_rms_floor(got, ref)
        assert e <= FP32_REL_TOL, f"{what}: fp32 relative error {e:.3e} > {FP32_REL_TOL}"
    else:
        e = abs_err_over_rms(got, ref)
        assert e <= BF16_RMS_TOL, f"{what}: bf16 abs error / RMS {e:.3e} > {BF16_RMS_TOL}"
    return e


BF16_U = 2.0 ** -8


def _bound_ratio(got, ref, scale, stored_bf16):
    got = np.asarray(got, np.float64); ref = np.asarray(ref, np.float64); scale = np.asarray(scale, np.float64)
    excess = np.abs(got - ref) - (BF16_U * np.abs(ref) if stored_bf16 else 0.0)
    return float(np.max(excess / np.where(scale > 0, scale, 1.0))) / BF16_U if ref.size else 0.0


def assert_within_rounding_bound(got, ref, M, what="", units=3.25):
    """Unnormalised bf16-path output: |got - ref| <= 3.25u M + u |ref|.  Under sum
    normalisation on tensor cores the values enter as bf16(v / sigma_k), one
    rounding more: units = 4.25, M the sum-normalised output for |v|."""
    k = _bound_ratio(got, ref, M, True)
    assert k <= units, f"{what}: error {k:.2f} u M > {units} u M"
    return k


def assert_normalised_within_rounding_bound(got, ref, Mbar, what=""):
    """Normalised bf16-path output: |got - ref| <= 3.25u (Mbar + |ref|) + u |ref|, Mbar = M / den."""
    k = _bound_ratio(got, ref, np.asarray(Mbar, np.float64) + np.abs(np.asarray(ref, np.float64)), True)
    assert k <= 3.25, f"{what}: error {k:.2f} u (M/den + |out|) > 3.25 u"
    return k


def assert_state_within_rounding_bound(got, ref, M, what=""):
    """bf16-path state (fp32 sums of bf16 features): |got - ref| <= 1.25u M."""
    k = _bound_ratio(got, ref, M, False)
    assert k <= 1.25, f"{what}: state error {k:.2f} u M > 1.25 u M"
    return k


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
