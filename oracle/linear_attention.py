"""Plain fp64 CPU oracle for kernelized linear attention.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import or run this module.  It shares no code
with the CUDA library and the library never calls it.

Everything is computed in float64 with numpy, straight from the definitions on
the source pages, one sequence and one head at a time:

* feature maps: identity and ELU+1 ("The Kernel Zoo", running example and
  §2.5 table; "Linear attention & kernelized approximations", item 2) and the
  FAVOR+ positive random features phi+(x) = exp(Omega x - |x|^2/2)/sqrt(m)
  ("The Kernel Zoo", §4.2 boxed map and §5.4; "Performer", §2 Step 3 and the
  §3 sketch);
* the DPFP-nu map phi(x) = concat_s (x~ * x~^(s)), x~ = relu([x, -x]),
  x~^(s)_i = x~_{(i+s) mod 2d}, s = 1..nu ("The Kernel Zoo", §6.3 boxed map and
  the §6.5 worked examples; map names "dpfp1", "dpfp2", ... give nu);
* orthogonal random features by Gram-Schmidt on Gaussian blocks, rows scaled
  to Gaussian (chi) lengths ("The Kernel Zoo", §5.1 and §5.3 Steps 1-4;
  "Performer", §2 Step 4);
* bidirectional attention S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j),
  out_i = phi(q_i)^T S / max(phi(q_i)^T z, eps) ("Reassociate a feature-map
  kernel", ¶1-2; "Performer", §2 Step 5 and §3 sketch, whose denominator is
  clamped from below at 1e-6);
* causal attention by the prefix recurrence S_i = S_{i-1} + phi(k_i) v_i^T,
  z_i = z_{i-1} + phi(k_i), with the diagonal included ("The Kernel Zoo",
  §1.3 and §5.4; "Reassociate a feature-map kernel", ¶4), with the state reset
  at every packed-sequence boundary (same paragraph);
* the quadratic rescan form, for cross-checks on tiny inputs ("Linear
  attention & kernelized approximations", "The naive way");
* normalisation variants: attention normalisation (the default above), none
  (the unnormalised fast-weight output of "The Kernel Zoo" §1.2-1.4) and sum
  normalisation phi'(x) = phi(x) / sum_f phi(x)_f applied to every query and
  key feature vector, with no attention denominator ("The Kernel Zoo",
  §7.2-7.4);
* a state carried in from an earlier segment of each sequence and out to the
  next ("The Kernel Zoo" §9.3, fast weights carried across training segments),
  and the one-token decode step of the recurrence ("Reassociate a feature-map
  kernel", ¶4);
* the backward pass: gradients of sum(dout * out) with respect to q, k and v,
  by the chain rule on the quadratic form ("Reassociate a feature-map kernel",
  ¶5: errors in outputs and gradients).

Every function here is pinned by tests against values the pages print,
closed forms or brute force (see tests/test_oracle_pins.py).
"""
from __future__ import annotations

import numpy as np

MAPS = ("identity", "elu1", "favor", "dpfp1")
NORMS = ("attention", "none", "sum")


def dpfp_nu(kind: str):
    """nu of a "dpfp<nu>" map name, else None."""
    if isinstance(kind, str) and kind.startswith("dpfp") and kind[4:].isdigit():
        return int(kind[4:])
    return None


# ----------------------------------------------------------------------------
# Feature maps
# ----------------------------------------------------------------------------
def feature_map(x, kind: str, omega=None) -> np.ndarray:
    """phi(x) over the last axis, in float64.

    identity: phi(x) = x                      ("The Kernel Zoo", §1.3, FWP baseline)
    elu1:     phi(x) = elu(x) + 1 = x + 1 for x > 0, exp(x) for x <= 0
              (ELU with alpha = 1; "The Kernel Zoo", running example)
    favor:    phi(x) = exp(omega x - |x|^2 / 2) / sqrt(m), omega of shape [m, d]
              ("The Kernel Zoo", §4.2 boxed feature map)
    dpfp<nu>: x~ = relu([x, -x]) in R^{2d}; for s = 1..nu the products
              x~_i * x~_{(i+s) mod 2d}, i = 0..2d-1; the nu blocks concatenated in
              order of s, so feature (s-1) * 2d + i ("The Kernel Zoo", §6.3, the
              DPFP-nu boxed map, d_dot = 2 d nu)
    """
    x = np.asarray(x, dtype=np.float64)
    if kind == "identity":
        return x.copy()
    if kind == "elu1":
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    if kind == "favor":
        if omega is None:
            raise ValueError("favor map needs omega")
        om = np.asarray(omega, dtype=np.float64)
        m = om.shape[0]
        proj = x @ om.T                                    # omega_i^T x for every i
        half_sq = 0.5 * np.sum(x * x, axis=-1, keepdims=True)   # |x|^2 / 2
        return np.exp(proj - half_sq) / np.sqrt(m)
    nu = dpfp_nu(kind)
    if nu is not None:
        d = x.shape[-1]
        if not 1 <= nu <= 2 * d - 1:
            raise ValueError(f"DPFP needs 1 <= nu <= 2d - 1, got nu = {nu}, d = {d}")
        xt = np.maximum(np.concatenate([x, -x], axis=-1), 0.0)          # step 1: relu([x, -x])
        blocks = [xt * np.roll(xt, -s, axis=-1) for s in range(1, nu + 1)]   # step 2: x~ * x~^(s)
        return np.concatenate(blocks, axis=-1)
    raise ValueError(f"unknown feature map {kind!r}")


def feature_dim(kind: str, d: int, omega=None) -> int:
    if kind == "favor":
        return int(np.asarray(omega).shape[0])
    nu = dpfp_nu(kind)
    return 2 * d * nu if nu is not None else d


# ----------------------------------------------------------------------------
# Orthogonal random features
# ----------------------------------------------------------------------------
def sum_normalise(phi, eps: float = 1e-6) -> np.ndarray:
    """phi'(x) = phi(x) / sum_f phi(x)_f over the last axis ("The Kernel Zoo"
    §7.2), so that the components of every row sum to 1.

    The pages assume non-negative features with a positive sum.  A sum below
    eps (a DPFP vector of an all-zero input, or underflow) is clamped to eps,
    the same floor the attention denominator gets, so such a row stays finite.
    """
    phi = np.asarray(phi, np.float64)
    return phi / np.maximum(phi.sum(axis=-1, keepdims=True), eps)


def features(x, kind: str, omega=None, norm: str = "attention", eps: float = 1e-6) -> np.ndarray:
    """The feature vectors attention uses: phi(x), sum-normalised under norm "sum"."""
    if norm not in NORMS:
        raise ValueError(norm)
    p = feature_map(x, kind, omega)
    return sum_normalise(p, eps) if norm == "sum" else p


def gram_schmidt(rows) -> np.ndarray:
    """Orthonormalise the rows of one or a batch of square blocks, in order.

    Row i has its components along the already finished rows 0..i-1 removed
    (the projection step of "The Kernel Zoo" §5.3 Step 2) and is then scaled
    to unit length (Steps 1 and 3).  The removal is applied twice, which
    leaves the exact-arithmetic result unchanged and keeps fp64 rounding from
    eroding orthogonality for ill-conditioned Gaussian draws.
    """
    Q = np.array(rows, dtype=np.float64, copy=True)
    squeeze = Q.ndim == 2
    if squeeze:
        Q = Q[None]
    n = Q.shape[1]
    for i in range(n):
        row = Q[:, i, :]
        if i > 0:
            prev = Q[:, :i, :]
            for _ in range(2):
                coef = prev @ row[:, :, None]                  # [b, i, 1]: q_j . row
                row = row - (coef.transpose(0, 2, 1) @ prev)[:, 0, :]
        row = row / np.linalg.norm(row, axis=-1, keepdims=True)
        Q[:, i, :] = row
    return Q[0] if squeeze else Q


def orthogonal_random_features(blocks, norm_vectors=None, r=None, norm: str = "chi") -> np.ndarray:
    """Orthogonal random projection matrix Omega of shape [r, d].

    blocks: [nb, d, d] iid N(0,1).  Each block's rows are orthonormalised by
    Gram-Schmidt ("The Kernel Zoo" §5.1: m <= d orthogonal rows per draw);
    the blocks are stacked and the first r rows kept (r > d is reached by
    stacking independent orthogonal blocks).
    norm = "chi":   row i is scaled to |norm_vectors[i]|, the length of a
                    fresh N(0, I_d) vector, so every row has the length
                    distribution of a Gaussian vector ("Performer" §2 Step 4).
    norm = "sqrt_d": every row scaled to sqrt(d) ("The Kernel Zoo" §5.3 Step 4).
    """
    B = np.asarray(blocks, dtype=np.float64)
    if B.ndim == 2:
        B = B[None]
    nb, d, d2 = B.shape
    assert d == d2
    if r is None:
        r = nb * d if norm_vectors is None else np.asarray(norm_vectors).shape[0]
    Q = gram_schmidt(B).reshape(nb * d, d)[:r]
    if norm == "chi":
        lengths = np.linalg.norm(np.asarray(norm_vectors, dtype=np.float64)[:r], axis=-1)
    elif norm == "sqrt_d":
        lengths = np.full(r, np.sqrt(d))
    else:
        raise ValueError(norm)
    return Q * lengths[:, None]


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------
def _bounds(cu_seqlens, T):
    if cu_seqlens is None:
        return [0, T]
    cu = [int(c) for c in np.asarray(cu_seqlens).ravel()]
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0, end at T and not decrease")
    return cu


def normalise(num, den, eps: float, eps_mode: str = "clamp"):
    """out = num / max(den, eps) (clamp, as the "Performer" §3 sketch does).

    eps_mode "add" gives num / (den + eps) and "none" returns the numerator
    alone (the unnormalised fast-weight output of "The Kernel Zoo" §1.2).
    """
    num = np.asarray(num, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    if eps_mode == "none":
        return num
    if eps_mode == "clamp":
        d = np.maximum(den, eps)
    elif eps_mode == "add":
        d = den + eps
    else:
        raise ValueError(eps_mode)
    return num / d[..., None]


def _out(num, den, eps, eps_mode, norm):
    """Attention normalisation divides by the denominator; "none" and "sum" return the numerator."""
    if norm == "attention":
        return normalise(num, den, eps, eps_mode)
    if norm in ("none", "sum"):
        return np.asarray(num, np.float64)
    raise ValueError(norm)


def _state_in(state_in, s, h, r, dv):
    """(S, z) that sequence s, head h starts from: zero, or copies of state_in[0][s, h], state_in[1][s, h]."""
    if state_in is None:
        return np.zeros((r, dv)), np.zeros(r)
    S0, z0 = state_in
    return np.array(S0[s, h], np.float64), np.array(z0[s, h], np.float64)


def bidir(q, k, v, kind, omega=None, cu_seqlens=None, eps=1e-6, eps_mode="clamp",
          return_parts=False, norm="attention", state_in=None):
    """Bidirectional kernelized attention over packed sequences.

    q, k: [T, H, dk]; v: [T, H, dv].  For each sequence and head:
    S = Phi_K^T V, z = Phi_K^T 1, num = Phi_Q S, den = Phi_Q z,
    out = num / max(den, eps)   ("Performer" §2 Step 5 and §3 sketch;
    "Linear attention & kernelized approximations", "Build the state once").
    norm "none" returns num, norm "sum" uses sum-normalised features and
    returns num ("The Kernel Zoo" §7.2-7.4).  state_in = (S0 [nseq, H, r, dv],
    z0 [nseq, H, r]) is added to every sequence's sums (memory from earlier
    segments, all of it visible).
    Returns out [T, H, dv] (and num, den, per-(sequence, head) S and z).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _bounds(cu_seqlens, T)
    r = feature_dim(kind, dk, omega)
    num = np.zeros((T, H, dv)); den = np.zeros((T, H))
    states = {}
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            pq = features(q[a:b, h], kind, omega, norm, eps).reshape(b - a, r)
            pk = features(k[a:b, h], kind, omega, norm, eps).reshape(b - a, r)
            S, z = _state_in(state_in, s, h, r, dv)
            S = S + pk.T @ v[a:b, h]      # sum_j phi(k_j) v_j^T   [r, dv]
            z = z + pk.sum(axis=0)        # sum_j phi(k_j)         [r]
            num[a:b, h] = pq @ S
            den[a:b, h] = pq @ z
            states[(s, h)] = (S, z)
    out = _out(num, den, eps, eps_mode, norm)
    if return_parts:
        return out, num, den, states
    return out


def causal(q, k, v, kind, omega=None, cu_seqlens=None, eps=1e-6, eps_mode="clamp",
           return_parts=False, norm="attention", state_in=None):
    """Causal kernelized attention by the prefix recurrence, token by token.

    For each sequence and head, starting from S = 0, z = 0 at the sequence's
    first token (or from state_in = (S0 [nseq, H, r, dv], z0 [nseq, H, r])):
    S += phi(k_i) v_i^T;  z += phi(k_i);  num_i = phi(q_i)^T S;
    den_i = phi(q_i)^T z; out_i = num_i / max(den_i, eps).  Key i is added
    before query i reads the state (inclusive prefix, "The Kernel Zoo" §1.3
    sum over j = 1..i; "Reassociate a feature-map kernel" ¶4).  norm as for
    bidir.  The parts include each (sequence, head)'s final (S, z).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = _bounds(cu_seqlens, T)
    r = feature_dim(kind, dk, omega)
    num = np.zeros((T, H, dv)); den = np.zeros((T, H))
    finals = {}
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            pq = features(q[a:b, h], kind, omega, norm, eps).reshape(b - a, r)   # one token at a time
            pk = features(k[a:b, h], kind, omega, norm, eps).reshape(b - a, r)
            S, z = _state_in(state_in, s, h, r, dv)
            for i in range(b - a):
                S += np.outer(pk[i], v[a + i, h])
                z += pk[i]
                num[a + i, h] = pq[i] @ S
                den[a + i, h] = pq[i] @ z
            finals[(s, h)] = (S.copy(), z.copy())
    out = _out(num, den, eps, eps_mode, norm)
    if return_parts:
        return out, num, den, finals
    return out


def decode_step(q, k, v, kind, S, z, omega=None, eps=1e-6, norm="attention"):
    """One token of causal attention for each of B independent sequences.

    q, k: [B, H, dk]; v: [B, H, dv]; S: [B, H, r, dv]; z: [B, H, r].  The
    recurrence's single step ("Reassociate a feature-map kernel" ¶4; "The
    Kernel Zoo" §1.3): S' = S + phi(k) v^T, z' = z + phi(k), then the query
    reads the updated state: out = phi(q)^T S' / max(phi(q)^T z', eps)
    (numerator alone under norm "none" and "sum").  Returns (out, S', z');
    the inputs are not modified.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    B, H, _ = q.shape
    S2 = np.array(S, np.float64); z2 = np.array(z, np.float64)
    out = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            pq = features(q[b, h], kind, omega, norm, eps)
            pk = features(k[b, h], kind, omega, norm, eps)
            S2[b, h] += np.outer(pk, v[b, h])
            z2[b, h] += pk
            num = pq @ S2[b, h]
            out[b, h] = num / max(pq @ z2[b, h], eps) if norm == "attention" else num
    return out, S2, z2


def rescan(q, k, v, kind, omega=None, cu_seqlens=None, eps=1e-6, eps_mode="clamp",
           causal_mask=True, norm="attention"):
    """Quadratic form: every query rescans its keys ("Linear attention &
    kernelized approximations", "The naive way: rescan every key").

    out_i = sum_j w_ij v_j / max(sum_j w_ij, eps), w_ij = phi(q_i) . phi(k_j),
    j over the whole sequence (bidirectional) or j <= i (causal); norm as
    for bidir.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, H, _ = q.shape
    dv = v.shape[2]
    cu = _bounds(cu_seqlens, T)
    num = np.zeros((T, H, dv)); den = np.zeros((T, H))
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            pq = features(q[a:b, h], kind, omega, norm, eps)
            pk = features(k[a:b, h], kind, omega, norm, eps)
            for i in range(b - a):
                last = i + 1 if causal_mask else b - a
                w = np.array([pq[i] @ pk[j] for j in range(last)])
                num[a + i, h] = w @ v[a:a + last, h]
                den[a + i, h] = w.sum()
    return _out(num, den, eps, eps_mode, norm)


def causal_rows(q, k, v, kind, omega, start, end, head, rows, eps=1e-6, eps_mode="clamp",
                norm="attention", state0=None):
    """Causal outputs of selected rows of one sequence [start, end) and head.

    Each requested row i gets S_i = S_0 + sum_{start <= j <= i} phi(k_j) v_j^T
    and z_i = z_0 + sum phi(k_j) computed directly from its definition (S_0,
    z_0 = state0, the carried state, or zero), so single rows of very long
    sequences can be checked without running the whole recurrence.
    Returns an array [len(rows), dv].
    """
    kk = np.asarray(k[start:end, head], np.float64)
    vv = np.asarray(v[start:end, head], np.float64)
    pk = features(kk, kind, omega, norm, eps)
    S0, z0 = (0.0, 0.0) if state0 is None else (np.asarray(state0[0], np.float64), np.asarray(state0[1], np.float64))
    outs = []
    for i in rows:
        j = int(i) - start
        assert 0 <= j < end - start
        S = S0 + pk[: j + 1].T @ vv[: j + 1]
        z = z0 + pk[: j + 1].sum(axis=0)
        pq = features(np.asarray(q[int(i), head], np.float64), kind, omega, norm, eps)
        outs.append(_out(pq @ S, np.asarray(pq @ z), eps, eps_mode, norm))
    return np.array(outs)


def bidir_rows(q, k, v, kind, omega, start, end, head, rows, eps=1e-6, eps_mode="clamp",
               norm="attention"):
    """Bidirectional outputs of selected rows of one sequence and head."""
    pk = features(np.asarray(k[start:end, head], np.float64), kind, omega, norm, eps)
    S = pk.T @ np.asarray(v[start:end, head], np.float64)
    z = pk.sum(axis=0)
    pq = features(np.asarray(q[np.asarray(rows, int), head], np.float64), kind, omega, norm, eps)
    return _out(pq @ S, pq @ z, eps, eps_mode, norm)


def feature_map_vjp(x, kind: str, omega, dphi) -> np.ndarray:
    """dL/dx given dL/dphi for phi = feature_map(x) (the chain rule through each map).

    identity: dx = dphi.  elu1: phi' = 1 for x > 0, exp(x) otherwise.
    favor: d phi_f / dx = phi_f (omega_f - x), so dx = Omega^T (dphi * phi)
           - x sum_f dphi_f phi_f.
    dpfp<nu>: phi_f = x~_a x~_b with b = (a + s) mod 2d gives dx~_a += dphi_f
           x~_b and dx~_b += dphi_f x~_a; x~ = relu([x, -x]) passes dx~_i for
           x_i > 0 and -dx~_{i+d} for x_i < 0.
    """
    x = np.asarray(x, np.float64)
    dphi = np.asarray(dphi, np.float64)
    nu = dpfp_nu(kind)
    if kind == "identity":
        return dphi.copy()
    if kind == "elu1":
        return dphi * np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))
    if kind == "favor":
        om = np.asarray(omega, np.float64)
        u = dphi * feature_map(x, "favor", om)
        return u @ om - x * u.sum(axis=-1, keepdims=True)
    if nu is not None:
        d = x.shape[-1]
        xt = np.maximum(np.concatenate([x, -x], axis=-1), 0.0)
        dxt = np.zeros_like(xt)
        for s_ in range(1, nu + 1):
            g = dphi[..., (s_ - 1) * 2 * d:s_ * 2 * d]
            partner = np.roll(xt, -s_, axis=-1)           # x~_{(i+s) mod 2d}
            dxt += g * partner                              # d/dx~_a of x~_a x~_b
            dxt += np.roll(g * xt, s_, axis=-1)             # d/dx~_b, moved back to index b
        return dxt[..., :d] * (x > 0) - dxt[..., d:] * (x < 0)
    raise ValueError(kind)


def features_vjp(x, kind: str, omega, norm: str, eps: float, dfeat) -> np.ndarray:
    """dL/dx given dL/dphi' for the features attention uses (sum-normalised
    under norm "sum": phi' = phi / sigma, sigma = max(sum_f phi_f, eps), so
    dphi = (dphi' - (dphi' . phi') 1) / sigma when the sum exceeds eps and
    dphi' / eps when it was clamped)."""
    dfeat = np.asarray(dfeat, np.float64)
    if norm == "sum":
        phi = feature_map(x, kind, omega)
        tot = phi.sum(axis=-1, keepdims=True)
        sig = np.maximum(tot, eps)
        p = phi / sig
        dot = np.where(tot > eps, (dfeat * p).sum(axis=-1, keepdims=True), 0.0)
        dphi = (dfeat - dot) / sig
    else:
        dphi = dfeat
    return feature_map_vjp(x, kind, omega, dphi)


def backward(q, k, v, dout, kind, causal_form, omega=None, cu_seqlens=None, eps=1e-6, norm="attention"):
    """Gradients (dq, dk, dv) of L = sum(dout * out) for the forward of the
    same arguments ("Reassociate a feature-map kernel" ¶5 asks for errors in
    outputs and gradients), from the quadratic form of one sequence and head:
    W = Phi_Q Phi_K^T (lower triangle, diagonal included, when causal),
    num = W V, den = W 1, out = num / max(den, eps).  By the chain rule
    dnum = dout / max(den, eps), dden = -(dout . out) / den where den > eps
    (0 where the clamp holds), dW = dnum V^T + dden 1^T (masked like W),
    dPhi_Q = dW Phi_K, dPhi_K = dW^T Phi_Q, dV = W^T dnum; then through the
    features (features_vjp).  norm "none" and "sum" have dnum = dout and no
    denominator term.  Omega is a constant (sampled once and frozen).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    T, H, dk_ = q.shape
    cu = _bounds(cu_seqlens, T)
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        for h in range(H):
            pq = features(q[a:b, h], kind, omega, norm, eps)
            pk = features(k[a:b, h], kind, omega, norm, eps)
            W = pq @ pk.T
            if causal_form:
                W = np.tril(W)
            vv = v[a:b, h]
            g = dout[a:b, h]
            num = W @ vv
            den = W.sum(axis=1)
            if norm == "attention":
                dc = np.maximum(den, eps)
                out = num / dc[:, None]
                dnum = g / dc[:, None]
                dden = np.where(den > eps, -(g * out).sum(axis=1) / np.where(den > eps, den, 1.0), 0.0)
            else:
                dnum = g
                dden = np.zeros(b - a)
            dW = dnum @ vv.T + dden[:, None]
            if causal_form:
                dW = np.tril(dW)
            dq[a:b, h] = features_vjp(q[a:b, h], kind, omega, norm, eps, dW @ pk)
            dk[a:b, h] = features_vjp(k[a:b, h], kind, omega, norm, eps, dW.T @ pq)
            dv[a:b, h] = W.T @ dnum
    return dq, dk, dv


def forward(q, k, v, kind, causal_form, omega=None, cu_seqlens=None, eps=1e-6, norm="attention",
            state_in=None):
    """Dispatch to the bidirectional or causal oracle."""
    f = causal if causal_form else bidir
    return f(q, k, v, kind, omega=omega, cu_seqlens=cu_seqlens, eps=eps, norm=norm, state_in=state_in)


def softmax_kernel_estimate(x, y, omega):
    """phi+(x)^T phi+(y), the FAVOR+ estimate of exp(x^T y) ("The Kernel Zoo" §4.2)."""
    return float(feature_map(x, "favor", omega) @ feature_map(y, "favor", omega))
