"""Pins of the fp64 oracle against what the source pages and mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print for their worked examples (tests/golden/, each citing its
passage), closed forms, library routines, invariants and brute force.  The
pins are chosen so that a plausible slip (a dropped 1/sqrt(m), a sign in the
|x|^2/2 term, a transposed projection, an exclusive prefix, a missed state
reset, add-eps instead of clamp) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import synthetic


def _one_head(a):
    """[n, d] -> [n, 1, d]"""
    return np.asarray(a, np.float64)[:, None, :]


# ----------------------------------------------------------------------------
# Worked examples printed on the pages
# ----------------------------------------------------------------------------
def test_identity_bidir_worked_example(golden):
    g = golden("identity_bidir_worked_example.txt")
    K = g["k"]
    v = g["v"].reshape(4, 1)
    q = np.zeros((4, 2)); q[0] = g["q0"]
    out, num, den, states = oracle.bidir(_one_head(q), _one_head(K), _one_head(v), "identity",
                                         return_parts=True)
    S, z = states[(0, 0)]
    assert np.allclose(S[:, 0], g["s"], atol=g["tol"], rtol=0)
    assert np.allclose(z, g["z"], atol=g["tol"], rtol=0)
    assert abs(num[0, 0, 0] - g["num"]) <= g["tol"]
    assert abs(den[0, 0] - g["den"]) <= g["tol"]
    assert abs(out[0, 0, 0] - g["out"]) <= g["tol"]
    # the naive rescan gives the same number
    scores = K @ g["q0"]
    assert np.allclose(scores, g["scores"], atol=0)
    resc = oracle.rescan(_one_head(q), _one_head(K), _one_head(v), "identity", causal_mask=False)
    assert abs(resc[0, 0, 0] - g["out"]) <= g["tol"]


def test_elu1_maps_of_running_example(golden):
    g = golden("elu_running_example.txt")
    assert np.array_equal(oracle.feature_map(g["Q"], "elu1"), g["phiQ"])
    assert np.array_equal(oracle.feature_map(g["K"], "elu1"), g["phiK"])


def test_elu1_causal_state_retrieval_and_o4(golden):
    g = golden("elu_running_example.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    # state after two causal steps
    _, _, _, finals = oracle.causal(Q[:2], K[:2], V[:2], "elu1", return_parts=True)
    S2, z2 = finals[(0, 0)]
    assert np.allclose(S2, g["S2"], atol=g["tol_exact"], rtol=0)
    retrieved = S2.T @ g["phiK"][0]
    assert np.allclose(retrieved, g["retrieve_k1"], atol=g["tol_exact"], rtol=0)
    assert np.allclose(retrieved / retrieved.sum(), g["retrieve_k1_normalised"],
                       atol=g["tol_printed"], rtol=0)
    out = oracle.causal(Q, K, V, "elu1")
    assert np.allclose(out[3, 0], [25 / 26, 15 / 26], atol=g["tol_exact"], rtol=0)
    assert np.allclose(out[3, 0], g["o4"], atol=g["tol_printed"], rtol=0)


def test_fast_weight_programmer_trace(golden):
    g = golden("fwp_identity_trace.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    y, _, _, finals = oracle.causal(Q, K, V, "identity", eps_mode="none", return_parts=True)
    assert np.allclose(y[:, 0], g["y"], atol=g["tol"], rtol=0)
    S4, _ = finals[(0, 0)]
    assert np.allclose(S4.T, g["W4"], atol=g["tol"], rtol=0)


def test_identity_causal_zero_denominator_gives_zero(golden):
    # token 1 of the running example: q1 . k1 = 0 and the numerator is 0 too.
    g = golden("fwp_identity_trace.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    out = oracle.causal(Q, K, V, "identity", eps=1e-6)
    expect = np.array([[0, 0], [1, 0], [0.75, 0.75], [0.5, 1.0]])
    assert np.allclose(out[:, 0], expect, atol=1e-12, rtol=0)


def test_negative_denominator_is_clamped_not_shifted():
    # "Performer" §3 sketch clamps the denominator from below at 1e-6; adding
    # eps would give a very different number for a negative identity-map score.
    q = _one_head([[1.0, 0.0]]); k = _one_head([[-1.0, 0.0]]); v = _one_head([[2.0]])
    clamp = oracle.bidir(q, k, v, "identity", eps=1e-6)
    add = oracle.bidir(q, k, v, "identity", eps=1e-6, eps_mode="add")
    assert clamp[0, 0, 0] == pytest.approx(-2.0 / 1e-6, rel=1e-12)
    assert add[0, 0, 0] == pytest.approx(-2.0 / (-1.0 + 1e-6), rel=1e-12)


def test_favor_m4_worked_example(golden):
    g = golden("favor_m4_worked_example.txt")
    om = g["omega"]
    pq1 = oracle.feature_map(g["q1"], "favor", om)
    pk1 = oracle.feature_map(g["k1"], "favor", om)
    pk2 = oracle.feature_map(g["k2"], "favor", om)
    # exact: exp(-1/2) * exp(1/2) / sqrt(4)
    assert pq1[0] == pytest.approx(0.5, abs=1e-15)
    assert np.allclose(pq1, g["phi_q1"], atol=g["tol"], rtol=0)
    assert np.allclose(pk1, g["phi_k1"], atol=g["tol"], rtol=0)
    assert np.array_equal(pk2, pq1)
    assert abs(pq1 @ pk1 - g["dot_q1_k1"]) <= g["tol"]
    assert abs(pq1 @ pk2 - g["dot_q1_k2"]) <= g["tol"]
    assert np.all(pq1 > 0) and np.all(pk1 > 0)


def test_orf_gram_schmidt_worked_example(golden):
    g = golden("orf_gram_schmidt_worked_example.txt")
    om = oracle.orthogonal_random_features(g["omega_raw"][None], norm="sqrt_d")
    assert np.allclose(om, g["omega_ort"], atol=g["tol"], rtol=0)
    assert abs(om[0] @ om[1]) < 1e-14
    assert np.allclose(np.linalg.norm(om, axis=1), math.sqrt(2), atol=1e-14)
    phi = oracle.feature_map(g["q1"], "favor", om)
    assert np.allclose(phi, g["phi_ort_q1"], atol=g["tol"], rtol=0)


# ----------------------------------------------------------------------------
# Closed forms, library routines, invariants
# ----------------------------------------------------------------------------
def test_elu1_matches_library_elu_plus_one():
    torch = pytest.importorskip("torch")
    x = np.linspace(-12, 6, 2001)
    ref = (torch.nn.functional.elu(torch.tensor(x, dtype=torch.float64), alpha=1.0) + 1).numpy()
    # elu(x) + 1 = (exp(x) - 1) + 1 cancels for x << 0: absolute error ~ 2^-53
    assert np.allclose(oracle.feature_map(x, "elu1"), ref, rtol=1e-15, atol=4e-16)
    assert oracle.feature_map(np.array([-1.0]), "elu1")[0] == pytest.approx(math.exp(-1), rel=1e-15)


def test_dpfp1_worked_examples(golden):
    """DPFP-1 of the running example's keys and of the mixed-sign keys k_A,
    k_B ("The Kernel Zoo", §6.5-6.6)."""
    g = golden("dpfp_worked_example.txt")
    phi = oracle.feature_map(g["K"], "dpfp1")
    assert phi.shape == (6, 4)
    assert np.allclose(phi, g["phiK"], rtol=0, atol=g["tol_exact"])
    assert abs(g["K"][4] @ g["K"][5] - g["kA_dot_kB"]) < g["tol_exact"]
    assert abs(phi[4] @ phi[5] - g["phikA_dot_phikB"]) < g["tol_exact"]
    assert oracle.feature_dim("dpfp1", 2) == 4


def test_dpfp_invariants():
    """Properties the DPFP-nu construction fixes ("The Kernel Zoo", §6.3-6.4):
    d_dot = 2 d nu, non-negative features, the shift-d block is zero (it pairs
    relu(x_i) with relu(-x_i)), degree-2 homogeneity, and phi(-x) equals phi(x)
    with every 2d block rotated by d (x~(-x) is x~(x) rotated by d)."""
    rng = np.random.default_rng(21)
    d, nu = 3, 4
    x = rng.standard_normal((50, d))
    phi = oracle.feature_map(x, f"dpfp{nu}")
    assert phi.shape == (50, 2 * d * nu) and oracle.feature_dim(f"dpfp{nu}", d) == 2 * d * nu
    assert np.all(phi >= 0) and np.count_nonzero(phi) > phi.size // 8
    blocks = phi.reshape(50, nu, 2 * d)
    assert np.array_equal(blocks[:, d - 1], np.zeros((50, 2 * d)))          # s = d
    assert np.count_nonzero(blocks[:, :d - 1]) > 0 and np.count_nonzero(blocks[:, d:]) > 0
    assert np.allclose(oracle.feature_map(2.5 * x, f"dpfp{nu}"), 6.25 * phi, rtol=1e-14, atol=0)
    neg = oracle.feature_map(-x, f"dpfp{nu}").reshape(50, nu, 2 * d)
    assert np.array_equal(neg, np.roll(blocks, d, axis=-1))
    # shift s pairs element i with element i + s: a plausible off-by-one (i - s,
    # or s from 0) breaks the printed k_A / k_B values, pinned above, and this:
    e = np.zeros((1, d)); e[0, 0] = 1.0; e[0, 1] = 1.0                  # x~ = e_0 + e_1
    f1 = oracle.feature_map(e, "dpfp1")[0]
    assert f1[0] == 1.0 and np.count_nonzero(f1) == 1


def test_identity_map_is_identity():
    x = np.random.default_rng(0).standard_normal((5, 7))
    assert np.array_equal(oracle.feature_map(x, "identity"), x)


def test_feature_maps_are_positive():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, 64)) * 2
    om = rng.standard_normal((256, 64))
    assert np.all(oracle.feature_map(x, "elu1") > 0)
    assert np.all(oracle.feature_map(x * 0.3, "favor", om) > 0)


def _chi_orf_batch(rng, nbatch, r, d):
    nb = -(-r // d)
    blocks = rng.standard_normal((nbatch, nb, d, d))
    norms = np.linalg.norm(rng.standard_normal((nbatch, r, d)), axis=-1)
    Q = oracle.gram_schmidt(blocks.reshape(nbatch * nb, d, d)).reshape(nbatch, nb * d, d)[:, :r]
    return Q * norms[..., None]


@pytest.mark.parametrize("xy", [0.5, -0.4])
def test_lemma1_monte_carlo_unbiased_with_chi_orf(xy):
    """Mean over 10^4 independent chi-norm orthogonal draws (d=64, r=256) of
    phi+(x)^T phi+(y) matches exp(x^T y) within 3 standard errors
    ("The Kernel Zoo" §4.1 Lemma 1; "Performer" §2 Steps 3-4)."""
    d, r, nseeds = 64, 256, 10_000
    rng = np.random.default_rng(12345)
    x = rng.standard_normal(d); x /= np.linalg.norm(x)
    w = rng.standard_normal(d); w -= (w @ x) * x; w /= np.linalg.norm(w)
    y = xy * x + math.sqrt(1 - xy * xy) * w            # |x| = |y| = 1, x^T y = xy
    est = []
    for _ in range(nseeds // 500):
        om = _chi_orf_batch(rng, 500, r, d)
        px = np.exp(om @ x - 0.5 * x @ x) / math.sqrt(r)
        py = np.exp(om @ y - 0.5 * y @ y) / math.sqrt(r)
        est.append(np.sum(px * py, axis=-1))
    est = np.concatenate(est)
    se = est.std(ddof=1) / math.sqrt(len(est))
    assert abs(est.mean() - math.exp(xy)) <= 3 * se
    # and the oracle's own feature map gives the same estimate on one draw
    om = _chi_orf_batch(rng, 1, r, d)[0]
    direct = np.exp(om @ x - 0.5) / 16 @ (np.exp(om @ y - 0.5) / 16)
    assert oracle.softmax_kernel_estimate(x, y, om) == pytest.approx(direct, rel=1e-12)


def test_lemma2_iid_positive_estimator_variance():
    """Variance of the i.i.d. positive estimator with m features equals
    SM(x,y)^2 (exp(|x+y|^2) - 1) / m, derived from the Gaussian moment
    generating function used in "The Kernel Zoo" §4.1 (the same quantity as
    §4.4's positive-MSE line, whose last factor is printed with x - y)."""
    d, m, n = 8, 16, 40_000
    rng = np.random.default_rng(7)
    x = rng.standard_normal(d); x *= 0.5 / np.linalg.norm(x)
    y = rng.standard_normal(d); y *= 0.5 / np.linalg.norm(y)
    om = rng.standard_normal((n, m, d))
    est = np.array([oracle.softmax_kernel_estimate(x, y, om[i]) for i in range(n)])
    sm = math.exp(x @ y)
    var = sm * sm * (math.exp((x + y) @ (x + y)) - 1) / m
    assert abs(est.mean() - sm) <= 4 * est.std(ddof=1) / math.sqrt(n)
    assert est.var(ddof=1) == pytest.approx(var, rel=0.08)


def test_sampled_omega_is_block_orthogonal_with_chi_lengths():
    r, d = 256, 64
    blocks, normv = synthetic.omega_gaussians(r, d, seed=7)
    om = oracle.orthogonal_random_features(blocks, normv, r=r)
    lengths = np.linalg.norm(normv, axis=1)
    assert np.allclose(np.linalg.norm(om, axis=1), lengths, rtol=1e-13, atol=0)
    for b in range(r // d):
        blk = om[b * d:(b + 1) * d]
        G = blk @ blk.T
        off = G - np.diag(np.diag(G))
        assert np.max(np.abs(off)) <= 1e-11 * np.max(np.diag(G))
    # each block spans the same space as its Gaussian draw (Gram-Schmidt keeps
    # the leading subspaces): row i lies in span(draw rows 0..i)
    B0 = blocks[0]
    for i in (0, 5, 31, 63):
        coef, *_ = np.linalg.lstsq(B0[: i + 1].T, om[i], rcond=None)
        assert np.allclose(B0[: i + 1].T @ coef, om[i], atol=1e-9)


def test_chi_lengths_have_chi_mean():
    """E|g| for g ~ N(0, I_d) is sqrt(2) Gamma((d+1)/2) / Gamma(d/2) (chi mean)."""
    from scipy.special import gammaln
    d, n = 64, 20_000
    lengths = np.linalg.norm(np.random.default_rng(3).standard_normal((n, d)), axis=1)
    mean = math.sqrt(2) * math.exp(gammaln((d + 1) / 2) - gammaln(d / 2))
    assert abs(lengths.mean() - mean) <= 3 * lengths.std() / math.sqrt(n)


@pytest.mark.parametrize("kind", ["identity", "elu1", "favor", "dpfp2"])
@pytest.mark.parametrize("causal_form", [True, False])
def test_linear_form_equals_quadratic_rescan(kind, causal_form):
    """Reassociation: the state form equals every query rescanning its keys
    ("Linear attention & kernelized approximations"; "The Kernel Zoo" §1.3)."""
    rng = np.random.default_rng(11)
    lengths = [5, 1, 10]
    T, H, d, dv = sum(lengths), 2, 4, 3
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q = rng.standard_normal((T, H, d)) * 0.6
    k = rng.standard_normal((T, H, d)) * 0.6
    v = rng.standard_normal((T, H, dv))
    om = rng.standard_normal((12, d))
    fast = oracle.forward(q, k, v, kind, causal_form, omega=om, cu_seqlens=cu)
    slow = oracle.rescan(q, k, v, kind, omega=om, cu_seqlens=cu, causal_mask=causal_form)
    if kind in ("identity", "dpfp2"):
        # identity scores can make den <= eps (and DPFP features can all vanish);
        # compare with a tolerance relative to the largest output
        assert np.allclose(fast, slow, rtol=1e-9, atol=1e-9 * np.abs(slow).max())
    else:
        assert np.allclose(fast, slow, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal_form", [True, False])
def test_packed_sequences_reset_state(causal_form):
    """A packed batch equals each sequence run alone ("Reassociate a
    feature-map kernel" ¶4: packing must reset the state at the boundary)."""
    rng = np.random.default_rng(5)
    lengths = [7, 3, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d = cu[-1], 2, 4
    q, k, v = (rng.standard_normal((T, H, d)) * 0.5 for _ in range(3))
    om = rng.standard_normal((8, d))
    packed = oracle.forward(q, k, v, "favor", causal_form, omega=om, cu_seqlens=cu)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        alone = oracle.forward(q[a:b], k[a:b], v[a:b], "favor", causal_form, omega=om)
        assert np.array_equal(packed[a:b], alone)
    # a missed reset would leak the previous sequence: check that it matters
    joined = oracle.forward(q, k, v, "favor", causal_form, omega=om)
    assert not np.allclose(joined[cu[1]:cu[2]], packed[cu[1]:cu[2]])


def test_last_causal_row_equals_bidirectional_row():
    rng = np.random.default_rng(9)
    T, H, d = 12, 3, 5
    q, k, v = (rng.standard_normal((T, H, d)) * 0.5 for _ in range(3))
    om = rng.standard_normal((16, d))
    c = oracle.causal(q, k, v, "favor", omega=om)
    b = oracle.bidir(q, k, v, "favor", omega=om)
    assert np.allclose(c[-1], b[-1], rtol=1e-12, atol=0)
    assert not np.allclose(c[0], b[0])


def test_row_sampler_matches_recurrence():
    rng = np.random.default_rng(2)
    T, H, d = 40, 2, 6
    q, k, v = (rng.standard_normal((T, H, d)) * 0.5 for _ in range(3))
    om = rng.standard_normal((16, d))
    cu = [0, 13, 40]
    full_c = oracle.causal(q, k, v, "favor", omega=om, cu_seqlens=cu)
    full_b = oracle.bidir(q, k, v, "favor", omega=om, cu_seqlens=cu)
    rows = [13, 14, 27, 39]
    got_c = oracle.causal_rows(q, k, v, "favor", om, 13, 40, 1, rows)
    got_b = oracle.bidir_rows(q, k, v, "favor", om, 13, 40, 1, rows)
    assert np.allclose(got_c, full_c[rows, 1], rtol=1e-12, atol=1e-14)
    assert np.allclose(got_b, full_b[rows, 1], rtol=1e-12, atol=1e-14)


def test_favor_kernel_matrix_is_unbiased_for_exp_scores():
    """Averaged over independent chi-norm orthogonal draws, the FAVOR+ score
    matrix Phi_Q Phi_K^T matches the softmax kernel exp(Q K^T) entrywise
    within 4 standard errors ("Performer" §2 Steps 3-5)."""
    rng = np.random.default_rng(4)
    n, d, r, draws = 6, 8, 64, 4000
    q = rng.standard_normal((n, d)) * d ** -0.25
    k = rng.standard_normal((n, d)) * d ** -0.25
    om = _chi_orf_batch(rng, draws, r, d)
    est = np.stack([oracle.feature_map(q, "favor", om[t]) @ oracle.feature_map(k, "favor", om[t]).T
                    for t in range(draws)])
    mean = est.mean(axis=0)
    se = est.std(axis=0, ddof=1) / np.sqrt(draws)
    assert np.all(np.abs(mean - np.exp(q @ k.T)) <= 4 * se)


# ----------------------------------------------------------------------------
# Normalisation variants, state carry and the decode step
# ----------------------------------------------------------------------------
def test_sum_normalisation_worked_example(golden):
    g = golden("sum_normalisation_example.txt")
    assert np.array_equal(oracle.feature_map(g["q1"], "elu1"), g["phi_q1"])
    assert np.array_equal(oracle.feature_map(g["k1"], "elu1"), g["phi_k1"])
    pq = oracle.features(g["q1"], "elu1", norm="sum")
    pk = oracle.features(g["k1"], "elu1", norm="sum")
    assert np.allclose(pq, g["phi_q1_sum"], atol=g["tol"], rtol=0)
    assert np.allclose(pk, g["phi_k1_sum"], atol=g["tol"], rtol=0)
    assert abs(pq @ pk - g["sim_sum"]) <= g["tol"]
    assert abs(pq @ pk - g["sim_sum_printed"]) <= g["tol_printed"]
    assert oracle.feature_map(g["q1"], "elu1") @ oracle.feature_map(g["k1"], "elu1") == g["sim"]
    # the other norms leave the features alone
    assert np.array_equal(oracle.features(g["q1"], "elu1", norm="none"), g["phi_q1"])


@pytest.mark.parametrize("kind", ["elu1", "favor", "dpfp2"])
def test_sum_normalised_features_sum_to_one(kind):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((9, 4)) * 0.7
    om = rng.standard_normal((8, 4))
    p = oracle.features(x, kind, om, norm="sum")
    assert np.allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p >= 0)
    # proportional to phi: the direction is unchanged
    raw = oracle.feature_map(x, kind, om)
    assert np.allclose(p * raw.sum(axis=-1, keepdims=True), raw, rtol=1e-13, atol=0)


def test_sum_normalisation_of_a_zero_feature_vector_is_zero():
    # DPFP of x = 0 has no positive part: every feature is 0 and the sum is
    # clamped at eps instead of dividing 0 by 0.
    p = oracle.features(np.zeros(3), "dpfp1", norm="sum", eps=1e-6)
    assert np.array_equal(p, np.zeros(6))


def test_sum_normalised_output_is_a_convex_combination():
    """Under sum normalisation the output is phi'(q)-weighted columns of the
    fast weights with weights summing to 1 ("The Kernel Zoo" §7.4): with one
    stored pair (k, c) the output is (phi'(q) . phi'(k)) c, a weight strictly
    between 0 and 1 for dense positive features, and no denominator."""
    c = np.array([0.5, -2.0, 3.0])
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 1, 2)); k = rng.standard_normal((1, 1, 2))
    v = c[None, None, :]
    out = oracle.causal(q, k, v, "elu1", norm="sum")
    w = oracle.features(q[0, 0], "elu1", norm="sum") @ oracle.features(k[0, 0], "elu1", norm="sum")
    assert 0 < w < 1
    assert np.allclose(out[0, 0], w * c, rtol=1e-14, atol=0)


@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
@pytest.mark.parametrize("causal_form", [True, False])
def test_norm_variants_equal_quadratic_rescan(norm, causal_form):
    rng = np.random.default_rng(12)
    lengths = [6, 0, 9]
    T, H, d, dv = sum(lengths), 2, 4, 3
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k = (rng.standard_normal((T, H, d)) * 0.6 for _ in range(2))
    v = rng.standard_normal((T, H, dv))
    om = rng.standard_normal((12, d))
    for kind in ("elu1", "favor"):
        fast = oracle.forward(q, k, v, kind, causal_form, omega=om, cu_seqlens=cu, norm=norm)
        slow = oracle.rescan(q, k, v, kind, omega=om, cu_seqlens=cu, causal_mask=causal_form, norm=norm)
        assert np.allclose(fast, slow, rtol=1e-12, atol=1e-14)


def test_norm_none_is_the_fast_weight_trace(golden):
    g = golden("fwp_identity_trace.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    y = oracle.causal(Q, K, V, "identity", norm="none")
    assert np.allclose(y[:, 0], g["y"], atol=g["tol"], rtol=0)
    # attention normalisation of the same trace differs (token 3: (0.75, 0.75))
    assert not np.allclose(oracle.causal(Q, K, V, "identity")[:, 0], g["y"])


def _state_pair(finals, nseq, H):
    S = np.stack([np.stack([finals[(s, h)][0] for h in range(H)]) for s in range(nseq)])
    z = np.stack([np.stack([finals[(s, h)][1] for h in range(H)]) for s in range(nseq)])
    return S, z


def test_state_carry_continues_the_running_example(golden):
    """Carrying S_2 (printed) and z_2 = phi(k_1) + phi(k_2) (printed maps)
    into a second segment of tokens 3-4 gives the page's o_4."""
    g = golden("elu_running_example.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    S2 = np.asarray(g["S2"])[None, None]
    z2 = (g["phiK"][0] + g["phiK"][1])[None, None]
    out, _, _, finals = oracle.causal(Q[2:], K[2:], V[2:], "elu1", state_in=(S2, z2), return_parts=True)
    assert np.allclose(out[1, 0], [25 / 26, 15 / 26], atol=g["tol_exact"], rtol=0)
    assert np.allclose(out[1, 0], g["o4"], atol=g["tol_printed"], rtol=0)
    # without the carried state the second segment starts from zero and differs
    assert not np.allclose(oracle.causal(Q[2:], K[2:], V[2:], "elu1")[1, 0], g["o4"], atol=1e-2)


def test_state_carry_reaches_the_printed_fast_weights(golden):
    g = golden("fwp_identity_trace.txt")
    Q, K, V = (_one_head(g[n]) for n in ("Q", "K", "V"))
    _, _, _, f1 = oracle.causal(Q[:2], K[:2], V[:2], "identity", norm="none", return_parts=True)
    y, _, _, f2 = oracle.causal(Q[2:], K[2:], V[2:], "identity", norm="none",
                                state_in=_state_pair(f1, 1, 1), return_parts=True)
    assert np.allclose(y[:, 0], g["y"][2:], atol=g["tol"], rtol=0)
    assert np.allclose(f2[(0, 0)][0].T, g["W4"], atol=g["tol"], rtol=0)


@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
@pytest.mark.parametrize("causal_form", [True, False])
def test_split_segments_with_carried_state_equal_the_whole(norm, causal_form):
    """Running every sequence in two segments, the second starting from the
    first's final state, equals one run over the whole sequences (causal: the
    recurrence continues; bidirectional: the sums add)."""
    rng = np.random.default_rng(31)
    first, second = [4, 0, 6], [5, 3, 0]
    H, d, dv = 2, 3, 2
    om = rng.standard_normal((8, d))
    seqs = [(rng.standard_normal((a + b, H, d)) * 0.6, rng.standard_normal((a + b, H, d)) * 0.6,
             rng.standard_normal((a + b, H, dv))) for a, b in zip(first, second)]
    cat = lambda parts: np.concatenate(parts, axis=0)
    cu1 = np.concatenate([[0], np.cumsum(first)]); cu2 = np.concatenate([[0], np.cumsum(second)])
    cuw = np.concatenate([[0], np.cumsum(np.add(first, second))])
    f = oracle.causal if causal_form else oracle.bidir
    for kind in ("elu1", "favor"):
        qw, kw, vw = (cat([s[i] for s in seqs]) for i in range(3))
        q1, k1, v1 = (cat([s[i][:a] for s, a in zip(seqs, first)]) for i in range(3))
        q2, k2, v2 = (cat([s[i][a:] for s, a in zip(seqs, first)]) for i in range(3))
        _, _, _, f1 = f(q1, k1, v1, kind, omega=om, cu_seqlens=cu1, norm=norm, return_parts=True)
        out2, _, _, f2 = f(q2, k2, v2, kind, omega=om, cu_seqlens=cu2, norm=norm,
                           state_in=_state_pair(f1, 3, H), return_parts=True)
        whole, _, _, fw = f(qw, kw, vw, kind, omega=om, cu_seqlens=cuw, norm=norm, return_parts=True)
        for s, (a, b) in enumerate(zip(first, second)):
            assert np.allclose(out2[cu2[s]:cu2[s + 1]], whole[cuw[s] + a:cuw[s + 1]], rtol=1e-12, atol=1e-14)
            for h in range(H):
                assert np.allclose(f2[(s, h)][0], fw[(s, h)][0], rtol=1e-12, atol=1e-14)
                assert np.allclose(f2[(s, h)][1], fw[(s, h)][1], rtol=1e-12, atol=1e-14)


def test_decode_steps_replay_the_running_example(golden):
    """One decode step per token from a zero state gives the page's outputs:
    the fast-weight trace y (identity, no normalisation), o_4 (ELU+1) and W_4."""
    gy = golden("fwp_identity_trace.txt")
    ge = golden("elu_running_example.txt")
    for kind, norm, g, check in (("identity", "none", gy, "y"), ("elu1", "attention", ge, "o4")):
        Q, K, V = g["Q"], g["K"], g["V"]
        S = np.zeros((1, 1, 2, 2)); z = np.zeros((1, 1, 2))
        outs = []
        for t in range(4):
            o, S, z = oracle.decode_step(Q[t][None, None], K[t][None, None], V[t][None, None], kind, S, z,
                                         norm=norm)
            outs.append(o[0, 0])
        if check == "y":
            assert np.allclose(outs, g["y"], atol=g["tol"], rtol=0)
            assert np.allclose(S[0, 0].T, g["W4"], atol=g["tol"], rtol=0)
        else:
            assert np.allclose(outs[3], [25 / 26, 15 / 26], atol=g["tol_exact"], rtol=0)


@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
def test_decode_steps_equal_the_causal_recurrence(norm):
    rng = np.random.default_rng(17)
    B, H, n, d, dv = 3, 2, 7, 4, 3
    om = rng.standard_normal((8, d))
    q, k = (rng.standard_normal((B, n, H, d)) * 0.6 for _ in range(2))
    v = rng.standard_normal((B, n, H, dv))
    for kind in ("elu1", "favor", "dpfp1"):
        r = oracle.feature_dim(kind, d, om)
        S = np.zeros((B, H, r, dv)); z = np.zeros((B, H, r))
        steps = []
        for t in range(n):
            o, S2, z2 = oracle.decode_step(q[:, t], k[:, t], v[:, t], kind, S, z, omega=om, norm=norm)
            assert not np.shares_memory(S2, S)
            S, z = S2, z2
            steps.append(o)
        steps = np.stack(steps, axis=1)            # [B, n, H, dv]
        cu = np.arange(B + 1) * n
        ref, _, _, finals = oracle.causal(q.reshape(B * n, H, d), k.reshape(B * n, H, d), v.reshape(B * n, H, dv),
                                          kind, omega=om, cu_seqlens=cu, norm=norm, return_parts=True)
        assert np.allclose(steps.reshape(B * n, H, dv), ref, rtol=1e-12, atol=1e-13)
        Sf, zf = _state_pair(finals, B, H)
        assert np.allclose(S, Sf, rtol=1e-12, atol=1e-14) and np.allclose(z, zf, rtol=1e-12, atol=1e-14)


def test_row_sampler_with_carried_state_matches_recurrence():
    rng = np.random.default_rng(6)
    T, H, d = 30, 2, 5
    q, k, v = (rng.standard_normal((T, H, d)) * 0.5 for _ in range(3))
    om = rng.standard_normal((8, d))
    S0 = rng.standard_normal((1, H, 8, d)); z0 = rng.uniform(1, 2, size=(1, H, 8))
    full = oracle.causal(q, k, v, "favor", omega=om, state_in=(S0, z0))
    rows = [0, 7, 29]
    got = oracle.causal_rows(q, k, v, "favor", om, 0, T, 1, rows, state0=(S0[0, 1], z0[0, 1]))
    assert np.allclose(got, full[rows, 1], rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# Backward pass
# ----------------------------------------------------------------------------
def _loss(q, k, v, dout, kind, causal_form, om, cu, norm):
    return float(np.sum(dout * oracle.forward(q, k, v, kind, causal_form, omega=om, cu_seqlens=cu, norm=norm)))


def _finite_difference_grads(q, k, v, dout, kind, causal_form, om, cu, norm, h=1e-6):
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(args[which])
        it = np.nditer(args[which], flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            base = args[which][i]
            args[which][i] = base + h
            lp = _loss(*args, dout, kind, causal_form, om, cu, norm)
            args[which][i] = base - h
            lm = _loss(*args, dout, kind, causal_form, om, cu, norm)
            args[which][i] = base
            g[i] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("kind", ["identity", "elu1", "favor", "dpfp1"])
@pytest.mark.parametrize("causal_form", [True, False])
@pytest.mark.parametrize("norm", ["attention", "none", "sum"])
def test_backward_matches_finite_differences(kind, causal_form, norm):
    """Central differences of sum(dout * out), element by element, on tiny
    packed inputs (two sequences, one of them a single token)."""
    if kind == "identity" and norm == "sum":
        pytest.skip("sum normalisation needs non-negative features")
    rng = np.random.default_rng(41)
    lengths = [4, 1]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d, dv = cu[-1], 1, 3, 2
    q, k = (rng.standard_normal((T, H, d)) * 0.7 for _ in range(2))
    if kind == "identity":   # keep the identity-map denominators well away from the eps clamp
        q, k = np.abs(q) + 0.2, np.abs(k) + 0.2
    v = rng.standard_normal((T, H, dv))
    dout = rng.standard_normal((T, H, dv))
    om = rng.standard_normal((5, d))
    got = oracle.backward(q, k, v, dout, kind, causal_form, omega=om, cu_seqlens=cu, norm=norm)
    want = _finite_difference_grads(q, k, v, dout, kind, causal_form, om, cu, norm)
    for g, w, name in zip(got, want, ("dq", "dk", "dv")):
        scale = max(1.0, np.abs(w).max())
        assert np.allclose(g, w, rtol=0, atol=2e-7 * scale), f"{name}: {np.abs(g - w).max():.2e}"


def test_backward_value_gradient_sums_to_upstream_gradient():
    """Attention-normalised outputs are convex combinations of the values
    (weights w_ij / den_i summing to 1 over j), so sum_j dL/dv_j equals
    sum_i dL/dout_i within every sequence and head."""
    rng = np.random.default_rng(42)
    lengths = [6, 3]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d = cu[-1], 2, 4
    q, k = (rng.standard_normal((T, H, d)) * 0.5 for _ in range(2))
    v, dout = (rng.standard_normal((T, H, 3)) for _ in range(2))
    om = rng.standard_normal((8, d))
    for causal_form in (True, False):
        _, _, dv = oracle.backward(q, k, v, dout, "favor", causal_form, omega=om, cu_seqlens=cu)
        for s in range(2):
            a, b = cu[s], cu[s + 1]
            assert np.allclose(dv[a:b].sum(axis=0), dout[a:b].sum(axis=0), rtol=1e-12, atol=1e-12)


def test_backward_of_packed_batch_equals_each_sequence_alone():
    rng = np.random.default_rng(43)
    lengths = [5, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d = cu[-1], 2, 3
    q, k, v, dout = (rng.standard_normal((T, H, d)) * 0.6 for _ in range(4))
    om = rng.standard_normal((6, d))
    packed = oracle.backward(q, k, v, dout, "favor", True, omega=om, cu_seqlens=cu)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        alone = oracle.backward(q[a:b], k[a:b], v[a:b], dout[a:b], "favor", True, omega=om)
        for x, y in zip(packed, alone):
            assert np.array_equal(x[a:b], y)
