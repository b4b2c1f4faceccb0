"""Pins for the oracle's Attention Matching fits (mass fit for beta, value fit for V_C).

Source: "Practical Online KV Cache Compaction for LLM Agents: An Empirical Study" (agifrontier
tutorial page), section on the two compaction families: after keeping the top-m keys, AM fits
an additive bias beta, min ||exp(Q K_C^T + beta) 1_m - exp(Q K^T) 1_n||^2, and compact values
V_C, min ||A_hat(Q; K_C, beta, V_C) - A(Q; K, V)||_F^2.

The oracle reads the open solver as cyclic coordinate descent from token eviction's answer.
These tests pin it to things other than itself: the non-negative least-squares optimum by brute
force over supports and by scipy's active-set solver, the least-squares optimum by numpy's
lstsq, one-key closed forms, the keep-all fixed point, monotone descent, and the token-eviction
score oracle (a separate C implementation) for the targets.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import am


def rng(seed):
    return np.random.default_rng(seed)


def nnls_brute_force(E, s):
    """min_{w >= 0} ||E w - s||^2 by trying every support: least squares on the support, kept
    if it is non-negative and the gradient outside it is >= 0 (the KKT conditions)."""
    m = E.shape[1]
    best, best_f = None, np.inf
    for k in range(m + 1):
        for S in itertools.combinations(range(m), k):
            w = np.zeros(m)
            if S:
                w[list(S)] = np.linalg.lstsq(E[:, S], s, rcond=None)[0]
            if np.any(w < -1e-12):
                continue
            g = E.T @ (E @ w - s)
            out = [j for j in range(m) if j not in S]
            if out and np.any(g[out] < -1e-9):
                continue
            f = float(np.sum((E @ w - s) ** 2))
            if f < best_f - 1e-15:
                best, best_f = w, f
    return best, best_f


@pytest.mark.parametrize("seed", range(6))
def test_mass_fit_reaches_the_nnls_optimum(seed):
    """Well-conditioned E (R = 9 > m = 4) with a target that forces some w_j = 0: many sweeps
    of the projected coordinate descent land on the brute-force and scipy optimum."""
    g = rng(seed)
    E = np.abs(g.standard_normal((9, 4))) + 0.1 * np.eye(9, 4)
    w_true = np.array([1.5, 0.0, 0.7, 0.0])
    s = E @ w_true + 0.3 * g.standard_normal(9)
    w_bf, f_bf = nnls_brute_force(E, s)
    w = am.mass_fit(E, s, 3000)
    np.testing.assert_allclose(w, w_bf, atol=1e-8)
    assert am.mass_objective(E, s, w) == pytest.approx(f_bf, rel=1e-10, abs=1e-14)
    scipy_opt = pytest.importorskip("scipy.optimize")
    w_sp, _ = scipy_opt.nnls(E, s)
    np.testing.assert_allclose(w, w_sp, atol=1e-8)
    assert np.all(w >= 0)


def test_mass_fit_active_constraint_is_exact_zero():
    """A key whose column points away from the target is clipped to w = 0 exactly (beta = -inf)."""
    E = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]])
    s = np.array([2.0, -1.0, 0.0])
    w = am.mass_fit(E, s, 3)
    assert w[0] == pytest.approx(2.0, abs=1e-15) and w[1] == 0.0
    beta = am.beta_of(w)
    assert beta[0] == pytest.approx(np.log(2.0)) and beta[1] == -np.inf


def test_mass_fit_one_key_closed_form():
    """m = 1: w = max(0, e.s / e.e) after one sweep."""
    g = rng(3)
    for _ in range(20):
        e = np.abs(g.standard_normal(7))
        s = g.standard_normal(7) + 0.5
        w = am.mass_fit(e[:, None], s, 1)
        assert w[0] == pytest.approx(max(0.0, e @ s / (e @ e)), rel=1e-13, abs=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_value_fit_reaches_least_squares(seed):
    """Full column rank Ph (R = 12 > m = 5): many sweeps reach numpy's lstsq solution."""
    g = rng(10 + seed)
    Ph = np.abs(g.standard_normal((12, 5)))
    Ph /= Ph.sum(axis=1, keepdims=True)
    Y = g.standard_normal((12, 3))
    X = am.value_fit(Ph, Y, g.standard_normal((5, 3)), 4000)
    X_ls = np.linalg.lstsq(Ph, Y, rcond=None)[0]
    np.testing.assert_allclose(X, X_ls, atol=1e-7)


def test_value_fit_one_key_is_the_mean_target():
    """m = 1: every row of Ph is 1 (rows normalised), so V_C is the mean of the target rows."""
    g = rng(4)
    Y = g.standard_normal((6, 4))
    X = am.value_fit(np.ones((6, 1)), Y, np.zeros((1, 4)), 1)
    np.testing.assert_allclose(X[0], Y.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_keep_all_is_a_fixed_point():
    """With every key kept, w = 1 matches the mass exactly and V_C = V reproduces the output:
    both gradients vanish and token eviction's start is returned unchanged."""
    g = rng(5)
    Q, K, V = g.standard_normal((6, 4)), g.standard_normal((9, 4)), g.standard_normal((9, 4))
    u = am.unit(Q, K, V, np.arange(9), 0.5, 6)
    np.testing.assert_allclose(u["w"], 1.0, atol=1e-12)
    np.testing.assert_allclose(u["vc"], V, atol=1e-10)
    assert am.mass_objective(u["E"], u["s"], u["w"]) < 1e-25
    assert np.all(u["beta"] == pytest.approx(0.0, abs=1e-12))


@pytest.mark.parametrize("seed", range(4))
def test_fits_never_increase_their_objective(seed):
    """Coordinate descent takes the exact minimiser along each coordinate: each sweep lowers (or
    keeps) the objective, starting from token eviction's w = 1 and V_C = V_keep."""
    g = rng(20 + seed)
    Q, K, V = g.standard_normal((16, 8)), g.standard_normal((40, 8)), g.standard_normal((40, 8))
    keep = np.sort(g.choice(40, size=9, replace=False))
    lse, Y = am.targets(Q, K, V, 0.7)
    c = lse.max()
    s = np.exp(lse - c)
    E = np.exp(am.logits(Q, K[keep], 0.7) - c)
    prev = am.mass_objective(E, s, np.ones(9))
    for t in range(1, 6):
        f = am.mass_objective(E, s, am.mass_fit(E, s, t))
        assert f <= prev * (1 + 1e-12) + 1e-300
        prev = f
    w = am.mass_fit(E, s, 5)
    prev = am.value_objective(E, Y, w, V[keep])
    for t in range(1, 6):
        f = am.value_objective(E, Y, w, am.value_fit(am.compact_probs(E, w), Y, V[keep], t))
        assert f <= prev * (1 + 1e-12) + 1e-300
        prev = f


def test_common_shift_leaves_the_fits_unchanged():
    """Scaling E and s by one constant (a common shift of all logits) changes neither w nor V_C."""
    g = rng(6)
    E = np.abs(g.standard_normal((10, 4)))
    s = np.abs(g.standard_normal(10)) + 1.0
    Y = g.standard_normal((10, 3))
    for k in (1e-30, 1e5):
        np.testing.assert_allclose(am.mass_fit(E * k, s * k, 7), am.mass_fit(E, s, 7), rtol=1e-10)
        np.testing.assert_allclose(am.compact_probs(E * k, np.ones(4)), am.compact_probs(E, np.ones(4)),
                                   rtol=1e-13)


def test_targets_match_the_score_oracle():
    """The targets' LSE is the C oracle's LSE; with V = identity, Y is the attention matrix,
    whose per-column root-mean-square is the C oracle's token-eviction score."""
    g = rng(7)
    Q, K = g.standard_normal((5, 6)), g.standard_normal((11, 6))
    lse, Y = am.targets(Q, K, np.eye(11), 0.4)
    s_ref, lse_ref = oracle.score_dense(Q, K, 0.4)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)
    np.testing.assert_allclose(np.sqrt((Y ** 2).mean(axis=0)), s_ref, rtol=1e-12)
    np.testing.assert_allclose(Y.sum(axis=1), 1.0, rtol=1e-13)


def test_cache_walks_pages_like_dense():
    """The paged driver gathers K, V, Q through a shuffled block table and gives the same fits
    as the dense unit on the gathered operands."""
    import torch

    import workloads
    sp = workloads.custom(L=2, H=2, G=2, d=16, P=8, q=3, lengths=(37, 20), shuffle_pages=True)
    case = workloads.build(sp, 3, "cpu")
    kb = case.k_pool.view(torch.int16).numpy().view(np.uint16)
    vb = case.v_pool.view(torch.int16).numpy().view(np.uint16)
    qb = case.q.view(torch.int16).numpy().view(np.uint16)
    m = [8, 5]
    g = rng(8)
    keep = np.zeros((2, 2, 13), np.int32)
    for l in range(2):
        for h in range(2):
            keep[l, h, :8] = np.sort(g.choice(37, 8, replace=False))
            keep[l, h, 8:] = np.sort(g.choice(20, 5, replace=False))
    bt = case.block_table.numpy()
    w, vc, units = am.cache(kb, vb, qb, bt, [0, 0], [37, 20], keep, m, sp.scale, 4)
    for (b, l, h), u in units.items():
        s0, n = 0, (37, 20)[b]
        K = workloads.gather_keys(case, b, s0, n)[l, h].double().numpy()
        slots = np.arange(n)
        pages = bt[b][slots // sp.P]
        V = case.v_pool[l, pages, h, slots % sp.P].double().numpy()
        Q = case.q[b, l, h].double().numpy()
        off = (0, 8)[b]
        kp = keep[l, h, off:off + m[b]]
        ref = am.unit(Q, K, V, kp, sp.scale, 4)
        np.testing.assert_array_equal(w[l, h, off:off + m[b]], ref["w"])
        np.testing.assert_array_equal(vc[l, h, off:off + m[b]], ref["vc"])


def test_concentrated_attention_keeps_token_eviction_residuals():
    """Concentrated attention (each proxy row aims at one kept key): token eviction already
    reproduces the mass and the output to fp64 rounding.  The plain fits may take steps of
    rounding size here, but neither residual may rise above the start's, and both stay at the
    rounding level of the targets."""
    g = rng(12)
    K = g.standard_normal((30, 16)) * 3
    V = g.standard_normal((30, 16))
    keep = np.array([2, 7, 11, 19, 23])
    Q = np.repeat(K[keep], 4, axis=0) * 3 + 0.01 * g.standard_normal((20, 16))
    u = am.unit(Q, K, V, keep, 1.0, 8)
    m0 = am.mass_objective(u["E"], u["s"], np.ones(5))
    v0 = am.value_objective(u["E"], u["Y"], np.ones(5), V[keep])
    assert am.mass_objective(u["E"], u["s"], u["w"]) <= m0 * (1 + 1e-9) + 1e-30
    assert am.value_objective(u["E"], u["Y"], u["w"], u["vc"]) <= v0 * (1 + 1e-9) + 1e-30
    assert np.sqrt(am.mass_objective(u["E"], u["s"], u["w"])) <= 1e-12 * np.linalg.norm(u["s"])
    assert np.sqrt(am.value_objective(u["E"], u["Y"], u["w"], u["vc"])) <= 1e-10 * np.linalg.norm(u["Y"])
