"""Pins for the oracle's lossless accept / resample step (no GPU).

"TriForce: Hierarchical Speculative Decoding for LLMs", section "Dual
Rejection Sampling: Mathematical Losslessness": accept x when
min(1, p(x)/q(x)) >= u, otherwise resample from max(0, p - q) normalised; the
two levels telescope so the emitted tokens follow the target distribution.

Pins: the losslessness theorem itself (chi-square on a 16-token vocabulary with
10^6 trials, for one level and for the two-level r -> q -> p composition), an
exact quadrature case, a hand-worked fixture, the acceptance-rate identity
P(accept) = sum_x min(p(x), q(x)) and the degenerate cases.
"""

import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle import triforce as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _probs(logits):
    e = np.exp(logits - logits.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def _draw(rng, probs, n):
    """n tokens from each row of probs [R, V] -> [n, R] (numpy's sampler)."""
    return np.stack([rng.choice(probs.shape[-1], size=n, p=probs[i]) for i in range(probs.shape[0])], axis=1)


def _chi2_pvalue(tokens, p):
    """Chi-square goodness of fit; bins of probability zero must stay empty."""
    counts = np.bincount(tokens, minlength=len(p))
    nz = p > 0
    assert counts[~nz].sum() == 0
    return stats.chisquare(counts[nz], p[nz] / p[nz].sum() * counts.sum()).pvalue


def test_golden_hand_cases():
    with open(os.path.join(GOLDEN, "spec_accept_hand.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        r = O.spec_accept(np.array(fx["tgt_logits"])[None], np.array(fx["drf_logits"])[None],
                          np.array([case["x"]]), np.array([case["u_acc"]]), np.array([case["u_res"]]))
        assert int(r["n_acc"][0]) == case["n_acc"], case
        assert int(r["next"][0]) == case["next"], case
        assert r["out_tokens"][0].tolist() == case["out_tokens"], case


def _lossless_setup(seed, V=16, gamma=4):
    rng = np.random.default_rng(seed)
    tgt = rng.standard_normal((gamma + 1, V)) * 2.0
    drf = tgt[:gamma] + rng.standard_normal((gamma, V))
    return rng, tgt, drf


def test_single_level_is_lossless_chi_square():
    N, V, gamma = 1_000_000, 16, 4
    rng, tgt, drf = _lossless_setup(0, V, gamma)
    p, q = _probs(tgt), _probs(drf)
    x = _draw(rng, q, N)
    r = O.spec_accept(tgt[None], drf[None], x, rng.random((N, gamma)), rng.random(N))
    assert _chi2_pvalue(r["out_tokens"][:, 0], p[0]) > 1e-3
    # Given position 0 was accepted, the token emitted at position 1 follows p_1.
    m = r["n_acc"] >= 1
    assert _chi2_pvalue(r["out_tokens"][m, 1], p[1]) > 1e-3
    # Acceptance-rate identity at position 0: P(accept) = sum_x min(p0, q0).
    rate = m.mean()
    want = np.minimum(p[0], q[0]).sum()
    assert abs(rate - want) < 5 * np.sqrt(want * (1 - want) / N)


def test_two_level_composition_is_lossless_chi_square():
    """r -> q (tiny drafter checked by the retrieval drafter), then q -> p
    (retrieval drafter checked by the target): the first emitted token follows p."""
    N, V, g1 = 1_000_000, 16, 4
    rng = np.random.default_rng(1)
    p_log = rng.standard_normal((g1 + 2, V)) * 2.0
    q_log = p_log[: g1 + 1] + rng.standard_normal((g1 + 1, V))
    r_log = q_log[:g1] + rng.standard_normal((g1, V))
    x = _draw(rng, _probs(r_log), N)
    lvl1 = O.spec_accept(q_log[None], r_log[None], x, rng.random((N, g1)), rng.random(N))
    y = lvl1["out_tokens"]  # accepted drafts + next token, -1 padded: the level-2 draft
    lvl2 = O.spec_accept(p_log[None], q_log[None], y, rng.random((N, g1 + 1)), rng.random(N))
    assert _chi2_pvalue(lvl1["out_tokens"][:, 0], _probs(q_log)[0]) > 1e-3
    assert _chi2_pvalue(lvl2["out_tokens"][:, 0], _probs(p_log)[0]) > 1e-3


def test_quadrature_exact_case():
    """p0 = (1/2, 1/4, 1/8, 1/8), q0 uniform: ratios (2, 1, 1/2, 1/2) and residual
    (1/4, 0, 0, 0).  On a midpoint grid of uniforms the emitted-token mass is
    exactly p0, enumerating every draft token with weight q0(x)."""
    p0 = np.array([0.5, 0.25, 0.125, 0.125])
    q0 = np.full(4, 0.25)
    tgt = np.log(np.stack([p0, p0]))
    drf = np.log(q0)[None]
    n = 200
    grid = (np.arange(n) + 0.5) / n
    X, UA, UR = np.meshgrid(np.arange(4), grid, grid, indexing="ij")
    r = O.spec_accept(tgt[None], drf[None], X.reshape(-1, 1), UA.reshape(-1, 1), UR.reshape(-1))
    w = q0[X.reshape(-1)] / (n * n)
    mass = np.bincount(r["out_tokens"][:, 0], weights=w, minlength=4)
    np.testing.assert_allclose(mass, p0, rtol=0, atol=1e-12)


def test_quadrature_random_case():
    rng = np.random.default_rng(5)
    V = 5
    tgt = rng.standard_normal((2, V)) * 2
    drf = rng.standard_normal((1, V)) * 2
    n = 500
    grid = (np.arange(n) + 0.5) / n
    X, UA, UR = np.meshgrid(np.arange(V), grid, grid, indexing="ij")
    r = O.spec_accept(tgt[None], drf[None], X.reshape(-1, 1), UA.reshape(-1, 1), UR.reshape(-1))
    w = _probs(drf)[0][X.reshape(-1)] / (n * n)
    mass = np.bincount(r["out_tokens"][:, 0], weights=w, minlength=V)
    # Midpoint-grid error: at most one grid cell per decision boundary.
    np.testing.assert_allclose(mass, _probs(tgt)[0], rtol=0, atol=2.0 * V / n)


def test_identical_distributions_accept_everything():
    rng, tgt, _ = _lossless_setup(2, 32, 4)
    N = 2000
    x = _draw(rng, _probs(tgt[:4]), N)
    r = O.spec_accept(tgt[None], tgt[None, :4], x, rng.random((N, 4)), rng.random(N))
    assert np.all(r["n_acc"] == 4)
    assert np.array_equal(r["out_tokens"][:, :4], x)


def test_point_mass_draft_where_target_is_zero():
    V, N = 8, 200_000
    rng = np.random.default_rng(3)
    tgt = rng.standard_normal((2, V))
    tgt[0, 3] = -1e4  # p0(3) = 0 (underflows even in float64)
    drf = np.full((1, V), -1e4)
    drf[0, 3] = 0.0  # q0 is a point mass on token 3
    r = O.spec_accept(tgt[None], drf[None], np.full((N, 1), 3), rng.random((N, 1)), rng.random(N))
    assert np.all(r["n_acc"] == 0)
    assert _chi2_pvalue(r["next"], _probs(tgt)[0]) > 1e-3


def test_empty_draft_samples_target_row_zero():
    tgt = np.log(np.array([[0.5, 0.5], [0.1, 0.9]]))
    r = O.spec_accept(tgt[None], np.zeros((1, 1, 2)), np.array([[-1], [-1]]), np.zeros((2, 1)), np.array([0.2, 0.7]))
    assert r["n_acc"].tolist() == [0, 0]
    assert r["next"].tolist() == [0, 1]


@pytest.mark.parametrize("temperature", [0.5, 2.0])
def test_temperature_is_a_logit_rescale(temperature):
    rng, tgt, drf = _lossless_setup(4, 16, 3)
    N = 5000
    x = _draw(rng, _probs(drf / temperature), N)
    ua, ur = rng.random((N, 3)), rng.random(N)
    a = O.spec_accept(tgt[None], drf[None], x, ua, ur, temperature=temperature)
    b = O.spec_accept(tgt[None] / temperature, drf[None] / temperature, x, ua, ur, temperature=1.0)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])


def test_inverse_cdf_strict_boundary():
    w = np.array([[1.0, 2.0, 3.0, 4.0]])
    for u, t in [(0.0, 0), (0.05, 0), (0.1, 1), (0.29, 1), (0.3, 2), (0.6, 3), (0.999, 3)]:
        got, _ = O.inverse_cdf(w, np.array([u]))
        assert int(got[0]) == t, (u, t)
