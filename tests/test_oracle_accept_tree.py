"""Pins for the oracle's tree form of accept / resample (no GPU).

"TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
TriForce" (a candidate tree verified in one pass) and "Dual Rejection
Sampling: Mathematical Losslessness" (the per-candidate test and residual).
Reading: siblings drawn independently from their parent's drafter
distribution are tested one at a time with the printed rule, each rejection
turning the target into the normalised residual.

Pins: the losslessness property (chi-square on a 16-token vocabulary with 10^6
trials for two- and three-way branching, and for the second token of a
two-level tree given the first level kept a candidate), exact quadrature over
every draw of a two-sibling tree, a hand-worked fixture, the chain as the
special case that reproduces the chain call decision for decision, and the
degenerate cases.
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


def _chi2_pvalue(tokens, p):
    counts = np.bincount(tokens, minlength=len(p))
    nz = p > 0
    assert counts[~nz].sum() == 0
    return stats.chisquare(counts[nz], p[nz] / p[nz].sum() * counts.sum()).pvalue


def test_golden_hand_cases():
    with open(os.path.join(GOLDEN, "spec_accept_tree_hand.json")) as f:
        fx = json.load(f)
    tgt, drf = np.array(fx["tgt_logits"])[None], np.array(fx["drf_logits"])[None]
    for case in fx["cases"]:
        parent = np.array([case.get("parent", fx["parent"])])
        r = O.spec_accept_tree(tgt, drf, np.array([case["x"]]), parent, np.array([case["u_acc"]]),
                               np.array([case["u_res"]]))
        assert int(r["n_acc"][0]) == case["n_acc"], case["name"]
        assert int(r["next"][0]) == case["next"], case["name"]
        assert r["out_tokens"][0].tolist() == case["out_tokens"], case["name"]
        assert r["acc_nodes"][0].tolist() == case["acc_nodes"], case["name"]


def test_chain_reproduces_the_chain_call():
    """parent[j] = j - 1: the same decisions, tokens and margins as spec_accept,
    with drafts cut short by tokens outside the vocabulary."""
    rng = np.random.default_rng(11)
    B, T, V = 3000, 6, 40
    tgt = rng.standard_normal((B, T + 1, V)) * 2.0
    drf = tgt[:, :T] + rng.standard_normal((B, T, V))
    q = _probs(drf)
    x = np.stack([[rng.choice(V, p=q[b, i]) for i in range(T)] for b in range(B)])
    x[::7, 3] = -1
    x[::11, 0] = V
    ua, ur = rng.random((B, T)), rng.random(B)
    chain = np.tile(np.arange(T) - 1, (B, 1))
    a = O.spec_accept(tgt, drf, x, ua, ur)
    b = O.spec_accept_tree(tgt, drf, x, chain, ua, ur)
    for k in ("n_acc", "next", "out_tokens"):
        assert np.array_equal(a[k], b[k]), k
    np.testing.assert_allclose(a["margin"], b["margin"], rtol=0, atol=1e-12)  # the residual is normalised first
    kept = np.arange(T)[None, :] < a["n_acc"][:, None]
    assert np.array_equal(b["acc_nodes"], np.where(kept, np.arange(T)[None, :], -1))


def _siblings_setup(seed, V, k):
    rng = np.random.default_rng(seed)
    tgt = rng.standard_normal((k + 1, V)) * 2.0  # row 0 the prefix, rows 1..k after each sibling
    q_root = tgt[0] + rng.standard_normal(V)
    drf = np.tile(q_root, (k, 1))  # every sibling drawn from the root's drafter distribution
    return rng, tgt, drf


@pytest.mark.parametrize("k", [2, 3])
def test_branching_root_is_lossless_chi_square(k):
    N, V = 1_000_000, 16
    rng, tgt, drf = _siblings_setup(20 + k, V, k)
    q = _probs(drf[0])
    x = rng.choice(V, size=(N, k), p=q)
    parent = np.full((1, k), -1)
    r = O.spec_accept_tree(tgt[None], drf[None], x, np.broadcast_to(parent, (N, k)), rng.random((N, k)),
                           rng.random(N))
    assert _chi2_pvalue(r["out_tokens"][:, 0], _probs(tgt[0])) > 1e-3
    # Kept sibling j emits its bonus token from the verifier row after it.
    for j in range(k):
        m = r["acc_nodes"][:, 0] == j
        assert m.sum() > 1000
        assert _chi2_pvalue(r["out_tokens"][m, 1], _probs(tgt[1 + j])) > 1e-3


def test_two_level_tree_second_token_chi_square():
    """Root -> candidates 0, 1; candidate 0 -> 2, 3; candidate 1 -> 4, 5 (all
    siblings drawn from their parent's drafter row).  The first emitted token
    follows the prefix row; given candidate c was kept first, the second
    emitted token follows the verifier row after c."""
    N, V = 1_000_000, 16
    rng = np.random.default_rng(7)
    tgt = rng.standard_normal((7, V)) * 2.0
    q_root = tgt[0] + rng.standard_normal(V)
    q_after = [tgt[1 + c] + rng.standard_normal(V) for c in (0, 1)]
    drf = np.stack([q_root, q_root, q_after[0], q_after[0], q_after[1], q_after[1]])
    parent = np.array([-1, -1, 0, 0, 1, 1])
    qs = _probs(drf)
    x = np.stack([rng.choice(V, size=N, p=qs[j]) for j in range(6)], axis=1)
    r = O.spec_accept_tree(tgt[None], drf[None], x, np.broadcast_to(parent, (N, 6)), rng.random((N, 6)),
                           rng.random(N))
    assert _chi2_pvalue(r["out_tokens"][:, 0], _probs(tgt[0])) > 1e-3
    for c in (0, 1):
        m = r["acc_nodes"][:, 0] == c
        assert _chi2_pvalue(r["out_tokens"][m, 1], _probs(tgt[1 + c])) > 1e-3
    assert r["n_acc"].max() == 2 and set(np.unique(r["acc_nodes"][:, 1])) <= {-1, 2, 3, 4, 5}


def test_quadrature_two_siblings_exact():
    """p0 = (1/2, 1/4, 1/8, 1/8), q0 uniform, two siblings from q0: enumerate
    both tokens with weight q0(a) q0(b) and every uniform on a midpoint grid
    that no decision boundary crosses; the emitted-token mass is p0 exactly."""
    p0 = np.array([0.5, 0.25, 0.125, 0.125])
    q0 = np.full(4, 0.25)
    tgt = np.log(np.stack([p0, p0, p0]))
    drf = np.log(np.stack([q0, q0]))
    n = 40
    grid = (np.arange(n) + 0.5) / n
    A, Bt, U1, U2, UR = np.meshgrid(np.arange(4), np.arange(4), grid, grid, grid, indexing="ij")
    N = A.size
    x = np.stack([A.reshape(-1), Bt.reshape(-1)], axis=1)
    r = O.spec_accept_tree(tgt[None], drf[None], x, np.broadcast_to([-1, -1], (N, 2)),
                           np.stack([U1.reshape(-1), U2.reshape(-1)], axis=1), UR.reshape(-1))
    w = q0[A.reshape(-1)] * q0[Bt.reshape(-1)] / n ** 3
    mass = np.bincount(r["out_tokens"][:, 0], weights=w, minlength=4)
    np.testing.assert_allclose(mass, p0, rtol=0, atol=1e-10)  # a 10^6-term float sum


def test_quadrature_three_siblings_random():
    rng = np.random.default_rng(9)
    V, k, n = 4, 3, 16
    tgt = rng.standard_normal((k + 1, V)) * 2
    qr = rng.standard_normal(V) * 2
    drf = np.tile(qr, (k, 1))
    q = _probs(qr)
    grid = (np.arange(n) + 0.5) / n
    axes = np.meshgrid(*([np.arange(V)] * k + [grid] * (k + 1)), indexing="ij")
    flat = [a.reshape(-1) for a in axes]
    N = flat[0].size
    x = np.stack(flat[:k], axis=1)
    r = O.spec_accept_tree(tgt[None], drf[None], x, np.broadcast_to([-1] * k, (N, k)), np.stack(flat[k:2 * k], 1),
                           flat[2 * k])
    w = np.prod([q[f] for f in flat[:k]], axis=0) / n ** (k + 1)
    mass = np.bincount(r["out_tokens"][:, 0], weights=w, minlength=V)
    # Midpoint-grid error: at most one grid cell per decision boundary crossed.
    np.testing.assert_allclose(mass, _probs(tgt[0]), rtol=0, atol=(2 * k + 2) * V / n * 0.5)


def test_identical_distributions_keep_the_first_sibling():
    rng = np.random.default_rng(3)
    V, N = 20, 5000
    tgt = rng.standard_normal((4, V))
    drf = np.tile(tgt[0], (3, 1))
    x = rng.choice(V, size=(N, 3), p=_probs(tgt[0]))
    r = O.spec_accept_tree(tgt[None], drf[None], x, np.broadcast_to([-1, -1, -1], (N, 3)), rng.random((N, 3)),
                           rng.random(N))
    assert np.all(r["acc_nodes"][:, 0] == 0) and np.all(r["n_acc"] == 1)
    assert np.array_equal(r["out_tokens"][:, 0], x[:, 0])


def test_no_candidates_and_all_invalid_draw_from_the_prefix_row():
    tgt = np.log(np.array([[0.5, 0.5], [0.1, 0.9], [0.1, 0.9]]))
    drf = np.zeros((2, 2))
    for x in (np.array([[-1, -1], [-1, -1]]), np.array([[2, -5], [2, 7]])):
        r = O.spec_accept_tree(tgt[None], drf[None], x, np.array([[-1, 0], [-1, -1]]), np.zeros((2, 2)),
                               np.array([0.2, 0.7]))
        assert r["n_acc"].tolist() == [0, 0] and r["next"].tolist() == [0, 1]
    r = O.spec_accept_tree(tgt[None, :1], np.zeros((1, 0, 2)), np.zeros((2, 0), dtype=int),
                           np.zeros((2, 0), dtype=int), np.zeros((2, 0)), np.array([0.2, 0.7]))
    assert r["n_acc"].tolist() == [0, 0] and r["next"].tolist() == [0, 1]
