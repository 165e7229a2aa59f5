"""Pins for the oracle's attention over position sets (no GPU).

Covers Force 2's sparse decode attention, Force 1's sink + window attention and
Force 3's full-cache verification ("TriForce: Hierarchical Speculative Decoding
for LLMs", "The Three Forces of TriForce").  Pins: torch's float64 scaled-dot-
product attention as a textbook cross-check, closed forms, a hand-worked
fixture, the split-K merge identity, set-builder statements of the position
sets, and the reductions the method implies (sparse == full when the budget
covers the context, window == full when the context fits the window, verify
row j == decode attention on the truncated cache).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import triforce as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def test_attend_matches_torch_sdpa_float64():
    rng = np.random.default_rng(0)
    for n, m, D in [(1, 1, 8), (3, 17, 16), (6, 300, 128), (24, 77, 128)]:
        q = rng.standard_normal((n, D))
        K = rng.standard_normal((m, D)) * 2
        V = rng.standard_normal((m, D))
        scale = 1 / math.sqrt(D)
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=scale)[0].numpy()
        np.testing.assert_allclose(O.attend(q, K, V, scale), want, rtol=1e-12, atol=1e-12)


def test_attend_golden_fixture():
    with open(os.path.join(GOLDEN, "attention_hand.json")) as f:
        fx = json.load(f)
    got = O.attend(np.array(fx["q"], float), np.array(fx["K"], float), np.array(fx["V"], float), fx["scale"])
    np.testing.assert_allclose(got, np.array(fx["out"]), rtol=1e-14, atol=1e-14)


def test_closed_forms():
    rng = np.random.default_rng(1)
    D = 128
    q = rng.standard_normal((2, D))
    V = rng.standard_normal((9, D))
    # Identical keys: uniform weights, output = mean of V.
    K = np.repeat(rng.standard_normal((1, D)), 9, axis=0)
    np.testing.assert_allclose(O.attend(q, K, V, 0.1), np.repeat(V.mean(0, keepdims=True), 2, 0), atol=1e-12)
    # A single key: output = its value row.
    np.testing.assert_allclose(O.attend(q, K[:1], V[:1], 0.1), np.repeat(V[:1], 2, 0), atol=1e-14)
    # One key dominating by a wide margin: output = that value row.
    K2 = rng.standard_normal((9, D)) * 0.01
    K2[4] = q[0] * 100
    np.testing.assert_allclose(O.attend(q[:1], K2, V, 1.0), V[4:5], atol=1e-12)
    # Empty key set: zeros.
    assert np.all(O.attend(q, K[:0], V[:0], 1.0) == 0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_merge_identity(seed):
    rng = np.random.default_rng(seed)
    n, m, D = 6, 257, 128
    q = rng.standard_normal((n, D))
    K = rng.standard_normal((m, D))
    V = rng.standard_normal((m, D))
    full = O.attend(q, K, V, 0.09)
    for nsplit in [1, 2, 5, 64]:
        cuts = np.sort(rng.choice(np.arange(1, m), size=nsplit - 1, replace=False)) if nsplit > 1 else []
        bounds = [0, *cuts, m]
        parts = [O.attend_partial(q, K[a:b], V[a:b], 0.09) for a, b in zip(bounds[:-1], bounds[1:])]
        parts.append(O.attend_partial(q, K[:0], V[:0], 0.09))  # an empty split changes nothing
        np.testing.assert_allclose(O.merge_partials(parts), full, rtol=1e-12, atol=1e-12)


def test_position_sets_against_set_builder():
    for L in [0, 1, 3, 4, 5, 100, 255, 256, 257, 300, 4096]:
        for ns, W in [(4, 252), (0, 8), (4, 0), (8, 3)]:
            want = sorted({t for t in range(L) if t < ns or t >= L - W})
            assert O.window_positions(L, ns, W).tolist() == want
        for T in [1, 5, 6]:
            for j in range(T):
                assert O.verify_positions(L, T, j).tolist() == [t for t in range(L) if t <= L - T + j]
    idx = np.array([3, 0, 7, -1, 99])
    for L in [0, 5, 20, 31, 64]:
        want = [t for c in [3, 0, 7] if c < -(-L // 4) for t in range(4 * c, 4 * c + 4) if t < L]
        assert O.sparse_positions(idx, 5, L, 4, 64).tolist() == want


def test_sparse_equals_full_when_budget_covers_context():
    B, Hq, Hkv, L, D, chunk = 2, 4, 2, 61, 128, 8
    q = _rand_bf16((B, Hq, D), 1)
    K = _rand_bf16((B, Hkv, L, D), 2)
    V = _rand_bf16((B, Hkv, L, D), 3)
    seq = np.array([61, 40])
    M = O.build_chunk_means(_bits(K), seq, chunk)
    kc = 8  # 8 chunks x 8 tokens >= 61
    idx, n_sel, *_ = O.chunk_scores_topk(_bits(q), M, seq, L, chunk, kc, Hkv)
    sp = O.sparse_decode_attn(_bits(q), _bits(K), _bits(V), seq, idx, n_sel, chunk, 0.088)
    # Full decode attention = verification with a single query token.
    full = O.verify_attn(_bits(q)[:, :, None, :], _bits(K), _bits(V), seq, 0.088)[:, :, 0]
    np.testing.assert_allclose(sp, full, rtol=1e-12, atol=1e-12)


def test_window_equals_full_when_context_fits():
    B, Hq, Hkv, L, D = 1, 2, 1, 200, 128
    q = _rand_bf16((B, Hq, D), 4)
    K = _rand_bf16((B, Hkv, L, D), 5)
    V = _rand_bf16((B, Hkv, L, D), 6)
    for Lb in [1, 100, 200]:
        seq = np.array([Lb])
        win = O.stream_window_attn(_bits(q), _bits(K), _bits(V), seq, 4, 252, 0.088)
        full = O.verify_attn(_bits(q)[:, :, None, :], _bits(K), _bits(V), seq, 0.088)[:, :, 0]
        np.testing.assert_allclose(win, full, rtol=1e-12, atol=1e-12)


def test_verify_row_equals_decode_on_truncated_cache():
    B, Hq, Hkv, L, D, T = 1, 4, 2, 90, 128, 5
    Q = _rand_bf16((B, Hq, T, D), 7)
    K = _rand_bf16((B, Hkv, L, D), 8)
    V = _rand_bf16((B, Hkv, L, D), 9)
    out = O.verify_attn(_bits(Q), _bits(K), _bits(V), np.array([L]), 0.088)
    for j in range(T):
        Lj = L - T + 1 + j
        dec = O.verify_attn(_bits(Q)[:, :, j : j + 1], _bits(K), _bits(V), np.array([Lj]), 0.088)[:, :, 0]
        np.testing.assert_allclose(out[:, :, j], dec, rtol=1e-12, atol=1e-12)
    # Rows with no visible key (context shorter than the candidate count) are zero.
    short = O.verify_attn(_bits(Q), _bits(K), _bits(V), np.array([2]), 0.088)
    assert np.all(short[:, :, :2] == 0) and np.all(np.isfinite(short))


def test_positions_beyond_length_are_never_read():
    B, Hq, Hkv, L, D = 1, 2, 2, 48, 128
    q = _rand_bf16((B, Hq, D), 10)
    K = _rand_bf16((B, Hkv, L, D), 11)
    V = _rand_bf16((B, Hkv, L, D), 12)
    K[:, :, 37:] = float("nan")
    V[:, :, 37:] = float("nan")
    seq = np.array([37])
    M = O.build_chunk_means(_bits(K), seq, 8)
    idx, n_sel, *_ = O.chunk_scores_topk(_bits(q), M, seq, L, 8, 6, Hkv)
    assert np.all(np.isfinite(O.bf16_to_f64(M)[:, :, :5]))
    assert np.all(np.isfinite(O.sparse_decode_attn(_bits(q), _bits(K), _bits(V), seq, idx, n_sel, 8, 0.1)))
    assert np.all(np.isfinite(O.stream_window_attn(_bits(q), _bits(K), _bits(V), seq, 4, 16, 0.1)))
    Q = _rand_bf16((B, Hq, 3, D), 13)
    assert np.all(np.isfinite(O.verify_attn(_bits(Q), _bits(K), _bits(V), seq, 0.1)))


# ---------------------------------------------------------------- level-1 verification over the retrieval cache


def _compacted_verify(Q, K, V, b, g, rows_pre, L, T, scale):
    """Verification over a cache rebuilt as [retrieved prefix rows, the T candidate
    rows]: query j then sees the prefix and candidates 0..j by verify_positions."""
    cand = list(range(max(L - T, 0), L))
    keep = list(rows_pre) + cand
    Kc = K[b : b + 1, g : g + 1, keep]
    Vc = V[b : b + 1, g : g + 1, keep]
    return O.verify_attn(_bits(Q[b : b + 1]), _bits(Kc), _bits(Vc), np.array([len(keep)]), scale)[0]


def test_sparse_verify_equals_verify_when_every_prefix_chunk_is_selected():
    B, Hq, Hkv, L, D, T, chunk = 2, 4, 2, 77, 128, 5, 8
    Q = _rand_bf16((B, Hq, T, D), 31)
    K = _rand_bf16((B, Hkv, L, D), 32)
    V = _rand_bf16((B, Hkv, L, D), 33)
    seq = np.array([77, 50])
    kc = 10
    idx = np.full((B, Hkv, kc), -1)
    n_sel = np.zeros((B, Hkv), dtype=np.int64)
    for b in range(B):
        C = -(-seq[b] // chunk)
        for g in range(Hkv):
            ids = np.random.default_rng(b * 7 + g).permutation(C)  # any order
            idx[b, g, :C] = ids
            n_sel[b, g] = C
    sv = O.sparse_verify_attn(_bits(Q), _bits(K), _bits(V), seq, idx, n_sel, chunk, 0.088)
    full = O.verify_attn(_bits(Q), _bits(K), _bits(V), seq, 0.088)
    np.testing.assert_allclose(sv, full, rtol=1e-12, atol=1e-12)


def test_sparse_verify_equals_verify_on_the_compacted_cache():
    """A selection with a chunk straddling the candidates, an invalid id and a
    partial last chunk: the result is verification over [retrieved prefix rows,
    candidates] (rows of selected chunks at or past L-T are not counted twice)."""
    B, Hq, Hkv, L, D, T, chunk = 1, 6, 2, 90, 128, 6, 8
    Q = _rand_bf16((B, Hq, T, D), 34)
    K = _rand_bf16((B, Hkv, L, D), 35)
    V = _rand_bf16((B, Hkv, L, D), 36)
    seq = np.array([86])  # candidates at 80..85; chunk 10 holds 80..85 (partial), chunk 9 72..79
    idx = np.array([[[3, 10, 0, 99, 9], [5, -1, 7, 1, 2]]])
    n_sel = np.array([[5, 5]])
    sv = O.sparse_verify_attn(_bits(Q), _bits(K), _bits(V), seq, idx, n_sel, chunk, 0.07)
    for g in range(Hkv):
        rows = []
        for c in idx[0, g]:
            if 0 <= c < -(-seq[0] // chunk):
                rows += [t for t in range(c * chunk, min(c * chunk + chunk, seq[0])) if t < seq[0] - T]
        ref = _compacted_verify(Q[:, g * 3 : (g + 1) * 3], K, V, 0, g, rows, seq[0], T, 0.07)
        np.testing.assert_allclose(sv[0, g * 3 : (g + 1) * 3], ref, rtol=1e-12, atol=1e-12)


def test_sparse_verify_with_an_empty_selection_sees_only_the_candidates():
    B, Hq, Hkv, L, D, T = 1, 2, 1, 40, 128, 4
    Q = _rand_bf16((B, Hq, T, D), 37)
    K = _rand_bf16((B, Hkv, L, D), 38)
    V = _rand_bf16((B, Hkv, L, D), 39)
    seq = np.array([40])
    sv = O.sparse_verify_attn(_bits(Q), _bits(K), _bits(V), seq, np.full((1, 1, 4), -1), np.zeros((1, 1)), 8, 0.1)
    tail = O.verify_attn(_bits(Q), _bits(K[:, :, 36:]), _bits(V[:, :, 36:]), np.array([4]), 0.1)
    np.testing.assert_allclose(sv, tail, rtol=1e-12, atol=1e-12)
    # the first candidate sees only itself: its output is its own V row
    np.testing.assert_allclose(sv[0, :, 0], np.broadcast_to(O.bf16_to_f64(_bits(V))[0, 0, 36], (Hq, D)), rtol=0,
                               atol=0)


# ------------------------------------------------------------------ candidate trees


def test_tree_ancestors_hand_worked():
    # 0 and its children 1, 2; 3 under 1: ancestors-or-self of each candidate
    parent = [-1, 0, 0, 1]
    assert O.tree_ancestors(parent, 0) == [0]
    assert O.tree_ancestors(parent, 1) == [1, 0]
    assert O.tree_ancestors(parent, 2) == [2, 0]
    assert O.tree_ancestors(parent, 3) == [3, 1, 0]
    # a link to itself, to a later candidate or below -1 ends the walk
    bad = [-1, 5, -3, 2, 4]
    assert O.tree_ancestors(bad, 1) == [1]
    assert O.tree_ancestors(bad, 2) == [2]
    assert O.tree_ancestors(bad, 3) == [3, 2]
    assert O.tree_ancestors(bad, 4) == [4]
    # positions: prefix, then the candidates in position order, clipped to [0, L)
    np.testing.assert_array_equal(O.tree_verify_positions(10, 4, 3, parent), [0, 1, 2, 3, 4, 5, 6, 7, 9])
    np.testing.assert_array_equal(O.tree_verify_positions(2, 4, 3, parent), [1])


def _tree_case(B=2, Hq=4, Hkv=2, T=6, L=40, D=32, seed=3):
    Q = _rand_bf16((B, Hq, T, D), seed)
    K = _rand_bf16((B, Hkv, L, D), seed + 1)
    V = _rand_bf16((B, Hkv, L, D), seed + 2)
    return Q, K, V


def test_tree_with_chain_parents_is_the_chain_verify():
    Q, K, V = _tree_case()
    B, T = Q.shape[0], Q.shape[2]
    seq = np.array([40, 23])
    chain = np.tile(np.arange(T) - 1, (B, 1))
    got = O.tree_verify_attn(_bits(Q), _bits(K), _bits(V), seq, chain, 0.2)
    want = O.verify_attn(_bits(Q), _bits(K), _bits(V), seq, 0.2)
    np.testing.assert_array_equal(got, want)


def test_tree_matches_sdpa_with_a_closure_mask():
    # the mask comes from the transitive closure of the parent adjacency
    # matrix, not from walking the parent links
    rng = np.random.default_rng(7)
    Q, K, V = _tree_case(T=7, L=30, seed=11)
    B, Hq, T, D = Q.shape
    Hkv, Lmax = K.shape[1], K.shape[2]
    seq = np.array([30, 12])
    parent = np.stack([np.array([rng.integers(-1, j) if j > 0 else -1 for j in range(T)]) for _ in range(B)])
    got = O.tree_verify_attn(_bits(Q), _bits(K), _bits(V), seq, parent, 0.17)
    Qf, Kf, Vf = (t.to(torch.float64) for t in (Q, K, V))
    for b in range(B):
        L = int(seq[b])
        A = np.eye(T, dtype=np.int64)  # A[j, i] = 1: i is j or an ancestor of j
        for j in range(T):
            if parent[b, j] >= 0:
                A[j, parent[b, j]] = 1
        R = A.copy()
        for _ in range(T):
            R = np.minimum(R @ A, 1)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            mask = np.zeros((T, Lmax), dtype=bool)
            mask[:, : max(L - T, 0)] = True
            for j in range(T):
                for i in range(T):
                    if R[j, i] and 0 <= L - T + i < L:
                        mask[j, L - T + i] = True
            want = torch.nn.functional.scaled_dot_product_attention(
                Qf[b, h][None], Kf[b, g][None], Vf[b, g][None], attn_mask=torch.from_numpy(mask)[None],
                scale=0.17)[0].numpy()
            np.testing.assert_allclose(got[b, h], want, rtol=1e-10, atol=1e-12)


def test_tree_relabelling_permutes_the_outputs():
    # the same tree with its candidates renumbered (parents still earlier):
    # queries, candidate keys and values move together, outputs follow
    Q, K, V = _tree_case(B=1, Hq=2, Hkv=1, T=5, L=20, seed=21)
    T, L = 5, 20
    parent = np.array([[-1, 0, -1, 1, 2]])
    perm = [0, 2, 1, 4, 3]  # new index -> old index; old parents map to earlier new indices
    inv = {old: new for new, old in enumerate(perm)}
    parent2 = np.array([[inv[parent[0, o]] if parent[0, o] >= 0 else -1 for o in perm]])
    assert all(parent2[0, j] < j for j in range(T))
    Q2 = Q[:, :, perm]
    K2, V2 = K.clone(), V.clone()
    K2[:, :, L - T:] = K[:, :, [L - T + o for o in perm]]
    V2[:, :, L - T:] = V[:, :, [L - T + o for o in perm]]
    seq = np.array([L])
    a = O.tree_verify_attn(_bits(Q), _bits(K), _bits(V), seq, parent, 0.3)
    b = O.tree_verify_attn(_bits(Q2), _bits(K2), _bits(V2), seq, parent2, 0.3)
    np.testing.assert_allclose(b, a[:, :, perm], rtol=1e-12, atol=1e-14)
