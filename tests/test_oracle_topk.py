"""Pins for the oracle's chunk scoring and top-k selection (no GPU).

Force 2 keeps the KV blocks with the highest key-query similarity ("TriForce:
Hierarchical Speculative Decoding for LLMs", "The Three Forces of TriForce").
The pins: a rank-count brute force of the selection rule, a hand-worked score
fixture, the GQA-sum invariant, and recovery of planted relevant chunks.
"""

import json
import os

import numpy as np
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _brute_topk(s, kc):
    """Chunk c is selected iff fewer than kc chunks beat it, where d beats c when
    s[d] > s[c], or s[d] == s[c] and d < c (ties to the lower id)."""
    C = len(s)
    sel = []
    for c in range(C):
        beaten_by = sum(1 for d in range(C) if s[d] > s[c] or (s[d] == s[c] and d < c))
        if beaten_by < kc:
            sel.append(c)
    return sel


def test_topk_matches_rank_count_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(300):
        C = int(rng.integers(0, 40))
        kc = int(rng.integers(1, 20))
        s = rng.integers(-4, 5, size=C).astype(np.float64)  # many exact ties
        if trial % 3 == 0:
            s = rng.standard_normal(C)
        ids, cut, gap = O.topk_chunks(s, kc)
        assert ids.tolist() == _brute_topk(s.tolist(), kc)
        if C > kc:
            assert cut == min(s[i] for i in ids)
            rest = [s[i] for i in range(C) if i not in set(ids.tolist())]
            assert gap == cut - max(rest)


def test_scores_golden_fixture():
    with open(os.path.join(GOLDEN, "chunk_scores_small.json")) as f:
        fx = json.load(f)
    q = torch.tensor(fx["q"], dtype=torch.bfloat16)  # [B, Hq, D]
    M = torch.tensor(fx["M"], dtype=torch.bfloat16)  # [B, Hkv, C, D]
    chunk = fx["chunk"]
    seq_lens = np.array(fx["seq_lens"])
    Lmax = M.shape[2] * chunk
    idx, n_sel, s_cut, gap, scores = O.chunk_scores_topk(
        _bits(q), _bits(M), seq_lens, Lmax, chunk, fx["kc"], M.shape[1])
    assert [s.tolist() for s in scores[0]] == fx["scores"][0]
    assert idx[0].tolist() == fx["idx"][0]
    assert n_sel[0].tolist() == fx["n_sel"][0]


def test_gqa_score_is_sum_of_member_head_scores():
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, D, C, chunk = 2, 8, 2, 16, 10, 8
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    M = torch.randn((B, Hkv, C, D), generator=g).to(torch.bfloat16)
    seq_lens = np.array([C * chunk, C * chunk - 5])
    gqa = O.chunk_scores(_bits(q), _bits(M), seq_lens, C * chunk, chunk, Hkv)
    # Same problem as MHA: every query head gets its own copy of its group's means.
    M_rep = M.repeat_interleave(Hq // Hkv, dim=1)
    mha = O.chunk_scores(_bits(q), _bits(M_rep), seq_lens, C * chunk, chunk, Hq)
    for b in range(B):
        summed = mha[b].reshape(Hkv, Hq // Hkv, -1).sum(axis=1)
        np.testing.assert_allclose(gqa[b], summed, rtol=1e-12, atol=1e-12)


def test_partial_last_chunk_is_a_candidate():
    s_len = 8 * 5 + 3  # five full chunks and one partial chunk
    q = torch.ones((1, 1, 4), dtype=torch.bfloat16)
    M = torch.zeros((1, 1, 6, 4), dtype=torch.bfloat16)
    M[0, 0, 5] = 2.0  # only the partial chunk scores high
    idx, n_sel, *_ = O.chunk_scores_topk(_bits(q), _bits(M), np.array([s_len]), 48, 8, 1, 1)
    assert idx[0, 0, 0] == 5 and n_sel[0, 0] == 1


def test_planted_chunks_are_retrieved_tiny_workload():
    w = synth.TINY
    seq = synth.seq_lens_for(w)
    q, _ = synth.decode_queries(w, 0)
    K, V, planted = synth.kv_cache(w, 0, q, seq)
    M = O.build_chunk_means(_bits(K), seq.numpy(), w.chunk)
    idx, n_sel, s_cut, gap, _ = O.chunk_scores_topk(_bits(q), M, seq.numpy(), w.L, w.chunk, w.kc, w.Hkv)
    for h in range(w.Hkv):
        pl = set(planted[0][h].tolist())
        assert 0 < len(pl) <= w.kc
        assert pl <= set(idx[0, h, : n_sel[0, h]].tolist())
        assert n_sel[0, h] == w.kc
