"""GPU parity of the fused retrieval-drafter call (scores + top-k + sparse
attention in one launch) against the float64 oracle.

The selection must pass the same checks as the top-k call (identical ids
except at oracle cut gaps below 1e-4) and must equal the separate top-k call's
selection exactly (same scores, same rule); the attention output is checked
against the oracle's sparse attention over the selection the call made
(max abs error <= 2e-3) and against the separate sparse-attention call.
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

from test_gpu_parity import ATOL, bits, check_topk, make_case, scale_for, small_workload

pytestmark = pytest.mark.gpu


def run_fused(cuda_lib, w, c, M, kc=None, scale=None):
    kc = kc or w.kc
    scale = scale if scale is not None else scale_for(w.D)
    s_cut = torch.empty((w.B, w.Hkv), dtype=torch.float32, device="cuda")
    idx, nsel, out = cuda_lib.tf_retrieval_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], kc, scale, s_cut=s_cut)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), nsel.cpu().numpy(), s_cut.cpu().numpy(), out.cpu().double().numpy()


def check_against_oracle(cuda_lib, w, c, M_bits, kc=None, scale=None):
    kc = kc or w.kc
    scale = scale if scale is not None else scale_for(w.D)
    seq = c["seq_cpu"].numpy()
    M = torch.from_numpy(M_bits.view(np.int16)).view(torch.bfloat16).cuda()
    idx, nsel, s_cut, out = run_fused(cuda_lib, w, c, M, kc, scale)
    idx_o, nsel_o, cut_o, gap_o, scores_o = O.chunk_scores_topk(bits(c["q_cpu"]), M_bits, seq, w.L, w.chunk, kc,
                                                                w.Hkv)
    check_topk(idx, nsel, idx_o, nsel_o, gap_o, scores_o)
    np.testing.assert_allclose(s_cut, cut_o, rtol=1e-5, atol=1e-4)
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, idx, nsel, w.chunk,
                                scale)
    err = np.abs(out - want).max()
    assert err <= ATOL, err
    # the two-call path on the same inputs: same selection, same attention
    idx2, nsel2 = cuda_lib.tf_chunk_scores_topk(c["q"], M, c["seq"], w.L, kc)
    out2 = cuda_lib.tf_sparse_decode_attn(c["q"], c["K"], c["V"], c["seq"], idx2, nsel2, scale)
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), idx) and np.array_equal(nsel2.cpu().numpy(), nsel)
    assert np.abs(out2.cpu().double().numpy() - out).max() <= ATOL
    return idx, nsel, out


@pytest.mark.parametrize("w", [
    synth.TINY,
    small_workload(),
    small_workload(budget=8 * 2000),
    small_workload(B=1, Hq=8, Hkv=8, L=32768, budget=4096, ragged=False, planted_frac=0.01),
    small_workload(B=2, Hq=8, Hkv=4, L=20000, budget=8 * 2048, L_min=17000),
    small_workload(B=3, Hq=6, Hkv=2, L=5000, budget=8 * 37, L_min=9),
    small_workload(B=1, Hq=2, Hkv=2, L=32768, budget=4096, ragged=False, planted_frac=0.01),
], ids=["tiny", "ragged-gqa", "budget-covers-all", "mha-32k", "kc-2048", "g3-odd-budget", "two-units-16-ctas"])
def test_retrieval_draft_parity(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan"))
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    idx, nsel, _ = check_against_oracle(cuda_lib, w, c, M_bits)
    for b in range(w.B):
        for g in range(w.Hkv):
            assert set(c["planted"][b][g].tolist()) <= set(idx[b, g, : nsel[b, g]].tolist())


def test_retrieval_draft_empty_and_tiny_contexts(cuda_lib):
    w = small_workload(B=3, ragged=False, L=64)
    c = make_case(w)
    c["seq"] = torch.tensor([0, 1, 64], dtype=torch.int32, device="cuda")
    c["seq_cpu"] = torch.tensor([0, 1, 64], dtype=torch.int32)
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), 8)
    for kc in (4, 8, 100):
        idx, nsel, out = check_against_oracle(cuda_lib, w, c, M_bits, kc=kc)
        assert nsel[0].tolist() == [0, 0] and np.all(out[0] == 0)


def test_retrieval_draft_all_equal_scores(cuda_lib):
    """6000 equal scores per unit: more threshold-bin keys than the on-chip
    candidate buffer holds, so the cut is resolved bin by bin; ties go to the
    lowest ids and the attention covers exactly chunks 0..511."""
    w = small_workload(B=1, ragged=False, L=8 * 6000)
    c = make_case(w)
    M_bits = np.zeros((1, w.Hkv, 6000, 128), dtype=np.uint16)
    idx, nsel, out = check_against_oracle(cuda_lib, w, c, M_bits, kc=512)
    for g in range(w.Hkv):
        assert idx[0, g].tolist() == list(range(512)) and nsel[0, g] == 512


def test_retrieval_draft_repeated_calls_agree(cuda_lib):
    """No state survives a call: the same inputs give the same selection
    (bit-identical) and the same attention up to the summation order, which
    follows the order in which chunks reach the consumer warps."""
    w = small_workload(B=2, Hq=8, Hkv=2, L=30000, budget=4096, L_min=20000)
    c = make_case(w)
    Cmax = -(-w.L // w.chunk)
    M = torch.empty((w.B, w.Hkv, Cmax, w.D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq"], M)
    a = run_fused(cuda_lib, w, c, M)
    b = run_fused(cuda_lib, w, c, M)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)
    np.testing.assert_allclose(a[3], b[3], rtol=1e-5, atol=1e-6)


def _level_means(w, C, levels, seed):
    """Means that are zero except dimension 0, set to level / 8 (exact in bf16):
    every score is q_sum[0] * level / 8 exactly, in fp32 and in float64, so
    equal levels are exact ties on both sides."""
    M = np.zeros((w.B, w.Hkv, C, 128), dtype=np.float32)
    M[..., 0] = levels / 8.0
    return (M.view(np.uint32) >> 16).astype(np.uint16)


def _exact_topk(scores_bg, kc):
    order = np.lexsort((np.arange(len(scores_bg)), -scores_bg))  # score descending, then lower id
    return np.sort(order[:kc])


def test_retrieval_draft_exact_ties_at_the_cut(cuda_lib):
    """Scores on 64 levels (about 256 chunks each): the cut falls inside a
    level with hundreds of exact ties spread over the CTAs of the cluster,
    which must go to the lower chunk ids."""
    C = 16384
    w = small_workload(B=1, Hq=2, Hkv=2, L=8 * C, ragged=False)
    c = make_case(w)
    rng = np.random.default_rng(4)
    M_bits = _level_means(w, C, rng.integers(0, 64, (w.B, w.Hkv, C)).astype(np.float32), 4)
    idx, nsel, out = check_against_oracle(cuda_lib, w, c, M_bits, kc=512)
    scores = O.chunk_scores(bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, 8, w.Hkv)
    for g in range(w.Hkv):
        assert np.array_equal(idx[0, g, :512], _exact_topk(scores[0][g], 512)), g


def test_retrieval_draft_top_chunks_fill_the_budget(cuda_lib):
    """Exactly kc chunks share the top score and the rest score far lower:
    the tied top level is the whole selection and s_cut its score."""
    C, kc = 16384, 512
    w = small_workload(B=1, Hq=2, Hkv=2, L=8 * C, ragged=False)
    c = make_case(w)
    rng = np.random.default_rng(6)
    q0 = bits(c["q_cpu"])  # make q_sum[0] > 0 so the high level scores highest
    levels = rng.integers(0, 40, (w.B, w.Hkv, C)).astype(np.float32)
    top = np.stack([rng.choice(C, kc, replace=False) for _ in range(w.Hkv)])
    for g in range(w.Hkv):
        levels[0, g, top[g]] = 100.0
    qs = O.bf16_to_f64(q0).reshape(w.B, w.Hkv, -1, 128).sum(axis=2)[..., 0]
    levels = np.where(qs[..., None] > 0, levels, -levels)
    M_bits = _level_means(w, C, levels, 6)
    idx, nsel, out = check_against_oracle(cuda_lib, w, c, M_bits, kc=kc)
    for g in range(w.Hkv):
        assert np.array_equal(idx[0, g], np.sort(top[g]))


def test_retrieval_draft_context_just_above_the_budget(cuda_lib):
    """600 chunks for a budget of 512: nearly every chunk is selected and the
    cut sits near the bottom of the score range."""
    w = small_workload(B=2, Hq=8, Hkv=2, L=8 * 600, budget=4096, ragged=False)
    c = make_case(w, fill_invalid=float("nan"))
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    check_against_oracle(cuda_lib, w, c, M_bits)


def _hinted(cuda_lib, w, c, M, hint, kc):
    s_cut = torch.empty((w.B, w.Hkv), dtype=torch.float32, device="cuda")
    idx, nsel, out = cuda_lib.tf_retrieval_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], kc, scale_for(w.D),
                                                      s_cut=s_cut, cut_hint=hint)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), nsel.cpu().numpy(), s_cut.cpu().numpy(), out.cpu().double().numpy()


def _hints(scores, s_cut, kc):
    """Per-unit bounds of every kind: below the cut with kc + 40 keys above it
    (or with as many as fit 2048), at the cut, one ulp above it, so far below
    that more than 4096 keys reach it (or every chunk, when there are fewer),
    and the special values."""
    B, Hkv = s_cut.shape
    below = np.full((B, Hkv), np.nan, np.float32)
    far = np.full((B, Hkv), np.nan, np.float32)
    for b in range(B):
        for g in range(Hkv):
            s = np.sort(np.asarray(scores[b][g], dtype=np.float32))[::-1]
            if len(s) > kc:
                below[b, g] = s[min(kc + 40, 2047, len(s) - 1)]
                far[b, g] = s[min(4200, len(s) - 1)] if len(s) > 4200 else -1e30
    at = s_cut.astype(np.float32)
    above = np.nextafter(at, np.float32(np.inf))
    mixed = np.where((np.arange(B)[:, None] + np.arange(Hkv)[None, :]) % 3 == 0, below,
                     np.where((np.arange(B)[:, None] + np.arange(Hkv)[None, :]) % 3 == 1, above, np.nan))
    return {"below": below, "at": at, "above": above, "far-below": far, "nan": np.full_like(at, np.nan),
            "+inf": np.full_like(at, np.inf), "-inf": np.full_like(at, -np.inf), "mixed": mixed.astype(np.float32)}


@pytest.mark.parametrize("w", [
    small_workload(),
    small_workload(B=1, Hq=8, Hkv=8, L=32768, budget=4096, ragged=False, planted_frac=0.01),
    small_workload(B=2, Hq=8, Hkv=4, L=20000, budget=8 * 2048, L_min=17000),
    small_workload(B=3, Hq=6, Hkv=2, L=5000, budget=8 * 37, L_min=9),
    small_workload(B=1, Hq=2, Hkv=2, L=32768, budget=4096, ragged=False, planted_frac=0.01),
], ids=["ragged-gqa", "mha-32k", "kc-2048", "g3-odd-budget", "two-units-16-ctas"])
def test_retrieval_draft_cut_hint_changes_nothing(cuda_lib, w):
    """A lower bound on the cut changes only the time: with bounds below, at
    and just above the cut, admitting more than 4096 keys, NaN, +-inf and a
    per-unit mix of them, the selection and s_cut equal the unhinted call's
    bit for bit and the attention matches the oracle over that selection."""
    c = make_case(w, fill_invalid=float("nan"))
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    M = torch.from_numpy(M_bits.view(np.int16)).view(torch.bfloat16).cuda()
    idx0, nsel0, cut0, out0 = run_fused(cuda_lib, w, c, M)
    scores = O.chunk_scores(bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, w.chunk, w.Hkv)
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx0,
                                nsel0, w.chunk, scale_for(w.D))
    for name, h in _hints(scores, cut0, w.kc).items():
        idx, nsel, cut, out = _hinted(cuda_lib, w, c, M, torch.from_numpy(h).cuda(), w.kc)
        assert np.array_equal(idx, idx0) and np.array_equal(nsel, nsel0), name
        assert np.array_equal(cut.view(np.uint32), cut0.view(np.uint32)), name
        assert np.abs(out - want).max() <= ATOL, name


def test_retrieval_draft_cut_hint_at_exact_ties(cuda_lib):
    """Scores on 64 levels (hundreds of exact ties per level): a bound equal to
    the cut level admits the whole tied level, and the ties at the cut still go
    to the lower chunk ids."""
    C = 16384
    w = small_workload(B=1, Hq=2, Hkv=2, L=8 * C, ragged=False)
    c = make_case(w)
    rng = np.random.default_rng(4)
    M_bits = _level_means(w, C, rng.integers(0, 64, (w.B, w.Hkv, C)).astype(np.float32), 4)
    M = torch.from_numpy(M_bits.view(np.int16)).view(torch.bfloat16).cuda()
    idx0, nsel0, cut0, out0 = run_fused(cuda_lib, w, c, M, kc=512)
    scores = O.chunk_scores(bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, 8, w.Hkv)
    for h in (cut0, np.nextafter(cut0, np.float32(-np.inf))):
        idx, nsel, cut, out = _hinted(cuda_lib, w, c, M, torch.from_numpy(h.astype(np.float32)).cuda(), 512)
        assert np.array_equal(idx, idx0) and np.array_equal(cut.view(np.uint32), cut0.view(np.uint32))
        for g in range(w.Hkv):
            assert np.array_equal(idx[0, g, :512], _exact_topk(scores[0][g], 512)), g
        assert np.abs(out - out0).max() <= ATOL


def test_retrieval_draft_cut_hint_one_cta_over_its_list(cuda_lib):
    """2500 chunks reach the bound, all in the first slice of the cluster:
    within the 4096 the cluster may gather, but more than one CTA may list,
    so the unhinted path runs; the selection is unchanged."""
    C = 40000
    w = small_workload(B=1, Hq=1, Hkv=1, L=8 * C, ragged=False)
    c = make_case(w)
    levels = np.zeros((1, 1, C), dtype=np.float32)
    levels[0, 0, :2500] = 50.0
    levels[0, 0, 100:400] = 60.0
    qs = O.bf16_to_f64(bits(c["q_cpu"])).reshape(1, 1, -1, 128).sum(axis=2)[..., 0]
    levels = np.where(qs[..., None] > 0, levels, -levels)
    M_bits = _level_means(w, C, levels, 0)
    M = torch.from_numpy(M_bits.view(np.int16)).view(torch.bfloat16).cuda()
    idx0, nsel0, cut0, out0 = run_fused(cuda_lib, w, c, M, kc=512)
    scores = O.chunk_scores(bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, 8, w.Hkv)
    assert np.array_equal(idx0[0, 0, :512], _exact_topk(scores[0][0], 512))
    bound = np.float32(np.sort(np.asarray(scores[0][0], dtype=np.float32))[::-1][2499])
    idx, nsel, cut, out = _hinted(cuda_lib, w, c, M, torch.full((1, 1), float(bound)).cuda(), 512)
    assert np.array_equal(idx, idx0) and np.array_equal(cut.view(np.uint32), cut0.view(np.uint32))
    assert np.abs(out - out0).max() <= ATOL


@pytest.mark.parametrize("w", [
    small_workload(),
    small_workload(B=2, Hq=8, Hkv=4, L=20000, budget=8 * 512, L_min=17000),
    small_workload(B=3, Hq=6, Hkv=2, L=5000, budget=8 * 37, L_min=9),
    small_workload(B=2, Hq=8, Hkv=2, L=600, budget=8 * 100, ragged=False),
], ids=["gqa4-ragged", "g2", "g3-short", "all-selected"])
@pytest.mark.parametrize("hinted", [False, True], ids=["cold", "bounded"])
def test_retrieval_window_draft(cuda_lib, w, hinted):
    """The drafter and the window in one launch: the selection is the plain
    call's bit for bit, the attention over it and the window attention match
    the oracle."""
    c = make_case(w, fill_invalid=float("nan") if w.ragged else None)
    scale = scale_for(w.D)
    M = torch.empty((w.B, w.Hkv, -(-w.L // w.chunk), w.D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq"], M)
    s_cut = torch.empty((w.B, w.Hkv), dtype=torch.float32, device="cuda")
    idx0, nsel0, _ = cuda_lib.tf_retrieval_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], w.kc, scale, s_cut=s_cut)
    hint = (s_cut - 0.3 * s_cut.abs()) if hinted else None
    idx, nsel, out, wout = cuda_lib.tf_retrieval_window_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], w.kc, scale,
                                                                   w.n_sink, w.window, cut_hint=hint)
    torch.cuda.synchronize()
    idx_h, nsel_h = idx.cpu().numpy(), nsel.cpu().numpy()
    assert np.array_equal(idx_h, idx0.cpu().numpy()) and np.array_equal(nsel_h, nsel0.cpu().numpy())
    seq = c["seq_cpu"].numpy()
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, idx_h, nsel_h, w.chunk,
                                scale)
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
    wwant = O.stream_window_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, w.n_sink, w.window,
                                 scale)
    assert np.abs(wout.cpu().double().numpy() - wwant).max() <= ATOL


def test_retrieval_window_draft_short_contexts(cuda_lib):
    """Contexts shorter than a chunk, than the sinks plus the window, and empty."""
    w = small_workload(B=4, Hq=8, Hkv=2, L=700, budget=8 * 16, ragged=False)
    c = make_case(w)
    seq = np.array([3, 0, 50, 700], dtype=np.int32)
    c["seq"] = torch.from_numpy(seq).cuda()
    scale = scale_for(w.D)
    M = torch.empty((w.B, w.Hkv, -(-w.L // w.chunk), w.D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq"], M)
    idx0, nsel0, _ = cuda_lib.tf_retrieval_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], w.kc, scale)
    idx, nsel, out, wout = cuda_lib.tf_retrieval_window_draft_attn(c["q"], M, c["K"], c["V"], c["seq"], w.kc, scale,
                                                                   w.n_sink, w.window)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx0.cpu().numpy()) and np.array_equal(nsel.cpu().numpy(),
                                                                                     nsel0.cpu().numpy())
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, idx.cpu().numpy(),
                                nsel.cpu().numpy(), w.chunk, scale)
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
    wwant = O.stream_window_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, w.n_sink, w.window,
                                 scale)
    assert np.abs(wout.cpu().double().numpy() - wwant).max() <= ATOL
    assert np.all(wout.cpu().numpy()[1] == 0)
