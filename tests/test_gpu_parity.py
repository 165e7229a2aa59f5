"""GPU parity of every library call against the float64 oracle.

Inputs come from the seeded generators (never from the CUDA path); both sides
read the same bf16 bits.  Tolerances:
  * chunk means: bit-exact (the definition rounds once; the kernel sums exactly);
  * top-k ids: identical except where the oracle's score gap at the cut is
    below 1e-4 (counted, and every swapped chunk must sit within 1e-4 of the cut);
  * attention outputs: max abs error <= 2e-3 (bf16 inputs, fp32 accumulation);
  * accept/resample: n_acc / next / out_tokens bit-exact except sequences whose
    uniforms fall within 1e-6 of a decision boundary (counted).
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

pytestmark = pytest.mark.gpu

ATOL = 2e-3
GAP = 1e-4
EDGE = 1e-6


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def scale_for(D):
    return D ** -0.5


def make_case(w, layer=0, fill_invalid=None, device="cuda"):
    seq = synth.seq_lens_for(w)
    q, Q = synth.decode_queries(w, layer)
    K, V, planted = synth.kv_cache(w, layer, q, seq, fill_invalid=fill_invalid)
    return dict(seq_cpu=seq, q_cpu=q, Q_cpu=Q, K_cpu=K, V_cpu=V, planted=planted,
                seq=seq.to(device), q=q.to(device), Q=Q.to(device), K=K.to(device), V=V.to(device))


def small_workload(**kw):
    base = dict(name="small", B=2, Hq=8, Hkv=2, D=128, L=1000, layers=1, chunk=8, budget=256, n_sink=4,
                window=60, T=6, gamma=4, vocab=1000, planted_frac=0.02, seed=21, ragged=True, L_min=200)
    base.update(kw)
    return synth.Workload(**base)


def check_topk(idx_g, nsel_g, idx_o, nsel_o, gap_o, scores_o):
    """Top-k parity: identical sets except at near-ties of the cut."""
    near_ties = 0
    B, Hkv, _ = idx_o.shape
    for b in range(B):
        for g in range(Hkv):
            assert nsel_g[b, g] == nsel_o[b, g]
            n = nsel_o[b, g]
            a = idx_g[b, g, :n]
            assert np.all(np.diff(a) > 0), "ids must be ascending and distinct"
            assert np.all(idx_g[b, g, n:] == -1)
            o = idx_o[b, g, :n]
            if np.array_equal(a, o):
                continue
            assert gap_o[b, g] < GAP, f"top-k mismatch at (b={b}, g={g}) with oracle gap {gap_o[b, g]}"
            s = scores_o[b][g]
            cut = min(s[o])
            for c in set(a.tolist()) ^ set(o.tolist()):
                assert abs(s[c] - cut) < GAP
            near_ties += 1
    return near_ties


# ------------------------------------------------------------------ a1


@pytest.mark.parametrize("w", [synth.TINY, small_workload()], ids=["tiny", "ragged-gqa"])
def test_chunk_means_bit_exact(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan"))
    Cmax = -(-w.L // w.chunk)
    M = torch.full((w.B, w.Hkv, Cmax, w.D), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq"], M)
    want = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    got = bits(M)
    assert np.array_equal(got, want), f"{(got != want).sum()} mismatching means"


def _bf16_bits(x):
    return bits(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def test_chunk_means_rounding_edge_cases(cuda_lib):
    """Chunks whose column sums sit on a bf16 rounding midpoint, a hair off it,
    behind heavy cancellation, so small that a rounding-error bound would
    underflow, so large that it would overflow, or hold +-inf and NaN: the
    exact sum must decide every one of them, bit for bit against the oracle."""
    rng = np.random.default_rng(11)
    C, D = 96, 128
    rows = np.zeros((C, 8, D), dtype=np.float32)
    for c in range(C):
        kind = c % 8
        for d in range(D):
            if kind == 0:    # sum / 8 exactly a midpoint: 1 + 2^-8 (tie, to even) or 1 + 3 * 2^-8
                v = [1.0] * 7 + [1.0 + (2 ** -5 if d % 2 else 3 * 2 ** -5)]
            elif kind == 1:  # sum 8 + 2^-5 + e: the midpoint 1 + 2^-8 plus or minus e / 8
                e = float(rng.choice([-1, 1])) * 2.0 ** -int(rng.integers(10, 24))
                v = [1.0] * 5 + [1.0 + 2 ** -5, 2.0, e]
            elif kind == 2:  # heavy cancellation around a small remainder
                big = float(2 ** int(rng.integers(4, 12)))
                v = [big, -big, big, -big] + list(rng.normal(0, 1e-3, 4))
            elif kind == 3:  # tiny: subnormal means, bounds below the normal range
                v = list(rng.normal(0, 1e-38, 8))
            elif kind == 4:  # huge: near the top of the range
                v = list(rng.normal(0, 1e37, 8))
            elif kind == 5:  # infinities and NaN
                v = list(rng.normal(0, 1, 8))
                v[d % 8] = [np.inf, -np.inf, np.nan][d % 3]
            elif kind == 6:  # exact zeros and signed zeros
                v = [0.0, -0.0] * 4
            else:            # ordinary values with widely spread exponents
                v = list(rng.normal(0, 1, 8) * 2.0 ** rng.integers(-30, 30, 8))
            rows[c, :, d] = np.asarray(v, dtype=np.float32)
    Kb = _bf16_bits(rows.reshape(1, 1, C * 8, D))
    K = torch.from_numpy(Kb.view(np.int16)).view(torch.bfloat16).cuda()
    seq = torch.tensor([C * 8], dtype=torch.int32)
    M = torch.full((1, 1, C, D), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(K, seq.cuda(), M)
    want = O.build_chunk_means(Kb, seq.numpy(), 8)
    got = bits(M)
    bad = np.argwhere(got[0, 0] != want[0, 0])
    detail = [(int(c % 8), int(c), int(d), hex(got[0, 0, c, d]), hex(want[0, 0, c, d])) for c, d in bad[:8]]
    assert len(bad) == 0, f"{len(bad)} mismatching means (kind, chunk, dim, got, want): {detail}"


def test_chunk_means_subrange_only(cuda_lib):
    w = small_workload(ragged=False, B=1)
    c = make_case(w)
    Cmax = -(-w.L // w.chunk)
    M = torch.full((w.B, w.Hkv, Cmax, w.D), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq"], M, c_begin=10, c_end=37)
    got = bits(M)
    want = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk, 10, 37)
    assert np.array_equal(got[:, :, 10:37], want[:, :, 10:37])
    seven = bits(torch.tensor([7.0], dtype=torch.bfloat16))[0]
    assert np.all(got[:, :, :10] == seven) and np.all(got[:, :, 37:] == seven)


# ------------------------------------------------------------------ a2 + a3


def run_topk(cuda_lib, w, c, M_bits, kc=None):
    kc = kc or w.kc
    M = torch.from_numpy(M_bits.view(np.int16)).view(torch.bfloat16).cuda()
    s_cut = torch.empty((w.B, w.Hkv), dtype=torch.float32, device="cuda")
    idx, n_sel = cuda_lib.tf_chunk_scores_topk(c["q"], M, c["seq"], w.L, kc, s_cut=s_cut)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), n_sel.cpu().numpy(), s_cut.cpu().numpy()


@pytest.mark.parametrize("w", [synth.TINY, small_workload(), small_workload(budget=8 * 2000)],
                         ids=["tiny", "ragged-gqa", "budget-covers-all"])
def test_scores_topk(cuda_lib, w):
    c = make_case(w)
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    idx, nsel, s_cut = run_topk(cuda_lib, w, c, M_bits)
    idx_o, nsel_o, cut_o, gap_o, scores_o = O.chunk_scores_topk(
        bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, w.chunk, w.kc, w.Hkv)
    check_topk(idx, nsel, idx_o, nsel_o, gap_o, scores_o)
    np.testing.assert_allclose(s_cut, cut_o, rtol=1e-5, atol=1e-4)
    # planted relevant chunks are all retrieved
    for b in range(w.B):
        for g in range(w.Hkv):
            assert set(c["planted"][b][g].tolist()) <= set(idx[b, g, : nsel[b, g]].tolist())


def test_topk_ties_go_to_lower_ids(cuda_lib):
    w = small_workload(B=1, ragged=False, L=8 * 3000)
    c = make_case(w)
    Cmax = w.L // 8
    M_bits = np.zeros((1, w.Hkv, Cmax, 128), dtype=np.uint16)  # every score is exactly 0
    qsum = c["q_cpu"].double().reshape(w.Hkv, w.G, 128).sum(1)[1]
    winner = torch.where(qsum >= 0, 1.0, -1.0).to(torch.bfloat16)  # a strictly positive score
    M_bits[0, 1, 2999] = bits(winner)
    idx, nsel, _ = run_topk(cuda_lib, w, c, M_bits, kc=100)
    assert idx[0, 0].tolist() == list(range(100))
    assert idx[0, 1].tolist() == list(range(99)) + [2999]


def test_topk_all_equal_scores_many_chunks(cuda_lib):
    """6000 equal scores per unit: the threshold bin holds more keys than the
    on-chip candidate gather takes, so the cluster resolves it bin by bin."""
    w = small_workload(B=1, ragged=False, L=8 * 6000)
    c = make_case(w)
    M_bits = np.zeros((1, w.Hkv, 6000, 128), dtype=np.uint16)
    idx, nsel, s_cut = run_topk(cuda_lib, w, c, M_bits, kc=512)
    for g in range(w.Hkv):
        assert idx[0, g].tolist() == list(range(512))
        assert nsel[0, g] == 512 and s_cut[0, g] == 0.0


def test_topk_empty_and_tiny_contexts(cuda_lib):
    w = small_workload(B=3, ragged=False, L=64)
    c = make_case(w)
    c["seq"] = torch.tensor([0, 1, 64], dtype=torch.int32, device="cuda")
    seq = np.array([0, 1, 64])
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), seq, 8)
    idx, nsel, _ = run_topk(cuda_lib, w, c, M_bits, kc=4)
    idx_o, nsel_o, _, gap_o, scores_o = O.chunk_scores_topk(bits(c["q_cpu"]), M_bits, seq, 64, 8, 4, w.Hkv)
    check_topk(idx, nsel, idx_o, nsel_o, gap_o, scores_o)
    assert nsel[0].tolist() == [0, 0] and nsel[1].tolist() == [1, 1]


# ------------------------------------------------------------------ a4


def oracle_idx(w, c):
    M_bits = O.build_chunk_means(bits(c["K_cpu"]), c["seq_cpu"].numpy(), w.chunk)
    idx_o, nsel_o, *_ = O.chunk_scores_topk(bits(c["q_cpu"]), M_bits, c["seq_cpu"].numpy(), w.L, w.chunk, w.kc,
                                            w.Hkv)
    return idx_o, nsel_o


@pytest.mark.parametrize("w", [synth.TINY, small_workload()], ids=["tiny", "ragged-gqa"])
def test_sparse_decode_attn(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan"))
    idx_o, nsel_o = oracle_idx(w, c)
    idx = torch.from_numpy(idx_o.astype(np.int32)).cuda()
    nsel = torch.from_numpy(nsel_o.astype(np.int32)).cuda()
    out = cuda_lib.tf_sparse_decode_attn(c["q"], c["K"], c["V"], c["seq"], idx, nsel, scale_for(w.D))
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx_o,
                                nsel_o, w.chunk, scale_for(w.D))
    err = np.abs(out.cpu().double().numpy() - want).max()
    assert err <= ATOL, err


def test_sparse_edge_cases(cuda_lib):
    w = small_workload(B=2, ragged=False, L=200, budget=64)
    c = make_case(w)
    kc = w.kc
    idx_o = np.full((2, w.Hkv, kc), -1, dtype=np.int64)
    nsel_o = np.zeros((2, w.Hkv), dtype=np.int64)
    idx_o[0, 0, :3] = [24, 0, 5]  # L=200: chunks 0..24; any order is accepted
    nsel_o[0, 0] = 3
    idx_o[0, 1, :4] = [1, 999, -5, 2]  # invalid ids are skipped
    nsel_o[0, 1] = 4
    idx_o[1, 0, :kc] = np.arange(kc)  # full list
    nsel_o[1, 0] = kc
    nsel_o[1, 1] = 0  # empty set -> zeros
    out = cuda_lib.tf_sparse_decode_attn(c["q"], c["K"], c["V"], c["seq"],
                                         torch.from_numpy(idx_o.astype(np.int32)).cuda(),
                                         torch.from_numpy(nsel_o.astype(np.int32)).cuda(), 0.05)
    want = O.sparse_decode_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), idx_o,
                                nsel_o, 8, 0.05)
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


# ------------------------------------------------------------------ a6


@pytest.mark.parametrize("w", [synth.TINY, small_workload(), small_workload(L=150, L_min=1)],
                         ids=["tiny", "ragged-gqa", "short-contexts"])
def test_stream_window_attn(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan"))
    out = cuda_lib.tf_stream_window_attn(c["q"], c["K"], c["V"], c["seq"], w.n_sink, w.window, scale_for(w.D))
    want = O.stream_window_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(),
                                w.n_sink, w.window, scale_for(w.D))
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


# ------------------------------------------------------------------ a7


@pytest.mark.parametrize("w", [synth.TINY, small_workload(), small_workload(Hkv=8, T=6, L=3000, L_min=2000),
                               small_workload(T=5), small_workload(Hq=8, Hkv=4, T=5),
                               small_workload(B=1, Hq=16, Hkv=2, T=4, L=900, ragged=False),
                               small_workload(B=2, Hq=8, Hkv=2, T=16, L=700, L_min=100),
                               small_workload(T=5, L=40000, L_min=30000),
                               small_workload(B=2, Hq=16, Hkv=2, T=5, L=40000, L_min=30000),
                               small_workload(B=2, Hq=16, Hkv=2, T=4, L=40000, L_min=30000)],
                         ids=["tiny", "gqa-two-launches", "mha-6", "gqa-t5-padding-rows", "g2-t5-padding-rows",
                              "own-group-two-launches",
                              "three-groups-two-launches", "split", "window-warpgroup-split",
                              "own-group-two-launches-split"])
def test_verify_window_attn(cuda_lib, w):
    """Both outputs against the two oracle calls: window rows after the G*T
    verify rows in one launch (G*(T+1) rows fit the verify row groups), and the
    two-launch path where they would need a group of their own."""
    c = make_case(w, fill_invalid=float("nan") if w.ragged else None)
    ws = cuda_lib.workspace(cuda_lib.tf_verify_window_attn_workspace(w.B, w.Hq, w.Hkv, w.L, w.T, w.n_sink, w.window), "cuda")
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), scale_for(w.D))
    wwant = O.stream_window_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), w.n_sink,
                                 w.window, scale_for(w.D))
    for _ in range(2):  # a second call on the same workspace
        out, wout = cuda_lib.tf_verify_window_attn(c["Q"], c["q"], c["K"], c["V"], c["seq"], w.n_sink, w.window,
                                                   scale_for(w.D), ws=ws)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).item()) == 0, "pipeline status word set"
        assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
        assert np.abs(wout.cpu().double().numpy() - wwant).max() <= ATOL


def test_verify_window_attn_short_contexts(cuda_lib):
    """Contexts shorter than the candidates, than the sinks and the window, and
    empty: both outputs follow their oracle position sets."""
    w = small_workload(B=4, Hq=8, Hkv=2, T=6, L=700, ragged=False)
    c = make_case(w)
    seq = np.array([3, 0, 50, 700], dtype=np.int32)
    c["seq"] = torch.from_numpy(seq).cuda()
    out, wout = cuda_lib.tf_verify_window_attn(c["Q"], c["q"], c["K"], c["V"], c["seq"], w.n_sink, w.window, 0.1)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, 0.1)
    wwant = O.stream_window_attn(bits(c["q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, w.n_sink, w.window, 0.1)
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL
    assert np.abs(wout.cpu().double().numpy() - wwant).max() <= ATOL
    assert np.all(wout.cpu().numpy()[1] == 0)


@pytest.mark.parametrize("G,T", [(1, 1), (2, 3), (1, 16), (2, 5), (3, 7), (4, 6), (2, 16), (8, 4), (4, 9)],
                         ids=lambda v: str(v))
def test_verify_row_groups(cuda_lib, G, T):
    """Query-row groups: the rows of a KV head rounded up to 8, 16, 24 or 32 (full
    and partly filled), and more than 32 rows split into several groups."""
    w = small_workload(B=1, Hq=2 * G, Hkv=2, T=T, L=700, ragged=False)
    c = make_case(w)
    out = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], 0.09)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), 0.09)
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


@pytest.mark.parametrize("lens", [[900, 3000, 0, 3000, 17, 2500, 900], [5 + 37 * i for i in range(65)]],
                         ids=["ties-and-empty", "65-sequences"])
def test_verify_ragged_batch_order(cuda_lib, lens):
    """Ragged batches run their longest sequences first (block row r takes the
    r-th longest context, ties in batch order, up to 64 sequences; larger
    batches keep the batch order): every sequence's rows still land in its own
    output slots, with equal, empty and tiny contexts in the mix."""
    L = max(lens)
    w = small_workload(B=len(lens), Hq=8, Hkv=2, T=6, L=L, ragged=False)
    c = make_case(w)
    seq = np.array(lens, dtype=np.int32)
    c["seq"] = torch.from_numpy(seq).cuda()
    for t in ("K", "V"):  # rows past each context hold NaN
        x = c[t + "_cpu"].clone()
        for b, n in enumerate(lens):
            x[b, :, n:] = float("nan")
        c[t + "_cpu"], c[t] = x, x.cuda()
    out = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], 0.09)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), seq, 0.09)
    got = out.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    assert np.abs(got - want).max() <= ATOL


def test_verify_context_shorter_than_candidates(cuda_lib):
    w = small_workload(B=2, ragged=False, L=16, T=6)
    c = make_case(w)
    c["seq"] = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    out = cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], 0.1)
    want = O.verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), np.array([3, 0]), 0.1)
    got = out.cpu().double().numpy()
    assert np.all(got[1] == 0) and np.all(got[0, :, :3] == 0)
    assert np.abs(got - want).max() <= ATOL


# ------------------------------------------------------------------ a8


def run_accept(cuda_lib, tgt, drf, x, ua, ur, temperature=1.0):
    n_acc, nxt, out = cuda_lib.tf_spec_accept(tgt.cuda(), drf.cuda(), x.cuda(), ua.cuda(), ur.cuda(), temperature)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), nxt.cpu().numpy(), out.cpu().numpy()


def compare_accept(got, want):
    n_acc, nxt, out = got
    same = (n_acc == want["n_acc"]) & (nxt == want["next"]) & np.all(out == want["out_tokens"], axis=1)
    bad = ~same
    assert np.all(want["margin"][bad] < EDGE), f"{bad.sum()} mismatches not explained by boundary draws"
    return int(bad.sum())


@pytest.mark.parametrize("B,gamma,V,temp", [(1, 4, 32000, 1.0), (64, 4, 32000, 1.0), (256, 5, 1000, 0.7),
                                            (512, 3, 7, 1.3)])
def test_spec_accept_parity(cuda_lib, B, gamma, V, temp):
    tgt, drf, x, ua, ur = synth.accept_inputs(B, gamma, V, seed=B + V)
    got = run_accept(cuda_lib, tgt, drf, x, ua, ur, temp)
    want = O.spec_accept(tgt.double().numpy(), drf.double().numpy(), x.numpy(), ua.double().numpy(),
                         ur.double().numpy(), temp)
    compare_accept(got, want)


def test_spec_accept_short_and_empty_drafts(cuda_lib):
    tgt, drf, x, ua, ur = synth.accept_inputs(32, 4, 500, seed=77)
    x[0:8, 2] = -1  # drafts of length 2
    x[8:16, 0] = -1  # empty drafts
    x[16:24, 3] = 500  # out-of-range token ends the draft
    got = run_accept(cuda_lib, tgt, drf, x, ua, ur)
    want = O.spec_accept(tgt.double().numpy(), drf.double().numpy(), x.numpy(), ua.double().numpy(),
                         ur.double().numpy())
    compare_accept(got, want)


@pytest.mark.parametrize("gamma,V", [(33, 500), (70, 2048)])
def test_spec_accept_long_drafts(cuda_lib, gamma, V):
    """Drafts longer than one warp of tests: a close drafter keeps most tokens,
    so acceptance runs past position 32; some drafts also end early."""
    tgt, drf, x, ua, ur = synth.accept_inputs(96, gamma, V, seed=gamma + V, drf_noise=0.02)
    x[0:8, 40 % gamma] = -1
    got = run_accept(cuda_lib, tgt, drf, x, ua, ur)
    want = O.spec_accept(tgt.double().numpy(), drf.double().numpy(), x.numpy(), ua.double().numpy(),
                         ur.double().numpy())
    assert np.any(want["n_acc"] > 32)
    compare_accept(got, want)


def test_spec_accept_identical_distributions(cuda_lib):
    tgt, drf, x, ua, ur = synth.accept_inputs(128, 4, 300, seed=5)
    drf = tgt[:, :4].clone()
    got = run_accept(cuda_lib, tgt, drf, x, ua, ur)
    assert np.all(got[0] == 4)


def _chi2_ok(tokens, p):
    from scipy import stats
    counts = np.bincount(tokens, minlength=len(p))
    return stats.chisquare(counts, p * counts.sum()).pvalue > 1e-3


def test_spec_accept_lossless_chi_square_gpu(cuda_lib):
    """10^6 independent sequences in one call: the first emitted token follows p0,
    for one level and for the two-level r -> q -> p composition."""
    N, V, g1 = 1_000_000, 16, 4
    d = synth.two_level_inputs(1, g1, V, seed=99)
    gen = synth.generator(1234, "cuda")
    p, q, r = d["p"].cuda(), d["q"].cuda(), d["r"].cuda()
    pN, qN, rN = p.expand(N, -1, -1).contiguous(), q.expand(N, -1, -1).contiguous(), r.expand(N, -1, -1).contiguous()
    x = synth.sample_tokens(rN, gen)
    u1 = torch.rand((N, g1), generator=gen, device="cuda")
    ur1 = torch.rand((N,), generator=gen, device="cuda")
    n1, nx1, y = cuda_lib.tf_spec_accept(qN[:, : g1 + 1].contiguous(), rN, x, u1, ur1)
    u2 = torch.rand((N, g1 + 1), generator=gen, device="cuda")
    ur2 = torch.rand((N,), generator=gen, device="cuda")
    n2, nx2, z = cuda_lib.tf_spec_accept(pN, qN, y, u2, ur2)
    torch.cuda.synchronize()
    q0 = torch.softmax(q[0, 0].double(), -1).cpu().numpy()
    p0 = torch.softmax(p[0, 0].double(), -1).cpu().numpy()
    assert _chi2_ok(y[:, 0].cpu().numpy(), q0)
    assert _chi2_ok(z[:, 0].cpu().numpy(), p0)


# ------------------------------------------------------------------ candidate trees


def random_tree(B, T, seed):
    rng = np.random.default_rng(seed)
    return np.array([[int(rng.integers(-1, j)) if j > 0 else -1 for j in range(T)] for _ in range(B)], np.int32)


@pytest.mark.parametrize("w", [small_workload(), small_workload(Hkv=8, T=6, L=3000, L_min=2000),
                               small_workload(B=1, Hq=16, Hkv=2, T=9, L=900, ragged=False),
                               small_workload(B=2, Hq=8, Hkv=2, T=16, L=1300, L_min=600)],
                         ids=["ragged-gqa", "mha-6", "row-groups-72", "t16"])
def test_verify_tree(cuda_lib, w):
    c = make_case(w, fill_invalid=float("nan") if w.ragged else None)
    parent = random_tree(w.B, w.T, seed=w.T)
    out = cuda_lib.tf_verify_attn_tree(c["Q"], c["K"], c["V"], c["seq"], torch.from_numpy(parent).cuda(),
                                       scale_for(w.D))
    want = O.tree_verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]), c["seq_cpu"].numpy(), parent,
                              scale_for(w.D))
    assert np.abs(out.cpu().double().numpy() - want).max() <= ATOL


def test_verify_tree_special_shapes(cuda_lib):
    w = small_workload(L=1200, T=6, ragged=False)
    c = make_case(w)
    sc = scale_for(w.D)
    want_of = lambda parent: O.tree_verify_attn(bits(c["Q_cpu"]), bits(c["K_cpu"]), bits(c["V_cpu"]),  # noqa: E731
                                                c["seq_cpu"].numpy(), parent, sc)
    run = lambda parent: cuda_lib.tf_verify_attn_tree(c["Q"], c["K"], c["V"], c["seq"],  # noqa: E731
                                                      torch.from_numpy(parent).cuda(), sc)
    # the chain is tf_verify_attn, to the bit
    chain = np.tile(np.arange(w.T, dtype=np.int32) - 1, (w.B, 1))
    assert torch.equal(run(chain), cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq"], sc))
    # a star: every candidate extends the prefix
    star = np.full((w.B, w.T), -1, np.int32)
    assert np.abs(run(star).cpu().double().numpy() - want_of(star)).max() <= ATOL
    # links to itself, to later candidates or below -1 end the walk
    bad = np.array([[-1, 3, 1, -7, 2, 5], [0, 0, 1, 9, 3, 4]], np.int32)
    assert np.abs(run(bad).cpu().double().numpy() - want_of(bad)).max() <= ATOL
    # contexts shorter than the candidates (L = 5 < T for the shortest sequence)
    c["seq"] = torch.tensor([5, 1200], dtype=torch.int32, device="cuda")
    c["seq_cpu"] = torch.tensor([5, 1200], dtype=torch.int32)
    tree = random_tree(w.B, w.T, seed=1)
    assert np.abs(run(tree).cpu().double().numpy() - want_of(tree)).max() <= ATOL


@pytest.mark.parametrize("w", [small_workload(), small_workload(Hkv=8, T=6, L=3000, L_min=2000)],
                         ids=["gqa-two-launches", "mha-one-launch"])
def test_verify_window_attn_in_cuda_graph(cuda_lib, w):
    """Captured once and replayed, the call (one launch, or the window launch
    and the verify launch on one workspace) gives the eager call's outputs bit
    for bit."""
    c = make_case(w)
    ws = cuda_lib.workspace(cuda_lib.tf_verify_window_attn_workspace(w.B, w.Hq, w.Hkv, w.L, w.T, w.n_sink, w.window),
                            "cuda")
    out, wout = cuda_lib.tf_verify_window_attn(c["Q"], c["q"], c["K"], c["V"], c["seq"], w.n_sink, w.window, 0.1, ws=ws)
    g_out, g_wout = torch.empty_like(out), torch.empty_like(wout)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.tf_verify_window_attn(c["Q"], c["q"], c["K"], c["V"], c["seq"], w.n_sink, w.window, 0.1, out=g_out,
                                       wout=g_wout, ws=ws)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(g_out, out) and torch.equal(g_wout, wout)
    assert cuda_lib.tf_check_status(ws) == 0
