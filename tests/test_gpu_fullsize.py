"""Parity at the full workload sizes, one layer each, sampled (sequence, KV head)
units checked one by one against the float64 oracle.

Same launch configuration as the benchmark: the whole layer (every unit) goes
through each call; the oracle recomputes a few units, always including the
first and last KV head and, for ragged batches, the longest and the shortest
sequence.  The offloaded verify streams the same cache from pinned host
memory in the benchmark's 16K-position segments; the window + verify call runs as
the benchmark's step runs it.  Tolerances as in test_gpu_parity.py.
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O

pytestmark = pytest.mark.gpu

ATOL = 2e-3
GAP = 1e-4


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def layer_on_gpu(w, layer=0):
    seq_cpu = synth.seq_lens_for(w)
    q, Q = synth.decode_queries(w, layer, device="cuda")
    K, V, planted = synth.kv_cache(w, layer, q, seq_cpu, device="cuda")
    return seq_cpu, q, Q, K, V, planted


def sample_units(w, seq_cpu):
    bs = {0, w.B - 1, int(torch.argmax(seq_cpu)), int(torch.argmin(seq_cpu))}
    gs = {0, w.Hkv - 1}
    return sorted((b, g) for b in bs for g in gs)


@pytest.mark.parametrize("w", [synth.LLAMA2_7B_128K, synth.LLAMA3_8B_GQA_128K, synth.MIXED_BATCH],
                         ids=lambda w: w.name)
def test_full_size_layer(cuda_lib, w):
    seq_cpu, q, Q, K, V, planted = layer_on_gpu(w)
    seq = seq_cpu.cuda()
    Cmax = -(-w.L // w.chunk)
    scale = w.D ** -0.5
    M = torch.empty((w.B, w.Hkv, Cmax, w.D), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(K, seq, M)
    idx, nsel = cuda_lib.tf_chunk_scores_topk(q, M, seq, w.L, w.kc)
    sp = cuda_lib.tf_sparse_decode_attn(q, K, V, seq, idx, nsel, scale)
    wi = cuda_lib.tf_stream_window_attn(q, K, V, seq, w.n_sink, w.window, scale)
    ve = cuda_lib.tf_verify_attn(Q, K, V, seq, scale)
    vw_v, vw_w = cuda_lib.tf_verify_window_attn(Q, q, K, V, seq, w.n_sink, w.window, scale)  # as the bench step
    fidx, fnsel, fsp = cuda_lib.tf_retrieval_draft_attn(q, M, K, V, seq, w.kc, scale)
    # the benchmark's bound: 0.7 x the cut of another seeded query set
    q_other, _ = synth.decode_queries(w, 1000, device="cuda")
    cut_other = torch.empty((w.B, w.Hkv), dtype=torch.float32, device="cuda")
    cuda_lib.tf_retrieval_draft_attn(q_other, M, K, V, seq, w.kc, scale, s_cut=cut_other)
    hidx, hnsel, hsp = cuda_lib.tf_retrieval_draft_attn(q, M, K, V, seq, w.kc, scale, cut_hint=cut_other * 0.7)
    # two to four heads per KV head: the step's draft carries the window rows (tf_retrieval_window_draft_attn)
    in_draft = 2 <= w.G <= 4
    if in_draft:
        widx, wnsel, wsp, wwi = cuda_lib.tf_retrieval_window_draft_attn(q, M, K, V, seq, w.kc, scale, w.n_sink,
                                                                        w.window, cut_hint=cut_other * 0.7)
    sv = cuda_lib.tf_sparse_verify_attn(Q, K, V, seq, idx, nsel, scale)
    # offloaded verify as timed: pinned host K/V, 16K-position segments, copies on a side stream
    K_host = torch.empty(K.shape, dtype=K.dtype, pin_memory=True).copy_(K)
    V_host = torch.empty(V.shape, dtype=V.dtype, pin_memory=True).copy_(V)
    off = cuda_lib.tf_verify_attn_offload(Q, K_host, V_host, seq, int(seq_cpu.max()), scale,
                                          seg_rows=min(16384, w.L), copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    del K_host, V_host
    # every unit of the offloaded verify against the resident one (both oracle-checked on the samples)
    assert (off - ve).abs().max().item() <= ATOL
    # the fused retrieval drafter selects exactly what the top-k call selects
    assert np.array_equal(fidx.cpu().numpy(), idx.cpu().numpy())
    assert np.array_equal(fnsel.cpu().numpy(), nsel.cpu().numpy())
    # ... with or without the bound
    assert np.array_equal(hidx.cpu().numpy(), idx.cpu().numpy())
    assert np.array_equal(hnsel.cpu().numpy(), nsel.cpu().numpy())
    if in_draft:
        assert np.array_equal(widx.cpu().numpy(), idx.cpu().numpy())
        assert np.array_equal(wnsel.cpu().numpy(), nsel.cpu().numpy())
        wsp_h, wwi_h = wsp.cpu().double().numpy(), wwi.cpu().double().numpy()
    hsp_h = hsp.cpu().double().numpy()
    fsp_h = fsp.cpu().double().numpy()
    M_h, idx_h, nsel_h = bits(M), idx.cpu().numpy(), nsel.cpu().numpy()
    sp_h, wi_h, ve_h = sp.cpu().double().numpy(), wi.cpu().double().numpy(), ve.cpu().double().numpy()
    sv_h, off_h = sv.cpu().double().numpy(), off.cpu().double().numpy()
    vwv_h, vww_h = vw_v.cpu().double().numpy(), vw_w.cpu().double().numpy()
    q_h, Q_h = bits(q), bits(Q)
    G = w.G
    near_ties = 0
    for b, g in sample_units(w, seq_cpu):
        L = int(seq_cpu[b])
        Kb, Vb = bits(K[b : b + 1, g : g + 1]), bits(V[b : b + 1, g : g + 1])
        sl = np.array([L])
        # a1: bit-exact chunk means of this unit
        M_o = O.build_chunk_means(Kb, sl, w.chunk)
        assert np.array_equal(M_h[b, g][: -(-L // 8)], M_o[0, 0][: -(-L // 8)])
        # a2 + a3: same top-k set unless the oracle's cut gap is below 1e-4
        qg = q_h[b : b + 1, g * G : (g + 1) * G]
        idx_o, nsel_o, _, gap_o, scores_o = O.chunk_scores_topk(qg, M_o, sl, w.L, w.chunk, w.kc, 1)
        assert nsel_h[b, g] == nsel_o[0, 0]
        got = idx_h[b, g, : nsel_h[b, g]]
        if not np.array_equal(got, idx_o[0, 0, : nsel_o[0, 0]]):
            assert gap_o[0, 0] < GAP
            near_ties += 1
        assert set(planted[b][g].tolist()) <= set(got.tolist())
        # a4 on the GPU's own selection (the attention is checked, not the selection again)
        sp_o = O.sparse_decode_attn(qg, Kb, Vb, sl, idx_h[b : b + 1, g : g + 1], nsel_h[b : b + 1, g : g + 1],
                                    w.chunk, scale)
        assert np.abs(sp_h[b, g * G : (g + 1) * G] - sp_o[0]).max() <= ATOL
        assert np.abs(fsp_h[b, g * G : (g + 1) * G] - sp_o[0]).max() <= ATOL
        assert np.abs(hsp_h[b, g * G : (g + 1) * G] - sp_o[0]).max() <= ATOL
        if in_draft:
            assert np.abs(wsp_h[b, g * G : (g + 1) * G] - sp_o[0]).max() <= ATOL
        # a6
        wi_o = O.stream_window_attn(qg, Kb, Vb, sl, w.n_sink, w.window, scale)
        assert np.abs(wi_h[b, g * G : (g + 1) * G] - wi_o[0]).max() <= ATOL
        assert np.abs(vww_h[b, g * G : (g + 1) * G] - wi_o[0]).max() <= ATOL
        if in_draft:
            assert np.abs(wwi_h[b, g * G : (g + 1) * G] - wi_o[0]).max() <= ATOL
        # a7
        ve_o = O.verify_attn(Q_h[b : b + 1, g * G : (g + 1) * G], Kb, Vb, sl, scale)
        assert np.abs(ve_h[b, g * G : (g + 1) * G] - ve_o[0]).max() <= ATOL
        assert np.abs(off_h[b, g * G : (g + 1) * G] - ve_o[0]).max() <= ATOL
        assert np.abs(vwv_h[b, g * G : (g + 1) * G] - ve_o[0]).max() <= ATOL
        # level-1 verify over the GPU's own selection
        sv_o = O.sparse_verify_attn(Q_h[b : b + 1, g * G : (g + 1) * G], Kb, Vb, sl,
                                    idx_h[b : b + 1, g : g + 1], nsel_h[b : b + 1, g : g + 1], w.chunk, scale)
        assert np.abs(sv_h[b, g * G : (g + 1) * G] - sv_o[0]).max() <= ATOL
    assert near_ties <= 1


def test_two_level_accept_full_vocab(cuda_lib):
    """Mixed-batch workload: tiny drafter -> retrieval drafter -> target over
    vocab 32000, batch 8, seeded uniforms; both levels against the oracle."""
    B, g1, V = 8, 4, 32000
    d = synth.two_level_inputs(B, g1, V, seed=4)
    p, q, r, x = d["p"], d["q"], d["r"], d["x"]
    n1, nx1, y = cuda_lib.tf_spec_accept(q[:, : g1 + 1].contiguous().cuda(), r.cuda(), x.cuda(), d["u1"].cuda(),
                                         d["ur1"].cuda())
    n2, nx2, z = cuda_lib.tf_spec_accept(p.cuda(), q.cuda(), y, d["u2"].cuda(), d["ur2"].cuda())
    torch.cuda.synchronize()
    o1 = O.spec_accept(q[:, : g1 + 1].double().numpy(), r.double().numpy(), x.numpy(), d["u1"].double().numpy(),
                       d["ur1"].double().numpy())
    same1 = np.all(y.cpu().numpy() == o1["out_tokens"], axis=1)
    assert np.all(same1 | (o1["margin"] < 1e-6))
    # level 2 consumes the oracle's own level-1 output on the oracle side
    o2 = O.spec_accept(p.double().numpy(), q.double().numpy(), o1["out_tokens"], d["u2"].double().numpy(),
                       d["ur2"].double().numpy())
    same2 = np.all(z.cpu().numpy() == o2["out_tokens"], axis=1) | ~same1
    assert np.all(same2 | (o2["margin"] < 1e-6))
