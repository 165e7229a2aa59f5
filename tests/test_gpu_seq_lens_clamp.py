"""Sequence lengths outside [0, Lmax] are clamped by every call, as the oracle's
valid_len states the contract: a length above Lmax reads the whole cache, a
negative length reads nothing.

The cache is generated with the clamped lengths (NaN past each of them); every
call then receives the raw lengths and is compared with the oracle given the
same raw lengths (the oracle clamps them; tests/test_oracle_clamp.py pins that
against the clamped call itself).
"""

import numpy as np
import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth
from oracle import triforce as O
from test_gpu_parity import ATOL, bits, check_topk, scale_for

pytestmark = pytest.mark.gpu

LMAX = 700  # not a multiple of the chunk: the last chunk is partial


def clamp_case(Hq, Hkv, T):
    raw = np.array([LMAX + 37, -5, 333, 2 ** 30], dtype=np.int32)
    clamped = np.clip(raw, 0, LMAX).astype(np.int32)
    w = synth.Workload("clamp", len(raw), Hq, Hkv, 128, LMAX, 1, 8, 256, 4, 60, T, 4, 100, 0.02, 51)
    seq_cl = torch.from_numpy(clamped)
    q, Q = synth.decode_queries(w, 0)
    K, V, _ = synth.kv_cache(w, 0, q, seq_cl, fill_invalid=float("nan"))
    d = "cuda"
    return dict(w=w, raw=raw, seq_raw=torch.from_numpy(raw).to(d), q_cpu=q, Q_cpu=Q, K_cpu=K, V_cpu=V,
                q=q.to(d), Q=Q.to(d), K=K.to(d), V=V.to(d))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2)], ids=["mha", "gqa4"])
def test_every_call_clamps_seq_lens(cuda_lib, Hq, Hkv):
    c = clamp_case(Hq, Hkv, T=5)
    w, raw, s = c["w"], c["raw"], scale_for(128)
    Kb, Vb, qb, Qb = bits(c["K_cpu"]), bits(c["V_cpu"]), bits(c["q_cpu"]), bits(c["Q_cpu"])
    Cmax = -(-LMAX // 8)

    # a1: chunk means
    M = torch.full((w.B, Hkv, Cmax, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.tf_build_chunk_means(c["K"], c["seq_raw"], M)
    M_o = O.build_chunk_means(Kb, raw, 8)
    assert np.array_equal(bits(M), M_o)

    # a2 + a3: scores and top-k
    idx_o, nsel_o, _, gap_o, scores_o = O.chunk_scores_topk(qb, M_o, raw, LMAX, 8, w.kc, Hkv)
    idx, nsel = cuda_lib.tf_chunk_scores_topk(c["q"], M, c["seq_raw"], LMAX, w.kc)
    torch.cuda.synchronize()
    check_topk(idx.cpu().numpy(), nsel.cpu().numpy(), idx_o, nsel_o, gap_o, scores_o)
    idx_np, nsel_np = idx.cpu().numpy(), nsel.cpu().numpy()

    def close(got, want, name):
        g = got.cpu().double().numpy()
        assert np.isfinite(g).all(), name
        err = float(np.abs(g - want).max())
        assert err <= ATOL, (name, err)

    # a4: sparse decode attention over the selection
    close(cuda_lib.tf_sparse_decode_attn(c["q"], c["K"], c["V"], c["seq_raw"], idx, nsel, s),
          O.sparse_decode_attn(qb, Kb, Vb, raw, idx_np, nsel_np, 8, s), "sparse")
    # a2 + a3 + a4 fused
    f_idx, f_nsel, f_out = cuda_lib.tf_retrieval_draft_attn(c["q"], M, c["K"], c["V"], c["seq_raw"], w.kc, s)
    torch.cuda.synchronize()
    assert np.array_equal(f_idx.cpu().numpy(), idx_np) and np.array_equal(f_nsel.cpu().numpy(), nsel_np)
    close(f_out, O.sparse_decode_attn(qb, Kb, Vb, raw, idx_np, nsel_np, 8, s), "fused draft")
    # a6: sinks + window
    close(cuda_lib.tf_stream_window_attn(c["q"], c["K"], c["V"], c["seq_raw"], 4, 60, s),
          O.stream_window_attn(qb, Kb, Vb, raw, 4, 60, s), "window")
    # a7: verify, its tree form, its offloaded form
    ver_o = O.verify_attn(Qb, Kb, Vb, raw, s)
    close(cuda_lib.tf_verify_attn(c["Q"], c["K"], c["V"], c["seq_raw"], s), ver_o, "verify")
    parent = np.tile(np.array([-1, 0, 0, 1, 2], dtype=np.int32), (w.B, 1))
    close(cuda_lib.tf_verify_attn_tree(c["Q"], c["K"], c["V"], c["seq_raw"], torch.from_numpy(parent).cuda(), s),
          O.tree_verify_attn(Qb, Kb, Vb, raw, parent, s), "tree verify")
    off = cuda_lib.tf_verify_attn_offload(c["Q"], c["K_cpu"].contiguous().pin_memory(),
                                          c["V_cpu"].contiguous().pin_memory(), c["seq_raw"], LMAX, s,
                                          seg_rows=256, copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    close(off, ver_o, "offloaded verify")
    # level-1 verify over the selection
    close(cuda_lib.tf_sparse_verify_attn(c["Q"], c["K"], c["V"], c["seq_raw"], idx, nsel, s),
          O.sparse_verify_attn(Qb, Kb, Vb, raw, idx_np, nsel_np, 8, s), "sparse verify")
    # resident retrieval cache
    Kc, Vc, lens, _ = cuda_lib.tf_pack_retrieval_cache(c["K"], c["V"], c["seq_raw"], idx, nsel)
    torch.cuda.synchronize()
    oK, oV, olens = O.compact_retrieval_cache(Kb, Vb, raw, idx_np, nsel_np, 8, w.kc)
    assert np.array_equal(lens.cpu().numpy().reshape(w.B, Hkv), olens)
    gK, gV = bits(Kc), bits(Vc)
    for b in range(w.B):
        for g in range(Hkv):
            n = int(olens[b, g])
            assert np.array_equal(gK[b, g, :n], oK[b, g, :n]) and np.array_equal(gV[b, g, :n], oV[b, g, :n])
