"""The binding refuses buffers whose shapes disagree with the sizes it passes
to the library (which reads and writes whole buffers from those sizes and
cannot see the tensors): a ValueError before anything is launched, and the
destination buffers are left untouched."""

import pytest
import torch

from hierarchical_speculative_decoding_gb300 import synth

pytestmark = pytest.mark.gpu


def _case():
    w = synth.Workload("shapes", 2, 8, 2, 128, 256, 1, 8, 64, 4, 60, 6, 4, 1000, 0.02, 5, False, 0)
    seq = synth.seq_lens_for(w).cuda()
    q, Q = synth.decode_queries(w, 0, device="cuda")
    K, V, _ = synth.kv_cache(w, 0, q, synth.seq_lens_for(w), device="cuda")
    M = torch.empty((w.B, w.Hkv, w.L // 8, w.D), dtype=torch.bfloat16, device="cuda")
    return w, seq, q, Q, K, V, M


def test_attention_calls_refuse_mismatched_shapes(cuda_lib):
    tf = cuda_lib
    w, seq, q, Q, K, V, M = _case()
    short_v = V[:, :, : w.L // 2].contiguous()
    with pytest.raises(ValueError, match="V must be"):
        tf.tf_verify_attn(Q, K, short_v, seq, 0.1)
    sentinel = torch.full((w.B, w.Hq, w.T - 1, w.D), 7.0, device="cuda")
    with pytest.raises(ValueError, match="out must be"):
        tf.tf_verify_attn(Q, K, V, seq, 0.1, out=sentinel)
    assert bool((sentinel == 7.0).all())
    with pytest.raises(ValueError, match="seq_lens must be"):
        tf.tf_stream_window_attn(q, K, V, seq[:1].contiguous(), 4, 60, 0.1)
    with pytest.raises(ValueError, match="wout must be"):
        tf.tf_verify_window_attn(Q, q, K, V, seq, 4, 60, 0.1,
                                 wout=torch.empty((w.B, w.Hq - 1, w.D), device="cuda"))
    with pytest.raises(ValueError, match="M must be"):
        tf.tf_retrieval_draft_attn(q, M[:, :, :-1].contiguous(), K, V, seq, 8, 0.1)
    with pytest.raises(ValueError, match="M must be"):
        tf.tf_chunk_scores_topk(q, M[:, :, :-1].contiguous(), seq, w.L, 8)
    out_sentinel = torch.full((w.B, w.Hq, w.D), 7.0, device="cuda")
    with pytest.raises(ValueError, match="wout must be"):
        tf.tf_retrieval_window_draft_attn(q, M, K, V, seq, 8, 0.1, w.n_sink, w.window, out=out_sentinel,
                                          wout=torch.empty((w.B, w.Hq - 1, w.D), device="cuda"))
    with pytest.raises(ValueError, match="cut_hint must be"):
        tf.tf_retrieval_window_draft_attn(q, M, K, V, seq, 8, 0.1, w.n_sink, w.window, out=out_sentinel,
                                          cut_hint=torch.zeros((w.B, w.Hkv + 1), device="cuda"))
    assert bool((out_sentinel == 7.0).all())
    idx = torch.zeros((w.B, w.Hkv, 8), dtype=torch.int32, device="cuda")
    n_sel = torch.zeros((w.B, w.Hkv), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="n_sel must be"):
        tf.tf_sparse_decode_attn(q, K, V, seq, idx, n_sel[:1].contiguous(), 0.1)
    with pytest.raises(ValueError, match="K must be"):
        tf.tf_sparse_verify_attn(Q, K[:1].contiguous(), V[:1].contiguous(), seq, idx, n_sel, 0.1)
    torch.cuda.synchronize()


def test_accept_calls_refuse_mismatched_shapes(cuda_lib):
    tf = cuda_lib
    B, gamma, Vn = 2, 3, 50
    tgt = torch.zeros((B, gamma + 1, Vn), device="cuda")
    drf = torch.zeros((B, gamma, Vn), device="cuda")
    toks = torch.zeros((B, gamma), dtype=torch.int32, device="cuda")
    u_acc = torch.zeros((B, gamma), device="cuda")
    u_res = torch.zeros((B,), device="cuda")
    with pytest.raises(ValueError, match="u_res must be"):
        tf.tf_spec_accept(tgt, drf, toks, u_acc, u_res[:1].contiguous())
    with pytest.raises(ValueError, match="out_tokens must be"):
        tf.tf_spec_accept(tgt, drf, toks, u_acc, u_res,
                          out_tokens=torch.empty((B, gamma), dtype=torch.int32, device="cuda"))
    parent = torch.full((B, gamma), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="acc_nodes must be"):
        tf.tf_spec_accept_tree(tgt, drf, toks, parent, u_acc, u_res,
                               acc_nodes=torch.empty((B, gamma + 1), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
